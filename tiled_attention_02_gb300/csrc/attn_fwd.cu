// attn_fwd.cu -- tiled exact-attention forward for GB300 (sm_103a).
//
// One CTA computes one 128-row query tile of one (batch, query head):
//
//   for each 128-key tile j (keys <= the tile's last row when causal):
//       S_j  = Q K_j^T                       tcgen05.mma, fp32 in TMEM
//       t    = S_j * scale * log2(e)  [+ bias * log2(e)]   (+ mask: -inf)
//       m'   = max(m, rowmax t);  alpha = 2^(m - m')
//       P_j  = 2^(t - m')  -> bf16, written back into TMEM over S_j
//       l    = alpha l + rowsum P_j (fp32, before rounding P)
//       O    = alpha O   (only when some row's max grew)
//       O   += P_j V_j                       tcgen05.mma, A operand from TMEM
//   O /= l -> bf16; LSE = (m + log2 l) ln 2
//
// This is the online-softmax double loop of kwkr.cn/news/592482, sections
// 2.2-2.3 ("FlashAttention原理与Triton实战" 2.2, 3.3), with the additive
// pre-softmax bias and emitted logits of the block attention residual
// (Block Attention Residual Triton kernel, "v1: Fuse Residual 进 Attention
// Kernel").  exp is evaluated as 2^x with the scale folded in.
//
// Warp roles (192 threads, one CTA per SM):
//   warps 0-3  softmax: thread r owns query row r (TMEM lane r); also the
//              O rescale and the epilogue.
//   warp 4     TMA producer: Q once, then K_j / V_j through 2-3 stage rings.
//   warp 5     TMEM allocator and single-thread tcgen05.mma issuer.
// TMEM (512 columns): S/P double buffer at columns 0 and 128, O at 256.
// Issue order on the tensor core: S_0, S_1, PV_0, S_2, PV_1, ... so that the
// softmax of tile j overlaps the MMAs of tiles j+1 and j-1.
#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace tattn {
namespace {

constexpr int kBlockM = 128;   // query rows per CTA
constexpr int kBlockN = 128;   // keys per tile
constexpr int kThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Lazy-rescale threshold in log2 units: the reference max is only raised when
// a row's max grows by more than this (factor 2^8).
constexpr float kRescaleLog2 = 8.0f;

template <int D>
struct FwdCfg {
    static constexpr int kChunks = D / 64;              // 128-byte swizzle atoms per row
    static constexpr int kChunkBytes = kBlockM * 128;   // one atom column of a tile
    static constexpr int kTileBytes = kBlockM * D * 2;  // bf16 128 x D tile
    static constexpr int kKStages = (D == 64) ? 3 : 2;
    static constexpr int kVStages = (D == 64) ? 3 : 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kTileBytes;
    static constexpr int kOffV = kOffK + kKStages * kTileBytes;
    static constexpr int kOffBar = kOffV + kVStages * kTileBytes;
    // barrier indices
    static constexpr int kBarQFull = 0;
    static constexpr int kBarKFull = 1;
    static constexpr int kBarKEmpty = kBarKFull + kKStages;
    static constexpr int kBarVFull = kBarKEmpty + kKStages;
    static constexpr int kBarVEmpty = kBarVFull + kVStages;
    static constexpr int kBarSFull = kBarVEmpty + kVStages;   // 2
    static constexpr int kBarPFull = kBarSFull + 2;           // 2
    static constexpr int kBarODone = kBarPFull + 2;
    static constexpr int kBarOFinal = kBarODone + 1;
    static constexpr int kBarDrain = kBarOFinal + 1;
    static constexpr int kNumBars = kBarDrain + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;   // tmem slot, abort flag
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;   // + base alignment slack
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColO = 256;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct FwdParams {
    const float *bias;
    float *emit;
    float *lse;
    int *status;
    int N, Hq, Hkv, group, BH, n_qtiles;
    float scale;        // scale of QK^T
    float scale_log2;   // scale * log2(e)
    int vec4;           // bias/emit rows are 16-byte aligned (N % 4 == 0)
};

// Waits for the arrival of in-flight async work on the abort path only,
// ignoring the abort flag, with a short limit of its own.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > 20ull * 1000ull * 1000ull) break;
    }
}

template <int D, bool CAUSAL, bool EXT>
__global__ void __launch_bounds__(kThreads, 1)
fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
           const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
           const FwdParams p) {
    using C = FwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Heaviest causal tiles first: block 0 gets the last query tile.
    const int blk = blockIdx.x;
    const int qt = CAUSAL ? (p.n_qtiles - 1 - blk / p.BH) : (blk / p.BH);
    const int bh = blk % p.BH;
    const int bh_kv = (bh / p.Hq) * p.Hkv + (bh % p.Hq) / p.group;
    const int n_ktiles = (p.N + kBlockN - 1) / kBlockN;
    const int n_kv = CAUSAL ? min(qt + 1, n_ktiles) : n_ktiles;

    auto bar = [&](int i) -> uint32_t { return sb + C::kOffBar + 8u * i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
    const AbortCtl ac{abort_flag, p.status};

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        mbar_init(bar(C::kBarQFull), 1);
        for (int s = 0; s < C::kKStages; ++s) {
            mbar_init(bar(C::kBarKFull + s), 1);
            mbar_init(bar(C::kBarKEmpty + s), 1);
        }
        for (int s = 0; s < C::kVStages; ++s) {
            mbar_init(bar(C::kBarVFull + s), 1);
            mbar_init(bar(C::kBarVEmpty + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(C::kBarSFull + s), 1);
            mbar_init(bar(C::kBarPFull + s), kBlockM);
        }
        mbar_init(bar(C::kBarODone), 1);
        mbar_init(bar(C::kBarOFinal), 1);
        mbar_init(bar(C::kBarDrain), 1);
        fence_barrier_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmO);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 4) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            bool ok = true;
            mbar_arrive_expect_tx(bar(C::kBarQFull), C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_3d(sb + C::kOffQ + c * C::kChunkBytes, &tmQ, bar(C::kBarQFull), c * 64,
                            qt * kBlockM, bh);
            int k_issued = 0, v_issued = 0;
            for (int j = 0; j < n_kv; ++j) {
                const int ks = j % C::kKStages;
                if (j >= C::kKStages)
                    ok = mbar_wait(bar(C::kBarKEmpty + ks), ((j / C::kKStages) - 1) & 1, ac);
                if (!ok) break;
                mbar_arrive_expect_tx(bar(C::kBarKFull + ks), C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(sb + C::kOffK + ks * C::kTileBytes + c * C::kChunkBytes, &tmK,
                                bar(C::kBarKFull + ks), c * 64, j * kBlockN, bh_kv);
                k_issued = j + 1;
                const int vs = j % C::kVStages;
                if (j >= C::kVStages)
                    ok = mbar_wait(bar(C::kBarVEmpty + vs), ((j / C::kVStages) - 1) & 1, ac);
                if (!ok) break;
                mbar_arrive_expect_tx(bar(C::kBarVFull + vs), C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(sb + C::kOffV + vs * C::kTileBytes + c * C::kChunkBytes, &tmV,
                                bar(C::kBarVFull + vs), c * 64, j * kBlockN, bh_kv);
                v_issued = j + 1;
            }
            if (!ok) {
                // Let every copy already issued land before the CTA exits: the
                // last arm of each stage is the only one not yet consumed.
                drain_wait(bar(C::kBarQFull), 0);
                for (int j = max(k_issued - C::kKStages, 0); j < k_issued; ++j)
                    drain_wait(bar(C::kBarKFull + j % C::kKStages), (j / C::kKStages) & 1);
                for (int j = max(v_issued - C::kVStages, 0); j < v_issued; ++j)
                    drain_wait(bar(C::kBarVFull + j % C::kVStages), (j / C::kVStages) & 1);
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdS = idesc_bf16_f32(kBlockM, kBlockN, false, false);
            constexpr uint32_t kIdPV = idesc_bf16_f32(kBlockM, D, false, true);
            bool ok = mbar_wait(bar(C::kBarQFull), 0, ac);
            tc_fence_after();

            auto issue_pv = [&](int i, bool last) -> bool {
                const int pb = i & 1;
                if (!mbar_wait(bar(C::kBarPFull + pb), (i >> 1) & 1, ac)) return false;
                const int vs = i % C::kVStages;
                if (!mbar_wait(bar(C::kBarVFull + vs), (i / C::kVStages) & 1, ac)) return false;
                tc_fence_after();
                const uint32_t a_tmem = tmem + pb * kBlockN;   // P: bf16 pairs, cols 0..63
                const uint32_t v_base = sb + C::kOffV + vs * C::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk) {
                    const uint64_t bdesc = sdesc_sw128(v_base + kk * 2048, C::kChunkBytes, 1024);
                    mma_ts(tmem + C::kColO, a_tmem + kk * 8, bdesc, kIdPV,
                           (i > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar(C::kBarVEmpty + vs));
                mma_commit(bar(last ? C::kBarOFinal : C::kBarODone));
                return true;
            };

            for (int j = 0; j < n_kv && ok; ++j) {
                const int ks = j % C::kKStages;
                ok = mbar_wait(bar(C::kBarKFull + ks), (j / C::kKStages) & 1, ac);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + (j & 1) * kBlockN;
                const uint32_t k_base = sb + C::kOffK + ks * C::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
                    const uint64_t adesc = sdesc_sw128(sb + C::kOffQ + off, 16, 1024);
                    const uint64_t bdesc = sdesc_sw128(k_base + off, 16, 1024);
                    mma_ss(d_tmem, adesc, bdesc, kIdS, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(C::kBarSFull + (j & 1)));
                mma_commit(bar(C::kBarKEmpty + ks));
                if (j >= 1) ok = issue_pv(j - 1, false);
            }
            if (ok) ok = issue_pv(n_kv - 1, true);
            if (!ok) {
                mma_commit(bar(C::kBarDrain));
                drain_wait(bar(C::kBarDrain), 0);
            }
        }
        __syncwarp();
    } else {
        // ----------------------------------------------- softmax warpgroup
        const int r = threadIdx.x;             // row within the tile == TMEM lane
        const int q_row = qt * kBlockM + r;    // row within the head
        const bool row_valid = q_row < p.N;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        float m_run = -INFINITY;   // running max, log2 units
        float l_run = 0.f;
        bool ok = true;

        for (int j = 0; j < n_kv; ++j) {
            const int sbuf = j & 1;
            ok = mbar_wait_warp(bar(C::kBarSFull + sbuf), (j >> 1) & 1, ac);
            if (!ok) break;
            tc_fence_after();
            const uint32_t tS = tmem + lane_base + sbuf * kBlockN;
            float x[kBlockN];
            {
                uint32_t rr[kBlockN];
                tmem_ld128(tS, rr);
#pragma unroll
                for (int c = 0; c < kBlockN; ++c) x[c] = __uint_as_float(rr[c]);
            }
            const int key0 = j * kBlockN;
            const bool diag = CAUSAL && (j == qt);
            const bool ragged = key0 + kBlockN > p.N;
            // x holds raw q.k when `raw` (scale > 0, no bias): the max commutes
            // with the positive scale and the scale folds into the exp2 FMA.
            // Otherwise x is turned into log2-unit logits t here.
            bool raw = !EXT && p.scale_log2 > 0.f;

            if constexpr (EXT) {
                // Natural-unit logit = scale*qk + bias; emitted before the mask.
                const size_t roff = (static_cast<size_t>(bh) * p.N + q_row) * p.N + key0;
                const float *brow = (p.bias && row_valid) ? p.bias + roff : nullptr;
                float *erow = (p.emit && row_valid) ? p.emit + roff : nullptr;
                if (!diag && !ragged && p.vec4) {
#pragma unroll
                    for (int c = 0; c < kBlockN; c += 4) {
                        float4 bv = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (brow) bv = __ldg(reinterpret_cast<const float4 *>(brow + c));
                        float4 y;
                        y.x = fmaf(x[c + 0], p.scale, bv.x);
                        y.y = fmaf(x[c + 1], p.scale, bv.y);
                        y.z = fmaf(x[c + 2], p.scale, bv.z);
                        y.w = fmaf(x[c + 3], p.scale, bv.w);
                        if (erow) *reinterpret_cast<float4 *>(erow + c) = y;
                        x[c + 0] = y.x * kLog2e;
                        x[c + 1] = y.y * kLog2e;
                        x[c + 2] = y.z * kLog2e;
                        x[c + 3] = y.w * kLog2e;
                    }
                } else {
                    const int lim = diag ? min(r + 1, kBlockN) : kBlockN;
#pragma unroll
                    for (int c = 0; c < kBlockN; ++c) {
                        const bool inside = (c < lim) && (key0 + c < p.N);
                        float bval = 0.f;
                        if (brow && inside) bval = __ldg(brow + c);
                        const float y = fmaf(x[c], p.scale, bval);
                        if (erow && inside) erow[c] = y;
                        x[c] = y * kLog2e;
                    }
                }
            } else {
                if (!raw) {
#pragma unroll
                    for (int c = 0; c < kBlockN; ++c) x[c] *= p.scale_log2;
                }
            }

            if (diag || ragged) {
#pragma unroll
                for (int c = 0; c < kBlockN; ++c) {
                    const bool keep = (!diag || c <= r) && (key0 + c < p.N);
                    x[c] = keep ? x[c] : -INFINITY;
                }
            }
            // Row max as a tree (8 independent chains of 3-input max).
            float mx[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = x[i];
#pragma unroll
            for (int c = 8; c < kBlockN; c += 16) {
#pragma unroll
                for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], x[c + i], x[c + 8 + i]);
            }
            // (c runs 8, 24, ..., 120: elements 8..127 are all covered.)
            const float mt_x = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                     fmaxf(mx[6], mx[7]));
            const float m_tile = raw ? mt_x * p.scale_log2 : mt_x;
            // Lazy rescale: keep the previous reference max while the new row
            // max exceeds it by at most kRescaleLog2 (p stays <= 2^8); O/l and
            // LSE are unchanged by the choice of reference.
            float m_new = fmaxf(m_run, m_tile);
            if (m_new - m_run <= kRescaleLog2) m_new = m_run;
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = ex2(m_run - m_use);   // 0 on the first tile

            const float cmul = raw ? p.scale_log2 : 1.f;
            const uint64_t cm2 = f2pack(cmul, cmul);
            const uint64_t nm2 = f2pack(-m_use, -m_use);
            uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};   // (+0.0f, +0.0f) pairs
            {
                uint32_t pk[kBlockN / 2];
#pragma unroll
                for (int c = 0; c < kBlockN / 2; ++c) {
                    float t0, t1;
                    f2unpack(ffma2(f2pack(x[2 * c], x[2 * c + 1]), cm2, nm2), t0, t1);
                    const float p0 = ex2(t0), p1 = ex2(t1);
                    acc[c & 3] = fadd2(acc[c & 3], f2pack(p0, p1));
                    pk[c] = pack_bf16x2(p0, p1);
                }
                tmem_st64(tS, pk);
            }
            float sum;
            {
                const uint64_t a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
                float u0, u1;
                f2unpack(fadd2(a01, a23), u0, u1);
                sum = u0 + u1;
            }
            l_run = fmaf(l_run, alpha, sum);

            const bool need = (j > 0) && (alpha < 1.f);
            if (__any_sync(0xffffffffu, need)) {
                // O holds PV_0..PV_{j-1}; PV_{j-1} must have landed first.
                ok = mbar_wait_warp(bar(C::kBarODone), (j - 1) & 1, ac);
                if (!ok) break;
                tc_fence_after();
                const uint32_t tO = tmem + lane_base + C::kColO;
                const uint64_t a2 = f2pack(alpha, alpha);
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    uint32_t rr[64];
                    tmem_ld64(tO + c * 64, rr);
#pragma unroll
                    for (int e = 0; e < 64; e += 2) {
                        float o0 = __uint_as_float(rr[e]), o1 = __uint_as_float(rr[e + 1]);
                        f2unpack(fmul2(f2pack(o0, o1), a2), o0, o1);
                        rr[e] = __float_as_uint(o0);
                        rr[e + 1] = __float_as_uint(o1);
                    }
                    tmem_st64(tO + c * 64, rr);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(C::kBarPFull + sbuf));
            m_run = m_new;
        }

        // ------------------------------------------------------- epilogue
        if (ok) ok = mbar_wait_warp(bar(C::kBarOFinal), 0, ac);
        if (ok) {
            tc_fence_after();
            const float inv_l = 1.f / l_run;
            const uint32_t tO = tmem + lane_base + C::kColO;
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t rr[64];
                tmem_ld64(tO + c * 64, rr);
#pragma unroll
                for (int pc = 0; pc < 8; ++pc) {       // 16-byte pieces of this 64-column atom
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = pack_bf16x2(__uint_as_float(rr[pc * 8 + 2 * e]) * inv_l,
                                           __uint_as_float(rr[pc * 8 + 2 * e + 1]) * inv_l);
                    const uint32_t addr = sb + C::kOffQ + c * C::kChunkBytes + r * 128 +
                                          (static_cast<uint32_t>(pc ^ (r & 7)) << 4);
                    st_shared_v4(addr, w[0], w[1], w[2], w[3]);
                }
            }
            if (p.lse && row_valid)
                p.lse[static_cast<size_t>(bh) * p.N + q_row] = (m_run + log2f(l_run)) * kLn2;
            fence_proxy_async_smem();
        }
        tc_fence_before();
        named_bar_sync(1, kBlockM);
        if (threadIdx.x == 0 && *abort_flag == 0) {
            for (int c = 0; c < C::kChunks; ++c)
                tma_store_3d(&tmO, sb + C::kOffQ + c * C::kChunkBytes, c * 64, qt * kBlockM, bh);
            tma_store_commit();
            tma_store_wait_read();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, bool CAUSAL, bool EXT>
cudaError_t launch_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                     const CUtensorMap &to, const FwdParams &prm, unsigned grid,
                     cudaStream_t stream) {
    using C = FwdCfg<D>;
    auto kern = fwd_kernel<D, CAUSAL, EXT>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, to, prm);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(bool causal, bool ext, const CUtensorMap &tq, const CUtensorMap &tk,
                     const CUtensorMap &tv, const CUtensorMap &to, const FwdParams &prm,
                     unsigned grid, cudaStream_t stream) {
    if (causal)
        return ext ? launch_t<D, true, true>(tq, tk, tv, to, prm, grid, stream)
                   : launch_t<D, true, false>(tq, tk, tv, to, prm, grid, stream);
    return ext ? launch_t<D, false, true>(tq, tk, tv, to, prm, grid, stream)
               : launch_t<D, false, false>(tq, tk, tv, to, prm, grid, stream);
}

}  // namespace

cudaError_t launch_fwd(const FwdProblem &pb, int *status, cudaStream_t stream) {
    const long long BH = static_cast<long long>(pb.B) * pb.Hq;
    const long long BHkv = static_cast<long long>(pb.B) * pb.Hkv;
    CUtensorMap tq, tk, tv, to;
    if (!encode_bf16_rows(&tq, pb.q, pb.D, pb.N, BH, kBlockM) ||
        !encode_bf16_rows(&tk, pb.k, pb.D, pb.N, BHkv, kBlockN) ||
        !encode_bf16_rows(&tv, pb.v, pb.D, pb.N, BHkv, kBlockN) ||
        !encode_bf16_rows(&to, pb.o, pb.D, pb.N, BH, kBlockM))
        return cudaErrorInvalidValue;
    FwdParams prm;
    prm.bias = pb.bias;
    prm.emit = pb.emit;
    prm.lse = pb.lse;
    prm.status = status;
    prm.N = pb.N;
    prm.Hq = pb.Hq;
    prm.Hkv = pb.Hkv;
    prm.group = pb.Hq / pb.Hkv;
    prm.BH = static_cast<int>(BH);
    prm.n_qtiles = (pb.N + kBlockM - 1) / kBlockM;
    prm.scale = pb.scale;
    prm.scale_log2 = pb.scale * kLog2e;
    prm.vec4 = (pb.N % 4 == 0) &&
               (reinterpret_cast<uintptr_t>(pb.bias) % 16 == 0) &&
               (reinterpret_cast<uintptr_t>(pb.emit) % 16 == 0);
    const unsigned grid = static_cast<unsigned>(prm.n_qtiles * BH);
    const bool ext = (pb.bias != nullptr) || (pb.emit != nullptr);
    if (pb.D == 64) return launch_d<64>(pb.causal, ext, tq, tk, tv, to, prm, grid, stream);
    return launch_d<128>(pb.causal, ext, tq, tk, tv, to, prm, grid, stream);
}

}  // namespace tattn
