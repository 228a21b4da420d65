// attn_decode.cu -- single-query decode attention (flash decode) for GB300.
//
// One new query row per (batch, query head) attends to the N cached keys of
// its kv head.  The query sits at position N-1, so the causal mask keeps
// every key and the result equals the last row of causal attention.
//
// The work is the sequence of (kv head, 128-key stage) pairs; a persistent
// block per SM takes an equal contiguous run of it (stream-K), streams those
// K/V stages through a TMA ring and, for every query head of the group (G =
// Hq / Hkv rows share one K/V stream), keeps the online-softmax state of the
// run's part in each kv head -- a segment: m (log2 units), l and the
// unnormalised O.  A second kernel merges a head's segments with the
// block-merge rule of the online softmax (kwkr.cn/news/592482, 2.2):
//   M = max_s m_s,   L = sum_s l_s 2^(m_s - M),   O = sum_s O_s 2^(m_s - M) / L,
//   LSE = (M + log2 L) ln 2.
// "FlashAttention原理与Triton实战" section 7 names flash decode as an
// extension of the fused kernel.
//
// Every K/V byte serves only G query rows, so the kernel is bound by HBM
// bandwidth; the two contractions still run on the tensor cores, in
// transposed form so that the M dimension is the 128 keys of a stage (S^T =
// K q^T) and the 128 (padded) columns of V (O^T = V^T P^T), with the G <= 16
// heads as N.  On the CUDA cores that leaves one exp2 per key and head.
//
// Threads (192): warps 0-3 softmax and output (thread t = TMEM lane t),
// warp 4 TMA producer (128-key K/V stages), warp 5 TMEM allocation and MMA.
#include <cuda_bf16.h>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace tattn {
namespace {

// Programmatic dependent launch.  griddep_launch_dependents lets a kernel
// launched after this one with programmatic stream serialization start its
// blocks now (once every block of this grid has signalled or exited);
// griddep_wait blocks until the grids this one depends on have completed and
// their memory operations are visible (a no-op without the dependency).
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

constexpr int kKeys = 128;           // keys per stage: the MMA M of S^T
constexpr int kHeads = 16;           // query heads of a group, padded: the MMA N
constexpr int kThreads = 192;        // warps 0-3 softmax / output, 4 producer, 5 MMA
constexpr int kWarpProducer = 4;
constexpr int kWarpMma = 5;
constexpr float kLn2 = 0.6931471805599453f;
// Lazy rescale (as in the forward): the reference max of a head only moves
// when the head's max grows by more than 2^8.
constexpr float kRescaleLog2 = 8.0f;

template <int D>
struct DecCfg {
    // K and V move through separate rings, so that a K slot is refilled as
    // soon as the score MMA has read it (V waits for the PV MMA).  A slot
    // holds the 128-byte atoms (64 columns) that cover D; TMA fills columns
    // D .. 127 of the last one with zeros at D = 80, 96.  The PV MMA runs
    // with M = 128: at D = 64 its second 64-row block of V^T is a shared
    // dummy atom, whose (arbitrary) contents only reach output rows >= 64,
    // which are never stored.
    static constexpr int kAtomBytes = kKeys * 128;               // 16 KB
    static constexpr int kLoadAtoms = (D + 63) / 64;
    static constexpr int kSlotBytes = kLoadAtoms * kAtomBytes;   // K or V of one stage
    static constexpr int kDummyBytes = kLoadAtoms == 1 ? kAtomBytes : 0;
    static constexpr int kHAtom = kHeads * 128;                  // 16 rows of one atom: 2 KB
    static constexpr int kOther = 2 * 2 * kHAtom + 2 * 2 * kHAtom + kHeads * kKeys * 4 +
                                  kHeads * 4 + 1024 + 512;
    static constexpr int kStagesFit = (227 * 1024 - kOther - kDummyBytes) / (2 * kSlotBytes);
    static constexpr int kStages = kStagesFit > 6 ? 6 : kStagesFit;
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kStages * kSlotBytes;
    static constexpr int kOffDummy = kOffV + kStages * kSlotBytes;
    static constexpr int kOffQ = kOffDummy + kDummyBytes;              // 2 x bf16 [16][128]
    static constexpr int kOffP = kOffQ + 2 * 2 * kHAtom;               // 2 x bf16 [16][128]
    static constexpr int kOffScore = kOffP + 2 * 2 * kHAtom;           // fp32 [16][128]
    static constexpr int kOffAlpha = kOffScore + kHeads * kKeys * 4;   // fp32 [16]
    static constexpr int kOffBar = kOffAlpha + kHeads * 4;
    static constexpr int kBarKFull = 0;
    static constexpr int kBarKEmpty = kStages;
    static constexpr int kBarVFull = 2 * kStages;
    static constexpr int kBarVEmpty = 3 * kStages;
    static constexpr int kBarQFull = 4 * kStages;
    static constexpr int kBarQEmpty = kBarQFull + 2;
    static constexpr int kBarDrain = kBarQEmpty + 2;
    static constexpr int kNumBars = kBarDrain + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;            // tmem slot, abort flag
    static constexpr int kUsed = kOffMisc + 16;
    static constexpr int kSmemBytes = kUsed + 1023 <= 227 * 1024 ? kUsed + 1023 : 227 * 1024;
    static_assert(kStages >= 2 && kUsed <= 227 * 1024, "shared memory budget");
    // TMEM: S^T buffers at columns 0 and 32, O^T at 64 (16 columns each)
    static constexpr uint32_t kTmemCols = 128;
    static constexpr uint32_t kColO = 64;
};

struct DecParams {
    float *m_part;            // [slots, G]     log2-unit reference max of a segment
    float *l_part;            // [slots, G]     row sum relative to it
    float *o_part;            // [slots, G, D]  unnormalised output relative to it
    int *status;
    int N, G, spg;            // spg = 128-key stages per kv head
    long long T;              // total stages: B * Hkv * spg
    int grid;
    float scale_log2;
};

// Work split (stream-K): block c of `grid` takes the stages
// [c T / grid, (c+1) T / grid) of the flattened (kv head, stage) order, so
// every block streams the same number of K/V bytes.  A kv head's stages that
// fall in one block form a segment with its own softmax state; the segment
// of block c and kv head bg writes slot c + bg (both indices grow along the
// order, so the slot is unique and below grid + heads - 1).
__host__ __device__ __forceinline__ long long range_begin(int c, long long T, int grid) {
    return static_cast<long long>(c) * T / grid;
}
// The block whose range holds stage x.
__device__ __forceinline__ int block_of(long long x, long long T, int grid) {
    return static_cast<int>(((x + 1) * grid + T - 1) / T - 1);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > 20ull * 1000ull * 1000ull) break;
    }
}

__device__ __forceinline__ void st_shared_v2(uint32_t addr, uint32_t a, uint32_t b) {
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}

// Byte offset of element (row, col) in a [16 rows][128 cols] bf16 tile of
// two 128-byte-swizzled atoms (64 columns each, `atom` bytes apart).
__device__ __forceinline__ uint32_t sw_off(int row, int col, int atom) {
    return (col / 64) * atom + row * 128 +
           (static_cast<uint32_t>(((col % 64) / 8) ^ (row & 7)) << 4) + (col % 8) * 2;
}

// Position of a block's walk along its stages: kv head and stage within it.
struct Walk {
    int bg, ks, spg;
    __device__ void step() {
        if (++ks == spg) {
            ks = 0;
            ++bg;
        }
    }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
decode_split_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const DecParams p) {
    using C = DecCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    if (smem - smem_raw + C::kUsed > C::kSmemBytes) {
        if (threadIdx.x == 0) atomicCAS(p.status, kStatusOk, kStatusDeviceCheck);
        return;
    }
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = threadIdx.x;

    const int c = blockIdx.x;
    const long long x0 = range_begin(c, p.T, p.grid);
    const int n_it = static_cast<int>(range_begin(c + 1, p.T, p.grid) - x0);
    const Walk start{static_cast<int>(x0 / p.spg), static_cast<int>(x0 % p.spg), p.spg};

    auto bar = [&](int i) -> uint32_t { return sb + C::kOffBar + 8u * i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
    const AbortCtl ac{abort_flag, p.status, kWaitLimitNs};
    float *sScore = reinterpret_cast<float *>(smem + C::kOffScore);   // [16 heads][128 keys]
    float *sAlpha = reinterpret_cast<float *>(smem + C::kOffAlpha);   // [16]

    if (t == 0) {
        *abort_flag = 0;
        // KEmpty[s] completes when the score MMA of the stage in K slot s
        // is done (the softmax waits on it too); VFull[s] when V has landed
        // AND the 128 softmax threads have written P^T of that stage (one
        // wait for the MMA thread); VEmpty[s] when the PV MMA is done (the
        // softmax waits on it before reusing a P^T buffer).
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar(C::kBarKFull + s), 1);
            mbar_init(bar(C::kBarKEmpty + s), 1);
            mbar_init(bar(C::kBarVFull + s), 1 + 128);
            mbar_init(bar(C::kBarVEmpty + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(C::kBarQFull + s), 1);
            mbar_init(bar(C::kBarQEmpty + s), 1);
        }
        mbar_init(bar(C::kBarDrain), 1);
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // The merge kernel's blocks may be scheduled beside this grid's from now
    // on; they wait (griddep_wait) until this grid has finished.
    if (t == 0) griddep_launch_dependents();

    if (warp == kWarpProducer) {
        // ------------------------------------------------------ TMA producer
        // Per segment the 16 query rows of its kv head (rows of the next
        // head, or zero fill past the last one, pad a group smaller than 16);
        // per stage 128 keys of K and of V.  (K slots free up after the score
        // MMA, V slots after the PV MMA; issuing the two together measured
        // faster than running K a stage ahead.)
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            int k_issued = 0, v_issued = 0, seg = -1;
            Walk wk = start, wv = start;
            auto load_k = [&](int j) -> bool {
                if (j == 0 || wk.ks == 0) {
                    const int qb = (++seg) & 1;
                    if (seg >= 2 && !mbar_wait(bar(C::kBarQEmpty + qb), ((seg - 2) >> 1) & 1, ac))
                        return false;
                    const uint32_t qfull = bar(C::kBarQFull + qb);
                    mbar_arrive_expect_tx(qfull, C::kLoadAtoms * C::kHAtom);
                    for (int a = 0; a < C::kLoadAtoms; ++a)
                        tma_load_3d(sb + C::kOffQ + qb * 2 * C::kHAtom + a * C::kHAtom, &tmQ, qfull,
                                    a * 64, wk.bg * p.G, 0);
                }
                const int st = j % C::kStages;
                if (j >= C::kStages &&
                    !mbar_wait(bar(C::kBarKEmpty + st), ((j / C::kStages) - 1) & 1, ac))
                    return false;
                const uint32_t full = bar(C::kBarKFull + st);
                mbar_arrive_expect_tx(full, C::kSlotBytes);
                for (int a = 0; a < C::kLoadAtoms; ++a)
                    tma_load_3d(sb + C::kOffK + st * C::kSlotBytes + a * C::kAtomBytes, &tmK, full,
                                a * 64, wk.ks * kKeys, wk.bg);
                wk.step();
                k_issued = j + 1;
                return true;
            };
            auto load_v = [&](int j) -> bool {
                const int st = j % C::kStages;
                if (j >= C::kStages &&
                    !mbar_wait(bar(C::kBarVEmpty + st), ((j / C::kStages) - 1) & 1, ac))
                    return false;
                const uint32_t full = bar(C::kBarVFull + st);
                mbar_arrive_expect_tx(full, C::kSlotBytes);
                for (int a = 0; a < C::kLoadAtoms; ++a)
                    tma_load_3d(sb + C::kOffV + st * C::kSlotBytes + a * C::kAtomBytes, &tmV, full,
                                a * 64, wv.ks * kKeys, wv.bg);
                wv.step();
                v_issued = j + 1;
                return true;
            };
            bool ok = true;
            for (int j = 0; j < n_it && ok; ++j) {
                if (!(ok = load_k(j))) break;
                ok = load_v(j);
            }
            if (!ok) {
                for (int j = max(k_issued - C::kStages, 0); j < k_issued; ++j)
                    drain_wait(bar(C::kBarKFull + j % C::kStages), (j / C::kStages) & 1);
                for (int j = max(v_issued - C::kStages, 0); j < v_issued; ++j)
                    drain_wait(bar(C::kBarVFull + j % C::kStages), (j / C::kStages) & 1);
                for (int k = max(seg - 1, 0); k <= seg; ++k)
                    drain_wait(bar(C::kBarQFull + (k & 1)), (k >> 1) & 1);
            }
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------- MMA issuer
        // Per stage: S^T = K q^T (M = 128 keys, N = 16 heads, K = D), then,
        // once the softmax has written P^T: O^T += V^T P^T (M = 128 columns
        // of V, N = 16 heads, K = 128 keys; V is the MN-major A operand).
        // S^T of the next stage is issued before P^T of this one is awaited,
        // so the score MMA overlaps the softmax.  (Each MMA instruction takes
        // about as long to issue at N = 16 as at N = 128, and each barrier
        // wait costs about as much as one even when the phase is complete:
        // the loop keeps both counts down.)
        if (lane == 0) {
            constexpr uint32_t kIdS = idesc_bf16_f32(kKeys, kHeads, false, false);
            constexpr uint32_t kIdPV = idesc_bf16_f32(128, kHeads, true, false);
            Walk ws = start, wv = start;
            int seg = -1;
            auto issue_s = [&](int j) -> bool {
                const bool first = j == 0 || ws.ks == 0;
                const bool last = j == n_it - 1 || ws.ks == p.spg - 1;
                ws.step();
                if (first) ++seg;
                const int qb = seg & 1;
                if (first && !mbar_wait(bar(C::kBarQFull + qb), (seg >> 1) & 1, ac)) return false;
                const int st = j % C::kStages;
                if (!mbar_wait(bar(C::kBarKFull + st), (j / C::kStages) & 1, ac)) return false;
                tc_fence_after();
                const uint32_t kbase = sb + C::kOffK + st * C::kSlotBytes;
                const uint32_t qbase = sb + C::kOffQ + qb * 2 * C::kHAtom;
                const uint32_t tS = tmem + (j & 1) * 32;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t adesc = sdesc_sw128(
                        kbase + (kk >> 2) * C::kAtomBytes + (kk & 3) * 32, 16, 1024);
                    const uint64_t bdesc =
                        sdesc_sw128(qbase + (kk >> 2) * C::kHAtom + (kk & 3) * 32, 16, 1024);
                    mma_ss(tS, adesc, bdesc, kIdS, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(C::kBarKEmpty + st));
                if (last) mma_commit(bar(C::kBarQEmpty + qb));
                return true;
            };
            bool ok = n_it > 0 && issue_s(0);
            for (int it = 0; it < n_it && ok; ++it, wv.step()) {
                if (it + 1 < n_it && !(ok = issue_s(it + 1))) break;
                const int st = it % C::kStages;
                if (!(ok = mbar_wait(bar(C::kBarVFull + st), (it / C::kStages) & 1, ac))) break;
                tc_fence_after();
                const bool first = it == 0 || wv.ks == 0;
                const uint32_t voff = C::kOffV + st * C::kSlotBytes;
                const uint32_t vbase = sb + voff;
                // distance to the second 64-row block of V^T
                const uint32_t lbo = C::kLoadAtoms == 2 ? C::kAtomBytes : C::kOffDummy - voff;
                const uint32_t pbase = sb + C::kOffP + (it & 1) * 2 * C::kHAtom;
#pragma unroll
                for (int kk = 0; kk < kKeys / 16; ++kk) {
                    const uint64_t adesc = sdesc_sw128(vbase + kk * 2048, lbo, 1024);
                    const uint64_t bdesc = sdesc_sw128(
                        pbase + (kk >> 2) * C::kHAtom + (kk & 3) * 32, 16, 1024);
                    mma_ss(tmem + C::kColO, adesc, bdesc, kIdPV, (!first || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar(C::kBarVEmpty + st));
            }
            if (!ok && n_it > 0) {
                mma_commit(bar(C::kBarDrain));
                drain_wait(bar(C::kBarDrain), 0);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------ softmax and output (128)
        // Thread t is TMEM lane t: key t of the stage for S^T, column t of V
        // (output column d = t) for O^T.  Warp w keeps the softmax state of
        // heads w, w + 4, w + 8, w + 12; the four are processed side by side
        // (padded heads too: they are finite and never stored) so that their
        // shuffle reductions overlap.
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        float m_run[4], l_run[4];
        Walk w = start;
        for (int it = 0; it < n_it; ++it, w.step()) {
            const bool first = it == 0 || w.ks == 0;
            const bool last = it == n_it - 1 || w.ks == p.spg - 1;
            if (first) {
#pragma unroll
                for (int i = 0; i < 4; ++i) { m_run[i] = -INFINITY; l_run[i] = 0.f; }
            }
            const int st = it % C::kStages;
            const uint32_t ph = (it / C::kStages) & 1;
            bool got = mbar_wait_warp(bar(C::kBarKEmpty + st), ph, ac);   // S^T(it) done
            if (got) {
                tc_fence_after();
                uint32_t sr[16];
                tmem_ld16(tmem + lane_base + (it & 1) * 32, sr);
                const bool valid = w.ks * kKeys + t < p.N;
#pragma unroll
                for (int h = 0; h < kHeads; ++h)   // transposed: [head][key], conflict-free
                    sScore[h * kKeys + t] =
                        valid ? __uint_as_float(sr[h]) * p.scale_log2 : -INFINITY;
                tc_fence_before();
            }
            if (named_bar_or(1, 128, !got)) break;
            // P^T(it) overwrites P^T(it-2): PV(it-2) must be done with it.
            if (it >= 2)
                got = mbar_wait_warp(bar(C::kBarVEmpty + (it - 2) % C::kStages),
                                     ((it - 2) / C::kStages) & 1, ac);
            const uint32_t pbase = sb + C::kOffP + (it & 1) * 2 * C::kHAtom;
            bool need = false;
            if (got) {
                // Lane l takes keys 4l .. 4l+3: one 16-byte score read and
                // one 8-byte store of four bf16 probabilities per head (the
                // four share a 16-byte swizzle chunk).
                float4 sv[4];
                float mt[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    sv[i] = *reinterpret_cast<const float4 *>(&sScore[(warp + 4 * i) * kKeys + 4 * lane]);
                    mt[i] = fmaxf(fmaxf(sv[i].x, sv[i].y), fmaxf(sv[i].z, sv[i].w));
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        mt[i] = fmaxf(mt[i], __shfl_xor_sync(0xffffffffu, mt[i], o));
                float ps[4], al[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int h = warp + 4 * i;
                    float m_new = fmaxf(m_run[i], mt[i]);
                    if (m_new - m_run[i] <= kRescaleLog2) m_new = m_run[i];
                    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                    al[i] = ex2(m_run[i] - m_use);   // 0 at a segment's first stage
                    const float p0 = ex2(sv[i].x - m_use), p1 = ex2(sv[i].y - m_use);
                    const float p2 = ex2(sv[i].z - m_use), p3 = ex2(sv[i].w - m_use);
                    const __nv_bfloat162 b01 = __floats2bfloat162_rn(p0, p1);
                    const __nv_bfloat162 b23 = __floats2bfloat162_rn(p2, p3);
                    st_shared_v2(pbase + sw_off(h, 4 * lane, C::kHAtom),
                                 *reinterpret_cast<const uint32_t *>(&b01),
                                 *reinterpret_cast<const uint32_t *>(&b23));
                    ps[i] = (p0 + p1) + (p2 + p3);
                    m_run[i] = m_new;
                    need = need || (h < p.G && !first && al[i] < 1.f);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                    for (int i = 0; i < 4; ++i) ps[i] += __shfl_xor_sync(0xffffffffu, ps[i], o);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    l_run[i] = l_run[i] * al[i] + ps[i];
                    if (lane == 0) sAlpha[warp + 4 * i] = al[i];
                }
            }
            // Rare events (a head's reference max moved, or a wait failed)
            // cost a second barrier; every thread takes part in each.
            if (named_bar_or(2, 128, need || !got)) {
                if (named_bar_or(1, 128, !got)) break;
                // Rescale O^T (column h by alpha_h) once PV(it-1) is in it.
                bool okr = mbar_wait_warp(bar(C::kBarVEmpty + (it - 1) % C::kStages),
                                          ((it - 1) / C::kStages) & 1, ac);
                if (okr) {
                    tc_fence_after();
                    uint32_t orr[16];
                    tmem_ld16(tmem + lane_base + C::kColO, orr);
#pragma unroll
                    for (int h = 0; h < kHeads; ++h)
                        orr[h] = __float_as_uint(__uint_as_float(orr[h]) * sAlpha[h]);
                    tmem_st16(tmem + lane_base + C::kColO, orr);
                    tmem_st_wait();
                }
                if (named_bar_or(1, 128, !okr)) break;
            }
            fence_proxy_async_smem();   // P^T for the MMA (async proxy)
            tc_fence_before();
            mbar_arrive(bar(C::kBarVFull + st));
            if (last) {
                // Segment done: its partial state goes to slot c + bg.
                const bool okd = mbar_wait_warp(bar(C::kBarVEmpty + st), ph, ac);
                if (named_bar_or(1, 128, !okd)) break;
                tc_fence_after();
                const size_t slot = static_cast<size_t>(c + w.bg) * p.G;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int h = warp + 4 * i;
                    if (h < p.G && lane == 0) {
                        p.m_part[slot + h] = m_run[i];
                        p.l_part[slot + h] = l_run[i];
                    }
                }
                uint32_t orr[16];
                tmem_ld16(tmem + lane_base + C::kColO, orr);
                tc_fence_before();
                if (t < D) {
#pragma unroll
                    for (int h = 0; h < kHeads; ++h)
                        if (h < p.G) p.o_part[(slot + h) * D + t] = __uint_as_float(orr[h]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// One warp per (batch, query head): merges the partial states of the
// segments its kv head was split into.
__global__ void __launch_bounds__(256)
decode_merge_kernel(const float *__restrict__ m_part, const float *__restrict__ l_part,
                    const float *__restrict__ o_part, __nv_bfloat16 *__restrict__ o,
                    float *__restrict__ lse, int rows, int G, int D, int spg, long long T,
                    int grid) {
    // Launched as a programmatic dependent of the split kernel: its partials
    // are complete and visible once this returns.
    griddep_wait();
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int bg = row / G, h = row % G;
    const int c0 = block_of(static_cast<long long>(bg) * spg, T, grid);
    const int c1 = block_of(static_cast<long long>(bg) * spg + spg - 1, T, grid);
    float M = -INFINITY;
    for (int cc = c0 + lane; cc <= c1; cc += 32)
        M = fmaxf(M, m_part[static_cast<size_t>(cc + bg) * G + h]);
    M = warp_max(M);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float L = 0.f;
    for (int cc = c0 + lane; cc <= c1; cc += 32) {
        const size_t s = static_cast<size_t>(cc + bg) * G + h;
        L += l_part[s] * ex2(m_part[s] - Mu);
    }
    L = warp_sum(L);
    const float inv_l = 1.f / L;
    for (int d = lane; d < D; d += 32) {
        float acc = 0.f;
        for (int cc = c0; cc <= c1; ++cc) {
            const size_t s = static_cast<size_t>(cc + bg) * G + h;
            acc = fmaf(o_part[s * D + d], ex2(m_part[s] - Mu), acc);
        }
        o[static_cast<size_t>(row) * D + d] = __float2bfloat16_rn(acc * inv_l);
    }
    if (lse && lane == 0) lse[row] = (Mu + log2f(L)) * kLn2;
}

template <int D>
cudaError_t launch_d(const DecProblem &pb, int *status, cudaStream_t stream) {
    using C = DecCfg<D>;
    const long long BHkv = static_cast<long long>(pb.B) * pb.Hkv;
    CUtensorMap tq, tk, tv;
    if (!encode_bf16_rows(&tq, pb.q, D, pb.B * pb.Hq, 1, kHeads) ||
        !encode_bf16_rows(&tk, pb.k, D, pb.N, BHkv, kKeys) ||
        !encode_bf16_rows(&tv, pb.v, D, pb.N, BHkv, kKeys))
        return cudaErrorInvalidValue;
    DecParams prm;
    prm.m_part = pb.m_part;
    prm.l_part = pb.l_part;
    prm.o_part = pb.o_part;
    prm.status = status;
    prm.N = pb.N;
    prm.G = pb.Hq / pb.Hkv;
    prm.spg = (pb.N + kKeys - 1) / kKeys;
    prm.T = BHkv * prm.spg;
    prm.grid = pb.grid;
    prm.scale_log2 = pb.scale * 1.4426950408889634f;
    auto kern = decode_split_kernel<D>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(pb.grid), kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, prm);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int rows = pb.B * pb.Hq;
    // Programmatic stream serialization: the merge's blocks start while the
    // split kernel runs and wait in the kernel for it to finish, which hides
    // the second launch's latency.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((rows + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, decode_merge_kernel, static_cast<const float *>(pb.m_part),
                           static_cast<const float *>(pb.l_part),
                           static_cast<const float *>(pb.o_part),
                           static_cast<__nv_bfloat16 *>(pb.o), pb.lse, rows, prm.G, static_cast<int>(D),
                           prm.spg, prm.T, static_cast<int>(pb.grid));
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

long long decode_stages(int B, int Hkv, int N) {
    return static_cast<long long>(B) * Hkv * ((static_cast<long long>(N) + kKeys - 1) / kKeys);
}

cudaError_t launch_decode(const DecProblem &pb, int *status, cudaStream_t stream) {
    switch (pb.D) {
    case 64: return launch_d<64>(pb, status, stream);
    case 80: return launch_d<80>(pb, status, stream);
    case 96: return launch_d<96>(pb, status, stream);
    default: return launch_d<128>(pb, status, stream);
    }
}

}  // namespace tattn
