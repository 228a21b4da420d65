// attn_decode.cu -- single-query decode attention (flash decode) for GB300.
//
// One new query row per (batch, query head) attends to the N cached keys of
// its kv head.  The query sits at position N-1, so the causal mask keeps
// every key and the result equals the last row of causal attention.
//
// The keys of each kv head are split over S CTAs (split-K).  Each CTA
// streams its K/V chunk through a TMA ring and, for every query head of the
// group (G = Hq / Hkv rows share one K/V stream), keeps the online-softmax
// state of its chunk: m (log2 units), l and the unnormalised O.  A second
// kernel merges the S partial states with the block-merge rule of the online
// softmax (kwkr.cn/news/592482, 2.2):
//   M = max_s m_s,   L = sum_s l_s 2^(m_s - M),   O = sum_s O_s 2^(m_s - M) / L,
//   LSE = (M + log2 L) ln 2.
// "FlashAttention原理与Triton实战" section 7 names flash decode as an
// extension of the fused kernel.
//
// Every K/V byte is used by G query rows only, so the kernel is bound by HBM
// bandwidth; its arithmetic runs on the CUDA cores from 128-byte swizzled
// shared memory (conflict-free row reads), not on the tensor cores.
//
// Threads (288): warps 0-7 compute, warp 8 is the TMA producer.
//   scores   thread t takes key t % 64 of the 64-key stage and query heads
//            t / 64, t / 64 + 4, ... (G <= 16)
//   softmax  warp w takes heads w and w + 8: row max / sum over the stage,
//   and PV   then O += p V with lane l holding the bf16 column pairs l, l+32, ...
#include <cuda_bf16.h>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace tattn {
namespace {

constexpr int kKeys = 64;            // keys per stage
constexpr int kMaxGroup = 16;        // query heads per kv head
constexpr int kWorkers = 256;        // compute threads
constexpr int kThreads = kWorkers + 32;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct DecCfg {
    static constexpr int kChunks = (D + 63) / 64;                // 128-byte atoms per row
    static constexpr int kAtomBytes = kKeys * 128;               // one atom column of a stage tile
    static constexpr int kTileBytes = kChunks * kAtomBytes;      // K (or V) of one stage
    // One block per SM with a deep ring: the kernel streams HBM, and every
    // stage but the one being read is a load in flight.
    static constexpr int kOther = kMaxGroup * D * 4 + 2 * kMaxGroup * kKeys * 4 + 1024 + 256;
    static constexpr int kStages = (200 * 1024 - kOther) / (2 * kTileBytes);
    static constexpr int kOffRing = 0;                           // stage s: K then V
    static constexpr int kOffQ = kOffRing + kStages * 2 * kTileBytes;   // fp32 [16][D]
    static constexpr int kOffScore = kOffQ + kMaxGroup * D * 4;         // fp32 [2][16][64]
    static constexpr int kOffBar = kOffScore + 2 * kMaxGroup * kKeys * 4;
    static constexpr int kNumBars = 2 * kStages;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;             // abort flag
    static constexpr int kUsed = kOffMisc + 16;
    static constexpr int kSmemBytes = kUsed + 1023;                     // base alignment slack
    static_assert(kStages >= 2 && kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct DecParams {
    const __nv_bfloat16 *q;   // [B*Hq, D]
    float *m_part;            // [B*Hq, S]   log2-unit running max of each split
    float *l_part;            // [B*Hq, S]   row sum relative to m
    float *o_part;            // [B*Hq, S, D] unnormalised output relative to m
    int *status;
    int N, Hq, Hkv, G, S, chunk;
    float scale_log2;
};

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

__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
decode_split_kernel(const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const DecParams p) {
    using C = DecCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = threadIdx.x;

    const int bg = blockIdx.x / p.S;          // (batch, kv head)
    const int split = blockIdx.x % p.S;
    const int b = bg / p.Hkv, g = bg % p.Hkv;
    const int bh0 = b * p.Hq + g * p.G;       // first query head row of the group
    const int k_begin = split * p.chunk;
    const int k_end = min(p.N, k_begin + p.chunk);
    const int n_it = (k_end - k_begin + kKeys - 1) / kKeys;

    auto bar = [&](int i) -> uint32_t { return sb + C::kOffBar + 8u * i; };
    const int kFull = 0, kEmpty = C::kStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc);
    const AbortCtl ac{abort_flag, p.status};
    float *sQ = reinterpret_cast<float *>(smem + C::kOffQ);
    float *sScore = reinterpret_cast<float *>(smem + C::kOffScore);

    if (t == 0) {
        *abort_flag = 0;
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar(kFull + s), 1);
            mbar_init(bar(kEmpty + s), kWorkers);
        }
        fence_barrier_init();
    }
    // The group's query rows, widened to fp32 (scale applied in the scores).
    for (int i = t; i < p.G * D; i += kThreads) {
        const int h = i / D, d = i % D;
        sQ[h * D + d] = __bfloat162float(p.q[static_cast<size_t>(bh0 + h) * D + d]);
    }
    __syncthreads();

    if (warp == kWorkers / 32) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            bool ok = true;
            int issued = 0;
            for (int it = 0; it < n_it; ++it) {
                const int st = it % C::kStages;
                if (it >= C::kStages)
                    ok = mbar_wait(bar(kEmpty + st), ((it / C::kStages) - 1) & 1, ac);
                if (!ok) break;
                const uint32_t full = bar(kFull + st);
                const uint32_t base = sb + C::kOffRing + st * 2 * C::kTileBytes;
                mbar_arrive_expect_tx(full, 2 * C::kTileBytes);
                const int key0 = k_begin + it * kKeys;
                for (int c = 0; c < C::kChunks; ++c) {
                    tma_load_3d(base + c * C::kAtomBytes, &tmK, full, c * 64, key0, bg);
                    tma_load_3d(base + C::kTileBytes + c * C::kAtomBytes, &tmV, full, c * 64,
                                key0, bg);
                }
                issued = it + 1;
            }
            if (!ok) {
                for (int it = max(issued - C::kStages, 0); it < issued; ++it)
                    drain_wait(bar(kFull + it % C::kStages), (it / C::kStages) & 1);
            }
        }
        __syncwarp();
        return;
    }

    // ------------------------------------------------------------ compute
    // scores: thread t takes key t % 64 and heads t/64, t/64 + 4, ... (< G).
    // softmax and PV: with G <= 8, each head has 8/G warps that split the
    // stage's keys between them (each recomputes the head's row max and sum,
    // which are the same in all of them); with G > 8 each warp takes heads w
    // and w + 8 over all 64 keys.
    const int kk = t & (kKeys - 1);
    const int hs = t >> 6;
    const bool small_group = p.G <= 8;
    const int wph = small_group ? 8 / p.G : 1;            // warps per head
    const int h0 = small_group ? warp / wph : warp;       // this warp's (first) head
    const int kper = kKeys / wph;                         // keys per warp
    const int kfirst = small_group ? (warp % wph) * kper : 0;
    const bool active = h0 < p.G;
    const bool two = !small_group && warp + 8 < p.G;      // second head w + 8
    // PV layout: lane l owns 16-byte column piece l % kLPK (8 columns) of
    // key kq + l / kLPK for kq = 0, kKPI, 2 kKPI, ...; the kKPI partial sums
    // of a piece are added across lanes at the end.
    constexpr int kPieces = D / 8;
    constexpr int kLPK = kPieces <= 8 ? 8 : 16;           // lanes per key
    constexpr int kKPI = 32 / kLPK;                       // keys per warp step
    const int piece = lane % kLPK;
    const int ksub_lane = lane / kLPK;
    const bool piece_ok = piece < kPieces;
    const uint32_t sQaddr = sb + C::kOffQ;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    uint64_t o_acc[2][4];                                 // 8 columns as 4 fp32 pairs
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int j = 0; j < 4; ++j) o_acc[a][j] = 0ull;
    bool ok = true;

    for (int it = 0; it < n_it; ++it) {
        const int st = it % C::kStages;
        const int par = it & 1;
        float *score = sScore + par * kMaxGroup * kKeys;
        const bool got = mbar_wait(bar(kFull + st), (it / C::kStages) & 1, ac);
        const uint32_t kbase = sb + C::kOffRing + st * 2 * C::kTileBytes;
        const uint32_t vbase = kbase + C::kTileBytes;
        const int key0 = k_begin + it * kKeys;

        // --- scores s_h(key) = q_h . k in log2 units, -inf past the chunk
        if (got && hs < p.G) {
            uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
            for (int pc = 0; pc < D / 8; ++pc) {   // 16-byte pieces of the key row
                const uint32_t addr = kbase + (pc / 8) * C::kAtomBytes + kk * 128 +
                                      (static_cast<uint32_t>((pc % 8) ^ (kk & 7)) << 4);
                const float4 raw = ld_shared_f4(addr);
                const uint32_t w[4] = {__float_as_uint(raw.x), __float_as_uint(raw.y),
                                       __float_as_uint(raw.z), __float_as_uint(raw.w)};
                uint64_t kp[4];   // bf16 pairs widened to fp32 pairs
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    kp[e] = f2pack(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xffff0000u));
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int h = hs + 4 * i;
                    if (h < p.G) {
                        const uint32_t qa = sQaddr + (h * D + pc * 8) * 4;
                        const float4 qa4 = ld_shared_f4(qa), qb4 = ld_shared_f4(qa + 16);
                        acc[i] = ffma2(kp[0], f2pack(qa4.x, qa4.y), acc[i]);
                        acc[i] = ffma2(kp[1], f2pack(qa4.z, qa4.w), acc[i]);
                        acc[i] = ffma2(kp[2], f2pack(qb4.x, qb4.y), acc[i]);
                        acc[i] = ffma2(kp[3], f2pack(qb4.z, qb4.w), acc[i]);
                    }
                }
            }
            const bool valid = key0 + kk < k_end;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int h = hs + 4 * i;
                if (h < p.G) {
                    float lo, hi;
                    f2unpack(acc[i], lo, hi);
                    score[h * kKeys + kk] = valid ? (lo + hi) * p.scale_log2 : -INFINITY;
                }
            }
        }
        // Every worker reaches the barrier; a failed wait leaves through it.
        if (named_bar_or(1, kWorkers, !got)) {
            ok = false;
            break;
        }

        if (active) {
            // --- online softmax over the stage's 64 keys (whole row)
            float pk0[2], pk1[2], alpha[2] = {1.f, 1.f};
#pragma unroll
            for (int a = 0; a < 2; ++a) {
                pk0[a] = pk1[a] = 0.f;
                if (a == 1 && !two) continue;
                const float *sh = score + (a == 0 ? h0 : warp + 8) * kKeys;
                const float s0 = sh[lane], s1 = sh[lane + 32];
                const float mt = warp_max(fmaxf(s0, s1));
                const float m_new = fmaxf(m_run[a], mt);
                const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                alpha[a] = ex2(m_run[a] - m_use);
                pk0[a] = ex2(s0 - m_use);
                pk1[a] = ex2(s1 - m_use);
                l_run[a] = l_run[a] * alpha[a] + warp_sum(pk0[a] + pk1[a]);
                m_run[a] = m_new;
            }
#pragma unroll
            for (int a = 0; a < 2; ++a) {
                const uint64_t al = f2pack(alpha[a], alpha[a]);
#pragma unroll
                for (int j = 0; j < 4; ++j) o_acc[a][j] = fmul2(o_acc[a][j], al);
            }
            // --- O += p V over this warp's keys
            const uint32_t vpiece = vbase + (piece / 8) * C::kAtomBytes;
#pragma unroll 4
            for (int kq = 0; kq < kper; kq += kKPI) {
                const int key = kfirst + kq + ksub_lane;
                // kKPI consecutive keys starting at a multiple of kKPI lie on the
                // same side of 32, so one select serves the whole warp.
                const bool lo_half = kfirst + kq < 32;
                const float pa = __shfl_sync(0xffffffffu, lo_half ? pk0[0] : pk1[0], key & 31);
                const float pb = __shfl_sync(0xffffffffu, lo_half ? pk0[1] : pk1[1], key & 31);
                if (piece_ok) {
                    const uint32_t addr =
                        vpiece + key * 128 + (static_cast<uint32_t>((piece % 8) ^ (key & 7)) << 4);
                    const float4 raw = ld_shared_f4(addr);
                    const uint32_t w[4] = {__float_as_uint(raw.x), __float_as_uint(raw.y),
                                           __float_as_uint(raw.z), __float_as_uint(raw.w)};
                    const uint64_t pa2 = f2pack(pa, pa), pb2 = f2pack(pb, pb);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint64_t vf = f2pack(__uint_as_float(w[j] << 16),
                                                   __uint_as_float(w[j] & 0xffff0000u));
                        o_acc[0][j] = ffma2(pa2, vf, o_acc[0][j]);
                        if (two) o_acc[1][j] = ffma2(pb2, vf, o_acc[1][j]);
                    }
                }
            }
        }
        mbar_arrive(bar(kEmpty + st));   // this worker is done with the stage's K and V
    }

    // ------------------------------------------------ partial state out
    // Add the kKPI key lanes of each piece, then, with G <= 8, the warps of a
    // head (disjoint key subsets, same reference max) through shared memory.
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int off = kLPK; off < 32; off <<= 1) {
                float lo, hi;
                f2unpack(o_acc[a][j], lo, hi);
                lo += __shfl_xor_sync(0xffffffffu, lo, off);
                hi += __shfl_xor_sync(0xffffffffu, hi, off);
                o_acc[a][j] = f2pack(lo, hi);
            }
        }
    float *red = sScore;   // [8 warps][D], free after the last stage
    named_bar_sync(1, kWorkers);
    if (ok && active && small_group && wph > 1 && lane < kLPK && piece_ok) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float lo, hi;
            f2unpack(o_acc[0][j], lo, hi);
            red[warp * D + piece * 8 + 2 * j] = lo;
            red[warp * D + piece * 8 + 2 * j + 1] = hi;
        }
    }
    named_bar_sync(1, kWorkers);
    if (ok && active && (!small_group || warp % wph == 0)) {
#pragma unroll
        for (int a = 0; a < 2; ++a) {
            if (a == 1 && !two) continue;
            const int h = a == 0 ? h0 : warp + 8;
            const size_t ps = static_cast<size_t>(bh0 + h) * p.S + split;
            if (lane == 0) {
                p.m_part[ps] = m_run[a];
                p.l_part[ps] = l_run[a];
            }
            if (lane < kLPK && piece_ok) {
                float out[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) f2unpack(o_acc[a][j], out[2 * j], out[2 * j + 1]);
                if (small_group) {
                    for (int w2 = 1; w2 < wph; ++w2)
#pragma unroll
                        for (int e = 0; e < 8; ++e) out[e] += red[(warp + w2) * D + piece * 8 + e];
                }
                float4 *dst = reinterpret_cast<float4 *>(p.o_part + ps * D + piece * 8);
                dst[0] = make_float4(out[0], out[1], out[2], out[3]);
                dst[1] = make_float4(out[4], out[5], out[6], out[7]);
            }
        }
    }
}

// One warp per (batch, query head): merges the S partial states.
__global__ void __launch_bounds__(256)
decode_merge_kernel(const float *__restrict__ m_part, const float *__restrict__ l_part,
                    const float *__restrict__ o_part, __nv_bfloat16 *__restrict__ o,
                    float *__restrict__ lse, int rows, int S, int D) {
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float *mr = m_part + static_cast<size_t>(row) * S;
    const float *lr = l_part + static_cast<size_t>(row) * S;
    float M = -INFINITY;
    for (int s = lane; s < S; s += 32) M = fmaxf(M, mr[s]);
    M = warp_max(M);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float L = 0.f;
    for (int s = lane; s < S; s += 32) L += lr[s] * ex2(mr[s] - Mu);
    L = warp_sum(L);
    const float inv_l = 1.f / L;
    for (int d = lane; d < D; d += 32) {
        float acc = 0.f;
        for (int s = 0; s < S; ++s)
            acc = fmaf(o_part[(static_cast<size_t>(row) * S + s) * D + d], ex2(mr[s] - Mu), acc);
        o[static_cast<size_t>(row) * D + d] = __float2bfloat16_rn(acc * inv_l);
    }
    if (lse && lane == 0) lse[row] = (Mu + log2f(L)) * kLn2;
}

template <int D>
cudaError_t launch_d(const DecProblem &pb, int *status, cudaStream_t stream) {
    using C = DecCfg<D>;
    const long long BHkv = static_cast<long long>(pb.B) * pb.Hkv;
    CUtensorMap tk, tv;
    if (!encode_bf16_rows(&tk, pb.k, D, pb.N, BHkv, kKeys) ||
        !encode_bf16_rows(&tv, pb.v, D, pb.N, BHkv, kKeys))
        return cudaErrorInvalidValue;
    DecParams prm;
    prm.q = static_cast<const __nv_bfloat16 *>(pb.q);
    prm.m_part = pb.m_part;
    prm.l_part = pb.l_part;
    prm.o_part = pb.o_part;
    prm.status = status;
    prm.N = pb.N;
    prm.Hq = pb.Hq;
    prm.Hkv = pb.Hkv;
    prm.G = pb.Hq / pb.Hkv;
    prm.S = pb.splits;
    prm.chunk = pb.chunk;
    prm.scale_log2 = pb.scale * 1.4426950408889634f;
    auto kern = decode_split_kernel<D>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(BHkv * pb.splits), kThreads, C::kSmemBytes, stream>>>(tk, tv,
                                                                                        prm);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int rows = pb.B * pb.Hq;
    decode_merge_kernel<<<(rows + 7) / 8, 256, 0, stream>>>(
        pb.m_part, pb.l_part, pb.o_part, static_cast<__nv_bfloat16 *>(pb.o), pb.lse, rows,
        pb.splits, D);
    return cudaGetLastError();
}

}  // namespace

int decode_max_splits(int N) {
    const int s = (N + 127) / 128;
    return s < 64 ? s : 64;
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
