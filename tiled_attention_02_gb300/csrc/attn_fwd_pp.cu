// attn_fwd_pp.cu -- tiled exact-attention forward, two query tiles per CTA.
//
// The same computation as attn_fwd.cu (the online-softmax double loop of
// kwkr.cn/news/592482, sections 2.2-2.3; "FlashAttention原理与Triton实战"
// 2.2, 3.3), for the plain forward without bias or emitted logits.  A work
// item is a pair of adjacent 128-row query tiles, A and B, of one (batch,
// query head); both consume the same K_j / V_j tiles from shared memory.
// Each tile has its own softmax warps, S/P buffer and O accumulator in TMEM,
// and the tensor core alternates between the tiles:
//
//   S_A(j)  PV_B(j-1)  S_B(j)  PV_A(j)  S_A(j+1)  PV_B(j)  S_B(j+1) ...
//
// so that while tile A's softmax turns S_A(j) into P_A(j), the tensor core
// runs tile B's PV and score MMAs, and the other way round.  With one query
// tile per CTA the tensor core waits for each softmax; here it mostly does
// not.
//
// Warp roles (352 threads, one CTA per SM, persistent):
//   warps 0-3    tile A softmax: thread r owns query row r (TMEM lane r) and
//                all 128 keys of every key tile, so a row's max, sum and
//                rescale need no exchange between threads;
//   warps 4-7    tile B softmax, the same;
//   warp 8       TMA producer: Q_A / Q_B per item, then K_j, V_j rings;
//   warp 9       TMEM allocator and tcgen05.mma issuer (one thread): tile
//                A's MMAs at D = 64, both tiles' otherwise;
//   warp 10      tile B's tcgen05.mma issuer at D = 64.
// A thread that issues tcgen05.mma waits some 60-80 cycles per instruction
// whatever its size (measured on this GPU: one thread issues an M = 128,
// N = 64 MMA every ~78 cycles, two threads in different warps together one
// every ~40).  At D = 64, where the PV MMAs are N = 64 and the tiles' score
// and PV MMAs are decoupled by the separate P buffers below, each tile has
// an issuer of its own; both issuers wait for every K / V stage and each
// commits the stage's release once (two arrivals), which keeps their ring
// phases from mixing.  With P written over S, one issuer keeps each tile's
// MMA groups whole (interleaving two issuers' instructions would delay
// every score tile, and with it the next softmax).
// TMEM (512 columns): S/P of A at 0, of B at 128; O of A at 256, of B at 384.
//
// An S_T(j) commit tracks every MMA issued before it, PV_T(j-1) included,
// so the softmax of S_T(j) may rescale O_T in TMEM without a further wait.
//
// At D = 64 TMEM also holds a separate P buffer per tile (S at 0 / 128, P
// at 256 / 320, O at 384 / 448).  The softmax then releases S_T(j) as soon
// as it has loaded it into registers, and the tile's issuer runs one key
// tile ahead: S_T(j+1), then PV_T(j).  S_T(j+1) is computed while the
// softmax still works on S_T(j), so the softmax of a tile runs back to back
// instead of waiting for PV_T(j) and S_T(j+1) in turn.
// The output rows are written from registers straight to global memory
// (16-byte stores, rows past N skipped), which frees the Q buffers as soon
// as an item's last score MMA is done.
#include "attn_internal.h"
#include "sm103_ptx.cuh"

#include <algorithm>

namespace tattn {
namespace {

constexpr int kBlockM = 128;   // query rows per tile
constexpr int kBlockN = 128;   // keys per tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Lazy-rescale threshold in log2 units (see attn_fwd.cu): the reference max
// is raised only when a row's max grows by more than 2^8.
constexpr float kRescaleLog2 = 8.0f;
constexpr int kSmemBudget = 227 * 1024;

constexpr int kTileThreads = 128;          // softmax threads per query tile
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;    // tile A issuer (also allocates TMEM); tile B: kWarpMma + 1
constexpr int kThreads = 11 * 32;
constexpr int kOChunk = 32;                // O columns per TMEM load in rescale / store

// MERGE: K_j and V_j share one stage ring (see kMergeKV).
template <int D, bool MERGE>
struct PPCfg {
    static constexpr int kChunks = (D + 63) / 64;           // 128-byte swizzle atoms per row
    static constexpr int kChunkBytes = kBlockM * 128;
    static constexpr int kTileBytes = kChunks * kChunkBytes;
    static constexpr int kKStages = D == 64 ? 4 : 2;
    static constexpr int kVStages = kKStages;   // (merged K / V stages need equal counts)
    static constexpr int kOffQ = 0;                          // Q_A, Q_B
    static constexpr int kOffK = kOffQ + 2 * kTileBytes;
    static constexpr int kOffV = kOffK + kKStages * kTileBytes;
    static constexpr int kOffBar = kOffV + kVStages * kTileBytes;
    // barrier indices (per tile T: base + T)
    static constexpr int kBarQFull = 0;
    static constexpr int kBarQEmpty = 2;
    static constexpr int kBarSFull = 4;
    static constexpr int kBarPFull = 6;
    static constexpr int kBarOFinal = 8;
    static constexpr int kBarDrain = 10;     // per issuer: 2
    static constexpr int kBarSCons = 12;     // (separate P) S_T read into registers
    static constexpr int kBarPVDone = 14;    // (separate P) PV_T done with P_T
    static constexpr int kBarKFull = 16;
    static constexpr int kBarKEmpty = kBarKFull + kKStages;
    static constexpr int kBarVFull = kBarKEmpty + kKStages;
    static constexpr int kBarVEmpty = kBarVFull + kVStages;
    static constexpr int kNumBars = kBarVEmpty + kVStages;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;   // tmem slot, abort flag
    static constexpr int kUsed = kOffMisc + 16;
    static constexpr int kSmemBytes = kUsed + 1023 <= kSmemBudget ? kUsed + 1023 : kSmemBudget;
    static constexpr uint32_t kTmemCols = 512;
    // Separate P buffers (D = 64 only: S 2 x 128 + P 2 x 64 + O 2 x 64
    // columns); otherwise P is written over S.
    static constexpr bool kSepP = D == 64;
    static constexpr uint32_t kColP = kSepP ? 256 : 0;
    static constexpr uint32_t kPStride = kSepP ? 64 : 128;
    static constexpr uint32_t kColO = kSepP ? 384 : 256;
    static constexpr uint32_t kOStride = kSepP ? 64 : 128;
    static constexpr int kIssuers = kSepP ? 2 : 1;   // MMA-issuing threads
    // K_j and V_j of a stage load together, under one barrier (the K
    // stage's), and the stage is released after its PVs: one wait and one
    // release commit per key tile fewer for each issuer.  Always with
    // separate P; at D >= 80 only for long rows of keys (chosen at launch):
    // a merged stage goes back one key tile later, and with two stages
    // that shortens K's lead over its score MMA -- measured +3-5% for
    // causal D = 128 from N = 8192 up, -7% at B4 H32 N4096.
    static constexpr bool kMergeKV = kSepP || MERGE;
    static_assert(kUsed <= kSmemBudget, "shared memory budget");
};

struct PPParams {
    float *lse;
    __nv_bfloat16 *o;
    int *status;
    int N, Hq, Hkv, group, BH, n_qtiles, n_pairs;
    float scale_log2;   // scale * log2(e)
    int window;         // causal sliding window W (key j kept iff i - W < j), 0 = none
    int hchunk;         // causal item order: heads per chunk (BH: a single chunk)
    unsigned long long wait_limit_ns;
    int inject_skip_k0; // tests of the timeout path: block 0 never loads its first K tile
};

// Waits for in-flight async work on the abort path only, ignoring the abort
// flag, with a short limit of its own.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > 20ull * 1000ull * 1000ull) break;
    }
}

// O *= alpha on NC consecutive TMEM columns of this thread's row.
template <int NC>
__device__ __forceinline__ void o_rescale_cols(uint32_t tO, float alpha) {
    const uint64_t a2 = f2pack(alpha, alpha);
    uint32_t rr[NC];
    tmem_ld_cols<NC>(tO, rr);
#pragma unroll
    for (int e = 0; e < NC; e += 2) {
        float o0 = __uint_as_float(rr[e]), o1 = __uint_as_float(rr[e + 1]);
        f2unpack(fmul2(f2pack(o0, o1), a2), o0, o1);
        rr[e] = __float_as_uint(o0);
        rr[e + 1] = __float_as_uint(o1);
    }
    tmem_st_cols<NC>(tO, rr);
}

// O *= alpha on the D columns of this thread's row, kOChunk at a time.
template <int D, int C0 = 0>
__device__ __forceinline__ void o_rescale(uint32_t tO, float alpha) {
    if constexpr (C0 < D) {
        constexpr int NC = D - C0 < kOChunk ? D - C0 : kOChunk;
        o_rescale_cols<NC>(tO + C0, alpha);
        o_rescale<D, C0 + NC>(tO, alpha);
    }
}

__device__ __forceinline__ void st_global_v4(void *ptr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// This thread's row of O, TMEM columns [C0, D), times 1/l, as bf16 (round
// to nearest even) straight to the output row in global memory, 16 bytes at
// a time, kOChunk columns per TMEM load.  Every thread of the warp loads
// (tcgen05.ld is warp-wide); only rows inside the tensor (`store`) write.
template <int D, int C0 = 0>
__device__ __forceinline__ void o_store(uint32_t tO, float inv_l, __nv_bfloat16 *dst,
                                        bool store) {
    if constexpr (C0 < D) {
        constexpr int NC = D - C0 < kOChunk ? D - C0 : kOChunk;
        uint32_t rr[NC];
        tmem_ld_cols<NC>(tO + C0, rr);
        if (store) {
#pragma unroll
            for (int pc = 0; pc < NC / 8; ++pc) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w[e] = pack_bf16x2(__uint_as_float(rr[pc * 8 + 2 * e]) * inv_l,
                                       __uint_as_float(rr[pc * 8 + 2 * e + 1]) * inv_l);
                st_global_v4(dst + C0 + pc * 8, w[0], w[1], w[2], w[3]);
            }
        }
        o_store<D, C0 + NC>(tO, inv_l, dst, store);
    }
}

// One item: a pair of query tiles (A = 2p, B = 2p + 1 when it exists) of one
// (batch, query head), and the key tiles each of them needs.
struct PPItem {
    int bh, bh_kv;
    int qt_a, lo_a, hi_a;   // tile A: query tile, key tiles lo..hi (inclusive)
    int qt_b, lo_b, hi_b;   // tile B, when it exists
    bool b_on;              // tile B exists (N has a query tile 2p + 1)
    int lo_u, hi_u;         // key tiles of the item (union)
    __device__ int qt(int T) const { return T ? qt_b : qt_a; }
    __device__ int lo(int T) const { return T ? lo_b : lo_a; }
    __device__ int hi(int T) const { return T ? hi_b : hi_a; }
};

template <int D, bool CAUSAL, bool MERGE>
__global__ void __launch_bounds__(kThreads, 1)
fwd_pp_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const PPParams p) {
    using C = PPCfg<D, MERGE>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    if (smem - smem_raw + C::kUsed > C::kSmemBytes) {
        if (threadIdx.x == 0) atomicCAS(p.status, kStatusOk, kStatusDeviceCheck);
        return;
    }
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_ktiles = (p.N + kBlockN - 1) / kBlockN;
    const int n_items = p.n_pairs * p.BH;

    // Items in rounds of gridDim.x, every other round in reverse block order
    // (heaviest causal items first, so the blocks' totals stay balanced).
    auto item_at = [&](int rnd) -> int {
        const int G = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
        const int base = rnd * G;
        if (base >= n_items) return -1;
        const int k = base + ((rnd & 1) ? G - 1 - b : b);
        return k < n_items ? k : -1;
    };
    auto decode = [&](int k) -> PPItem {
        PPItem it;
        int pr;
        if (CAUSAL) {
            // Heaviest pairs first, heads fastest, within chunks of hchunk
            // heads (one chunk unless all heads' K/V is well over the L2).
            if (p.hchunk >= p.BH) {
                pr = p.n_pairs - 1 - k / p.BH;
                it.bh = k % p.BH;
            } else {
                const int per_chunk = p.hchunk * p.n_pairs;
                const int c = k / per_chunk;
                const int nh = min(p.hchunk, p.BH - c * p.hchunk);
                const int kk = k - c * per_chunk;
                pr = p.n_pairs - 1 - kk / nh;
                it.bh = c * p.hchunk + kk % nh;
            }
        } else {
            // Equal weights: pairs fastest, so the blocks running at once
            // share a few heads' K/V in L2.
            pr = k % p.n_pairs;
            it.bh = k / p.n_pairs;
        }
        it.bh_kv = (it.bh / p.Hq) * p.Hkv + (it.bh % p.Hq) / p.group;
        it.b_on = 2 * pr + 1 < p.n_qtiles;
        auto lo_of = [&](int qt) {
            return (CAUSAL && p.window > 0) ? max(0, qt * kBlockM - p.window + 1) / kBlockN : 0;
        };
        auto hi_of = [&](int qt) { return CAUSAL ? min(qt, n_ktiles - 1) : n_ktiles - 1; };
        it.qt_a = 2 * pr;
        it.lo_a = lo_of(it.qt_a);
        it.hi_a = hi_of(it.qt_a);
        it.qt_b = 2 * pr + 1;
        it.lo_b = lo_of(it.qt_b);
        it.hi_b = hi_of(it.qt_b);
        it.lo_u = it.lo_a;
        it.hi_u = it.b_on ? it.hi_b : it.hi_a;
        return it;
    };

    auto bar = [&](int i) -> uint32_t { return sb + C::kOffBar + 8u * i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
    const AbortCtl ac{abort_flag, p.status, p.wait_limit_ns};

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int T = 0; T < 2; ++T) {
            mbar_init(bar(C::kBarQFull + T), 1);
            mbar_init(bar(C::kBarQEmpty + T), 1);
            mbar_init(bar(C::kBarSFull + T), 1);
            mbar_init(bar(C::kBarPFull + T), kTileThreads);
            mbar_init(bar(C::kBarOFinal + T), 1);
            mbar_init(bar(C::kBarSCons + T), kTileThreads);
            mbar_init(bar(C::kBarPVDone + T), 1);
            mbar_init(bar(C::kBarDrain + T), 1);
        }
        // Stage releases: one commit from each issuer.
        for (int s = 0; s < C::kKStages; ++s) {
            mbar_init(bar(C::kBarKFull + s), 1);
            mbar_init(bar(C::kBarKEmpty + s), C::kIssuers);
        }
        for (int s = 0; s < C::kVStages; ++s) {
            mbar_init(bar(C::kBarVFull + s), 1);
            mbar_init(bar(C::kBarVEmpty + s), C::kIssuers);
        }
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == kWarpProducer && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kWarpProducer) {
        // ------------------------------------------------------ TMA producer
        // Per item: Q_A (and Q_B) once the previous item's last score MMA of
        // that tile is done, an L2 prefetch of the next item's Q tiles, then
        // K_j and V_j for every key tile of the item, in order.  The K and V
        // rings continue across items.
        if (lane == 0) {
            bool ok = true;
            int nq[2] = {0, 0};            // Q loads issued per tile
            int t = 0;                     // K / V tiles issued
            for (int rnd = 0; ok; ++rnd) {
                const int k = item_at(rnd);
                if (k < 0) break;
                const PPItem itm = decode(k);
                auto load_q = [&](int T, int qt) -> bool {
                    if (nq[T] > 0 && !mbar_wait(bar(C::kBarQEmpty + T), (nq[T] - 1) & 1, ac))
                        return false;
                    mbar_arrive_expect_tx(bar(C::kBarQFull + T), C::kTileBytes);
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(sb + C::kOffQ + T * C::kTileBytes + c * C::kChunkBytes, &tmQ,
                                    bar(C::kBarQFull + T), c * 64, qt * kBlockM, itm.bh);
                    ++nq[T];
                    return true;
                };
                ok = load_q(0, itm.qt_a) && (!itm.b_on || load_q(1, itm.qt_b));
                if (!ok) break;
                {   // the next item's Q tiles into L2 while this item runs
                    const int kn = item_at(rnd + 1);
                    if (kn >= 0) {
                        const PPItem nx = decode(kn);
                        for (int c = 0; c < C::kChunks; ++c) {
                            tma_prefetch_l2_3d(&tmQ, c * 64, nx.qt_a * kBlockM, nx.bh);
                            if (nx.b_on) tma_prefetch_l2_3d(&tmQ, c * 64, nx.qt_b * kBlockM, nx.bh);
                        }
                    }
                }
                for (int j = itm.lo_u; j <= itm.hi_u && ok; ++j, ++t) {
                    const int ks = t % C::kKStages;
                    if (t >= C::kKStages &&
                        !(ok = mbar_wait(bar(C::kBarKEmpty + ks), ((t / C::kKStages) - 1) & 1, ac)))
                        break;
                    // (Injected fault: block 0 never loads its first K tile;
                    // it still counts as issued, and the drain below waits
                    // for it with its own short limit.)
                    if (!(p.inject_skip_k0 && blockIdx.x == 0 && t == 0)) {
                        mbar_arrive_expect_tx(bar(C::kBarKFull + ks),
                                              C::kMergeKV ? 2 * C::kTileBytes : C::kTileBytes);
                        for (int c = 0; c < C::kChunks; ++c)
                            tma_load_3d(sb + C::kOffK + ks * C::kTileBytes + c * C::kChunkBytes,
                                        &tmK, bar(C::kBarKFull + ks), c * 64, j * kBlockN,
                                        itm.bh_kv);
                    }
                    const int vs = t % C::kVStages;
                    if (C::kMergeKV) {
                        // V_t on K_t's barrier (armed above for both tiles;
                        // the injected fault leaves out both).
                        if (!(p.inject_skip_k0 && blockIdx.x == 0 && t == 0))
                            for (int c = 0; c < C::kChunks; ++c)
                                tma_load_3d(sb + C::kOffV + vs * C::kTileBytes +
                                                c * C::kChunkBytes,
                                            &tmV, bar(C::kBarKFull + ks), c * 64, j * kBlockN,
                                            itm.bh_kv);
                        continue;
                    }
                    if (t >= C::kVStages &&
                        !(ok = mbar_wait(bar(C::kBarVEmpty + vs), ((t / C::kVStages) - 1) & 1, ac))) {
                        ++t;   // K_t was issued
                        break;
                    }
                    mbar_arrive_expect_tx(bar(C::kBarVFull + vs), C::kTileBytes);
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(sb + C::kOffV + vs * C::kTileBytes + c * C::kChunkBytes, &tmV,
                                    bar(C::kBarVFull + vs), c * 64, j * kBlockN, itm.bh_kv);
                }
            }
            if (!ok) {
                // Let every copy already issued land before the CTA exits.  K
                // tiles run up to t - 1; V tiles up to t - 1 too, except when
                // the V wait failed (then K_{t-1} has no V, and the V drain
                // below waits out its short limit on a phase never armed).
                for (int T = 0; T < 2; ++T)
                    if (nq[T] > 0) drain_wait(bar(C::kBarQFull + T), (nq[T] - 1) & 1);
                for (int u = max(t - C::kKStages, 0); u < t; ++u)
                    drain_wait(bar(C::kBarKFull + u % C::kKStages), (u / C::kKStages) & 1);
                if (!C::kMergeKV)
                    for (int u = max(t - C::kVStages, 0); u < t; ++u)
                        drain_wait(bar(C::kBarVFull + u % C::kVStages), (u / C::kVStages) & 1);
            }
        }
        __syncwarp();
    } else if (warp == kWarpMma || warp == kWarpMma + 1) {
        // ------------------------------------------------------ MMA issuers
        if (lane == 0 && warp - kWarpMma < C::kIssuers) {
            // The tile this thread issues for (with one issuer: both, T = 0
            // being the first of the pair).
            const int T = warp - kWarpMma;
            constexpr uint32_t kIdS = idesc_bf16_f32(kBlockM, kBlockN, false, false);
            constexpr uint32_t kIdPV = idesc_bf16_f32(kBlockM, D, false, true);
            const uint64_t dq = sdesc_sw128(sb + C::kOffQ + T * C::kTileBytes, 16, 1024);
            const uint64_t dk0 = sdesc_sw128(sb + C::kOffK, 16, 1024);
            const uint64_t dv0 = sdesc_sw128(sb + C::kOffV, C::kChunkBytes, 1024);
            const uint32_t s_tmem = tmem + T * kBlockN;
            const uint32_t p_tmem = tmem + C::kColP + T * C::kPStride;   // P: bf16 pairs
            const uint32_t o_tmem = tmem + C::kColO + T * C::kOStride;
            // Tile U's score MMA from K stage ks, and its PV MMA from V stage vs
            // (U = T except on the single-issuer path, which issues for both).
            auto issue_s_u = [&](int U, int ks) {
                const uint64_t dk = dk0 + ((ks * C::kTileBytes) >> 4);
                const uint64_t dqu = dq + ((U - T) * (C::kTileBytes >> 4));
                const uint32_t d_tmem = s_tmem + (U - T) * kBlockN;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
                    mma_ss(d_tmem, dqu + off, dk + off, kIdS, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(C::kBarSFull + U));
            };
            auto issue_pv_u = [&](int U, int vs, bool first) {
                const uint64_t dv = dv0 + ((vs * C::kTileBytes) >> 4);
                const uint32_t a_tmem = p_tmem + (U - T) * C::kPStride;
                const uint32_t d_tmem = o_tmem + (U - T) * C::kOStride;
                mma_ts(d_tmem, a_tmem, dv, kIdPV, first ? 0u : 1u);
#pragma unroll
                for (int kk = 1; kk < kBlockN / 16; ++kk)
                    mma_ts(d_tmem, a_tmem + kk * 8, dv + ((kk * 2048) >> 4), kIdPV, 1u);
            };
            auto issue_s = [&](int ks) { issue_s_u(T, ks); };
            auto issue_pv = [&](int vs, bool first) { issue_pv_u(T, vs, first); };
            // Steps: the key tiles of this block's items, in order; t counts
            // them (the K / V ring position).
            struct Step {
                bool valid;
                int rnd, j;
                PPItem itm;
            };
            auto step_at = [&](int rnd) -> Step {
                Step st{false, rnd, 0, PPItem{}};
                const int k = item_at(rnd);
                if (k >= 0) {
                    st.valid = true;
                    st.itm = decode(k);
                    st.j = st.itm.lo_u;
                }
                return st;
            };
            auto next_step = [&](const Step &st) -> Step {
                if (st.j < st.itm.hi_u) {
                    Step n = st;
                    ++n.j;
                    return n;
                }
                return step_at(st.rnd + 1);
            };
            // Tile T takes part in step st (tile B may not exist).
            auto in_tile = [&](const Step &st) -> bool {
                return T == 0 ? st.j <= st.itm.hi_a : (st.itm.b_on && st.j >= st.itm.lo_b);
            };
            int nq = 0;   // Q tiles waited for
            int sc = 0;   // S MMAs issued
            int pc = 0;   // PV MMAs issued
            // The S MMA of step st (K tile t): Q first when the step opens an
            // item, then the K stage; the stage's release is committed
            // whether or not this tile took part.
            auto issue_s_step = [&](const Step &st, int t) -> bool {
                const bool in = in_tile(st);
                if (st.j == st.itm.lo_u && (T == 0 || st.itm.b_on)) {
                    if (!mbar_wait(bar(C::kBarQFull + T), nq & 1, ac)) return false;
                    ++nq;
                }
                const int ks = t % C::kKStages;
                if (!mbar_wait(bar(C::kBarKFull + ks), (t / C::kKStages) & 1, ac)) return false;
                if (in) {
                    // With separate P, S_T's previous value must be in the
                    // softmax's registers; otherwise the previous PV_T (issued
                    // before by this thread) is the last reader of the buffer.
                    if (C::kSepP && sc > 0 &&
                        !mbar_wait(bar(C::kBarSCons + T), (sc - 1) & 1, ac))
                        return false;
                    tc_fence_after();
                    issue_s(ks);
                    if (st.j == st.itm.hi(T)) mma_commit(bar(C::kBarQEmpty + T));
                    ++sc;
                }
                if (!C::kMergeKV) mma_commit(bar(C::kBarKEmpty + ks));
                return true;
            };
            auto issue_pv_step = [&](const Step &st, int t) -> bool {
                const bool in = in_tile(st);
                const int vs = t % C::kVStages;
                if (!C::kMergeKV &&
                    !mbar_wait(bar(C::kBarVFull + vs), (t / C::kVStages) & 1, ac))
                    return false;
                if (in) {
                    if (!mbar_wait(bar(C::kBarPFull + T), pc & 1, ac)) return false;
                    tc_fence_after();
                    issue_pv(vs, st.j == st.itm.lo(T));
                    if (C::kSepP) mma_commit(bar(C::kBarPVDone + T));
                    if (st.j == st.itm.hi(T)) mma_commit(bar(C::kBarOFinal + T));
                    ++pc;
                }
                // (Merged stages: K_t and V_t go back together, after the PV;
                // this issuer waited for the stage in its S step.)
                mma_commit(bar(C::kMergeKV ? C::kBarKEmpty + vs : C::kBarVEmpty + vs));
                return true;
            };
            bool ok = true;
            Step cur = step_at(0);
            int t = 0;   // K / V tile of `cur`
            if constexpr (C::kSepP) {
                // S of the next key tile (of this item or the next) before
                // the PV of this one.
                if (cur.valid) ok = issue_s_step(cur, 0);
                while (ok && cur.valid) {
                    const Step nxt = next_step(cur);
                    if (nxt.valid && !(ok = issue_s_step(nxt, t + 1))) break;
                    if (!(ok = issue_pv_step(cur, t))) break;
                    cur = nxt;
                    ++t;
                }
            } else {
                // P is written over S, one issuer for both tiles, in the
                // order S_A(j), PV_B(j-1), S_B(j), PV_A(j): S_T(j+1) follows
                // PV_T(j), and while one tile's softmax runs the tensor core
                // works on the other tile's MMA groups.
                int nqb = 0, scb = 0, pcb = 0;   // tile B's counters
                struct Pend {
                    bool on;
                    int vs;
                    bool first, last;
                } pend{false, 0, false, false};   // tile B's PV of the previous key tile
                auto flush_b = [&]() -> bool {
                    if (!pend.on) return true;
                    if (!mbar_wait(bar(C::kBarPFull + 1), pcb & 1, ac)) return false;
                    tc_fence_after();
                    issue_pv_u(1, pend.vs, pend.first);
                    mma_commit(bar(C::kMergeKV ? C::kBarKEmpty + pend.vs : C::kBarVEmpty + pend.vs));
                    if (pend.last) mma_commit(bar(C::kBarOFinal + 1));
                    ++pcb;
                    pend.on = false;
                    return true;
                };
                while (ok && cur.valid) {
                    const PPItem &itm = cur.itm;
                    const bool a_in = cur.j <= itm.hi_a;
                    const bool b_in = itm.b_on && cur.j >= itm.lo_b;
                    const int ks = t % C::kKStages, vs = t % C::kVStages;
                    if (cur.j == itm.lo_u) {
                        if (!(ok = mbar_wait(bar(C::kBarQFull), nq & 1, ac))) break;
                        ++nq;
                        if (itm.b_on) {
                            if (!(ok = mbar_wait(bar(C::kBarQFull + 1), nqb & 1, ac))) break;
                            ++nqb;
                        }
                    }
                    if (!(ok = mbar_wait(bar(C::kBarKFull + ks), (t / C::kKStages) & 1, ac))) break;
                    tc_fence_after();
                    if (a_in) {
                        issue_s_u(0, ks);
                        if (cur.j == itm.hi_a) mma_commit(bar(C::kBarQEmpty));
                        ++sc;
                    }
                    if (!(ok = flush_b())) break;
                    if (b_in) {
                        issue_s_u(1, ks);
                        if (cur.j == itm.hi_b) mma_commit(bar(C::kBarQEmpty + 1));
                        ++scb;
                    }
                    if (!C::kMergeKV) {
                        mma_commit(bar(C::kBarKEmpty + ks));
                        if (!(ok = mbar_wait(bar(C::kBarVFull + vs), (t / C::kVStages) & 1, ac)))
                            break;
                    }
                    if (a_in) {
                        if (!(ok = mbar_wait(bar(C::kBarPFull), pc & 1, ac))) break;
                        tc_fence_after();
                        issue_pv_u(0, vs, cur.j == itm.lo_a);
                        if (cur.j == itm.hi_a) mma_commit(bar(C::kBarOFinal));
                        ++pc;
                    }
                    if (b_in) pend = Pend{true, vs, cur.j == itm.lo_b, cur.j == itm.hi_b};
                    else mma_commit(bar(C::kMergeKV ? C::kBarKEmpty + vs : C::kBarVEmpty + vs));
                    cur = next_step(cur);
                    ++t;
                }
                if (ok) ok = flush_b();
            }
            if (!ok) {
                mma_commit(bar(C::kBarDrain + T));
                drain_wait(bar(C::kBarDrain + T), 0);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------- softmax warpgroups
        // Tile T = warp / 4; thread r of the warpgroup owns query row r
        // (TMEM lane r) and all 128 keys of each key tile.  The warps of a
        // tile never wait for one another: each leaves on its own when a
        // wait fails.
        const int T = warp >> 2;
        const int r = ((warp & 3) << 5) | lane;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_base + T * kBlockN;
        const uint32_t tP = tmem + lane_base + C::kColP + T * C::kPStride;
        const uint32_t tO = tmem + lane_base + C::kColO + T * C::kOStride;
        bool ok = true;
        int t = 0;     // S/P iterations of this tile
        int nit = 0;   // items of this tile
        for (int rnd = 0; ok; ++rnd) {
            const int kitem = item_at(rnd);
            if (kitem < 0) break;
            const PPItem itm = decode(kitem);
            if (T == 1 && !itm.b_on) continue;
            const int qt = itm.qt(T), lo = itm.lo(T), hi = itm.hi(T);
            const int row_lo = qt * kBlockM;
            const int q_row = row_lo + r;
            const bool row_valid = q_row < p.N;
            float m_run = -INFINITY;   // running reference max, log2 units
            float l_run = 0.f;         // row sum
            for (int j = lo; j <= hi; ++j, ++t) {
                if (!(ok = mbar_wait_warp(bar(C::kBarSFull + T), t & 1, ac))) break;
                tc_fence_after();
                const int key0 = j * kBlockN;
                // x holds raw q.k; xmul (the scale in log2 units, when
                // positive) turns it into log2-unit logits and folds into
                // the exp2 FMA.
                float xmul = p.scale_log2;
                float x[kBlockN];
                {
                    uint32_t rr[kBlockN];
                    tmem_ld128(tS, rr);
#pragma unroll
                    for (int c = 0; c < kBlockN; ++c) x[c] = __uint_as_float(rr[c]);
                }
                if constexpr (C::kSepP) {
                    // S_T(j) is in registers: the issuer may compute S_T(j+1).
                    tc_fence_before();
                    mbar_arrive(bar(C::kBarSCons + T));
                }
                if (!(p.scale_log2 > 0.f)) {
#pragma unroll
                    for (int c = 0; c < kBlockN; ++c) x[c] *= p.scale_log2;
                    xmul = 1.f;
                }
                const bool diag = CAUSAL && (j == qt);
                const bool ragged = key0 + kBlockN > p.N;
                const bool wedge = CAUSAL && p.window > 0 && key0 < row_lo + kBlockM - p.window;
                if (diag && !ragged && !wedge) {
                    // The diagonal tile alone: key c kept iff c <= r (one
                    // compare per key; the general form below is several
                    // times slower and sits on every item's last tile).
#pragma unroll
                    for (int c = 0; c < kBlockN; ++c) x[c] = c <= r ? x[c] : -INFINITY;
                } else if (diag || ragged || wedge) {
                    const int klo = wedge ? q_row - p.window + 1 - key0 : -(1 << 30);
                    const int khi = diag ? r : (1 << 30);          // last kept key (causal)
                    const int kend = p.N - key0;                    // keys past N
#pragma unroll
                    for (int c = 0; c < kBlockN; ++c)
                        x[c] = (c <= khi && c < kend && c >= klo) ? x[c] : -INFINITY;
                }
                // Row max as a tree (8 independent chains of 3-input max).
                float mx[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mx[i] = x[i];
#pragma unroll
                for (int c = 8; c + 16 <= kBlockN; c += 16) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], x[c + i], x[c + 8 + i]);
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) mx[i] = fmaxf(mx[i], x[kBlockN - 8 + i]);
                const float m_tile =
                    fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                          fmaxf(mx[6], mx[7])) * xmul;
                // Lazy rescale: keep the previous reference max while the new
                // row max exceeds it by at most kRescaleLog2.
                float m_new = fmaxf(m_run, m_tile);
                if (m_new - m_run <= kRescaleLog2) m_new = m_run;
                const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                const float alpha = ex2(m_run - m_use);   // 0 on the item's first tile

                const uint64_t cm2 = f2pack(xmul, xmul);
                const uint64_t nm2 = f2pack(-m_use, -m_use);
                uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
                // P as packed bf16 pairs: keys 2c, 2c+1 of the tile in column c.
                uint32_t pk[kBlockN / 2];
#pragma unroll
                for (int c = 0; c < kBlockN / 2; ++c) {
                    float t0, t1;
                    f2unpack(ffma2(f2pack(x[2 * c], x[2 * c + 1]), cm2, nm2), t0, t1);
                    const float p0 = ex2(t0), p1 = ex2(t1);
                    acc[c & 3] = fadd2(acc[c & 3], f2pack(p0, p1));
                    pk[c] = pack_bf16x2(p0, p1);
                }
                if (C::kSepP && t > 0) {
                    // PV_T(j-1) must be done with the P buffer (and with O,
                    // which may be rescaled below).
                    if (!(ok = mbar_wait_warp(bar(C::kBarPVDone + T), (t - 1) & 1, ac))) break;
                    tc_fence_after();
                }
                tmem_st64(tP, pk);
                float sum;
                {
                    const uint64_t a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
                    float u0, u1;
                    f2unpack(fadd2(a01, a23), u0, u1);
                    sum = u0 + u1;
                }
                l_run = fmaf(l_run, alpha, sum);
                // O holds PV_T of the earlier key tiles, all complete (the
                // S_T(j) commit covered them; with separate P, the PV wait
                // above did).
                if (__any_sync(0xffffffffu, j > lo && alpha < 1.f)) o_rescale<D>(tO, alpha);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(C::kBarPFull + T));
                m_run = m_new;
            }
            if (!ok) break;

            // --------------------------------------------------- epilogue
            if (!(ok = mbar_wait_warp(bar(C::kBarOFinal + T), nit & 1, ac))) break;
            ++nit;
            tc_fence_after();
            const float inv_l = 1.f / l_run;
            __nv_bfloat16 *orow =
                p.o + (static_cast<size_t>(itm.bh) * p.N + (row_valid ? q_row : 0)) * D;
            o_store<D>(tO, inv_l, orow, row_valid);
            if (p.lse && row_valid)
                p.lse[static_cast<size_t>(itm.bh) * p.N + q_row] = (m_run + log2f(l_run)) * kLn2;
            tc_fence_before();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, bool CAUSAL, bool MERGE>
cudaError_t launch_t(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                     const PPParams &prm, unsigned grid, cudaStream_t stream) {
    using C = PPCfg<D, MERGE>;
    auto kern = fwd_pp_kernel<D, CAUSAL, MERGE>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, C::kSmemBytes, stream>>>(q, k, v, prm);
    return cudaGetLastError();
}

// Merged K / V stages from 64 key tiles per row up (always at D = 64).
constexpr int kMergeMinKeyTiles = 64;

template <int D>
cudaError_t launch_d(bool causal, const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                     const PPParams &prm, unsigned grid, cudaStream_t stream) {
    if constexpr (D != 64) {
        if ((prm.N + kBlockN - 1) / kBlockN < kMergeMinKeyTiles)
            return causal ? launch_t<D, true, false>(q, k, v, prm, grid, stream)
                          : launch_t<D, false, false>(q, k, v, prm, grid, stream);
    }
    return causal ? launch_t<D, true, true>(q, k, v, prm, grid, stream)
                  : launch_t<D, false, true>(q, k, v, prm, grid, stream);
}

}  // namespace

cudaError_t launch_fwd_pp(const FwdProblem &pb, int *status, cudaStream_t stream) {
    const long long BH = static_cast<long long>(pb.B) * pb.Hq;
    const long long BHkv = static_cast<long long>(pb.B) * pb.Hkv;
    CUtensorMap mq, mk, mv;
    if (!encode_bf16_rows(&mq, pb.q, pb.D, pb.N, BH, kBlockM) ||
        !encode_bf16_rows(&mk, pb.k, pb.D, pb.N, BHkv, kBlockN) ||
        !encode_bf16_rows(&mv, pb.v, pb.D, pb.N, BHkv, kBlockN))
        return cudaErrorInvalidValue;
    DeviceInfo di;
    if (!device_info(&di)) return cudaErrorInvalidValue;
    PPParams prm;
    prm.lse = pb.lse;
    prm.o = static_cast<__nv_bfloat16 *>(pb.o);
    prm.status = status;
    prm.N = pb.N;
    prm.Hq = pb.Hq;
    prm.Hkv = pb.Hkv;
    prm.group = pb.Hq / pb.Hkv;
    prm.BH = static_cast<int>(BH);
    prm.n_qtiles = (pb.N + kBlockM - 1) / kBlockM;
    prm.n_pairs = (prm.n_qtiles + 1) / 2;
    prm.scale_log2 = pb.scale * kLog2e;
    prm.window = pb.causal ? pb.window : 0;
    prm.wait_limit_ns = pb.wait_limit_ns ? pb.wait_limit_ns : kWaitLimitNs;
    prm.inject_skip_k0 = pb.inject_skip_k0;
    // Causal item order: one chunk of all heads unless their K/V is over
    // twice the L2; then chunks whose K/V is about half the L2 (as in the
    // one-tile forward).
    prm.hchunk = static_cast<int>(BH);
    {
        const double l2 = di.l2_bytes;
        const double head_kv = static_cast<double>(pb.N) * pb.D * 4.0 / (pb.Hq / pb.Hkv);
        if (pb.causal && head_kv * static_cast<double>(BH) > 2.0 * l2)
            prm.hchunk = static_cast<int>(std::max<long long>(
                1, std::min<long long>(BH, static_cast<long long>(0.5 * l2 / head_kv))));
    }
    const long long n_items = static_cast<long long>(prm.n_pairs) * BH;
    const unsigned grid = static_cast<unsigned>(n_items < di.sms ? n_items : di.sms);
    switch (pb.D) {
    case 64: return launch_d<64>(pb.causal, mq, mk, mv, prm, grid, stream);
    case 80: return launch_d<80>(pb.causal, mq, mk, mv, prm, grid, stream);
    case 96: return launch_d<96>(pb.causal, mq, mk, mv, prm, grid, stream);
    default: return launch_d<128>(pb.causal, mq, mk, mv, prm, grid, stream);
    }
}

}  // namespace tattn
