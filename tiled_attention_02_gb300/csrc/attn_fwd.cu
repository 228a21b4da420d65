// attn_fwd.cu -- tiled exact-attention forward with a logit bias and / or
// emitted logits (the block attention residual), for GB300 (sm_103a).  The
// plain forward, without either, is attn_fwd_pp.cu.
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
// Warp roles (one CTA per SM):
//   warps 0-7  two softmax warpgroups.  Thread r of warpgroup w owns query row
//              r (TMEM lane r) for keys [64 w, 64 w + 64) of every key tile;
//              the two swap partial row maxima through shared memory once per
//              tile, so both scale by the same reference max.  Each rescales
//              and stores its half of O's columns.
//   warp 8     TMA producer: Q once, then K_j / V_j through 1-3 stage rings.
//   warp 9     TMEM allocator and single-thread tcgen05.mma issuer.
//   warps 10-11  (staged residual only) fp32 bias loader and emitted-logit
//              storer, see below.
// TMEM (512 columns): S/P double buffer at columns 0 and 128, O at 256.
// Issue order on the tensor core: S_0, S_1, PV_0, S_2, PV_1, ... so that the
// softmax of tile j overlaps the MMAs of tiles j+1 and j-1.  Splitting a
// tile's keys over two warpgroups halves the per-tile softmax latency (TMEM
// load, 64 exp2 per thread instead of 128, P store), which is the critical
// path of every tile.
//
// The residual variants (bias and/or emitted logits) move 2 x 64 KB of fp32
// per 128 x 128 tile, several times the tile's MMA time at HBM bandwidth, so
// their data path is what bounds them.  Two variants (template EXT):
//   2  staged: the bias tile is cut into four 128 x 32 fp32 chunks (one
//      128-byte swizzle atom wide) that warp 10 TMA-loads into a ring of
//      shared-memory slots; each softmax thread reads its row of a chunk,
//      writes the emitted logit back over the bias in place, and warp 11
//      TMA-stores the chunk to the emit tensor before the slot is refilled.
//      Needs 16-byte rows (N % 4 == 0) and 16-byte aligned bases;
//   1  direct: per-thread global loads and stores of the row, for shapes
//      the staged variant cannot map.
#include "attn_internal.h"
#include "sm103_ptx.cuh"

#include <algorithm>

namespace tattn {
namespace {

constexpr int kBlockM = 128;   // query rows per CTA
constexpr int kBlockN = 128;   // keys per tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Lazy-rescale threshold in log2 units: the reference max is only raised when
// a row's max grows by more than this (factor 2^8).
constexpr float kRescaleLog2 = 8.0f;
constexpr int kSmemBudget = 227 * 1024;
constexpr int kResChunkCols = 32;                          // fp32 keys per chunk
constexpr int kResChunks = kBlockN / kResChunkCols;        // chunks per key tile
constexpr int kResChunkBytes = kBlockM * kResChunkCols * 4;

// Warp roles.  Warps 0-7 are two softmax warpgroups.
constexpr int kSoftWarps = 8;
constexpr int kSoftThreads = kSoftWarps * 32;
constexpr int kHalfN = kBlockN / 2;   // keys of a tile handled by one softmax warpgroup
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;
constexpr int kWarpLoader = 10;       // staged residual only
constexpr int kWarpStorer = 11;       // staged residual only

// (The plain forward, without bias or emitted logits, is attn_fwd_pp.cu.)
template <int EXT>
constexpr int fwd_threads() {
    static_assert(EXT == 1 || EXT == 2, "residual variants only");
    return EXT == 2 ? 384 : 320;
}

template <int D, int EXT>
struct FwdCfg {
    // A bf16 row of D elements occupies ceil(D/64) 128-byte swizzle atoms;
    // for D = 80 or 96 the second atom is zero-filled past D by TMA, the MMAs
    // use D/16 K-steps (QK^T) or N = D (PV), and stores are clipped at D.
    static constexpr int kChunks = (D + 63) / 64;         // 128-byte swizzle atoms per row
    static constexpr int kChunkBytes = kBlockM * 128;     // one atom column of a tile
    static constexpr int kTileBytes = kChunks * kChunkBytes;   // bf16 128 x D tile, padded
    // O columns [0, kOSplit) belong to softmax warpgroup 0, the rest to
    // warpgroup 1 (each TMEM access stays aligned to its own width).
    static constexpr int kOSplit = D > 64 ? 64 : D / 2;
    // The staged residual variant is bound by its fp32 stream: it gives part
    // of the K/V rings' shared memory to the residual slots (V_j is only
    // needed a whole softmax after its load is issued, so one V stage holds).
    static constexpr int kKStages = (D == 64) ? (EXT == 2 ? 2 : 3) : (EXT == 2 ? 1 : 2);
    static constexpr int kVStages = kKStages;
    static constexpr int kQBufs = 1;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQBufs * kTileBytes;
    static constexpr int kOffV = kOffK + kKStages * kTileBytes;
    static constexpr int kOffRes = kOffV + kVStages * kTileBytes;
    static constexpr int kRedBytes = 2 * 2 * kBlockM * 4;   // row-max exchange, 2 buffers
    static constexpr int kResSlots =
        EXT == 2 ? (kSmemBudget - 512 - 16 - kRedBytes - kOffRes) / kResChunkBytes : 0;
    static constexpr int kResRing = kResSlots > 0 ? kResSlots : 1;
    static constexpr int kOffBar = kOffRes + kResSlots * kResChunkBytes;
    // barrier indices
    static constexpr int kBarQFull = 0;                       // the Q tile
    static constexpr int kBarKFull = 1;
    static constexpr int kBarKEmpty = kBarKFull + kKStages;
    static constexpr int kBarVFull = kBarKEmpty + kKStages;
    static constexpr int kBarVEmpty = kBarVFull + kVStages;
    static constexpr int kBarSFull = kBarVEmpty + kVStages;   // 2
    static constexpr int kBarPFull = kBarSFull + 2;           // 2
    static constexpr int kBarODone = kBarPFull + 2;
    static constexpr int kBarOFinal = kBarODone + 1;
    static constexpr int kBarDrain = kBarOFinal + 1;
    static constexpr int kBarResFull = kBarDrain + 1;           // slot loaded (or granted)
    static constexpr int kBarResDone = kBarResFull + kResSlots;  // softmax finished the slot
    static constexpr int kBarResFree = kBarResDone + kResSlots;  // slot's store has read it
    static constexpr int kNumBars = kBarResFree + kResSlots;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;   // tmem slot, abort flag
    static constexpr int kOffRed = kOffMisc + 16;
    static constexpr int kUsed = kOffRed + kRedBytes;
    // Up to 1023 bytes of slack for aligning the base, as far as the budget allows.
    static constexpr int kSmemBytes = kUsed + 1023 <= kSmemBudget ? kUsed + 1023 : kSmemBudget;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColO = 256;
    static_assert(kUsed <= kSmemBudget, "shared memory budget");
    static_assert(EXT != 2 || kResSlots >= kResChunks, "residual ring holds a key tile");
};

struct FwdParams {
    const float *bias;
    float *emit;
    float *lse;
    int *status;
    int N, Hq, Hkv, group, BH, n_qtiles;
    float scale;        // scale of QK^T
    float scale_log2;   // scale * log2(e)
    int window;         // causal sliding window W (key j kept iff i - W < j), 0 = none
    int hchunk;         // causal item order: heads per chunk (BH: a single chunk)
    unsigned long long wait_limit_ns;   // bound of every pipeline wait
};

// O *= alpha on NC consecutive TMEM columns of this thread's row.
template <int NC>
__device__ __forceinline__ void o_rescale(uint32_t tO, float alpha) {
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

// Row r's O columns [C0, C0 + NC), times 1/l, as bf16 into the 128-byte
// swizzled output tile at `tile` (atoms of 64 columns, 128 rows each).
template <int NC, int C0>
__device__ __forceinline__ void o_stage(uint32_t tO, float inv_l, uint32_t tile, int r) {
    uint32_t rr[NC];
    tmem_ld_cols<NC>(tO, rr);
#pragma unroll
    for (int pc = 0; pc < NC / 8; ++pc) {   // 16-byte pieces
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            w[e] = pack_bf16x2(__uint_as_float(rr[pc * 8 + 2 * e]) * inv_l,
                               __uint_as_float(rr[pc * 8 + 2 * e + 1]) * inv_l);
        const int colg = C0 + pc * 8;   // first O column of the piece
        const uint32_t addr = tile + (colg / 64) * (kBlockM * 128) + r * 128 +
                              (static_cast<uint32_t>(((colg % 64) / 8) ^ (r & 7)) << 4);
        st_shared_v4(addr, w[0], w[1], w[2], w[3]);
    }
}

// Waits for the arrival of in-flight async work on the abort path only,
// ignoring the abort flag, with a short limit of its own.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > 20ull * 1000ull * 1000ull) break;
    }
}

template <int D, bool CAUSAL, int EXT>
__global__ void __launch_bounds__(fwd_threads<EXT>(), 1)
fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
           const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
           const __grid_constant__ CUtensorMap tmBias, const __grid_constant__ CUtensorMap tmEmit,
           const FwdParams p) {
    using C = FwdCfg<D, EXT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    // The layout needs a 1024-byte aligned base; refuse to run if the
    // allocation cannot hold it after alignment.
    if (smem - smem_raw + C::kUsed > C::kSmemBytes) {
        if (threadIdx.x == 0) atomicCAS(p.status, kStatusOk, kStatusDeviceCheck);
        return;
    }
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int n_ktiles = (p.N + kBlockN - 1) / kBlockN;
    const int n_items = p.n_qtiles * p.BH;
    // This block's items (query tile, head): rounds of gridDim.x items, every
    // other round in reverse block order, so that with the heaviest causal
    // tiles first the blocks' totals stay balanced.  Round 0 only, unless the
    // kernel is persistent (grid smaller than the item count).
    auto item_at = [&](int rnd) -> int {
        const int G = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
        const int base = rnd * G;
        if (base >= n_items) return -1;
        const int k = base + ((rnd & 1) ? G - 1 - b : b);
        return k < n_items ? k : -1;
    };
    struct Item {
        int qt, bh, bh_kv, row_lo, kv_lo, n_kv;
    };
    auto decode = [&](int k) -> Item {
        Item it;
        // Causal: heaviest tiles first (item 0 is the last query tile of
        // head 0), heads fastest, within chunks of hchunk heads taken one
        // after another (one chunk unless all heads' K/V is well over L2, so
        // that the items running at once share a few heads' K/V).  Otherwise
        // every item weighs the same, and query tiles go fastest so that the
        // blocks running at once share a few heads' K/V in L2 instead of each
        // streaming its own from HBM.
        if (CAUSAL) {
            if (p.hchunk >= p.BH) {
                it.qt = p.n_qtiles - 1 - k / p.BH;
                it.bh = k % p.BH;
            } else {
                const int per_chunk = p.hchunk * p.n_qtiles;
                const int c = k / per_chunk;
                const int nh = min(p.hchunk, p.BH - c * p.hchunk);   // heads of this chunk
                const int kk = k - c * per_chunk;
                it.qt = p.n_qtiles - 1 - kk / nh;
                it.bh = c * p.hchunk + kk % nh;
            }
        } else {
            it.qt = k % p.n_qtiles;
            it.bh = k / p.n_qtiles;
        }
        it.bh_kv = (it.bh / p.Hq) * p.Hkv + (it.bh % p.Hq) / p.group;
        // Key tiles kv_lo .. kv_lo + n_kv - 1: the causal mask ends them at
        // the diagonal tile, a sliding window starts them at the tile holding
        // key row_lo - W + 1 (the first key the tile's first row keeps).
        it.row_lo = it.qt * kBlockM;
        it.kv_lo = (CAUSAL && p.window > 0) ? max(0, it.row_lo - p.window + 1) / kBlockN : 0;
        it.n_kv = (CAUSAL ? min(it.qt + 1, n_ktiles) : n_ktiles) - it.kv_lo;
        return it;
    };
    // The item of a one-item block (the residual variants' chunk roles).
    const Item one = decode(max(item_at(0), 0));
    const int qt = one.qt, bh = one.bh, kv_lo = one.kv_lo, n_kv = one.n_kv;

    auto bar = [&](int i) -> uint32_t { return sb + C::kOffBar + 8u * i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
    const AbortCtl ac{abort_flag, p.status, p.wait_limit_ns};

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
            // the softmax threads' P, plus the producer's V_j (bytes)
            mbar_init(bar(C::kBarPFull + s), kSoftThreads + 1);
        }
        mbar_init(bar(C::kBarODone), 1);
        mbar_init(bar(C::kBarOFinal), 1);
        mbar_init(bar(C::kBarDrain), 1);
        for (int s = 0; s < C::kResSlots; ++s) {
            mbar_init(bar(C::kBarResFull + s), 1);
            mbar_init(bar(C::kBarResDone + s), kBlockM);
            mbar_init(bar(C::kBarResFree + s), 1);
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
        tma_prefetch_desc(&tmO);
        if constexpr (EXT == 2) {
            if (p.bias) tma_prefetch_desc(&tmBias);
            if (p.emit) tma_prefetch_desc(&tmEmit);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kWarpProducer) {
        // ------------------------------------------------------ TMA producer
        // Per item its Q tile (into Q buffer n_q % kQBufs, issued when the K
        // cursor enters the item), then K and V per key tile.  K runs one tile
        // ahead of V: K_{t+1} only waits for S_{t+1-KStages} to finish with its
        // stage, while V_t waits for PV_{t-VStages}, which needs the softmax of
        // that tile; issuing K first keeps the next S MMA from queueing behind
        // a V wait.  The tile counters run on across items, so the rings and
        // their barriers continue from one item to the next.
        if (lane == 0) {
            bool ok = true;
            int n_q = 0, k_issued = 0, v_issued = 0;
            int kr = 0, kj = 0, vr = 0, vj = 0;   // K / V cursors: round, tile of the item
            Item ki = decode(item_at(0)), vi = ki;
            bool k_done = false, v_done = false;
            auto advance = [&](int &rr, int &jj, Item &itm, bool &done) {
                if (++jj == itm.n_kv) {
                    jj = 0;
                    const int k = item_at(++rr);
                    if (k < 0) done = true;
                    else itm = decode(k);
                }
            };
            // (One item per block: its Q tile loads once, into the one buffer.)
            auto load_q = [&](const Item &itm) -> bool {
                const int qb = n_q % C::kQBufs;
                mbar_arrive_expect_tx(bar(C::kBarQFull + qb), C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(sb + C::kOffQ + qb * C::kTileBytes + c * C::kChunkBytes, &tmQ,
                                bar(C::kBarQFull + qb), c * 64, itm.row_lo, itm.bh);
                ++n_q;
                return true;
            };
            auto load_k = [&]() -> bool {
                if (kj == 0 && !load_q(ki)) return false;
                const int t = k_issued, ks = t % C::kKStages;
                if (t >= C::kKStages &&
                    !mbar_wait(bar(C::kBarKEmpty + ks), ((t / C::kKStages) - 1) & 1, ac))
                    return false;
                mbar_arrive_expect_tx(bar(C::kBarKFull + ks), C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(sb + C::kOffK + ks * C::kTileBytes + c * C::kChunkBytes, &tmK,
                                bar(C::kBarKFull + ks), c * 64, (ki.kv_lo + kj) * kBlockN,
                                ki.bh_kv);
                k_issued = t + 1;
                advance(kr, kj, ki, k_done);
                return true;
            };
            auto load_v = [&]() -> bool {
                const int t = v_issued, vs = t % C::kVStages;
                if (t >= C::kVStages &&
                    !mbar_wait(bar(C::kBarVEmpty + vs), ((t / C::kVStages) - 1) & 1, ac))
                    return false;
                // V_t completes on P_t's barrier: the MMA issuer waits once for
                // both.  The barrier's previous phase (tile t-2) must be over
                // before it is armed for tile t: wait for PV_{t-2} (implied by
                // the stage wait above when the V ring has at most 2 stages).
                if (C::kVStages > 2 && t >= 2) {
                    const int tp = t - 2;
                    if (!mbar_wait(bar(C::kBarVEmpty + tp % C::kVStages), (tp / C::kVStages) & 1,
                                   ac))
                        return false;
                }
                const uint32_t pv_bar = bar(C::kBarPFull + (t & 1));
                mbar_arrive_expect_tx(pv_bar, C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(sb + C::kOffV + vs * C::kTileBytes + c * C::kChunkBytes, &tmV,
                                pv_bar, c * 64, (vi.kv_lo + vj) * kBlockN, vi.bh_kv);
                v_issued = t + 1;
                advance(vr, vj, vi, v_done);
                return true;
            };
            ok = load_k();
            while (ok && !v_done) {
                // K of the next tile first -- unless it opens a new item, whose Q
                // may wait for an earlier item's output store: then V first.
                const bool k_opens = !k_done && kj == 0;
                if (!k_done && !k_opens) ok = load_k();
                if (ok) ok = load_v();
                if (ok && k_opens) ok = load_k();
            }
            if (!ok) {
                // Let every copy already issued land before the CTA exits: the
                // last arm of each buffer is the only one not yet consumed.
                for (int q = max(n_q - C::kQBufs, 0); q < n_q; ++q)
                    drain_wait(bar(C::kBarQFull + q % C::kQBufs), (q / C::kQBufs) & 1);
                for (int t = max(k_issued - C::kKStages, 0); t < k_issued; ++t)
                    drain_wait(bar(C::kBarKFull + t % C::kKStages), (t / C::kKStages) & 1);
                // (V loads complete on the P barriers, which may never fill
                // after an abort: the drain then waits out its short limit.)
                for (int t = max(v_issued - 2, 0); t < v_issued; ++t)
                    drain_wait(bar(C::kBarPFull + (t & 1)), (t >> 1) & 1);
            }
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdS = idesc_bf16_f32(kBlockM, kBlockN, false, false);
            constexpr uint32_t kIdPV = idesc_bf16_f32(kBlockM, D, false, true);
            // PV of tile i (counted across items): `first` starts the item's O
            // accumulator, `last` also signals the item's final O.  Every PV
            // completes on ODone (the softmax waits there before a rescale).
            auto issue_pv = [&](int i, bool first, bool last) -> bool {
                const int pb = i & 1;
                if (!mbar_wait(bar(C::kBarPFull + pb), (i >> 1) & 1, ac)) return false;
                const int vs = i % C::kVStages;
                tc_fence_after();
                const uint32_t a_tmem = tmem + pb * kBlockN;   // P: bf16 pairs, cols 0..63
                const uint32_t v_base = sb + C::kOffV + vs * C::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk) {
                    const uint64_t bdesc = sdesc_sw128(v_base + kk * 2048, C::kChunkBytes, 1024);
                    mma_ts(tmem + C::kColO, a_tmem + kk * 8, bdesc, kIdPV,
                           (!first || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar(C::kBarVEmpty + vs));
                mma_commit(bar(C::kBarODone));
                if (last) mma_commit(bar(C::kBarOFinal));
                return true;
            };

            bool ok = true;
            int n_q = 0, t = 0;   // items started, tiles whose S was issued
            bool prev_first = false, prev_last = false;
            for (int rnd = 0; ok; ++rnd) {
                const int k = item_at(rnd);
                if (k < 0) break;
                const Item itm = decode(k);
                const int qb = n_q % C::kQBufs;
                if (!(ok = mbar_wait(bar(C::kBarQFull + qb), (n_q / C::kQBufs) & 1, ac))) break;
                tc_fence_after();
                ++n_q;
                const uint32_t q_base = sb + C::kOffQ + qb * C::kTileBytes;
                for (int j = 0; j < itm.n_kv; ++j, ++t) {
                    const int ks = t % C::kKStages;
                    if (!(ok = mbar_wait(bar(C::kBarKFull + ks), (t / C::kKStages) & 1, ac))) break;
                    tc_fence_after();
                    const uint32_t d_tmem = tmem + (t & 1) * kBlockN;
                    const uint32_t k_base = sb + C::kOffK + ks * C::kTileBytes;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
                        const uint64_t adesc = sdesc_sw128(q_base + off, 16, 1024);
                        const uint64_t bdesc = sdesc_sw128(k_base + off, 16, 1024);
                        mma_ss(d_tmem, adesc, bdesc, kIdS, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(bar(C::kBarSFull + (t & 1)));
                    mma_commit(bar(C::kBarKEmpty + ks));
                    // The previous tile's PV (perhaps of the previous item).
                    if (t >= 1 && !(ok = issue_pv(t - 1, prev_first, prev_last))) break;
                    prev_first = j == 0;
                    prev_last = j == itm.n_kv - 1;
                }
            }
            if (ok && t >= 1) ok = issue_pv(t - 1, prev_first, prev_last);
            if (!ok) {
                mma_commit(bar(C::kBarDrain));
                drain_wait(bar(C::kBarDrain), 0);
            }
        }
        __syncwarp();
    } else if (EXT == 2 && warp == kWarpLoader) {
        // ------------------------------------------- residual chunk loader
        // Chunk g = 4 j + c covers keys [128 j + 32 c, +32) of this query
        // tile.  With a bias it is TMA-loaded (zero fill past N); without one
        // the slot is only handed to the softmax, which writes the emitted
        // logits into it.
        if (lane == 0) {
            const int n_chunks = n_kv * kResChunks;
            bool ok = true;
            int issued = 0;
            int slot = 0;
            uint32_t phase = 0;
            for (int g = 0; g < n_chunks; ++g) {
                if (g >= C::kResSlots) ok = mbar_wait(bar(C::kBarResFree + slot), phase ^ 1u, ac);
                if (!ok) break;
                const uint32_t full = bar(C::kBarResFull + slot);
                if (p.bias) {
                    mbar_arrive_expect_tx(full, kResChunkBytes);
                    tma_load_3d(sb + C::kOffRes + slot * kResChunkBytes, &tmBias, full,
                                (kv_lo + g / kResChunks) * kBlockN +
                                    (g % kResChunks) * kResChunkCols,
                                qt * kBlockM, bh);
                } else {
                    mbar_arrive(full);
                }
                issued = g + 1;
                if (++slot == C::kResSlots) { slot = 0; phase ^= 1u; }
            }
            if (!ok && p.bias) {
                for (int g = max(issued - C::kResRing, 0); g < issued; ++g)
                    drain_wait(bar(C::kBarResFull + g % C::kResRing),
                               static_cast<uint32_t>(g / C::kResRing) & 1u);
            }
        }
        __syncwarp();
    } else if (EXT == 2 && warp == kWarpStorer) {
        // ------------------------------------------- emitted-logit storer
        // Waits until the softmax has written a chunk, TMA-stores it (clipped
        // at N) and frees the slot once the store has read it.  While the
        // next chunk is already done, one store is left reading so that two
        // overlap.
        if (lane == 0) {
            const int n_chunks = n_kv * kResChunks;
            int slot = 0;
            uint32_t phase = 0;
            int pending = -1;   // slot whose store may still be reading
            for (int g = 0; g < n_chunks; ++g) {
                if (!mbar_wait(bar(C::kBarResDone + slot), phase, ac)) break;
                int nslot = slot + 1;
                uint32_t nphase = phase;
                if (nslot == C::kResSlots) { nslot = 0; nphase ^= 1u; }
                if (p.emit) {
                    tma_store_3d(&tmEmit, sb + C::kOffRes + slot * kResChunkBytes,
                                 (kv_lo + g / kResChunks) * kBlockN +
                                     (g % kResChunks) * kResChunkCols,
                                 qt * kBlockM, bh);
                    tma_store_commit();
                    const bool next_ready =
                        g + 1 < n_chunks && mbar_test(bar(C::kBarResDone + nslot), nphase);
                    if (next_ready) {
                        tma_store_wait_read_n<1>();
                        if (pending >= 0) mbar_arrive(bar(C::kBarResFree + pending));
                        pending = slot;
                    } else {
                        tma_store_wait_read();
                        if (pending >= 0) mbar_arrive(bar(C::kBarResFree + pending));
                        mbar_arrive(bar(C::kBarResFree + slot));
                        pending = -1;
                    }
                } else {
                    mbar_arrive(bar(C::kBarResFree + slot));
                }
                slot = nslot;
                phase = nphase;
            }
            tma_store_wait_read();
        }
        __syncwarp();
    } else {
        // ---------------------------------------------- softmax warpgroups
        // Warpgroup wg handles keys [64 wg, 64 wg + 64) of every key tile for
        // all 128 rows; the two exchange their partial row max through shared
        // memory once per tile, so they apply the same reference max, and each
        // keeps its own partial row sum.  Every named barrier below is reached
        // by all 256 threads the same number of times (failures are carried to
        // the next barrier and leave through it together).
        const int wg = warp >> 2;
        const int r = ((warp & 3) << 5) | lane;   // row within the tile == TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const int col0 = wg * kHalfN;             // first key of this warpgroup
        float *red = reinterpret_cast<float *>(smem + C::kOffRed);   // [2][2][128]
        bool ok = true;
        int t = 0;   // key tiles over this block's items (the S / P buffer sequence)
        for (int rnd = 0; ok; ++rnd) {
        const int kitem = item_at(rnd);
        if (kitem < 0) break;
        const Item itm = decode(kitem);
        const int qt = itm.qt, bh = itm.bh, kv_lo = itm.kv_lo, n_kv = itm.n_kv;
        const int row_lo = itm.row_lo;
        const int q_row = qt * kBlockM + r;       // row within the head
        const bool row_valid = q_row < p.N;
        float m_run = -INFINITY;   // running max, log2 units
        float l_run = 0.f;         // this warpgroup's part of the row sum

        for (int j = 0; j < n_kv; ++j, ++t) {
            const int sbuf = t & 1;
            const uint32_t tS = tmem + lane_base + sbuf * kBlockN;
            const int key0 = (kv_lo + j) * kBlockN;
            const bool diag = CAUSAL && (kv_lo + j == qt);
            const bool ragged = key0 + kBlockN > p.N;
            // Some row of the tile drops keys below its window start.
            const bool wedge = CAUSAL && p.window > 0 && key0 < row_lo + kBlockM - p.window;
            // x ends up holding the natural-unit logits y = scale q.k + bias,
            // whose row max commutes with the factor xmul = log2(e) that turns
            // them into log2-unit logits; xmul folds into the exp2 FMA.
            const float xmul = kLog2e;
            float x[kHalfN];
            float mt_x = -INFINITY;
            bool got = ok && mbar_wait_warp(bar(C::kBarSFull + sbuf), (t >> 1) & 1, ac);
            if (got) {
                tc_fence_after();
                {
                    uint32_t rr[kHalfN];
                    tmem_ld64(tS + col0, rr);
#pragma unroll
                    for (int c = 0; c < kHalfN; ++c) x[c] = __uint_as_float(rr[c]);
                }

                if constexpr (EXT == 2) {
                    const uint64_t sc2 = f2pack(p.scale, p.scale);
                    // Natural-unit logit y = scale*qk + bias, chunk by chunk
                    // from the staged ring; y goes back over the bias for the
                    // storer (before the mask: masked entries of a diagonal
                    // tile are written too, which the emit contract leaves
                    // unspecified).
                    const uint32_t row_off = static_cast<uint32_t>(r) * 128u;
#pragma unroll
                    for (int cc = 0; cc < kResChunks / 2; ++cc) {
                        const int g = j * kResChunks + wg * (kResChunks / 2) + cc;
                        const int slot = g % C::kResRing;
                        const uint32_t phase = static_cast<uint32_t>(g / C::kResRing) & 1u;
                        if (!mbar_wait_warp(bar(C::kBarResFull + slot), phase, ac)) {
                            got = false;
                            break;
                        }
                        const uint32_t base = sb + C::kOffRes + slot * kResChunkBytes + row_off;
#pragma unroll
                        for (int k = 0; k < kResChunkCols / 4; ++k) {
                            // 16-byte piece k of the row sits at k ^ (row % 8)
                            // (128-byte swizzle).
                            const uint32_t addr = base + (static_cast<uint32_t>(k ^ (r & 7)) << 4);
                            float4 bv = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (p.bias) bv = ld_shared_f4(addr);
                            const int col = cc * kResChunkCols + k * 4;
                            f2unpack(ffma2(f2pack(x[col], x[col + 1]), sc2, f2pack(bv.x, bv.y)),
                                     x[col], x[col + 1]);
                            f2unpack(
                                ffma2(f2pack(x[col + 2], x[col + 3]), sc2, f2pack(bv.z, bv.w)),
                                x[col + 2], x[col + 3]);
                            if (p.emit)
                                st_shared_v4(addr, __float_as_uint(x[col]),
                                             __float_as_uint(x[col + 1]),
                                             __float_as_uint(x[col + 2]),
                                             __float_as_uint(x[col + 3]));
                        }
                        if (p.emit) fence_proxy_async_smem();
                        mbar_arrive(bar(C::kBarResDone + slot));
                    }
                } else if constexpr (EXT == 1) {
                    // Natural-unit logit = scale*qk + bias; emitted before the mask.
                    const size_t roff =
                        (static_cast<size_t>(bh) * p.N + q_row) * p.N + key0 + col0;
                    const float *brow = (p.bias && row_valid) ? p.bias + roff : nullptr;
                    float *erow = (p.emit && row_valid) ? p.emit + roff : nullptr;
                    const int lim = diag ? r + 1 - col0 : kHalfN;   // keys < lim are kept
#pragma unroll
                    for (int c = 0; c < kHalfN; ++c) {
                        const bool inside = (c < lim) && (key0 + col0 + c < p.N);
                        float bval = 0.f;
                        if (brow && inside) bval = __ldg(brow + c);
                        x[c] = fmaf(x[c], p.scale, bval);
                        if (erow && inside) erow[c] = x[c];
                    }
                }

                if (diag || ragged || wedge) {
                    const int klo = wedge ? q_row - p.window + 1 - key0 : -(1 << 30);   // first kept key
#pragma unroll
                    for (int c = 0; c < kHalfN; ++c) {
                        const int key = col0 + c;
                        const bool keep =
                            (!diag || key <= r) && (key0 + key < p.N) && (key >= klo);
                        x[c] = keep ? x[c] : -INFINITY;
                    }
                }
                // Partial row max as a tree (8 independent chains of 3-input max).
                float mx[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mx[i] = x[i];
#pragma unroll
                for (int c = 8; c + 16 <= kHalfN; c += 16) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], x[c + i], x[c + 8 + i]);
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) mx[i] = fmaxf(mx[i], x[kHalfN - 8 + i]);
                // (c runs 8, 24, 40 over elements 8..55; the last pass adds 56..63.)
                mt_x = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                             fmaxf(mx[6], mx[7]));
                red[(sbuf * 2 + wg) * kBlockM + r] = mt_x;
                tc_fence_before();   // this warpgroup's S reads precede the other's P writes
            }
            if (named_bar_or(2, kSoftThreads, !got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float mt_other = red[(sbuf * 2 + (wg ^ 1)) * kBlockM + r];
            const float m_tile = fmaxf(mt_x, mt_other) * xmul;
            // Lazy rescale: keep the previous reference max while the new row
            // max exceeds it by at most kRescaleLog2 (p stays <= 2^8); O/l and
            // LSE are unchanged by the choice of reference.  Both warpgroups
            // compute the same m_new from the same inputs.
            float m_new = fmaxf(m_run, m_tile);
            if (m_new - m_run <= kRescaleLog2) m_new = m_run;
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = ex2(m_run - m_use);   // 0 on the first tile

            const uint64_t cm2 = f2pack(xmul, xmul);
            const uint64_t nm2 = f2pack(-m_use, -m_use);
            uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};   // (+0.0f, +0.0f) pairs
            {
                uint32_t pk[kHalfN / 2];
#pragma unroll
                for (int c = 0; c < kHalfN / 2; ++c) {
                    float t0, t1;
                    f2unpack(ffma2(f2pack(x[2 * c], x[2 * c + 1]), cm2, nm2), t0, t1);
                    const float p0 = ex2(t0), p1 = ex2(t1);
                    acc[c & 3] = fadd2(acc[c & 3], f2pack(p0, p1));
                    pk[c] = pack_bf16x2(p0, p1);
                }
                // P as packed bf16 pairs: keys 2c, 2c+1 of the tile in column c.
                tmem_st32(tS + col0 / 2, pk);
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
                // O holds PV_0..PV_{j-1}; PV_{j-1} must have landed first.  Each
                // warpgroup rescales its half of O's columns.
                if (!mbar_wait_warp(bar(C::kBarODone), (t - 1) & 1, ac)) {
                    ok = false;   // leaves at the next barrier, with the other warpgroup
                } else {
                    tc_fence_after();
                    const uint32_t tO = tmem + lane_base + C::kColO;
                    if (wg == 0) o_rescale<C::kOSplit>(tO, alpha);
                    else o_rescale<D - C::kOSplit>(tO + C::kOSplit, alpha);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            if (ok) mbar_arrive(bar(C::kBarPFull + sbuf));
            m_run = m_new;
        }

        // ------------------------------------------------------- epilogue
        // Both warpgroups reach the barriers below exactly once per item,
        // whatever happened in the loop.  O is staged (bf16, swizzled) in the
        // item's Q buffer, which its S MMAs are done with.
        if (ok) ok = mbar_wait_warp(bar(C::kBarOFinal), rnd & 1, ac);
        float *lsum = red + (t & 1) * 2 * kBlockM;   // the buffer the item's last tile did not use
        if (ok) lsum[wg * kBlockM + r] = l_run;
        const bool fail = named_bar_or(2, kSoftThreads, !ok);
        const uint32_t o_tile = sb + C::kOffQ + (rnd % C::kQBufs) * C::kTileBytes;
        if (!fail) {
            tc_fence_after();
            const float l_tot = l_run + lsum[(wg ^ 1) * kBlockM + r];
            const float inv_l = 1.f / l_tot;
            const uint32_t tO = tmem + lane_base + C::kColO;
            if (wg == 0) o_stage<C::kOSplit, 0>(tO, inv_l, o_tile, r);
            else o_stage<D - C::kOSplit, C::kOSplit>(tO + C::kOSplit, inv_l, o_tile, r);
            if (wg == 0 && p.lse && row_valid)
                p.lse[static_cast<size_t>(bh) * p.N + q_row] = (m_run + log2f(l_tot)) * kLn2;
            fence_proxy_async_smem();
        }
        tc_fence_before();
        // (Also keeps the next item's first row-max writes off the row sums
        // the other warpgroup reads above.)
        named_bar_sync(1, kSoftThreads);
        if (fail) {
            ok = false;
            break;
        }
        if (threadIdx.x == 0 && *abort_flag == 0) {
            for (int c = 0; c < C::kChunks; ++c)
                tma_store_3d(&tmO, o_tile + c * C::kChunkBytes, c * 64, row_lo, bh);
            tma_store_commit();
            tma_store_wait_read();
        }
        }   // items
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

struct FwdMaps {
    CUtensorMap q, k, v, o, bias, emit;
};

template <int D, bool CAUSAL, int EXT>
cudaError_t launch_t(const FwdMaps &m, const FwdParams &prm, unsigned grid, cudaStream_t stream) {
    using C = FwdCfg<D, EXT>;
    auto kern = fwd_kernel<D, CAUSAL, EXT>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, fwd_threads<EXT>(), C::kSmemBytes, stream>>>(m.q, m.k, m.v, m.o, m.bias, m.emit,
                                                               prm);
    return cudaGetLastError();
}

template <int D, bool CAUSAL>
cudaError_t launch_c(int ext, const FwdMaps &m, const FwdParams &prm, unsigned grid,
                     cudaStream_t stream) {
    if (ext == 2) return launch_t<D, CAUSAL, 2>(m, prm, grid, stream);
    return launch_t<D, CAUSAL, 1>(m, prm, grid, stream);
}

template <int D>
cudaError_t launch_d(bool causal, int ext, const FwdMaps &m, const FwdParams &prm, unsigned grid,
                     cudaStream_t stream) {
    return causal ? launch_c<D, true>(ext, m, prm, grid, stream)
                  : launch_c<D, false>(ext, m, prm, grid, stream);
}

}  // namespace

cudaError_t launch_fwd(const FwdProblem &pb, int *status, cudaStream_t stream) {
    // The plain forward runs two query tiles per thread block (attn_fwd_pp.cu).
    if (!pb.bias && !pb.emit) return launch_fwd_pp(pb, status, stream);
    const long long BH = static_cast<long long>(pb.B) * pb.Hq;
    const long long BHkv = static_cast<long long>(pb.B) * pb.Hkv;
    FwdMaps m;
    if (!encode_bf16_rows(&m.q, pb.q, pb.D, pb.N, BH, kBlockM) ||
        !encode_bf16_rows(&m.k, pb.k, pb.D, pb.N, BHkv, kBlockN) ||
        !encode_bf16_rows(&m.v, pb.v, pb.D, pb.N, BHkv, kBlockN) ||
        !encode_bf16_rows(&m.o, pb.o, pb.D, pb.N, BH, kBlockM))
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
    prm.window = pb.causal ? pb.window : 0;
    prm.wait_limit_ns = pb.wait_limit_ns ? pb.wait_limit_ns : kWaitLimitNs;
    const long long n_items = static_cast<long long>(prm.n_qtiles) * BH;
    // Causal item order: one chunk of all heads unless their K/V is over
    // twice the L2; then chunks whose K/V is about half the L2, so that the
    // items running at once share a few heads' K/V (measured, D128 causal:
    // B8 H32 N8192 4.78 -> 3.78 ms, where the 152 items running at once
    // were otherwise 152 different heads; B4 H16 N16384 and B1 H16 N65536
    // the same or slightly faster).
    DeviceInfo di;
    if (!device_info(&di)) return cudaErrorInvalidValue;
    prm.hchunk = static_cast<int>(BH);
    {
        const double l2 = di.l2_bytes;
        const double head_kv = static_cast<double>(pb.N) * pb.D * 4.0 / (pb.Hq / pb.Hkv);   // per query head
        if (pb.causal && head_kv * static_cast<double>(BH) > 2.0 * l2)
            prm.hchunk = static_cast<int>(
                std::max<long long>(1, std::min<long long>(BH, static_cast<long long>(0.5 * l2 / head_kv))));
    }
    int ext = 1;
    {
        // The staged variant maps the [N, N] planes as tensors of 128 x 32
        // fp32 boxes: rows must be 16-byte multiples, bases 16-byte aligned.
        const auto a16 = [](const void *ptr) { return reinterpret_cast<uintptr_t>(ptr) % 16 == 0; };
        ext = (pb.N % 4 == 0 && a16(pb.bias) && a16(pb.emit)) ? 2 : 1;
        // A map of one operand stands in for the one that is absent (never used).
        const float *rb = pb.bias ? pb.bias : pb.emit;
        const float *re = pb.emit ? pb.emit : pb.bias;
        if (ext == 2 && (!encode_f32_rows(&m.bias, rb, pb.N, pb.N, BH, kBlockM) ||
                         !encode_f32_rows(&m.emit, re, pb.N, pb.N, BH, kBlockM)))
            ext = 1;
    }
    if (ext != 2) m.bias = m.emit = m.q;   // unused by the kernel
    // One block per (query tile, head).
    const unsigned grid = static_cast<unsigned>(n_items);
    switch (pb.D) {
    case 64: return launch_d<64>(pb.causal, ext, m, prm, grid, stream);
    case 80: return launch_d<80>(pb.causal, ext, m, prm, grid, stream);
    case 96: return launch_d<96>(pb.causal, ext, m, prm, grid, stream);
    default: return launch_d<128>(pb.causal, ext, m, prm, grid, stream);
    }
}

}  // namespace tattn
