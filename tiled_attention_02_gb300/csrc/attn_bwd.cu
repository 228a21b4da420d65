// attn_bwd.cu -- recompute-based attention backward for GB300 (sm_103a).
//
// The backward of exact attention from the saved per-row log-sum-exp only
// (kwkr.cn/news/592482, section 2.4; "FlashAttention原理与Triton实战",
// sections 2.3 and 4.3): P is recomputed tile by tile, the chain rule gives
//   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - Delta),  Delta_i = dO_i . O_i,
//   dK = scale dS^T Q,  dQ = scale dS K.
//
// Three launches on the caller's stream:
//  1. bwd_pre_kernel    Delta_i (fp32, from the bf16 O and dO), LSE * log2(e)
//                       padded to whole 128-row tiles, and a zeroed fp32 dQ
//                       accumulator -- all in the caller's workspace.
//  2. bwd_main_kernel   one CTA per (batch, kv head, 128-key tile); loops over
//                       every 128-row query tile of every query head of the
//                       group that can see those keys.  Per query tile:
//                         S^T  = K Q^T       tcgen05.mma -> TMEM
//                         dP^T = V dO^T      tcgen05.mma -> TMEM
//                         P^T  = 2^(S^T scale log2e - LSE log2e)   (bf16 -> TMEM)
//                         dS^T = P^T o (dP^T - Delta) * scale     (bf16 -> smem)
//                         dV  += P^T dO      tcgen05.mma, A from TMEM
//                         dK  += dS^T Q      tcgen05.mma
//                         dQ   = dS K        tcgen05.mma -> TMEM, staged to
//                                            smem and added into the fp32
//                                            accumulator by TMA bulk
//                                            reductions
//                       dK, dV stay in TMEM for the whole loop (summed over the
//                       query heads of a kv group) and are stored once.
//  3. bwd_dq_kernel     fp32 dQ accumulator -> bf16 dQ.
//
// Warp roles of the main kernel (448 threads, one CTA per SM):
//   warps 0-7  two warpgroups; warpgroup w computes P^T and dS^T for query
//              columns 64w..64w+63 (thread r = key row r = TMEM lane r);
//              epilogue: warpgroup 0 stores dV, warpgroup 1 stores dK.
//   warps 8-11 thread r owns query row r of the dQ tile: TMEM -> smem -> TMA add.
//   warp 12    TMA producer (K, V once; Q, dO, LSE, Delta per query tile).
//   warp 13    TMEM allocator and tcgen05.mma issuer.
// TMEM columns: S^T/P^T 0..127, dP^T/dQ 128..255, dV 256.., dK 256+D...
// MMA order per query tile j: S^T(j), dP^T(j), dV(j), dK(j), dQ(j); the P^T
// work overlaps dP^T and the dS^T work overlaps dV.
#include "attn_internal.h"
#include "sm103_ptx.cuh"

#include <algorithm>

namespace tattn {
namespace {

constexpr int kTile = 128;
constexpr float kLog2e = 1.4426950408889634f;

// --------------------------------------------------------------- preprocess

template <int D>
__global__ void __launch_bounds__(256)
bwd_pre_kernel(const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ dO,
               const float *__restrict__ lse, float *__restrict__ lse2,
               float *__restrict__ delta, float *__restrict__ dq_acc, int N, int NP,
               int n_tiles) {
    constexpr int kVecs = D / 8;                           // 16-byte vectors (8 bf16) per row
    constexpr int kLanesPerRow = kVecs <= 8 ? 8 : 16;      // power of two >= kVecs
    constexpr int kRowsPerWarp = 32 / kLanesPerRow;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // One block per (head, row tile) on a 1D grid: B*Hq*tiles fits in 31 bits,
    // while either factor alone may pass the 65535 limit of gridDim.y.
    const int bh = static_cast<int>(blockIdx.x / static_cast<unsigned>(n_tiles));
    const int row0 = static_cast<int>(blockIdx.x % static_cast<unsigned>(n_tiles)) * kTile;
    const int sub = lane % kLanesPerRow;
    for (int rr = warp * kRowsPerWarp + lane / kLanesPerRow; rr < kTile; rr += 8 * kRowsPerWarp) {
        const int row = row0 + rr;
        const bool valid = row < N;
        float acc = 0.f;
        const size_t off = (static_cast<size_t>(bh) * N + row) * D + sub * 8;
        if (valid && sub < kVecs) {
            const uint4 a = *reinterpret_cast<const uint4 *>(o + off);
            const uint4 b = *reinterpret_cast<const uint4 *>(dO + off);
            const __nv_bfloat162 *pa = reinterpret_cast<const __nv_bfloat162 *>(&a);
            const __nv_bfloat162 *pb = reinterpret_cast<const __nv_bfloat162 *>(&b);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 fa = __bfloat1622float2(pa[e]);
                const float2 fb = __bfloat1622float2(pb[e]);
                acc = fmaf(fa.x, fb.x, acc);
                acc = fmaf(fa.y, fb.y, acc);
            }
            float4 *z = reinterpret_cast<float4 *>(dq_acc + off);
            z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int m = kLanesPerRow / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
        if (sub == 0) {
            const size_t prow = static_cast<size_t>(bh) * NP + row;
            lse2[prow] = valid ? lse[static_cast<size_t>(bh) * N + row] * kLog2e : INFINITY;
            delta[prow] = valid ? acc : 0.f;
        }
    }
}

// ----------------------------------------------- accumulator zero fill

__global__ void __launch_bounds__(256)
bwd_zero_kernel(float4 *__restrict__ p, size_t n4) {
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ------------------------------------------------------------ dQ convert

__global__ void __launch_bounds__(256)
bwd_dq_kernel(const float *__restrict__ acc, __nv_bfloat16 *__restrict__ dq, size_t n8) {
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n8;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const float4 a = reinterpret_cast<const float4 *>(acc)[2 * i];
        const float4 b = reinterpret_cast<const float4 *>(acc)[2 * i + 1];
        uint4 w;
        w.x = pack_bf16x2(a.x, a.y);
        w.y = pack_bf16x2(a.z, a.w);
        w.z = pack_bf16x2(b.x, b.y);
        w.w = pack_bf16x2(b.z, b.w);
        reinterpret_cast<uint4 *>(dq)[i] = w;
    }
}

// ------------------------------------------------------------ main kernel

constexpr int kMaxSmem = 232448;   // opt-in shared memory per block on sm_100/sm_103
// Block residual variant: fp32 [query][key] tiles of the bias, the incoming
// logit gradient and the outgoing one move in chunks of 32 query rows x 128
// keys (four 32 x 32 boxes of 128-byte swizzled rows).
constexpr int kResQ = 32;                      // query rows per chunk
constexpr int kResChunkBytes = kResQ * kTile * 4;
constexpr int kResChunks = kTile / kResQ;      // chunks per (query tile, key tile)
constexpr int kResSlots = 4;

template <bool RES>
constexpr int bwd_threads() { return RES ? 512 : 448; }

template <int D, bool RES = false>
struct BwdCfg {
    // A bf16 row of D elements occupies ceil(D/64) 128-byte swizzle atoms
    // (zero-filled past D by TMA); stores and reductions are clipped at D.
    static constexpr int kChunks = (D + 63) / 64;
    static constexpr int kChunkBytes = kTile * 128;
    static constexpr int kTileBytes = kChunks * kChunkBytes;
    static constexpr int kDQBoxes = (D + 31) / 32;   // fp32 dQ boxes of 32 columns
    // The residual variant keeps one {Q, dO} stage and gives the other's
    // shared memory to its fp32 chunk ring.  Its stage's two tile buffers
    // swap roles every item: Q(j) in buffer j % 2, dO(j) in buffer
    // (j + 1) % 2.  dO(j) is last read by dV(j), well before Q(j) is last
    // read by dK(j), so Q(j + 1) loads into dO(j)'s buffer while item j's
    // dS work runs, and dO(j + 1) into Q(j)'s buffer after dK(j).
    static constexpr int kQStages = RES ? 1 : 2;
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kTileBytes;
    static constexpr int kOffStage = 2 * kTileBytes;          // kQStages stages of {Q, dO}
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kOffRows = kOffStage + kQStages * kStageBytes;   // lse2[2][128], delta[2][128]
    static constexpr int kOffDS = ((kOffRows + 4 * kTile * 4) + 1023) & ~1023;
    static constexpr int kDSBytes = kTile * kTile * 2;
    static constexpr int kOffRes = kOffDS + kDSBytes;
    static constexpr int kNumResSlots = RES ? kResSlots : 0;
    static constexpr int kResRing = RES ? kResSlots : 1;
    static constexpr int kOffBar = kOffRes + kNumResSlots * kResChunkBytes;
    static constexpr int kBarKV = 0;
    // Per stage: QFull / QEmpty cover Q and the LSE / Delta rows (and dO too
    // in the one-stage residual variant); DOFull / DOEmpty cover dO (two-stage
    // variant), whose buffer also stages part of dQ.
    static constexpr int kBarQFull = 1;      // 2
    static constexpr int kBarQEmpty = 3;     // 2 (residual variant: per tile buffer)
    static constexpr int kBarSFull = 5;
    static constexpr int kBarDPFull = 6;
    static constexpr int kBarPReady = 7;
    static constexpr int kBarDSReady = 8;
    static constexpr int kBarDQFull = 9;
    static constexpr int kBarDQEmpty = 10;
    static constexpr int kBarDSFree = 11;
    static constexpr int kBarAccDone = 12;
    static constexpr int kBarDrain = 13;
    static constexpr int kBarDOFull = 14;    // 2
    static constexpr int kBarDOEmpty = 16;   // 2
    static constexpr int kBarResFull = 18;                        // kNumResSlots each
    static constexpr int kBarResDone = kBarResFull + kNumResSlots;
    static constexpr int kBarResFree = kBarResDone + kNumResSlots;
    static constexpr int kNumBars = kBarResFree + kNumResSlots;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kUsed = kOffMisc + 16;
    static constexpr int kSmemBytes = (kUsed + 1023 <= kMaxSmem) ? kUsed + 1023 : kMaxSmem;
    static constexpr uint32_t kTmemCols = 512;
    // dK starts on a 64-column boundary so that 64-column loads stay aligned.
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256;
    static constexpr uint32_t kColDK = D <= 64 ? 256 + 64 : 384;
    static_assert(kDQBoxes * kTile * 128 <= 2 * kTileBytes, "dQ staging fits a stage");
    static_assert(kResChunks == 4, "one chunk per P/dS warpgroup half");
    static_assert(kUsed <= kMaxSmem, "shared memory budget");
};

struct BwdParams {
    const float *lse2;
    const float *delta;
    float *dq_acc;
    int *status;
    int N, NP, Hq, Hkv, group, BHkv, n_tiles;
    float scale, scale_log2;
    int window;   // causal sliding window W (key j kept for query i iff i - W < j), 0 = none
    // residual variant: which of the three fp32 [B,Hq,N,N] tensors are given
    int has_bias, has_gin, has_gout;
    // blocks per (key tile, kv head): each takes group / hsplit query heads;
    // with hsplit > 1, dK and dV are fp32 partial sums added into accumulators
    int hsplit;
    // kv heads per block-order chunk: chunks go one after another, key tile 0
    // (the heaviest under the causal mask) first within each
    int hchunk;
};

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > 20ull * 1000ull * 1000ull) break;
    }
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}


// Writes 64 packed-bf16 words (128 columns) of row r into a 128-row tile
// staged in the 128-byte swizzled layout TMA and tcgen05 use.
__device__ __forceinline__ void stage_row64(uint32_t tile, int r, int atom, const uint32_t *w) {
#pragma unroll
    for (int pc = 0; pc < 8; ++pc) {
        const uint32_t addr = tile + atom * (kTile * 128) + r * 128 +
                              (static_cast<uint32_t>(pc ^ (r & 7)) << 4);
        st_shared_v4(addr, w[4 * pc], w[4 * pc + 1], w[4 * pc + 2], w[4 * pc + 3]);
    }
}

template <int D, bool CAUSAL, bool RES>
__global__ void __launch_bounds__(bwd_threads<RES>(), 1)
bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ CUtensorMap tmBias,
                const __grid_constant__ CUtensorMap tmGin, const __grid_constant__ CUtensorMap tmGout,
                const BwdParams p) {
    using C = BwdCfg<D, RES>;
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

    // Blocks go in chunks of hchunk kv heads (the last chunk may be smaller),
    // heaviest key tiles first within a chunk (under the causal mask tile 0
    // sees every query tile), so that the blocks running at once share a few
    // heads' Q, dO and dQ accumulator in L2.
    // blockIdx.y is the chunk of hchunk kv heads (chunks run one after
    // another: blocks are dispatched in order of their linear index).
    const int kt = blockIdx.x / (p.hchunk * p.hsplit);
    const int bh_kv = blockIdx.y * p.hchunk + (blockIdx.x % (p.hchunk * p.hsplit)) / p.hsplit;
    const int hs = blockIdx.x % p.hsplit;          // which share of the group's query heads
    const int hper = p.group / p.hsplit;           // query heads of this block
    const int b = bh_kv / p.Hkv, g = bh_kv % p.Hkv;
    // Query tiles q_lo .. q_lo + nq - 1 see this key tile: from the diagonal
    // (causal) to the tile holding query kt*128 + 127 + W - 1 (window).
    const int q_lo = CAUSAL ? kt : 0;
    const int q_end = (CAUSAL && p.window > 0)
                          ? min(p.n_tiles, (kt * kTile + kTile - 1 + p.window - 1) / kTile + 1)
                          : p.n_tiles;
    const int nq = q_end - q_lo;                  // query tiles per query head
    const int n_items = hper * nq;

    auto bar = [&](int i) -> uint32_t { return sb + C::kOffBar + 8u * i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffMisc + 4);
    const AbortCtl ac{abort_flag, p.status, kWaitLimitNs};
    auto item_qi = [&](int j) { return q_lo + j % nq; };
    auto item_bhq = [&](int j) { return b * p.Hq + g * p.group + hs * hper + j / nq; };
    const uint32_t s_rows = sb + C::kOffRows;   // lse2[s][128] then delta[s][128]
    // Residual chunk sequence of item j: the bias chunks c = 0..3 (if a bias
    // is given), then the logit-gradient chunks c = 0..3 (if one flows in or
    // out); chunk c covers query rows 32c..32c+31 of the item's query tile.
    const int res_bias = RES && p.has_bias ? kResChunks : 0;
    const int res_grad = RES && (p.has_gin || p.has_gout) ? kResChunks : 0;
    const int res_per_item = res_bias + res_grad;
    // Within the bias (and the gradient) chunks of an item, position pos
    // holds chunk 2 (pos % 2) + pos / 2, i.e. the order 0, 2, 1, 3: the
    // first-half chunks of both P/dS warpgroups (chunk 2w + h is warpgroup
    // w's query columns 32h..32h+31) come first.  A warpgroup hands its
    // first bias chunk back halfway through its P phase, so the first
    // gradient chunks can load while the P phase still runs.
    auto res_chunk_at = [](int pos) { return 2 * (pos & 1) + (pos >> 1); };

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        mbar_init(bar(C::kBarKV), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(C::kBarQFull + s), 1);
            mbar_init(bar(C::kBarQEmpty + s), 1);    // the MMA thread, after the item's MMAs
            mbar_init(bar(C::kBarDOFull + s), 1);
            mbar_init(bar(C::kBarDOEmpty + s), 4);   // the four drain warps (staged drain)
        }
        for (int s = 0; s < C::kNumResSlots; ++s) {
            mbar_init(bar(C::kBarResFull + s), 1);
            // Done: the P/dS warpgroup that wrote a gradient chunk.  Free:
            // the warpgroup that read a bias chunk, or the storer (one
            // arrival of kTile) once a gradient chunk's store has read it.
            mbar_init(bar(C::kBarResDone + s), kTile);
            mbar_init(bar(C::kBarResFree + s), kTile);
        }
        mbar_init(bar(C::kBarSFull), 1);
        mbar_init(bar(C::kBarDPFull), 1);
        mbar_init(bar(C::kBarPReady), 2 * kTile);
        mbar_init(bar(C::kBarDSReady), 2 * kTile);
        mbar_init(bar(C::kBarDQFull), 1);
        mbar_init(bar(C::kBarDQEmpty), kTile);
        // dS buffer free: the MMA thread (dK, dQ read it) and, with the staged
        // drain, the four drain warps (part of dQ is staged there).
        mbar_init(bar(C::kBarDSFree), RES ? 1 : 5);
        mbar_init(bar(C::kBarAccDone), 1);
        mbar_init(bar(C::kBarDrain), 1);
        fence_barrier_init();
    }
    if (warp == 13) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 12) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            bool ok = true;
            mbar_arrive_expect_tx(bar(C::kBarKV), 2 * C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c) {
                tma_load_3d(sb + C::kOffK + c * C::kChunkBytes, &tmK, bar(C::kBarKV), c * 64,
                            kt * kTile, bh_kv);
                tma_load_3d(sb + C::kOffV + c * C::kChunkBytes, &tmV, bar(C::kBarKV), c * 64,
                            kt * kTile, bh_kv);
            }
            int issued = 0, issued_do = 0;
            if constexpr (RES) {
                // Q(j) and the rows into buffer / row slot j % 2 once dO(j - 1)
                // (the buffer's previous use) is done; dO(j) into buffer
                // (j + 1) % 2 once Q(j - 1) is done.  Each buffer is used once
                // per item, so its empty barrier completes phase j at item j.
                for (int j = 0; j < n_items; ++j) {
                    const int qi = item_qi(j), bhq = item_bhq(j);
                    const int bq = j & 1, bd = bq ^ 1;
                    const uint32_t ph = static_cast<uint32_t>(j - 1) & 1u;
                    if (j > 0 && !(ok = mbar_wait(bar(C::kBarQEmpty + bq), ph, ac))) break;
                    const uint32_t fb = bar(C::kBarQFull);
                    mbar_arrive_expect_tx(fb, C::kTileBytes + 2 * kTile * 4);
                    const uint32_t sq = sb + C::kOffStage + bq * C::kTileBytes;
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(sq + c * C::kChunkBytes, &tmQ, fb, c * 64, qi * kTile, bhq);
                    const size_t prow = static_cast<size_t>(bhq) * p.NP + qi * kTile;
                    bulk_load(s_rows + bq * kTile * 4, p.lse2 + prow, kTile * 4, fb);
                    bulk_load(s_rows + (2 + bq) * kTile * 4, p.delta + prow, kTile * 4, fb);
                    issued = j + 1;
                    if (j > 0 && !(ok = mbar_wait(bar(C::kBarQEmpty + bd), ph, ac))) break;
                    const uint32_t db = bar(C::kBarDOFull);
                    mbar_arrive_expect_tx(db, C::kTileBytes);
                    const uint32_t sd = sb + C::kOffStage + bd * C::kTileBytes;
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(sd + c * C::kChunkBytes, &tmdO, db, c * 64, qi * kTile, bhq);
                    issued_do = j + 1;
                }
            }
            for (int j = 0; j < (RES ? 0 : n_items); ++j) {
                const int s = j % C::kQStages;
                const uint32_t ph = ((j / C::kQStages) - 1) & 1;
                if (j >= C::kQStages && !(ok = mbar_wait(bar(C::kBarQEmpty + s), ph, ac))) break;
                const int qi = item_qi(j), bhq = item_bhq(j);
                const uint32_t fb = bar(C::kBarQFull + s);
                // Q and the rows on QFull, dO on DOFull (so that S^T can
                // start before dO has landed)
                mbar_arrive_expect_tx(fb, C::kTileBytes + 2 * kTile * 4);
                const uint32_t st = sb + C::kOffStage + s * C::kStageBytes;
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(st + c * C::kChunkBytes, &tmQ, fb, c * 64, qi * kTile, bhq);
                const size_t prow = static_cast<size_t>(bhq) * p.NP + qi * kTile;
                bulk_load(s_rows + s * kTile * 4, p.lse2 + prow, kTile * 4, fb);
                bulk_load(s_rows + (2 + s) * kTile * 4, p.delta + prow, kTile * 4, fb);
                if constexpr (!RES) {
                    issued = j + 1;
                    if (j >= C::kQStages && !(ok = mbar_wait(bar(C::kBarDOEmpty + s), ph, ac)))
                        break;
                }
                // (With one stage dO's buffer goes back with Q's, on QEmpty.)
                const uint32_t db = bar(C::kBarDOFull + s);
                mbar_arrive_expect_tx(db, C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(st + C::kTileBytes + c * C::kChunkBytes, &tmdO, db, c * 64,
                                qi * kTile, bhq);
                issued = j + 1;
                issued_do = j + 1;
            }
            if (!ok) {
                // (Residual variant: one Q and one dO load in flight at most,
                // on barrier 0 of each.)
                drain_wait(bar(C::kBarKV), 0);
                for (int j = max(issued - C::kQStages, 0); j < issued; ++j)
                    drain_wait(bar(C::kBarQFull + j % C::kQStages), (j / C::kQStages) & 1);
                for (int j = max(issued_do - C::kQStages, 0); j < issued_do; ++j)
                    drain_wait(bar(C::kBarDOFull + j % C::kQStages), (j / C::kQStages) & 1);
            }
        }
        __syncwarp();
    } else if (warp == 13) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdS = idesc_bf16_f32(kTile, kTile, false, false);
            constexpr uint32_t kIdAcc = idesc_bf16_f32(kTile, D, false, true);   // dV, dK
            constexpr uint32_t kIdDQ = idesc_bf16_f32(kTile, D, true, true);     // dQ
            const uint32_t sK = sb + C::kOffK, sV = sb + C::kOffV, sDS = sb + C::kOffDS;
            auto stage_of = [&](int j) -> uint32_t {
                return sb + C::kOffStage + (j % C::kQStages) * C::kStageBytes;
            };
            // Q(j) and dO(j) tiles (the residual variant alternates buffers).
            auto q_of = [&](int j) -> uint32_t {
                return RES ? sb + C::kOffStage + (j & 1) * C::kTileBytes : stage_of(j);
            };
            auto do_of = [&](int j) -> uint32_t {
                return RES ? sb + C::kOffStage + ((j + 1) & 1) * C::kTileBytes
                           : stage_of(j) + C::kTileBytes;
            };
            auto wait_stage = [&](int j) -> bool {   // Q and the LSE / Delta rows
                if (!mbar_wait(bar(C::kBarQFull + j % C::kQStages), (j / C::kQStages) & 1, ac))
                    return false;
                tc_fence_after();
                return true;
            };
            auto wait_do = [&](int j) -> bool {
                if (!mbar_wait(bar(C::kBarDOFull + j % C::kQStages), (j / C::kQStages) & 1, ac))
                    return false;
                tc_fence_after();
                return true;
            };
            auto wait_on = [&](int b, int phase) -> bool {
                if (!mbar_wait(bar(b), phase & 1, ac)) return false;
                tc_fence_after();
                return true;
            };
            auto issue_st = [&](int j) {   // S^T = K Q^T (over P^T(j-1), read by dV(j-1))
                const uint32_t sQ = q_of(j);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
                    mma_ss(tmem + C::kColS, sdesc_sw128(sK + off, 16, 1024),
                           sdesc_sw128(sQ + off, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(C::kBarSFull));
            };
            auto issue_dpt = [&](int j) {   // dP^T = V dO^T (over dQ(j-1), drained)
                const uint32_t sdO = do_of(j);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
                    mma_ss(tmem + C::kColDP, sdesc_sw128(sV + off, 16, 1024),
                           sdesc_sw128(sdO + off, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(C::kBarDPFull));
            };
            auto issue_dv = [&](int j) {   // dV += P^T dO  (A in TMEM)
                const uint32_t sdO = do_of(j);
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk) {
                    // P^T of query columns 64w..64w+63 sits in TMEM columns
                    // 64w..64w+31 (over warpgroup w's own, already read, S^T).
                    mma_ts(tmem + C::kColDV, tmem + C::kColS + (kk >> 2) * 64 + (kk & 3) * 8,
                           sdesc_sw128(sdO + kk * 2048, C::kChunkBytes, 1024), kIdAcc,
                           (j > 0 || kk > 0) ? 1u : 0u);
                }
                // Residual variant: dO(j)'s buffer is free (Q(j + 1) loads there).
                if (RES) mma_commit(bar(C::kBarQEmpty + ((j + 1) & 1)));
            };
            auto issue_dk_dq = [&](int j) {   // dK += dS^T Q, then dQ = dS K (over dP^T(j), read)
                const uint32_t sQ = q_of(j);
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
                    mma_ss(tmem + C::kColDK, sdesc_sw128(sDS + off, 16, 1024),
                           sdesc_sw128(sQ + kk * 2048, C::kChunkBytes, 1024), kIdAcc,
                           (j > 0 || kk > 0) ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk) {   // both operands MN-major
                    mma_ss(tmem + C::kColDP, sdesc_sw128(sDS + kk * 2048, C::kChunkBytes, 1024),
                           sdesc_sw128(sK + kk * 2048, C::kChunkBytes, 1024), kIdDQ,
                           kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(C::kBarDQFull));   // also: every MMA of item j has completed
                mma_commit(bar(C::kBarDSFree));
                // Q of the item is free now (residual variant: Q(j)'s buffer,
                // where dO(j + 1) loads); with two stages the drain hands dO's
                // buffer back once its reductions have read the part of dQ
                // staged there.
                mma_commit(bar(C::kBarQEmpty + (RES ? (j & 1) : j % C::kQStages)));
            };
            bool ok = mbar_wait(bar(C::kBarKV), 0, ac);
            if constexpr (RES) {
                // One {Q, dO} stage: per query tile j,
                //   S^T(j)  dP^T(j)  [P ready] dV(j)  [dS ready] dK(j) dQ(j).
                // P is computed while dP^T runs and dS while dV runs.
                for (int j = 0; j < n_items && ok; ++j) {
                    if (!(ok = wait_stage(j))) break;
                    issue_st(j);
                    if (j > 0 && !(ok = wait_on(C::kBarDQEmpty, j - 1))) break;
                    if (!(ok = wait_do(j))) break;
                    issue_dpt(j);
                    if (!(ok = wait_on(C::kBarPReady, j))) break;
                    issue_dv(j);
                    if (!(ok = wait_on(C::kBarDSReady, j))) break;
                    issue_dk_dq(j);
                }
            } else {
                // Two stages, software-pipelined over query tiles:
                //   [P ready(j)] dV(j)  S^T(j+1)  [dS ready(j)] dK(j) dQ(j)
                //   [dQ(j) drained] dP^T(j+1)
                // so the P phase of tile j+1 runs while dK(j) and dQ(j) do.
                if (ok && n_items > 0 && (ok = wait_stage(0))) {
                    issue_st(0);
                    if ((ok = wait_do(0))) issue_dpt(0);
                }
                for (int j = 0; j < n_items && ok; ++j) {
                    if (!(ok = wait_on(C::kBarPReady, j))) break;
                    issue_dv(j);
                    if (j + 1 < n_items) {
                        if (!(ok = wait_stage(j + 1))) break;
                        issue_st(j + 1);
                    }
                    if (!(ok = wait_on(C::kBarDSReady, j))) break;
                    issue_dk_dq(j);
                    if (j + 1 < n_items) {
                        if (!(ok = wait_on(C::kBarDQEmpty, j))) break;
                        if (!(ok = wait_do(j + 1))) break;
                        issue_dpt(j + 1);
                    }
                }
            }
            if (ok) {
                mma_commit(bar(C::kBarAccDone));
            } else {
                mma_commit(bar(C::kBarDrain));
                drain_wait(bar(C::kBarDrain), 0);
            }
        }
        __syncwarp();
    } else if (RES && warp == 14) {
        // -------------------------------------- residual chunk loader
        // Bias and incoming-gradient chunks by TMA (zero fill past N); a
        // gradient chunk with no incoming gradient is only handed over.
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();   // each chunk is read once
            bool ok = true;
            int slot = 0, issued = 0, gi = 0;
            uint32_t phase = 0;
            for (int j = 0; j < n_items && ok; ++j) {
                const int qi = item_qi(j), bhq = item_bhq(j);
                for (int idx = 0; idx < res_per_item; ++idx, ++gi) {
                    if (gi >= kResSlots) ok = mbar_wait(bar(C::kBarResFree + slot), phase ^ 1u, ac);
                    if (!ok) break;
                    const bool is_bias = idx < res_bias;
                    const int c = res_chunk_at(is_bias ? idx : idx - res_bias);
                    const uint32_t full = bar(C::kBarResFull + slot);
                    const CUtensorMap *map = is_bias ? &tmBias : (p.has_gin ? &tmGin : nullptr);
                    if (map) {
                        mbar_arrive_expect_tx(full, kResChunkBytes);
                        for (int bx = 0; bx < kTile / kResQ; ++bx)
                            tma_load_3d_hint(sb + C::kOffRes + slot * kResChunkBytes +
                                                 bx * (kResQ * 128),
                                             map, full, kt * kTile + bx * kResQ,
                                             qi * kTile + c * kResQ, bhq, pol);
                    } else {
                        mbar_arrive(full);
                    }
                    issued = gi + 1;
                    if (++slot == kResSlots) { slot = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                for (int x = max(issued - kResSlots, 0); x < issued; ++x)
                    drain_wait(bar(C::kBarResFull + x % C::kResRing),
                               static_cast<uint32_t>(x / C::kResRing) & 1u);
            }
        }
        __syncwarp();
    } else if (RES && warp == 15) {
        // ---------------------------------- outgoing logit-gradient storer
        // Gradient chunks only (bias chunks go back to the loader straight
        // from the warpgroup that read them): wait until the chunk is
        // written, store it (when an outgoing gradient is wanted), and hand
        // the slot back once the store has read it.  The chunk sequence of
        // an item puts its gradient chunks in slots 0..3 (after the bias
        // chunks in 0..3, if any), so each slot's Done barrier completes once
        // per item.
        if (lane == 0 && res_grad) {
            const uint64_t pol = l2_policy_evict_first();   // written once
            bool ok = true;
            for (int j = 0; j < n_items && ok; ++j) {
                const int qi = item_qi(j), bhq = item_bhq(j);
                for (int pos = 0; pos < kResChunks; ++pos) {
                    const int c = res_chunk_at(pos);
                    const int slot = (j * res_per_item + res_bias + pos) % kResSlots;
                    if (!(ok = mbar_wait(bar(C::kBarResDone + slot), j & 1, ac))) break;
                    if (p.has_gout) {
                        for (int bx = 0; bx < kTile / kResQ; ++bx)
                            tma_store_3d_hint(&tmGout,
                                              sb + C::kOffRes + slot * kResChunkBytes +
                                                  bx * (kResQ * 128),
                                              kt * kTile + bx * kResQ, qi * kTile + c * kResQ, bhq,
                                              pol);
                        tma_store_commit();
                        tma_store_wait_read();
                    }
                    mbar_arrive_n(bar(C::kBarResFree + slot), kTile);
                }
            }
            tma_store_wait_read();
        }
        __syncwarp();
    } else if (warp >= 8 && warp < 12) {
        // ------------------------------------------------ dQ drain warpgroup
        if constexpr (RES) {
            // dQ(j) goes from TMEM straight into the fp32 accumulator with vector
            // reductions, so no shared memory holds it and the {Q, dO} stage (the
            // only one in this variant) is released as soon as the item's MMAs
            // are done (the MMA thread commits it).  The 16x256b load shape hands four consecutive threads one
            // 32-byte piece of a query row, so each red.global.add.v2.f32 of a
            // warp adds 8 whole sectors -- the same L2 work per byte as a TMA
            // reduction.  Warp 8 + w drains query rows 32w .. 32w + 31 (its TMEM
            // lanes) in two halves of 16; the TMEM columns are handed back after
            // the second half's load, before its reductions are issued.
            constexpr int kUnits = D / 8;
            const int wq = warp - 8;
            const int r_in = lane >> 2;          // row within a half (and + 8)
            const int c_in = 2 * (lane & 3);     // first of the thread's two columns in a unit
            for (int j = 0; j < n_items; ++j) {
                const bool got = mbar_wait_warp(bar(C::kBarDQFull), j & 1, ac);
                // All four drain warps leave together.
                if (named_bar_or(2, kTile, !got)) break;
                tc_fence_after();
                const int qi = item_qi(j), bhq = item_bhq(j);
                float *rows = p.dq_acc + (static_cast<size_t>(bhq) * p.N + qi * kTile) * D;
                const int valid = p.N - qi * kTile;   // rows of this tile inside N
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t v[4 * kUnits];
                    const int r0 = 32 * wq + 16 * hf + r_in;
                    tmem_ld_16x256b<kUnits>(
                        tmem + (static_cast<uint32_t>(32 * wq + 16 * hf) << 16) + C::kColDP, v);
                    if (hf == 1) {
                        tc_fence_before();
                        mbar_arrive(bar(C::kBarDQEmpty));   // TMEM columns of dQ are free
                    }
#pragma unroll
                    for (int u = 0; u < kUnits; ++u) {
                        if (r0 < valid)
                            red_add_v2_f32(rows + static_cast<size_t>(r0) * D + 8 * u + c_in,
                                           v[4 * u], v[4 * u + 1]);
                        if (r0 + 8 < valid)
                            red_add_v2_f32(rows + static_cast<size_t>(r0 + 8) * D + 8 * u + c_in,
                                           v[4 * u + 2], v[4 * u + 3]);
                    }
                }
            }
        } else {
            // dQ(j) is staged as fp32, 128-byte swizzled boxes of 32 columns --
            // boxes 0 and 1 in the dS buffer, the rest in item j's dO buffer,
            // both free once item j's MMAs are done (Q's buffer is not used, so
            // the next Q tile can load at once) -- and added into the fp32
            // accumulator with TMA bulk reductions.  Each warp stages its own
            // 32 query rows and reduces them with 32-row boxes, so the warps
            // never wait on one another.  The dS buffer is handed back first
            // (the P / dS warpgroups write the next dS there), then the dO
            // buffer (the producer loads a later dO there).  The TMEM columns
            // go back right after the last TMEM load (the next dP^T waits on
            // them).
            constexpr int kDsBoxes = C::kDQBoxes < 2 ? C::kDQBoxes : 2;
            const int qr = threadIdx.x - 256;
            const int wq = warp - 8;
            const uint32_t tDQ = tmem + (static_cast<uint32_t>(wq * 32) << 16) + C::kColDP;
            const uint32_t sDS = sb + C::kOffDS;
            for (int j = 0; j < n_items; ++j) {
                const int s = j % C::kQStages;
                const bool got = mbar_wait_warp(bar(C::kBarDQFull), j & 1, ac);
                // All four drain warps leave together.
                if (named_bar_or(2, kTile, !got)) break;
                tc_fence_after();
                const uint32_t sDO = sb + C::kOffStage + s * C::kStageBytes + C::kTileBytes;
                auto box_at = [&](int bx) -> uint32_t {
                    return bx < kDsBoxes ? sDS + bx * (kTile * 128)
                                         : sDO + (bx - kDsBoxes) * (kTile * 128);
                };
#pragma unroll
                for (int c = 0; c < C::kDQBoxes; c += 2) {
                    // Two 32-column boxes per 64-column load; a last odd box
                    // (D = 80, 96) takes a 32-column load, whose columns past D
                    // are clipped by the reduction.
                    constexpr int kPair = 2;
                    uint32_t rr[64];
                    const int nb = (c + 1 < C::kDQBoxes) ? kPair : 1;
                    if (nb == 2) tmem_ld64(tDQ + c * 32, rr);
                    else tmem_ld32(tDQ + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&rr[0]));
                    if (c + 2 >= C::kDQBoxes) {
                        tc_fence_before();
                        mbar_arrive(bar(C::kBarDQEmpty));   // TMEM columns of dQ are free
                    }
#pragma unroll
                    for (int hb = 0; hb < kPair; ++hb) {
                        if (hb >= nb) break;
                        const uint32_t box = box_at(c + hb) + qr * 128;
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch) {
                            const int e = hb * 32 + ch * 4;
                            st_shared_v4(box + (static_cast<uint32_t>(ch ^ (qr & 7)) << 4), rr[e],
                                         rr[e + 1], rr[e + 2], rr[e + 3]);
                        }
                    }
                    // Boxes 0 and 1 (the dS buffer) are reduced first, while
                    // the rest is loaded and staged; each box group is one
                    // bulk group of this warp's lane 0.
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const int row0 = item_qi(j) * kTile + wq * 32;
                        if (row0 < p.N) {   // (rows past N are clipped by the reduction)
                            for (int bx = c; bx < c + nb; ++bx)
                                tma_reduce_add_3d(&tmDQ, box_at(bx) + wq * (32 * 128), bx * 32,
                                                  row0, item_bhq(j));
                        }
                        tma_store_commit();
                    }
                }
                if (lane == 0) {
                    if constexpr (C::kDQBoxes <= 2) tma_store_commit();   // (no second group)
                    tma_store_wait_read_n<1>();
                    mbar_arrive(bar(C::kBarDSFree));          // this warp's dS-buffer part is read
                    tma_store_wait_read();
                    mbar_arrive(bar(C::kBarDOEmpty + s));     // and its dO-buffer part
                }
                __syncwarp();
            }
        }
        // Meet the P / dS warpgroups before their dK/dV epilogue (with the
        // staged drain: once its last reduction has read stage 0).
        named_bar_sync(3, 3 * kTile);
    } else {
        // ---------------------------------------- two P / dS warpgroups
        // Warpgroup w (warps 4w..4w+3) owns query columns 64w..64w+63; thread
        // kr is key row kr (TMEM lane kr).
        const int w = warp >> 2;
        const int kr = threadIdx.x & 127;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_base + C::kColS + w * 64;
        const uint32_t tDP = tmem + lane_base + C::kColDP + w * 64;
        const uint32_t sDS = sb + C::kOffDS;
        const uint64_t sc2 = f2pack(p.scale_log2, p.scale_log2);
        const uint64_t sm2 = f2pack(p.scale, p.scale);
        const uint64_t l2e2 = f2pack(kLog2e, kLog2e);
        // Four LSE or Delta values (the same for every key row, so a
        // broadcast).  As plain C++ loads the compiler may issue them ahead of
        // the arithmetic that needs them (the barrier waits before each phase
        // still order them after the TMA writes); that measured 9% faster on
        // long causal problems.  The residual variant, whose loop also reads
        // the bias, measured slower that way and keeps the in-order loads.
        auto ld_rows_f4 = [&](uint32_t addr) -> float4 {
            if constexpr (RES) return ld_shared_f4(addr);
            else return *reinterpret_cast<const float4 *>(smem + (addr - sb));
        };
        // Offsets of key row kr inside a residual chunk (four 32-key boxes,
        // 128-byte rows of 32 fp32, 16-byte pieces swizzled by row % 8).
        const uint32_t res_koff = (kr / kResQ) * (kResQ * 128) + (kr % 4) * 4;
        const int res_kpiece = (kr % kResQ) / 4;
        bool ok = true;
        for (int j = 0; j < n_items; ++j) {
            const int s = j % C::kQStages;
            // --- P^T(j) = 2^(S^T scale log2e - LSE log2e), bf16 into TMEM over S^T
            ok = mbar_wait_warp(bar(C::kBarSFull), j & 1, ac);
            if (ok) ok = mbar_wait_warp(bar(C::kBarQFull + s), (j / C::kQStages) & 1, ac);
            if (!ok) break;
            tc_fence_after();
            const bool diag = CAUSAL && (item_qi(j) == kt);
            // Some query column of the tile lies W or more rows past some key row.
            const int qoff = (item_qi(j) - kt) * kTile;   // query row - key row offset of the tiles
            const bool wedge = CAUSAL && p.window > 0 && qoff + kTile - 1 >= p.window;
            const int rs = RES ? (j & 1) : s;   // row slot (the residual variant alternates)
            const uint32_t s_lse = s_rows + rs * kTile * 4 + w * 256;
            const uint32_t s_dlt = s_rows + (2 + rs) * kTile * 4 + w * 256;
            uint32_t pw[32];   // P^T of this warpgroup's 64 columns, bf16 pairs
            // Residual chunks of this warpgroup: query columns 64w + 32h .. +31
            // are chunk 2w + h of the bias and of the logit gradient.
            uint32_t bslot[2] = {0u, 0u}, gslot[2] = {0u, 0u};
            int bsi[2] = {0, 0}, gsi[2] = {0, 0};
            if constexpr (RES) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int gb = j * res_per_item + 2 * h + w;   // position of chunk 2w + h
                    const int gg = gb + res_bias;
                    bsi[h] = gb % kResSlots;
                    gsi[h] = gg % kResSlots;
                    bslot[h] = sb + C::kOffRes + bsi[h] * kResChunkBytes + res_koff;
                    gslot[h] = sb + C::kOffRes + gsi[h] * kResChunkBytes + res_koff;
                    if (res_bias && ok)
                        ok = mbar_wait_warp(bar(C::kBarResFull + bsi[h]),
                                            static_cast<uint32_t>(gb / kResSlots) & 1u, ac);
                }
                if (!ok) break;
            }
            {
                uint32_t sr[64];
                tmem_ld64(tS, sr);
#pragma unroll
                for (int c = 0; c < 64; c += 4) {
                    const float4 l4 = ld_rows_f4(s_lse + c * 4);
#pragma unroll
                    for (int u = 0; u < 4; u += 2) {
                        const float la = u == 0 ? l4.x : l4.z, lb = u == 0 ? l4.y : l4.w;
                        float t0, t1;
                        uint64_t off2 = f2pack(-la, -lb);   // -LSE log2e
                        if constexpr (RES) {
                            if (res_bias) {   // + bias log2e, read transposed from the chunk
                                const int rq = (c + u) % kResQ;
                                const uint32_t ba = bslot[(c + u) / kResQ] + rq * 128;
                                const float b0 = ld_shared_f32(
                                    ba + (static_cast<uint32_t>(res_kpiece ^ (rq & 7)) << 4));
                                const float b1 = ld_shared_f32(
                                    ba + 128 + (static_cast<uint32_t>(res_kpiece ^ ((rq + 1) & 7)) << 4));
                                off2 = ffma2(f2pack(b0, b1), l2e2, off2);
                            }
                        }
                        f2unpack(ffma2(f2pack(__uint_as_float(sr[c + u]), __uint_as_float(sr[c + u + 1])),
                                       sc2, off2), t0, t1);
                        float p0 = ex2(t0), p1 = ex2(t1);
                        if (diag || wedge) {
                            // kept iff 0 <= query - key < W (no upper limit without a window)
                            const int dq0 = qoff + w * 64 + c + u - kr;
                            const int wl = wedge ? p.window : (1 << 30);
                            p0 = (dq0 >= 0 && dq0 < wl) ? p0 : 0.f;
                            p1 = (dq0 + 1 >= 0 && dq0 + 1 < wl) ? p1 : 0.f;
                        }
                        pw[(c + u) >> 1] = pack_bf16x2(p0, p1);
                    }
                    if constexpr (RES) {
                        // First bias chunk (columns 0..31) read: back to the loader.
                        if (c == kResQ - 4 && res_bias) mbar_arrive(bar(C::kBarResFree + bsi[0]));
                    }
                }
            }
            tmem_st32(tS, pw);   // columns 64w..64w+31, already read
            if constexpr (RES) {
                if (res_bias) mbar_arrive(bar(C::kBarResFree + bsi[1]));   // second bias chunk
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(C::kBarPReady));

            // --- dS^T(j) = P^T o (dP^T - Delta) * scale, bf16 into smem
            ok = mbar_wait_warp(bar(C::kBarDPFull), j & 1, ac);
            if (ok && j > 0) ok = mbar_wait_warp(bar(C::kBarDSFree), (j - 1) & 1, ac);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if constexpr (RES) {
                    if (res_grad && !mbar_wait_warp(bar(C::kBarResFull + gsi[h]),
                                                    static_cast<uint32_t>(
                                                        (j * res_per_item + res_bias + 2 * h + w) /
                                                        kResSlots) & 1u,
                                                    ac)) {
                        ok = false;
                        break;
                    }
                }
                uint32_t dr[32];
                tmem_ld32(tDP + h * 32, dr);
#pragma unroll
                for (int c = 0; c < 32; c += 8) {   // one 16-byte chunk of the dS^T row
                    const int cc = h * 32 + c;
                    const float4 da = ld_rows_f4(s_dlt + cc * 4);
                    const float4 db = ld_rows_f4(s_dlt + cc * 4 + 16);
                    const float dv[8] = {da.x, da.y, da.z, da.w, db.x, db.y, db.z, db.w};
                    uint32_t wv[4];
#pragma unroll
                    for (int u = 0; u < 8; u += 2) {
                        float e0, e1;   // dP - Delta
                        f2unpack(fadd2(f2pack(__uint_as_float(dr[c + u]), __uint_as_float(dr[c + u + 1])),
                                       f2pack(-dv[u], -dv[u + 1])), e0, e1);
                        // P as rounded to bf16 for the dV MMA (the same values in both).
                        const float2 pp = __bfloat1622float2(
                            *reinterpret_cast<const __nv_bfloat162 *>(&pw[(cc + u) >> 1]));
                        float d0, d1;
                        if constexpr (RES) {
                            // total logit gradient: P (dP - Delta) + incoming, 0 where masked
                            f2unpack(fmul2(f2pack(pp.x, pp.y), f2pack(e0, e1)), d0, d1);
                            const int rq = c + u;   // query row within chunk h
                            const uint32_t ga0 = gslot[h] + rq * 128 +
                                                 (static_cast<uint32_t>(res_kpiece ^ (rq & 7)) << 4);
                            const uint32_t ga1 = gslot[h] + (rq + 1) * 128 +
                                                 (static_cast<uint32_t>(res_kpiece ^ ((rq + 1) & 7)) << 4);
                            if (res_grad && p.has_gin) {
                                d0 += ld_shared_f32(ga0);
                                d1 += ld_shared_f32(ga1);
                            }
                            if (diag || wedge) {
                                const int dq0 = qoff + w * 64 + cc + u - kr;
                                const int wl = wedge ? p.window : (1 << 30);
                                d0 = (dq0 >= 0 && dq0 < wl) ? d0 : 0.f;
                                d1 = (dq0 + 1 >= 0 && dq0 + 1 < wl) ? d1 : 0.f;
                            }
                            if (res_grad && p.has_gout) {
                                st_shared_f32(ga0, d0);
                                st_shared_f32(ga1, d1);
                            }
                            wv[u >> 1] = pack_bf16x2(d0 * p.scale, d1 * p.scale);
                        } else {
                            f2unpack(fmul2(fmul2(f2pack(pp.x, pp.y), f2pack(e0, e1)), sm2), d0, d1);
                            wv[u >> 1] = pack_bf16x2(d0, d1);
                        }
                    }
                    const int chunk = cc >> 3;     // 16-byte chunk within the 64-query atom
                    st_shared_v4(sDS + w * (kTile * 128) + kr * 128 +
                                     (static_cast<uint32_t>(chunk ^ (kr & 7)) << 4),
                                 wv[0], wv[1], wv[2], wv[3]);
                }
                if constexpr (RES) {
                    if (res_grad) {   // chunk h done: written back for the storer
                        if (p.has_gout) fence_proxy_async_smem();
                        mbar_arrive(bar(C::kBarResDone + gsi[h]));
                    }
                }
            }
            if (!ok) break;
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(C::kBarDSReady));
        }

        // ------------------------------------------------ epilogue: dK, dV
        // Warpgroup 0 stores dV, warpgroup 1 stores dK (all D columns of each key row).
        if (ok) ok = mbar_wait_warp(bar(C::kBarAccDone), 0, ac);
        named_bar_sync(3, 3 * kTile);   // the drain warps are done
        const uint32_t stV = sb + C::kOffStage;                  // stage 0 Q buffer
        const uint32_t stK = sb + C::kOffStage + C::kTileBytes;  // stage 0 dO buffer
        if (p.hsplit > 1) {
            // Partial sums over this block's query heads: fp32 boxes of 32
            // columns (as the dQ drain), added into the accumulators by TMA.
            // With two stages dV and dK stage at once, else one after the other.
            constexpr int kRounds = C::kQStages >= 2 ? 1 : 2;
            for (int rd = 0; rd < kRounds; ++rd) {
                const uint32_t dst = sb + C::kOffStage + (kRounds == 1 ? w * C::kStageBytes : 0);
                if (ok && (kRounds == 1 || rd == w)) {
                    tc_fence_after();
                    const uint32_t tacc = tmem + lane_base + (w == 0 ? C::kColDV : C::kColDK);
#pragma unroll
                    for (int c = 0; c < C::kDQBoxes; c += 2) {
                        uint32_t rr[64];
                        const int nb = (c + 1 < C::kDQBoxes) ? 2 : 1;
                        if (nb == 2) tmem_ld64(tacc + c * 32, rr);
                        else tmem_ld32(tacc + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&rr[0]));
#pragma unroll
                        for (int hb = 0; hb < 2; ++hb) {
                            if (hb >= nb) break;
                            const uint32_t box = dst + (c + hb) * (kTile * 128) + kr * 128;
#pragma unroll
                            for (int ch = 0; ch < 8; ++ch) {
                                const int e = hb * 32 + ch * 4;
                                st_shared_v4(box + (static_cast<uint32_t>(ch ^ (kr & 7)) << 4),
                                             rr[e], rr[e + 1], rr[e + 2], rr[e + 3]);
                            }
                        }
                    }
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                named_bar_sync(1, 2 * kTile);
                if (threadIdx.x == 0 && *abort_flag == 0) {
                    for (int t2 = 0; t2 < 2; ++t2) {
                        if (kRounds == 2 && t2 != rd) continue;
                        const uint32_t src = sb + C::kOffStage + (kRounds == 1 ? t2 * C::kStageBytes : 0);
                        for (int bx = 0; bx < C::kDQBoxes; ++bx)
                            tma_reduce_add_3d(t2 == 0 ? &tmdV : &tmdK, src + bx * (kTile * 128),
                                              bx * 32, kt * kTile, bh_kv);
                    }
                    tma_store_commit();
                    tma_store_wait_read();
                }
                named_bar_sync(1, 2 * kTile);   // staging read before it is reused
            }
        } else {
        if (ok) {
            tc_fence_after();
            const uint32_t col = w == 0 ? C::kColDV : C::kColDK;
            const uint32_t dst = w == 0 ? stV : stK;
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c) {   // columns past D are clipped by the store
                uint32_t rr[64];
                tmem_ld64(tmem + lane_base + col + c * 64, rr);
                uint32_t wv[32];
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    wv[e] = pack_bf16x2(__uint_as_float(rr[2 * e]), __uint_as_float(rr[2 * e + 1]));
                stage_row64(dst, kr, c, wv);
            }
            fence_proxy_async_smem();
        }
        tc_fence_before();
        named_bar_sync(1, 2 * kTile);
        if (threadIdx.x == 0 && *abort_flag == 0) {
            for (int c = 0; c < C::kChunks; ++c) {
                tma_store_3d(&tmdV, stV + c * C::kChunkBytes, c * 64, kt * kTile, bh_kv);
                tma_store_3d(&tmdK, stK + c * C::kChunkBytes, c * 64, kt * kTile, bh_kv);
            }
            tma_store_commit();
            tma_store_wait_read();
        }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 13) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, bool RES>
cudaError_t launch_main(const CUtensorMap (&m)[10], const BwdParams &prm, dim3 grid,
                        bool causal, cudaStream_t stream) {
    using C = BwdCfg<D, RES>;
    auto kern = causal ? bwd_main_kernel<D, true, RES> : bwd_main_kernel<D, false, RES>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, bwd_threads<RES>(), C::kSmemBytes, stream>>>(m[0], m[1], m[2], m[3], m[4], m[5],
                                                              m[6], m[7], m[8], m[9], prm);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const BwdProblem &pb, int *status, cudaStream_t stream) {
    const long long BH = static_cast<long long>(pb.B) * pb.Hq;
    const long long BHkv = static_cast<long long>(pb.B) * pb.Hkv;
    const int n_tiles = pb.NP / kTile;

    // The host work (device queries, tensor maps) comes first and the three
    // launches back to back, so that the GPU does not wait between them.
    cudaError_t e = cudaSuccess;

    // Main kernel maps: q, k, v, dO, dK, dV, dQ accumulator, bias, incoming and outgoing
    // logit gradients (the last three: [B*Hq, N query rows, N keys] fp32 in
    // 32 x 32 boxes; a map of the first given one stands in for absent ones).
    CUtensorMap m[10];
    if (!encode_bf16_rows(&m[0], pb.q, D, pb.N, BH, kTile) ||
        !encode_bf16_rows(&m[1], pb.k, D, pb.N, BHkv, kTile) ||
        !encode_bf16_rows(&m[2], pb.v, D, pb.N, BHkv, kTile) ||
        !encode_bf16_rows(&m[3], pb.dO, D, pb.N, BH, kTile) ||
        !encode_bf16_rows(&m[4], pb.dk, D, pb.N, BHkv, kTile) ||
        !encode_bf16_rows(&m[5], pb.dv, D, pb.N, BHkv, kTile) ||
        !encode_f32_rows(&m[6], pb.dq_acc, D, pb.N, BH, 32))   // one drain warp's 32 rows
        return cudaErrorInvalidValue;
    const bool res = pb.bias || pb.grad_in || pb.grad_out;
    // Split a key tile's query heads over blocks when the grid would
    // otherwise leave SMs idle or run a few long blocks (grouped heads only).
    DeviceInfo di;
    if (!device_info(&di)) return cudaErrorInvalidValue;
    const int sms = di.sms;
    const int group = pb.Hq / pb.Hkv;
    const int hsplit =
        (group > 1 && pb.dk_acc && static_cast<long long>(n_tiles) * BHkv < 2LL * sms) ? group : 1;
    if (hsplit > 1) {
        // dK, dV through fp32 accumulators: zero them, map them in place of
        // the bf16 outputs, convert at the end.
        const size_t n_kv = static_cast<size_t>(BHkv) * pb.N * D;
        const size_t span = static_cast<size_t>(pb.dv_acc - pb.dk_acc) + n_kv;
        bwd_zero_kernel<<<static_cast<unsigned>(std::min<size_t>((span / 4 + 255) / 256, 152 * 8)),
                          256, 0, stream>>>(reinterpret_cast<float4 *>(pb.dk_acc), span / 4);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        if (!encode_f32_rows(&m[4], pb.dk_acc, D, pb.N, BHkv, kTile) ||
            !encode_f32_rows(&m[5], pb.dv_acc, D, pb.N, BHkv, kTile))
            return cudaErrorInvalidValue;
    }
    m[7] = m[8] = m[9] = m[6];
    if (res) {
        const float *any = pb.bias ? pb.bias : (pb.grad_in ? pb.grad_in : pb.grad_out);
        const float *src[3] = {pb.bias ? pb.bias : any, pb.grad_in ? pb.grad_in : any,
                               pb.grad_out ? pb.grad_out : any};
        for (int i = 0; i < 3; ++i)
            if (!encode_f32_rows(&m[7 + i], src[i], pb.N, pb.N, BH, kResQ))
                return cudaErrorInvalidValue;
    }
    BwdParams prm;
    prm.lse2 = pb.lse2;
    prm.delta = pb.delta;
    prm.dq_acc = pb.dq_acc;
    prm.status = status;
    prm.N = pb.N;
    prm.NP = pb.NP;
    prm.Hq = pb.Hq;
    prm.Hkv = pb.Hkv;
    prm.group = pb.Hq / pb.Hkv;
    prm.BHkv = static_cast<int>(BHkv);
    prm.n_tiles = n_tiles;
    prm.scale = pb.scale;
    prm.scale_log2 = pb.scale * kLog2e;
    prm.window = pb.causal ? pb.window : 0;
    prm.has_bias = pb.bias != nullptr;
    prm.has_gin = pb.grad_in != nullptr;
    prm.has_gout = pb.grad_out != nullptr;
    prm.hsplit = hsplit;
    // Block order: every kv head's key tile kt before tile kt + 1 while the
    // fp32 dQ accumulator is within twice the L2; past that, chunks of kv
    // heads whose accumulator part is about half the L2, so that the blocks
    // running at once keep theirs resident (measured, D128 causal: B1 H16
    // N65536 50.0 -> 40.9 ms, B4 H16 N16384 13.2 -> 10.7 ms; at B1 H16 N16384
    // and N32768, whose accumulators stay within twice the L2, the same).
    const double l2 = di.l2_bytes;
    const double acc_bytes = static_cast<double>(BH) * pb.N * D * 4.0;
    const double head_bytes = static_cast<double>(prm.group) * pb.N * D * 4.0;   // per kv head
    prm.hchunk = static_cast<int>(BHkv);
    // Chunked once the accumulator is over half the L2: a chunk's
    // accumulator takes a quarter of it, beside the chunk's Q and dO (as
    // large again in bf16), so that its reduce-adds stay in L2.  (Measured at
    // B1 H16 N16384 D128: DRAM traffic 2.9 GB -> 0.66 GB, 1.2x the
    // algorithmic bytes, time +1%; at B4 H32 N4096 D128: 22% faster.)
    if (acc_bytes > 0.5 * l2) {
        // (a divisor of the kv head count: every chunk is whole)
        long long hc = std::max<long long>(1, std::min<long long>(BHkv, static_cast<long long>(0.25 * l2 / head_bytes)));
        while (BHkv % hc != 0) --hc;
        // The chunks are gridDim.y (at most 65535); a head count with no
        // divisor near the target keeps the plain order.
        if (BHkv / hc <= 65535) prm.hchunk = static_cast<int>(hc);
    }
    // 1. Delta, LSE*log2(e), zeroed dQ accumulator.
    bwd_pre_kernel<D><<<static_cast<unsigned>(BH * n_tiles), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(pb.o), static_cast<const __nv_bfloat16 *>(pb.dO),
        pb.lse, pb.lse2, pb.delta, pb.dq_acc, pb.N, pb.NP, n_tiles);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // 2. x: key tiles (heaviest first) x the chunk's kv heads x head splits;
    // y: chunks of kv heads.
    const long long n_chunks = BHkv / prm.hchunk;
    const dim3 grid(static_cast<unsigned>(static_cast<long long>(n_tiles) * prm.hchunk * hsplit),
                    static_cast<unsigned>(n_chunks));
    e = res ? launch_main<D, true>(m, prm, grid, pb.causal, stream)
            : launch_main<D, false>(m, prm, grid, pb.causal, stream);
    if (e != cudaSuccess) return e;

    // 3. fp32 dQ accumulator -> bf16 dQ (and dK, dV when they were split).
    const size_t n8 = static_cast<size_t>(BH) * pb.N * D / 8;
    const unsigned blocks = static_cast<unsigned>(std::min<size_t>((n8 + 255) / 256, 152 * 16));
    bwd_dq_kernel<<<blocks, 256, 0, stream>>>(pb.dq_acc, static_cast<__nv_bfloat16 *>(pb.dq), n8);
    if (hsplit > 1) {
        const size_t k8 = static_cast<size_t>(BHkv) * pb.N * D / 8;
        const unsigned kb = static_cast<unsigned>(std::min<size_t>((k8 + 255) / 256, 152 * 16));
        bwd_dq_kernel<<<kb, 256, 0, stream>>>(pb.dk_acc, static_cast<__nv_bfloat16 *>(pb.dk), k8);
        bwd_dq_kernel<<<kb, 256, 0, stream>>>(pb.dv_acc, static_cast<__nv_bfloat16 *>(pb.dv), k8);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdProblem &pb, int *status, cudaStream_t stream) {
    if (pb.D == 64) return launch_d<64>(pb, status, stream);
    if (pb.D == 80) return launch_d<80>(pb, status, stream);
    if (pb.D == 96) return launch_d<96>(pb, status, stream);
    return launch_d<128>(pb, status, stream);
}

}  // namespace tattn
