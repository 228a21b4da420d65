/*
 * tattn.h -- C ABI of the tiled exact-attention library for GB300 (sm_103a).
 *
 * The library computes exact attention
 *
 *     O = softmax(scale * Q K^T  [+ bias]  [+ causal mask]) V
 *
 * tile by tile with an online softmax, so that the N x N score and
 * probability matrices never reach device memory, and saves one fp32
 * log-sum-exp per query row for a backward pass that recomputes the
 * probabilities from it.
 *
 * Sources of the operations (page title and section):
 *  - Standard attention S = QK^T / sqrt(d), P = softmax(S), O = PV and the
 *    N x N intermediates it materialises: "FlashAttention原理与Triton实战：
 *    突破Attention显存瓶颈", sections 1 and 2.1; kwkr.cn/news/592482, 1.1.
 *  - Online softmax block merge (m_new = max(m_old, m_blk), alpha =
 *    exp(m_old - m_new), l and O rescaled by alpha, divide by l at the end)
 *    and the tiled double loop: kwkr.cn/news/592482, 2.2 and 2.3.
 *  - Causal mask (key j kept for query i iff j <= i): kwkr.cn/news/592482,
 *    3.3 and 3.4; blog.ans20xx.com/posts/ai/day26, "最小 attention wrapper".
 *  - Sliding-window mask: see attn_fwd_window.
 *  - Additive pre-softmax logit bias read from the previous layer and the
 *    logits emitted for the next layer (block attention residual):
 *    Block Attention Residual Triton kernel (iqiancheng.github.io), sections
 *    "Block Attention Residual 做了什么" and "v1: Fuse Residual 进 Attention
 *    Kernel", "v2: 优化 torch.cat + SRAM 复用".
 *  - Backward by recomputation from saved row statistics:
 *    kwkr.cn/news/592482, 2.4; "FlashAttention原理与Triton实战", 2.3 and 4.3.
 *
 * Conventions shared by every entry point
 *  - Tensors are dense, contiguous, row-major:
 *      q, o, dO, dq : bf16 [B, Hq,  N, D]
 *      k, v, dk, dv : bf16 [B, Hkv, N, D]
 *      lse          : fp32 [B, Hq,  N]
 *      bias, logits : fp32 [B, Hq,  N, N]
 *  - Grouped heads: query head h reads key/value head h / (Hq / Hkv);
 *    Hq must be a multiple of Hkv (Hkv == Hq is plain multi-head).
 *  - D must be 64, 80, 96 or 128.  N, B, Hq, Hkv are any positive sizes (N need not
 *    be a multiple of the 128-row tile); a zero size is an empty problem and
 *    returns ATTN_OK without launching anything.
 *  - Every tensor pointer is a DEVICE pointer of the current CUDA device,
 *    owned by the caller; bf16 tensors must be 16-byte aligned, fp32 tensors
 *    4-byte aligned.  The library allocates no device memory for its
 *    kernels; the backward takes its scratch from a caller-provided
 *    workspace.  The only device state is one small status word per device,
 *    whose address is looked up once per device and cached: the library
 *    works in each device's primary context and does not support calls
 *    after cudaDeviceReset (or another teardown of that context).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls are asynchronous and stream-ordered: they return after
 *    the launches are queued.
 *  - Arguments are checked on the host before anything is launched; a bad
 *    argument returns ATTN_ERR_INVALID (or ATTN_ERR_UNSUPPORTED for a valid
 *    but unimplemented case) and touches no memory.  Sizes are limited by
 *    B*Hq*ceil(N/128) <= 2^31 - 1 (ATTN_ERR_UNSUPPORTED past it); within
 *    that bound every launch fits the grid limits.  A launch failure
 *    returns ATTN_ERR_CUDA.  Faults found on the device (a pipeline wait
 *    that ran out of time, a failed device-side check) do not trap: the
 *    kernel records a code in the status word and returns; read it with
 *    attn_last_device_status().
 */
#ifndef TATTN_H
#define TATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID = 1,      /* null/misaligned pointer, bad size or shape      */
    ATTN_ERR_UNSUPPORTED = 2,  /* valid request outside what is implemented       */
    ATTN_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed               */
    ATTN_ERR_TIMEOUT = 4,      /* a device pipeline wait exceeded its time limit  */
    ATTN_ERR_DEVICE_CHECK = 5  /* a device-side consistency check failed          */
} attn_status;

/*
 * Forward pass.
 *
 *   q            bf16 [B,Hq,N,D]   queries                          (in)
 *   k, v         bf16 [B,Hkv,N,D]  keys, values                     (in)
 *   bias         fp32 [B,Hq,N,N]   additive logit bias, or NULL     (in)
 *                Added, unscaled, to scale*QK^T before the mask and the
 *                softmax (the previous layer's pre-softmax logits in a
 *                block attention residual).  Under the causal mask the
 *                entries with j > i do not affect any result; the 128 x 128
 *                tiles strictly above the diagonal are never read, while
 *                entries above the diagonal inside the tiles that straddle
 *                it may be read.
 *   o            bf16 [B,Hq,N,D]   output, rounded to nearest even  (out)
 *   lse          fp32 [B,Hq,N]     LSE_i = m_i + ln l_i over the scaled,
 *                biased, masked logits (natural log), or NULL       (out)
 *   scale        multiplier of QK^T (usually 1/sqrt(D)); must be finite.
 *   causal       nonzero: key j is kept for query i iff j <= i.
 *   emit_logits  fp32 [B,Hq,N,N] or NULL                            (out)
 *                Receives s_ij = scale*q_i.k_j + bias_ij (bias term absent
 *                when bias is NULL) for every kept entry; under the causal
 *                mask, tiles strictly above the diagonal are not written and
 *                masked entries inside diagonal tiles hold unspecified
 *                values.  MAY be the same pointer as bias (in-place update
 *                of a preallocated residual buffer): each bias element is
 *                read by the only thread block that later overwrites it.
 *                Any other overlap between outputs and inputs is invalid.
 *
 * Returns ATTN_OK once the kernel is queued on `stream`.
 */
attn_status attn_fwd(const void *q, const void *k, const void *v, const float *bias,
                     void *o, float *lse,
                     int B, int Hq, int Hkv, int N, int D, float scale, int causal,
                     float *emit_logits, void *stream);

/*
 * Forward pass with a causal sliding window.
 *
 * The pages name a window mask stacked on the causal kernel
 * ("FlashAttention原理与Triton实战", sections 3.1 and 7) and a sliding-window
 * (SWA) baseline model (Block Attention Residual page, "实验结果"), without a
 * formula.  Here, key j is kept for query i iff  i - window < j <= i : the
 * `window` most recent keys, the query's own included.  window >= N is the
 * plain causal mask.
 *
 * Arguments, layouts, ownership and errors are those of attn_fwd with
 * causal = 1, plus:
 *   window       sliding-window length W >= 1 (ATTN_ERR_INVALID otherwise).
 * Only the 128 x 128 key tiles that hold a kept key are read (bias) or
 * written (emit_logits); masked entries inside those tiles hold
 * unspecified emitted values.
 */
attn_status attn_fwd_window(const void *q, const void *k, const void *v, const float *bias,
                            void *o, float *lse,
                            int B, int Hq, int Hkv, int N, int D, float scale, int window,
                            float *emit_logits, void *stream);

/*
 * Bytes of device workspace attn_bwd needs for this shape: an fp32 dQ
 * accumulator [B,Hq,N,D], plus two fp32 per-row arrays [B*Hq, NP]
 * (NP = N rounded up to a multiple of 128) holding LSE*log2(e) and
 * Delta_i = sum_d dO_id O_id, plus, with grouped heads (Hq > Hkv), fp32 dK
 * and dV accumulators [B,Hkv,N,D] (used when a key tile's query heads are
 * split over several thread blocks); each region rounded up to 256 bytes.
 * Returns 0 for an empty problem or invalid sizes.
 */
size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int N, int D);

/*
 * Backward pass by recomputation (no bias; the forward must have been run
 * without bias on the same q, k, v, scale and causal setting).
 *
 *   q, k, v      as for attn_fwd                                    (in)
 *   o            bf16 [B,Hq,N,D]  forward output                    (in)
 *   lse          fp32 [B,Hq,N]    forward log-sum-exp               (in)
 *   dO           bf16 [B,Hq,N,D]  gradient of the loss w.r.t. O     (in)
 *   dq           bf16 [B,Hq,N,D]                                    (out)
 *   dk, dv       bf16 [B,Hkv,N,D] (summed over each kv head's query
 *                heads when Hq > Hkv)                               (out)
 *   workspace    device scratch of at least attn_bwd_workspace_size()
 *                bytes, 256-byte aligned, owned by the caller; its contents
 *                on entry do not matter and are clobbered.
 *
 * Computes P_ij = exp(scale q_i.k_j - LSE_i), dV = P^T dO, dP = dO V^T,
 * Delta_i = sum_d dO_id O_id, dS = P o (dP - Delta), dQ = scale dS K,
 * dK = scale dS^T Q.
 */
attn_status attn_bwd(const void *q, const void *k, const void *v, const void *o,
                     const float *lse, const void *dO,
                     void *dq, void *dk, void *dv,
                     int B, int Hq, int Hkv, int N, int D, float scale, int causal,
                     void *workspace, size_t workspace_bytes, void *stream);

/*
 * Backward pass of one layer of a block attention residual chain.
 *
 * The layer computed  S = scale QK^T + bias  (bias = the previous layer's
 * emitted logits, or none for the first layer of a block) and, when it is
 * not the last layer, emitted S to the next layer, whose own logits add S
 * unscaled.  The gradient reaching S is therefore
 *     dS = P o (dP - Delta) + grad_in
 * (grad_in = the next layer's dS, absent for the last layer); dS gives
 * dq = scale dS K and dk = scale dS^T Q, dv = P^T dO, and dS itself is the
 * gradient of the bias, written to grad_out for the previous layer.  The
 * Block Attention Residual page ("v1: Fuse Residual 进 Attention Kernel")
 * says the backward keeps the LSE statistics, corrected for the residual:
 * lse must be the one attn_fwd returned with this bias.
 *
 *   bias      fp32 [B,Hq,N,N] the forward's bias, or NULL              (in)
 *   grad_in   fp32 [B,Hq,N,N] incoming logit gradient, or NULL         (in)
 *   grad_out  fp32 [B,Hq,N,N] dS on the kept entries, or NULL          (out)
 *             MAY be the same pointer as grad_in (in-place chain buffer):
 *             each element is read by the only thread block that later
 *             writes it.  Under the causal mask, tiles above the diagonal
 *             are not touched; masked entries inside the diagonal tiles
 *             hold unspecified values and are never read as grad_in.
 * Other arguments, layouts, workspace and errors are those of attn_bwd.
 * The residual tensors need 16-byte aligned bases and N % 4 == 0
 * (ATTN_ERR_UNSUPPORTED otherwise).
 */
attn_status attn_bwd_residual(const void *q, const void *k, const void *v, const void *o,
                              const float *lse, const void *dO, const float *bias,
                              const float *grad_in, void *dq, void *dk, void *dv, float *grad_out,
                              int B, int Hq, int Hkv, int N, int D, float scale, int causal,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * Backward pass of attn_fwd_window (same q, k, v, scale and window; no bias).
 * Arguments, workspace, layouts and errors are those of attn_bwd with
 * causal = 1, plus window >= 1 as in attn_fwd_window.
 */
attn_status attn_bwd_window(const void *q, const void *k, const void *v, const void *o,
                            const float *lse, const void *dO,
                            void *dq, void *dk, void *dv,
                            int B, int Hq, int Hkv, int N, int D, float scale, int window,
                            void *workspace, size_t workspace_bytes, void *stream);

/*
 * Size of the fixed device scratch behind attn_bwd_noalloc: 32 MiB.  A shape
 * fits when attn_bwd_workspace_size(B, Hq, Hkv, N, D) is at most this many
 * bytes -- about 64 thousand query rows (B*Hq*N) at D = 128, about 127
 * thousand at D = 64.
 */
#define ATTN_BWD_NOALLOC_SCRATCH_BYTES 33554432

/*
 * attn_bwd without a workspace argument, for callers that cannot allocate
 * device memory.  The pages have no counterpart to this entry point; it is
 * an addition of this library.
 *
 * Who needs it: a caller that cannot call cudaMalloc -- a host engine that
 * owns every device allocation and hands the libraries it loads no
 * allocator, or code that must not trigger the device-wide synchronisation
 * cudaMalloc and cudaFree can cause -- has no way to provide attn_bwd's
 * workspace.  This call allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.  Its scratch is one fixed array of
 * ATTN_BWD_NOALLOC_SCRATCH_BYTES in device memory, reserved on every device
 * that loads the library and held until the process exits.
 *
 * Arguments, layouts, results and error codes are those of attn_bwd, minus
 * the workspace.  In addition:
 *  - a shape whose workspace would exceed ATTN_BWD_NOALLOC_SCRATCH_BYTES is
 *    rejected with ATTN_ERR_UNSUPPORTED before anything is launched (use
 *    attn_bwd with your own workspace for it);
 *  - the first call on a device looks up that device's address of the
 *    scratch array (cudaGetSymbolAddress, with the device current) and
 *    caches it; make that first call before any stream capture.  The cached
 *    address belongs to the device's primary context: calls after
 *    cudaDeviceReset (or any other teardown of that context) are not
 *    supported;
 *  - every call shares the one array and the array keeps whatever the last
 *    call left in it; each call first rewrites everything it later reads, so
 *    leftover contents never change a result;
 *  - calls whose kernels overlap on the GPU (different streams, or several
 *    host threads) race on the shared scratch and give wrong results:
 *    order them, e.g. issue them on one stream.
 */
attn_status attn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                             const float *lse, const void *dO,
                             void *dq, void *dk, void *dv,
                             int B, int Hq, int Hkv, int N, int D, float scale, int causal,
                             void *stream);

/*
 * Bytes of device workspace attn_decode needs: an fp32 running max, row sum
 * and D-column partial output per query head and per segment (a run of one
 * kv head's keys inside one thread block), for up to 512 + B*Hkv - 1
 * segments of Hq/Hkv heads, each region rounded up to 256 bytes.  Returns 0
 * for an empty problem or invalid/unsupported sizes.
 */
size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int N, int D);

/*
 * Decode step (flash decode): one new query row per (batch, query head)
 * attends to an N-row key/value cache.  The query is at position N-1, so
 * the causal mask keeps all N keys; the result equals the last row of
 * attn_fwd with causal = 1 on the same cache.  The (kv head, 128-key) work
 * is spread evenly over one thread block per SM; a kv head whose keys span
 * several blocks has its partial softmax states merged with the
 * online-softmax block-merge rule (kwkr.cn/news/592482, 2.2);
 * "FlashAttention原理与Triton实战" section 7 names flash decode as an
 * extension of the fused kernel.
 *
 *   q            bf16 [B,Hq,D]      the new query rows                 (in)
 *   k, v         bf16 [B,Hkv,N,D]   key / value cache                  (in)
 *   o            bf16 [B,Hq,D]      output rows                        (out)
 *   lse          fp32 [B,Hq]        LSE of each row (natural log), or NULL (out)
 *   scale        multiplier of q.k (usually 1/sqrt(D)); must be finite.
 *   workspace    device scratch of at least attn_decode_workspace_size()
 *                bytes, 256-byte aligned; contents on entry do not matter.
 *
 * D is 64, 80, 96 or 128; Hq / Hkv (query heads per kv head) at most 16
 * (ATTN_ERR_UNSUPPORTED otherwise).  Other conventions as for attn_fwd.
 */
attn_status attn_decode(const void *q, const void *k, const void *v, void *o, float *lse,
                        int B, int Hq, int Hkv, int N, int D, float scale,
                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * Test hook for the bounded-wait failure path (the pages have no counterpart;
 * they only advise checking the -inf initialisation when NaNs appear,
 * "FlashAttention原理与Triton实战" 5.1).
 *
 * Runs attn_fwd (no bias, no emitted logits) with a fault injected: thread
 * block 0's TMA producer never issues its first K tile, so the MMA issuer's
 * wait for that tile cannot complete.  Every pipeline wait of the launch is
 * bounded by `wait_limit_ns` nanoseconds instead of the default 1 s.  The
 * first wait to run out records ATTN_ERR_TIMEOUT in the device status word
 * and raises the block's abort flag; the block's other roles give up their
 * waits, let their copies and MMAs in flight land (each with a 20 ms limit of
 * its own), free their tensor memory and return.  Nothing traps, and the
 * context stays usable.  The other blocks compute normally; the outputs of
 * block 0's query tiles are left unwritten.
 *
 *   wait_limit_ns  > 0 (ATTN_ERR_INVALID otherwise)
 * Other arguments, layouts and errors are those of attn_fwd.  Returns ATTN_OK
 * once queued; attn_last_device_status() then reports ATTN_ERR_TIMEOUT.
 */
attn_status attn_debug_fwd_timeout(const void *q, const void *k, const void *v, void *o,
                                   float *lse, int B, int Hq, int Hkv, int N, int D, float scale,
                                   int causal, unsigned long long wait_limit_ns, void *stream);

/* Static, human-readable name of a status code (never NULL). */
const char *attn_status_string(attn_status status);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word.  Returns ATTN_OK if no kernel since the last call recorded a fault,
 * else the first code recorded (ATTN_ERR_TIMEOUT, ATTN_ERR_DEVICE_CHECK), or
 * ATTN_ERR_CUDA if the synchronisation itself failed.
 */
attn_status attn_last_device_status(void *stream);

/* Library version as major*10000 + minor*100 + patch. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TATTN_H */
