// attn_internal.h -- host-side interface between the C-ABI layer and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace tattn {

// Validated forward problem (device pointers, sizes in elements).
struct FwdProblem {
    const void *q, *k, *v;
    const float *bias;
    void *o;
    float *lse;
    float *emit;
    int B, Hq, Hkv, N, D;
    float scale;
    bool causal;
    int window;      // sliding window W (causal only): key j kept iff i - W < j; 0 = none
    // Tests of the timeout path only (0 otherwise): the bound of each
    // pipeline wait (0 = the default) and the injected missing K load.
    unsigned long long wait_limit_ns = 0;
    int inject_skip_k0 = 0;
};

// Validated backward problem.
struct BwdProblem {
    const void *q, *k, *v, *o, *dO;
    const float *lse;
    void *dq, *dk, *dv;
    int B, Hq, Hkv, N, D;
    float scale;
    bool causal;
    int window;      // as in FwdProblem
    // block residual (all null for the plain backward): fp32 [B,Hq,N,N]
    const float *bias;       // the forward's logit bias
    const float *grad_in;    // gradient arriving at this layer's logits
    float *grad_out;         // total logit gradient (may alias grad_in)
    float *dq_acc;   // fp32 [B,Hq,N,D] inside the workspace
    float *lse2;     // fp32 [B*Hq, NP]: LSE * log2(e), +inf on padding rows
    float *delta;    // fp32 [B*Hq, NP]: rowsum(dO * O), 0 on padding rows
    float *dk_acc;   // fp32 [B,Hkv,N,D] (grouped heads only): dK summed over query heads
    float *dv_acc;   // fp32 [B,Hkv,N,D]  "   dV
    int NP;          // N rounded up to the 128-row tile
};

// Decode problem: one query row per (batch, query head) against an N-row
// key/value cache, the (kv head, 128-key stage) work spread evenly over
// `grid` persistent blocks.
struct DecProblem {
    const void *q, *k, *v;   // q [B,Hq,D], k/v [B,Hkv,N,D] bf16
    void *o;                 // [B,Hq,D] bf16
    float *lse;              // [B,Hq] or null
    int B, Hq, Hkv, N, D;
    float scale;
    int grid;
    // workspace: [slots, G] x2 and [slots, G, D] fp32, slots = grid + B*Hkv - 1
    float *m_part, *l_part, *o_part;
};

// Most blocks a decode launch uses (the workspace is sized for it).
constexpr int kDecodeMaxBlocks = 512;
// 128-key stages of a decode problem: B * Hkv * ceil(N / 128).
long long decode_stages(int B, int Hkv, int N);

// Byte offsets of the three workspace regions (each 256-byte aligned) and
// the total size, for a validated shape.
struct BwdWorkspace {
    size_t dq_acc, lse2, delta, dk_acc, dv_acc, total;
};
// dk_acc / dv_acc exist only with grouped heads (Hq > Hkv), where the
// backward may split a key tile's query heads over several blocks.
BwdWorkspace bwd_workspace_layout(int B, int Hq, int Hkv, int N, int D);

// Encodes a rank-3 bf16 tensor map over a [rows = N, cols = D] matrix per
// head (dims {D, N, heads}) with a {64, box_rows, 1} box and 128-byte
// swizzle.  Returns false if the driver rejects it.
bool encode_bf16_rows(CUtensorMap *map, const void *base, int D, int N, long long heads,
                      int box_rows);
// Same for an fp32 [heads, N, D] tensor with a {32, box_rows, 1} box.
bool encode_f32_rows(CUtensorMap *map, const void *base, int D, int N, long long heads,
                     int box_rows);

// Device status word of the current device (allocated statically).
int *device_status_ptr();

cudaError_t launch_fwd(const FwdProblem &pb, int *status, cudaStream_t stream);
// The plain forward (no bias, no emitted logits) with two query tiles per
// thread block (attn_fwd_pp.cu).
cudaError_t launch_fwd_pp(const FwdProblem &pb, int *status, cudaStream_t stream);
cudaError_t launch_bwd(const BwdProblem &pb, int *status, cudaStream_t stream);
cudaError_t launch_decode(const DecProblem &pb, int *status, cudaStream_t stream);

// SM count and L2 size of the current device, queried once per device.
struct DeviceInfo {
    int sms;
    int l2_bytes;
};
bool device_info(DeviceInfo *out);

}  // namespace tattn
