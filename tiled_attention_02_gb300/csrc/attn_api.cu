// attn_api.cu -- the C ABI declared in include/tattn.h: argument checks,
// TMA tensor-map encoding, the per-device status word, and dispatch to the
// kernel launchers.
#include <math.h>
#include <cudaTypedefs.h>
#include <mutex>

#include "attn_internal.h"
#include "tattn.h"

namespace tattn {
namespace {

// One status word per device; a kernel that meets a fault records the first
// code here instead of trapping.
__device__ int g_status_word;

constexpr int kMaxDevices = 64;
int *g_status_ptr[kMaxDevices] = {};
DeviceInfo g_dev_info[kMaxDevices] = {};   // sms == 0: not yet queried
std::mutex g_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    return g_encode;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Common size checks.  Returns ATTN_OK, or the code to return; sets *empty
// when there is nothing to compute.
attn_status check_sizes(int B, int Hq, int Hkv, int N, int D, float scale, bool *empty) {
    *empty = false;
    if (B < 0 || Hq < 0 || Hkv < 0 || N < 0) return ATTN_ERR_INVALID;
    if (!isfinite(scale)) return ATTN_ERR_INVALID;
    if (D != 64 && D != 80 && D != 96 && D != 128)
        return (D > 0) ? ATTN_ERR_UNSUPPORTED : ATTN_ERR_INVALID;
    if (B == 0 || Hq == 0 || N == 0) {
        *empty = true;
        return ATTN_OK;
    }
    if (Hkv == 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID;
    // Tile and head indices are 32-bit in the kernels; element offsets 64-bit.
    const long long BH = static_cast<long long>(B) * Hq;
    const long long ntiles = (static_cast<long long>(N) + 127) / 128;
    if (BH * ntiles > 0x7fffffffLL || BH > 0xffffffffLL) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

}  // namespace

namespace {
// Rank-3 tiled map over [heads, N, D] (dims {D, N, heads}), 128-byte rows in
// the box ({128 / elem_bytes, box_rows, 1}), 128-byte swizzle.
bool encode_rows(CUtensorMap *map, CUtensorMapDataType dtype, int elem_bytes, const void *base,
                 int D, int N, long long heads, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(heads)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * elem_bytes,
                             static_cast<cuuint64_t>(D) * elem_bytes * static_cast<cuuint64_t>(N)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / elem_bytes),
                         static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, dtype, 3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}
}  // namespace

bool encode_bf16_rows(CUtensorMap *map, const void *base, int D, int N, long long heads,
                      int box_rows) {
    return encode_rows(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, D, N, heads, box_rows);
}

bool encode_f32_rows(CUtensorMap *map, const void *base, int D, int N, long long heads,
                     int box_rows) {
    return encode_rows(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, D, N, heads, box_rows);
}

BwdWorkspace bwd_workspace_layout(int B, int Hq, int Hkv, int N, int D) {
    auto round256 = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const size_t rows = static_cast<size_t>(B) * Hq * N;
    const size_t prow = static_cast<size_t>(B) * Hq * (((static_cast<size_t>(N) + 127) / 128) * 128);
    const size_t kvrows = Hq > Hkv ? static_cast<size_t>(B) * Hkv * N : 0;
    BwdWorkspace w;
    w.dq_acc = 0;
    w.lse2 = round256(rows * D * sizeof(float));
    w.delta = w.lse2 + round256(prow * sizeof(float));
    w.dk_acc = w.delta + round256(prow * sizeof(float));
    w.dv_acc = w.dk_acc + round256(kvrows * D * sizeof(float));
    w.total = w.dv_acc + round256(kvrows * D * sizeof(float));
    return w;
}

bool device_info(DeviceInfo *out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &d = g_dev_info[dev];
    if (d.sms == 0) {
        int sms = 0, l2 = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            sms <= 0)
            return false;
        if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess || l2 <= 0)
            l2 = 128 << 20;
        d.l2_bytes = l2;
        d.sms = sms;
    }
    *out = d;
    return true;
}

int *device_status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int *>(p);
    }
    return g_status_ptr[dev];
}

}  // namespace tattn

using namespace tattn;

namespace {

// window: 0 for none, else W >= 1 (checked by the caller; implies causal).
attn_status fwd_impl(const void *q, const void *k, const void *v, const float *bias, void *o,
                     float *lse, int B, int Hq, int Hkv, int N, int D, float scale, int causal,
                     int window, float *emit_logits, void *stream,
                     unsigned long long wait_limit_ns = 0, int inject_skip_k0 = 0) {
    bool empty = false;
    attn_status st = check_sizes(B, Hq, Hkv, N, D, scale, &empty);
    if (st != ATTN_OK || empty) return st;
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
        return ATTN_ERR_INVALID;
    if ((bias && !aligned(bias, 4)) || (emit_logits && !aligned(emit_logits, 4)) ||
        (lse && !aligned(lse, 4)))
        return ATTN_ERR_INVALID;
    if (bias || emit_logits) {
        // [B,Hq,N,N] element offsets must fit in 64 bits.
        const double elems = static_cast<double>(B) * Hq * static_cast<double>(N) * N;
        if (elems > 9.0e18) return ATTN_ERR_UNSUPPORTED;
    }
    FwdProblem pb;
    pb.q = q;
    pb.k = k;
    pb.v = v;
    pb.bias = bias;
    pb.o = o;
    pb.lse = lse;
    pb.emit = emit_logits;
    pb.B = B;
    pb.Hq = Hq;
    pb.Hkv = Hkv;
    pb.N = N;
    pb.D = D;
    pb.scale = scale;
    pb.causal = causal != 0;
    pb.window = (window > 0 && window < N) ? window : 0;   // W >= N is the causal mask
    pb.wait_limit_ns = wait_limit_ns;
    pb.inject_skip_k0 = inject_skip_k0;
    int *status = device_status_ptr();
    if (!status) return ATTN_ERR_CUDA;
    cudaError_t e = launch_fwd(pb, status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}



attn_status bwd_impl(const void *q, const void *k, const void *v, const void *o, const float *lse,
                     const void *dO, void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int N,
                     int D, float scale, int causal, int window, void *workspace,
                     size_t workspace_bytes, void *stream, const float *bias = nullptr,
                     const float *grad_in = nullptr, float *grad_out = nullptr) {
    bool empty = false;
    attn_status st = check_sizes(B, Hq, Hkv, N, D, scale, &empty);
    if (st != ATTN_OK || empty) return st;
    if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv || !workspace)
        return ATTN_ERR_INVALID;
    const void *bf[] = {q, k, v, o, dO, dq, dk, dv};
    for (const void *p : bf)
        if (!aligned(p, 16)) return ATTN_ERR_INVALID;
    if (!aligned(lse, 4) || !aligned(workspace, 256)) return ATTN_ERR_INVALID;
    if (bias || grad_in || grad_out) {
        const float *res[3] = {bias, grad_in, grad_out};
        for (const float *r : res)
            if (r && !aligned(r, 4)) return ATTN_ERR_INVALID;
        // The residual tiles move as TMA boxes: 16-byte rows and bases.
        for (const float *r : res)
            if (r && (!aligned(r, 16) || N % 4 != 0)) return ATTN_ERR_UNSUPPORTED;
        const double elems = static_cast<double>(B) * Hq * static_cast<double>(N) * N;
        if (elems > 9.0e18) return ATTN_ERR_UNSUPPORTED;
    }
    const BwdWorkspace wl = bwd_workspace_layout(B, Hq, Hkv, N, D);
    if (workspace_bytes < wl.total) return ATTN_ERR_INVALID;
    BwdProblem pb;
    pb.q = q;
    pb.k = k;
    pb.v = v;
    pb.o = o;
    pb.dO = dO;
    pb.lse = lse;
    pb.dq = dq;
    pb.dk = dk;
    pb.dv = dv;
    pb.B = B;
    pb.Hq = Hq;
    pb.Hkv = Hkv;
    pb.N = N;
    pb.D = D;
    pb.scale = scale;
    pb.causal = causal != 0;
    pb.window = (window > 0 && window < N) ? window : 0;
    pb.bias = bias;
    pb.grad_in = grad_in;
    pb.grad_out = grad_out;
    char *ws = static_cast<char *>(workspace);
    pb.dq_acc = reinterpret_cast<float *>(ws + wl.dq_acc);
    pb.lse2 = reinterpret_cast<float *>(ws + wl.lse2);
    pb.delta = reinterpret_cast<float *>(ws + wl.delta);
    pb.dk_acc = Hq > Hkv ? reinterpret_cast<float *>(ws + wl.dk_acc) : nullptr;
    pb.dv_acc = Hq > Hkv ? reinterpret_cast<float *>(ws + wl.dv_acc) : nullptr;
    pb.NP = ((N + 127) / 128) * 128;
    int *status = device_status_ptr();
    if (!status) return ATTN_ERR_CUDA;
    cudaError_t e = launch_bwd(pb, status, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return ATTN_ERR_UNSUPPORTED;
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

struct DecWorkspace {
    size_t m, l, o, total;
};

DecWorkspace decode_workspace_layout(int B, int Hq, int Hkv, int D) {
    auto round256 = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    // One slot per (block, kv head) segment: at most blocks + kv heads - 1.
    const size_t slots = static_cast<size_t>(kDecodeMaxBlocks) + static_cast<size_t>(B) * Hkv - 1;
    const size_t parts = slots * static_cast<size_t>(Hq / Hkv);
    DecWorkspace w;
    w.m = 0;
    w.l = round256(parts * sizeof(float));
    w.o = w.l + round256(parts * sizeof(float));
    w.total = w.o + round256(parts * D * sizeof(float));
    return w;
}

constexpr int kDecodeMaxGroup = 16;

}  // namespace

extern "C" {

size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int N, int D) {
    bool empty = false;
    if (check_sizes(B, Hq, Hkv, N, D, 1.0f, &empty) != ATTN_OK || empty) return 0;
    if (Hq / Hkv > kDecodeMaxGroup) return 0;
    return decode_workspace_layout(B, Hq, Hkv, D).total;
}

attn_status attn_decode(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                        int Hq, int Hkv, int N, int D, float scale, void *workspace,
                        size_t workspace_bytes, void *stream) {
    bool empty = false;
    attn_status st = check_sizes(B, Hq, Hkv, N, D, scale, &empty);
    if (st != ATTN_OK || empty) return st;
    if (Hq / Hkv > kDecodeMaxGroup) return ATTN_ERR_UNSUPPORTED;
    if (!q || !k || !v || !o || !workspace) return ATTN_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
        (lse && !aligned(lse, 4)) || !aligned(workspace, 256))
        return ATTN_ERR_INVALID;
    const DecWorkspace wl = decode_workspace_layout(B, Hq, Hkv, D);
    if (workspace_bytes < wl.total) return ATTN_ERR_INVALID;
    DeviceInfo di;
    if (!device_info(&di)) return ATTN_ERR_CUDA;
    const int sms = di.sms;
    // One persistent block per SM (each holds most of an SM's shared
    // memory), never more blocks than 128-key stages.
    const long long stages = decode_stages(B, Hkv, N);
    long long grid = sms < kDecodeMaxBlocks ? sms : kDecodeMaxBlocks;
    if (grid > stages) grid = stages;
    DecProblem pb;
    pb.q = q;
    pb.k = k;
    pb.v = v;
    pb.o = o;
    pb.lse = lse;
    pb.B = B;
    pb.Hq = Hq;
    pb.Hkv = Hkv;
    pb.N = N;
    pb.D = D;
    pb.scale = scale;
    pb.grid = static_cast<int>(grid);
    char *ws = static_cast<char *>(workspace);
    pb.m_part = reinterpret_cast<float *>(ws + wl.m);
    pb.l_part = reinterpret_cast<float *>(ws + wl.l);
    pb.o_part = reinterpret_cast<float *>(ws + wl.o);
    int *status = device_status_ptr();
    if (!status) return ATTN_ERR_CUDA;
    cudaError_t e = launch_decode(pb, status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int N, int D) {
    bool empty = false;
    if (check_sizes(B, Hq, Hkv, N, D, 1.0f, &empty) != ATTN_OK || empty) return 0;
    return bwd_workspace_layout(B, Hq, Hkv, N, D).total;
}

attn_status attn_fwd(const void *q, const void *k, const void *v, const float *bias, void *o,
                     float *lse, int B, int Hq, int Hkv, int N, int D, float scale, int causal,
                     float *emit_logits, void *stream) {
    return fwd_impl(q, k, v, bias, o, lse, B, Hq, Hkv, N, D, scale, causal, 0, emit_logits,
                    stream);
}

attn_status attn_fwd_window(const void *q, const void *k, const void *v, const float *bias,
                            void *o, float *lse, int B, int Hq, int Hkv, int N, int D,
                            float scale, int window, float *emit_logits, void *stream) {
    if (window < 1) return ATTN_ERR_INVALID;
    return fwd_impl(q, k, v, bias, o, lse, B, Hq, Hkv, N, D, scale, 1, window, emit_logits,
                    stream);
}

attn_status attn_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
                     const void *dO, void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int N,
                     int D, float scale, int causal, void *workspace, size_t workspace_bytes,
                     void *stream) {
    return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, B, Hq, Hkv, N, D, scale, causal, 0,
                    workspace, workspace_bytes, stream);
}

attn_status attn_bwd_residual(const void *q, const void *k, const void *v, const void *o,
                              const float *lse, const void *dO, const float *bias,
                              const float *grad_in, void *dq, void *dk, void *dv, float *grad_out,
                              int B, int Hq, int Hkv, int N, int D, float scale, int causal,
                              void *workspace, size_t workspace_bytes, void *stream) {
    return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, B, Hq, Hkv, N, D, scale, causal, 0,
                    workspace, workspace_bytes, stream, bias, grad_in, grad_out);
}

attn_status attn_bwd_window(const void *q, const void *k, const void *v, const void *o,
                            const float *lse, const void *dO, void *dq, void *dk, void *dv,
                            int B, int Hq, int Hkv, int N, int D, float scale, int window,
                            void *workspace, size_t workspace_bytes, void *stream) {
    if (window < 1) return ATTN_ERR_INVALID;
    return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, B, Hq, Hkv, N, D, scale, 1, window,
                    workspace, workspace_bytes, stream);
}

attn_status attn_debug_fwd_timeout(const void *q, const void *k, const void *v, void *o,
                                   float *lse, int B, int Hq, int Hkv, int N, int D, float scale,
                                   int causal, unsigned long long wait_limit_ns, void *stream) {
    if (wait_limit_ns == 0) return ATTN_ERR_INVALID;
    return fwd_impl(q, k, v, nullptr, o, lse, B, Hq, Hkv, N, D, scale, causal, 0, nullptr,
                    stream, wait_limit_ns, 1);
}

const char *attn_status_string(attn_status s) {
    switch (s) {
        case ATTN_OK: return "ATTN_OK";
        case ATTN_ERR_INVALID: return "ATTN_ERR_INVALID: invalid argument";
        case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED: valid but unsupported request";
        case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA: a CUDA call failed";
        case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT: a device pipeline wait timed out";
        case ATTN_ERR_DEVICE_CHECK: return "ATTN_ERR_DEVICE_CHECK: a device-side check failed";
    }
    return "unknown attn_status";
}

attn_status attn_last_device_status(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    int *p = device_status_ptr();
    if (!p) return ATTN_ERR_CUDA;
    int h = 0;
    if (cudaMemcpy(&h, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
    if (h != 0) {
        const int zero = 0;
        if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return ATTN_ERR_CUDA;
    }
    return static_cast<attn_status>(h);
}

int attn_version(void) { return 100; }

}  // extern "C"
