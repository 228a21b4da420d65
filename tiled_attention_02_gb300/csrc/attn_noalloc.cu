// attn_noalloc.cu -- attn_bwd_noalloc: the backward pass for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: a host engine that owns every device
// allocation and gives the libraries it loads no allocator, or code that must
// never trigger the device-wide synchronisation that cudaMalloc / cudaFree can
// cause.  Such a caller cannot provide attn_bwd's workspace.  This entry point
// takes its scratch from one fixed array in device memory instead, reserved
// when the library's module is loaded on a device and held until the process
// exits.  It allocates nothing at call time.
#include <mutex>

#include "attn_internal.h"
#include "tattn.h"

namespace tattn {
namespace {

// The fixed scratch: fp32 dQ accumulator plus the two per-row arrays of the
// backward, laid out exactly as in a caller-provided attn_bwd workspace.
static __device__ __align__(256) unsigned char g_bwd_scratch[ATTN_BWD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_dev_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device.  In host code
// the array's name only stands for the symbol; the address a kernel may use
// comes from cudaGetSymbolAddress, looked up once per device with that
// device current and cached.
void *scratch_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_dev_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr)
            return nullptr;
        g_scratch_dev_ptr[dev] = p;
    }
    return g_scratch_dev_ptr[dev];
}

}  // namespace
}  // namespace tattn

extern "C" attn_status attn_bwd_noalloc(const void *q, const void *k, const void *v,
                                        const void *o, const float *lse, const void *dO, void *dq,
                                        void *dk, void *dv, int B, int Hq, int Hkv, int N, int D,
                                        float scale, int causal, void *stream) {
    const size_t need = attn_bwd_workspace_size(B, Hq, Hkv, N, D);
    if (need == 0) {
        // An empty problem, or invalid or unsupported sizes: attn_bwd's own
        // checks (D and scale included) give the same code it would give,
        // before it touches the missing workspace.
        return attn_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, Hq, Hkv, N, D, scale, causal,
                        nullptr, 0, stream);
    }
    if (need > static_cast<size_t>(ATTN_BWD_NOALLOC_SCRATCH_BYTES)) return ATTN_ERR_UNSUPPORTED;
    // Pointer checks come before the scratch lookup (a CUDA call), so that a
    // bad argument gives attn_bwd's code without touching the device.
    const void *bf[] = {q, k, v, o, dO, dq, dk, dv};
    for (const void *p : bf)
        if (!p || reinterpret_cast<uintptr_t>(p) % 16 != 0) return ATTN_ERR_INVALID;
    if (!lse || reinterpret_cast<uintptr_t>(lse) % 4 != 0) return ATTN_ERR_INVALID;
    void *scratch = tattn::scratch_ptr();
    if (!scratch) return ATTN_ERR_CUDA;
    // The backward's first kernel rewrites every scratch byte the later ones
    // read (zeroed dQ accumulator, per-row statistics), so what an earlier
    // call left in the array does not matter.
    return attn_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, Hq, Hkv, N, D, scale, causal, scratch,
                    static_cast<size_t>(ATTN_BWD_NOALLOC_SCRATCH_BYTES), stream);
}
