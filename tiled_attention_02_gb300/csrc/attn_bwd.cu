// attn_bwd.cu -- recompute-based attention backward (placeholder until the
// tcgen05 backward kernels land).
#include "attn_internal.h"

namespace tattn {

cudaError_t launch_bwd(const BwdProblem &, int *, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace tattn
