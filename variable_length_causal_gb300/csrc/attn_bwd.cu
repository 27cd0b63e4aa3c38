// attn_bwd.cu -- backward pass (placeholder until the kernels land).
#include "internal.h"

namespace vlc {

cudaError_t launch_attn_bwd(const BwdParams&, int, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace vlc
