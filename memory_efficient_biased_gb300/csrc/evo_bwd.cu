// evo_bwd.cu — backward kernels (placeholder until the sm_103a backward lands).
#include "evo_internal.h"

namespace evo {
cudaError_t launch_bwd(const BwdArgs&, int, bool, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace evo
