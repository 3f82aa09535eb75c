// Prompt rows of a mixed step (sequences contributing more than one query row).
#include "gw_internal.h"
namespace gw {
cudaError_t launch_local_prompt(int, int, const LocalArgs&, int, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_global_prompt(int, const LocalArgs&, int, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace gw
