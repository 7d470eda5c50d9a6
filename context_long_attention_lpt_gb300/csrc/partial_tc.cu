#include "launch.h"

namespace splitkv {
bool tc_supports(const PartialArgs&) { return false; }
cudaError_t launch_partial_tc(const PartialArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace splitkv
