#include "launch.h"

namespace splitkv {
bool decode_supports(const PartialArgs&) { return false; }
cudaError_t launch_partial_decode(const PartialArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace splitkv
