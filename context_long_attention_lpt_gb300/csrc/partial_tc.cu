#include "launch.h"

namespace splitkv {
bool tc_supports(const PartialArgs&) { return false; }
int launch_partial_tc(const PartialArgs&, cudaStream_t) { return SPLITKV_ERR_UNSUPPORTED; }
}  // namespace splitkv
