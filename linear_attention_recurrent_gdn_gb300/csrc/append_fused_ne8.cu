// Fused AppendDecode instances for merge intervals with M - 1 <= 8 log entries.
#include "append_launch.cuh"

namespace dl {
DL_DEFINE_FUSED(8)
}  // namespace dl
