// Fused AppendDecode instances for merge intervals with M - 1 <= 16 log entries.
#include "append_launch.cuh"

namespace dl {
DL_DEFINE_FUSED(16)
}  // namespace dl
