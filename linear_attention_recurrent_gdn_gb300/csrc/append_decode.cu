// AppendDecode: the two-kernel form's instances and the dispatch of the fused
// form to its per-bound translation units (kernel body in pipeline.cuh).
#include "append_launch.cuh"

namespace dl {

cudaError_t launch_append_decode(int op, int dk, const StepArgs& a, int grid, size_t smem,
                                 bool pdl, cudaStream_t s) {
  return launch_mode<APPEND, 0>(op, dk, a, grid, smem, pdl, s);
}

int fused_bound(int M) { return M - 1 <= 8 ? 8 : M - 1 <= 16 ? 16 : 32; }

cudaError_t launch_append_decode_fused(int op, int dk, const StepArgs& a, int grid, size_t smem,
                                       bool pdl, cudaStream_t s) {
  switch (fused_bound(a.M)) {
    case 8: return launch_fused_ne8(op, dk, a, grid, smem, pdl, s);
    case 16: return launch_fused_ne16(op, dk, a, grid, smem, pdl, s);
    default: return launch_fused_ne32(op, dk, a, grid, smem, pdl, s);
  }
}

int append_decode_regs(int op, int dk, bool fused, int M) {
  if (!fused) return regs_mode<APPEND, 0>(op, dk);
  switch (fused_bound(M)) {
    case 8: return regs_fused_ne8(op, dk);
    case 16: return regs_fused_ne16(op, dk);
    default: return regs_fused_ne32(op, dk);
  }
}

cudaError_t configure_append_decode(int op, int dk, size_t smem) {
  cudaError_t e = configure_mode<APPEND, 0>(op, dk, smem);
  if (e == cudaSuccess) e = configure_fused_ne8(op, dk, smem);
  if (e == cudaSuccess) e = configure_fused_ne16(op, dk, smem);
  if (e == cudaSuccess) e = configure_fused_ne32(op, dk, smem);
  return e;
}

}  // namespace dl
