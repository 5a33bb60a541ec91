// EagerStep instantiations and launcher (kernel body in pipeline.cuh): the
// dense step that reads and rewrites every state row of every active
// slot-head each token — the "state-update tax" the DeltaLog page describes
// in its "Problem" section, kept as the in-house comparison kernel.
#include "pipeline.cuh"
#include "launch.h"

namespace dl {

template <int OP, int DK>
static cudaError_t launch_ea(const StepArgs& a, int grid, size_t smem, cudaStream_t s) {
  pipe_kernel<OP, DK, DK, EAGER><<<grid, (a.ncw + 1) * 32, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_eager_step(int op, int dk, const StepArgs& a, int grid, size_t smem,
                              cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  if (dk == 64) {
    if (op == GDN) return launch_ea<GDN, 64>(a, grid, smem, s);
    if (op == KDA) return launch_ea<KDA, 64>(a, grid, smem, s);
    return launch_ea<RWKV6, 64>(a, grid, smem, s);
  }
  if (op == GDN) return launch_ea<GDN, 128>(a, grid, smem, s);
  if (op == KDA) return launch_ea<KDA, 128>(a, grid, smem, s);
  return launch_ea<RWKV6, 128>(a, grid, smem, s);
}

template <int OP, int DK>
static int regs_one() {
  cudaFuncAttributes fa;
  return cudaFuncGetAttributes(&fa, pipe_kernel<OP, DK, DK, EAGER>) == cudaSuccess ? fa.numRegs : 0;
}

int eager_step_regs(int op, int dk) {
  if (dk == 64) {
    if (op == GDN) return regs_one<GDN, 64>();
    if (op == KDA) return regs_one<KDA, 64>();
    return regs_one<RWKV6, 64>();
  }
  if (op == GDN) return regs_one<GDN, 128>();
  if (op == KDA) return regs_one<KDA, 128>();
  return regs_one<RWKV6, 128>();
}

template <int OP, int DK>
static cudaError_t cfg_one(size_t smem) {
  return raise_smem_limit(pipe_kernel<OP, DK, DK, EAGER>, smem);
}

cudaError_t configure_eager_step(int op, int dk, size_t smem) {
  if (dk == 64) {
    if (op == GDN) return cfg_one<GDN, 64>(smem);
    if (op == KDA) return cfg_one<KDA, 64>(smem);
    return cfg_one<RWKV6, 64>(smem);
  }
  if (op == GDN) return cfg_one<GDN, 128>(smem);
  if (op == KDA) return cfg_one<KDA, 128>(smem);
  return cfg_one<RWKV6, 128>(smem);
}

}  // namespace dl
