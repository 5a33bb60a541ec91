// Launch, attribute and register helpers of the pipelined AppendDecode
// instances (kernel body in pipeline.cuh), shared by the translation units
// that instantiate them: append_decode.cu (two-kernel form) and
// append_fused_ne{8,16,32}.cu (fused form, one per log-entry bound, compiled
// in parallel).
#pragma once
#include "pipeline.cuh"
#include "launch.h"

namespace dl {

template <int OP, int DK, int MODE, int NE>
static cudaError_t launch_ad(const StepArgs& a, int grid, size_t smem, bool pdl, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3((a.ncw + 1 + (MODE == FUSED ? a.npw : 0)) * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (pdl && MODE != EAGER) ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, pipe_kernel<OP, DK, DK, MODE, NE>, a);
}

template <int OP, int DK, int MODE, int NE>
static int regs_of() {
  cudaFuncAttributes fa;
  return cudaFuncGetAttributes(&fa, pipe_kernel<OP, DK, DK, MODE, NE>) == cudaSuccess ? fa.numRegs
                                                                                   : 0;
}

// Dispatch over (op, d_k) for one mode and log-entry bound.
template <int MODE, int NE>
static cudaError_t launch_mode(int op, int dk, const StepArgs& a, int grid, size_t smem, bool pdl,
                               cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  if (dk == 64) {
    if (op == GDN) return launch_ad<GDN, 64, MODE, NE>(a, grid, smem, pdl, s);
    if (op == KDA) return launch_ad<KDA, 64, MODE, NE>(a, grid, smem, pdl, s);
    return launch_ad<RWKV6, 64, MODE, NE>(a, grid, smem, pdl, s);
  }
  if (op == GDN) return launch_ad<GDN, 128, MODE, NE>(a, grid, smem, pdl, s);
  if (op == KDA) return launch_ad<KDA, 128, MODE, NE>(a, grid, smem, pdl, s);
  return launch_ad<RWKV6, 128, MODE, NE>(a, grid, smem, pdl, s);
}

// The attribute must be set on the kernel instances of the translation unit
// that launches them (each unit registers its own copy of a template kernel).
template <int MODE, int NE>
static cudaError_t configure_mode(int op, int dk, size_t smem) {
  if (dk == 64) {
    if (op == GDN) return raise_smem_limit(pipe_kernel<GDN, 64, 64, MODE, NE>, smem);
    if (op == KDA) return raise_smem_limit(pipe_kernel<KDA, 64, 64, MODE, NE>, smem);
    return raise_smem_limit(pipe_kernel<RWKV6, 64, 64, MODE, NE>, smem);
  }
  if (op == GDN) return raise_smem_limit(pipe_kernel<GDN, 128, 128, MODE, NE>, smem);
  if (op == KDA) return raise_smem_limit(pipe_kernel<KDA, 128, 128, MODE, NE>, smem);
  return raise_smem_limit(pipe_kernel<RWKV6, 128, 128, MODE, NE>, smem);
}

template <int MODE, int NE>
static int regs_mode(int op, int dk) {
  if (dk == 64) {
    if (op == GDN) return regs_of<GDN, 64, MODE, NE>();
    if (op == KDA) return regs_of<KDA, 64, MODE, NE>();
    return regs_of<RWKV6, 64, MODE, NE>();
  }
  if (op == GDN) return regs_of<GDN, 128, MODE, NE>();
  if (op == KDA) return regs_of<KDA, 128, MODE, NE>();
  return regs_of<RWKV6, 128, MODE, NE>();
}

// Entry points of one fused translation unit.
#define DL_DEFINE_FUSED(NE)                                                                   \
  cudaError_t launch_fused_ne##NE(int op, int dk, const StepArgs& a, int grid, size_t smem,   \
                                  bool pdl, cudaStream_t s) {                                 \
    return launch_mode<FUSED, NE>(op, dk, a, grid, smem, pdl, s);                             \
  }                                                                                           \
  cudaError_t configure_fused_ne##NE(int op, int dk, size_t smem) {                           \
    return configure_mode<FUSED, NE>(op, dk, smem);                                           \
  }                                                                                           \
  int regs_fused_ne##NE(int op, int dk) { return regs_mode<FUSED, NE>(op, dk); }

}  // namespace dl
