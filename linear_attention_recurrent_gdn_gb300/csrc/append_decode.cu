// AppendDecode instantiations and launcher (kernel body in pipeline.cuh).
#include "pipeline.cuh"
#include "launch.h"

namespace dl {

template <int OP, int DK, int MODE>
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
  return cudaLaunchKernelEx(&cfg, pipe_kernel<OP, DK, DK, MODE>, a);
}

cudaError_t launch_append_decode(int op, int dk, const StepArgs& a, int grid, size_t smem,
                                 bool pdl, cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  if (dk == 64) {
    if (op == GDN) return launch_ad<GDN, 64, APPEND>(a, grid, smem, pdl, s);
    if (op == KDA) return launch_ad<KDA, 64, APPEND>(a, grid, smem, pdl, s);
    return launch_ad<RWKV6, 64, APPEND>(a, grid, smem, pdl, s);
  }
  if (op == GDN) return launch_ad<GDN, 128, APPEND>(a, grid, smem, pdl, s);
  if (op == KDA) return launch_ad<KDA, 128, APPEND>(a, grid, smem, pdl, s);
  return launch_ad<RWKV6, 128, APPEND>(a, grid, smem, pdl, s);
}

cudaError_t launch_append_decode_fused(int op, int dk, const StepArgs& a, int grid, size_t smem,
                                       bool pdl, cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  if (dk == 64) {
    if (op == GDN) return launch_ad<GDN, 64, FUSED>(a, grid, smem, pdl, s);
    if (op == KDA) return launch_ad<KDA, 64, FUSED>(a, grid, smem, pdl, s);
    return launch_ad<RWKV6, 64, FUSED>(a, grid, smem, pdl, s);
  }
  if (op == GDN) return launch_ad<GDN, 128, FUSED>(a, grid, smem, pdl, s);
  if (op == KDA) return launch_ad<KDA, 128, FUSED>(a, grid, smem, pdl, s);
  return launch_ad<RWKV6, 128, FUSED>(a, grid, smem, pdl, s);
}

template <int OP, int DK>
static int regs_one(bool fused) {
  cudaFuncAttributes fa;
  const cudaError_t e = fused ? cudaFuncGetAttributes(&fa, pipe_kernel<OP, DK, DK, FUSED>)
                              : cudaFuncGetAttributes(&fa, pipe_kernel<OP, DK, DK, APPEND>);
  return e == cudaSuccess ? fa.numRegs : 0;
}

int append_decode_regs(int op, int dk, bool fused) {
  if (dk == 64) {
    if (op == GDN) return regs_one<GDN, 64>(fused);
    if (op == KDA) return regs_one<KDA, 64>(fused);
    return regs_one<RWKV6, 64>(fused);
  }
  if (op == GDN) return regs_one<GDN, 128>(fused);
  if (op == KDA) return regs_one<KDA, 128>(fused);
  return regs_one<RWKV6, 128>(fused);
}

// The attribute must be set on the kernel instance this translation unit
// launches (each translation unit registers its own copy of a template kernel).
template <int OP, int DK>
static cudaError_t cfg_one(size_t smem) {
  cudaError_t e = raise_smem_limit(pipe_kernel<OP, DK, DK, APPEND>, smem);
  if (e != cudaSuccess) return e;
  return raise_smem_limit(pipe_kernel<OP, DK, DK, FUSED>, smem);
}

cudaError_t configure_append_decode(int op, int dk, size_t smem) {
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
