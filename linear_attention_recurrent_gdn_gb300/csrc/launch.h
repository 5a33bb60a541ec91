// Host-side entry points of the kernel translation units (internal).
#pragma once
#include <cuda_runtime.h>
#include "dl_device.cuh"

namespace dl {

// ReplayPrep: one CTA per slot row.
cudaError_t launch_replay_prep(int op, int dk, const StepArgs& a, cudaStream_t s);

// AppendDecode (pipelined; merge fused).  `pdl` launches it as a programmatic
// dependent of the preceding ReplayPrep in the same stream.
cudaError_t launch_append_decode(int op, int dk, const StepArgs& a, int grid, size_t smem,
                                 bool pdl, cudaStream_t s);

// AppendDecode with the ReplayPrep stage fused in as a warp role (no ReplayPrep
// launch).  `pdl` launches it as a programmatic dependent of the preceding
// kernel in the stream (the previous step).
cudaError_t launch_append_decode_fused(int op, int dk, const StepArgs& a, int grid, size_t smem,
                                       bool pdl, cudaStream_t s);

// EagerStep: the dense read-modify-write step (the comparison kernel).
cudaError_t launch_eager_step(int op, int dk, const StepArgs& a, int grid, size_t smem,
                              cudaStream_t s);

// Raise a kernel's dynamic shared-memory limit to at least `smem` bytes; never
// lowers it, so contexts and calls that plan different shapes can share one
// kernel instance.
template <class Kernel>
inline cudaError_t raise_smem_limit(Kernel* kern, size_t smem) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess || (size_t)fa.maxDynamicSharedSizeBytes >= smem) return e;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

// Allow the pipelined kernels of (op, dk) to use at least `smem` bytes of
// dynamic shared memory.
cudaError_t configure_append_decode(int op, int dk, size_t smem);
cudaError_t configure_eager_step(int op, int dk, size_t smem);

// Registers per thread of the pipelined kernel instances (0 if unknown); the
// fused form's instance depends on the merge interval M.
int append_decode_regs(int op, int dk, bool fused, int M);

// The fused form's translation units, one per bound on log entries (M - 1 <= NE).
cudaError_t launch_fused_ne8(int op, int dk, const StepArgs& a, int grid, size_t smem, bool pdl,
                             cudaStream_t s);
cudaError_t launch_fused_ne16(int op, int dk, const StepArgs& a, int grid, size_t smem, bool pdl,
                              cudaStream_t s);
cudaError_t launch_fused_ne32(int op, int dk, const StepArgs& a, int grid, size_t smem, bool pdl,
                              cudaStream_t s);
cudaError_t configure_fused_ne8(int op, int dk, size_t smem);
cudaError_t configure_fused_ne16(int op, int dk, size_t smem);
cudaError_t configure_fused_ne32(int op, int dk, size_t smem);
int regs_fused_ne8(int op, int dk);
int regs_fused_ne16(int op, int dk);
int regs_fused_ne32(int op, int dk);
int eager_step_regs(int op, int dk);

// Standalone merge / read-state (S_out == nullptr: write back into S̄ and reset the log).
cudaError_t launch_merge(int op, int dk, const SlotListArgs& a, cudaStream_t s);
// Copy initial states into S̄ and reset the listed slots' table entries.
cudaError_t launch_set_state(int dk, int dv, const SlotListArgs& a, cudaStream_t s);
// Copy the source's log rows into each destination and point it at the source's base.
cudaError_t launch_fork(int op, int dk, const SlotListArgs& a, cudaStream_t s);

// Checkpoint records (one fixed-size record per listed slot, at buf + row *
// total): the dense base the slot reads [H, d_v, d_k] at offS, its log rows —
// value side at offA, keys at offK, log-decays at offL — and its log length at
// offN.  save = 1 copies the slots into the records (items[row].base names the
// base the slot reads); save = 0 restores them (the slot then owns its base).
struct CkptArgs {
  float* Sbar;
  void* alog;
  uint16_t* klog;
  float* Llog;
  int32_t* nlog;
  int32_t* base_of;
  unsigned char* buf;
  size_t total, offS, offA, offK, offL, offN;
  int32_t rows, H, Mcap, save;
  StepItem items[MAX_ROWS];
};
cudaError_t launch_checkpoint(int op, int dk, const CkptArgs& a, cudaStream_t s);

// Chunked prefill of T tokens: token-major inputs [T, rows, H, d]; `bonus`
// [H, d_k] for RWKV6.
// GDN and KDA at d_k = d_v = 128 and RWKV6 at 64 run on the tensor cores
// (prefill_tc.cu); a bounded wait there that runs out records DEV_TIMEOUT_MMA
// in `status`.
cudaError_t launch_prefill(int op, int dk, const SlotListArgs& a, const void* q, const void* k,
                           const void* v, const float* g, const float* beta, const float* bonus,
                           void* o, int T, int out_bf16, float scale, int32_t* status,
                           cudaStream_t s);
cudaError_t launch_prefill_gdn_tc(const SlotListArgs& a, const void* q, const void* k,
                                  const void* v, const float* g, const float* beta, void* o, int T,
                                  int out_bf16, float scale, int32_t* status, cudaStream_t s);
cudaError_t launch_prefill_kda_tc(const SlotListArgs& a, const void* q, const void* k,
                                  const void* v, const float* g, const float* beta, void* o, int T,
                                  int out_bf16, float scale, int32_t* status, cudaStream_t s);
// RWKV6 at d_k = d_v = 64: two slot-heads per CTA on the tensor cores (r in `r`).
cudaError_t launch_prefill_rwkv6_tc(const SlotListArgs& a, const void* r, const void* k,
                                    const void* v, const float* g, const float* bonus, void* o,
                                    int T, int out_bf16, float scale, int32_t* status,
                                    cudaStream_t s);

}  // namespace dl
