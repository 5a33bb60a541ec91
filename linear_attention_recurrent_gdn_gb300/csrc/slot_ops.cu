// Slot-level kernels outside the per-token hot loop:
//   * Merge / ReadState — materialise base + replayed log (DeltaLog page,
//     "Methodology — Base + Log", merge phase) into S̄ (forced merge) or into a
//     caller buffer (read-out; the context is unchanged);
//   * SetState — load initial states into S̄;
//   * Fork — Flide page, "Research method step by step", second step: a branch
//     indexes the source's saved state; only the source's log rows are copied;
//   * Checkpoint save / restore — Flide page, fourth step: a slot's exact
//     representation (the base it reads, its log rows and length) to and from a
//     caller-owned record.
#include "dl_device.cuh"
#include "layout.h"
#include "launch.h"

namespace dl {

// One CTA per (row, head): the slot-head's K̃ and value-side rows are staged
// once, then each of the 8 warps takes DV/8 rows in batches of 4, loading the
// next batch of the dense base while it finishes the current one.  The logical
// state of slot s with n log entries and cumulative log-decay Λ_{n-1} is
//   S = D ⊙ S̄[base] + Σ_{j<n} a_j K̃_j^T,  D = e^{Λ_{n-1}},  K̃_j = k_j ⊙ e^{Λ_{n-1} - Λ_j}
// (scalar decay for GDN, per key channel for KDA and RWKV6).
template <int OP, int DK, int DV>
__global__ void __launch_bounds__(256) merge_kernel(const __grid_constant__ SlotListArgs a) {
  constexpr int VEC = DK / 32, RPW = DV / 8, NB = RPW / 4;   // rows per warp, batches of 4
  constexpr bool PERKEY = OP != GDN;
  extern __shared__ __align__(16) float sm[];
  const int sh = blockIdx.x, h = sh % a.H, row = sh / a.H;
  const StepItem it = a.items[row];
  const int n = it.n, Mcap = a.Mcap;
  const size_t lh = (size_t)it.slot * a.H + h;
  float* Kt = sm;                    // [n][DK]
  float* U = sm + n * DK;            // [n][DV]
  float* sD = U + n * DV;            // [DK]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float* base = a.Sbar + ((size_t)it.base * a.H + h) * DV * DK + lane * VEC;
  float* dst = (a.S_out ? a.S_out + ((size_t)row * a.H + h) * DV * DK
                        : a.Sbar + ((size_t)it.slot * a.H + h) * DV * DK) + lane * VEC;

  // the first batch of this warp's rows loads while the log rows are staged
  float t[4][VEC], tn[4][VEC];
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) ldvec<VEC>(t[rr], base + (size_t)(warp * RPW + rr) * DK);

  if constexpr (PERKEY) {
    for (int i = tid; i < DK; i += 256) {
      const float Lc = n > 0 ? a.Llog[(lh * Mcap + n - 1) * DK + i] : 0.f;
      sD[i] = expf(Lc);
    }
#pragma unroll 4
    for (int idx = tid; idx < n * DK; idx += 256) {   // unrolled: the loads go out together
      const int j = idx / DK, i = idx - j * DK;
      const float Lc = a.Llog[(lh * Mcap + n - 1) * DK + i];
      Kt[idx] = bf16f(a.klog[(lh * Mcap + j) * DK + i]) * expf(Lc - a.Llog[(lh * Mcap + j) * DK + i]);
    }
  } else {
    const float Lc = n > 0 ? a.Llog[lh * Mcap + n - 1] : 0.f;
    for (int i = tid; i < DK; i += 256) sD[i] = expf(Lc);
#pragma unroll 4
    for (int idx = tid; idx < n * DK; idx += 256) {   // unrolled: the loads go out together
      const int j = idx / DK, i = idx - j * DK;
      Kt[idx] = bf16f(a.klog[(lh * Mcap + j) * DK + i]) * expf(Lc - a.Llog[lh * Mcap + j]);
    }
  }
#pragma unroll 4
  for (int idx = tid; idx < n * DV; idx += 256) {
    const size_t src = lh * Mcap * DV + idx;          // rows j of the slot-head, contiguous
    U[idx] = (OP == RWKV6) ? bf16f(static_cast<const uint16_t*>(a.alog)[src])
                           : static_cast<const float*>(a.alog)[src];
  }
  __syncthreads();

  float D[VEC];
  ldvec<VEC>(D, sD + lane * VEC);
#pragma unroll 1
  for (int b = 0; b < NB; ++b) {
    if (b + 1 < NB) {
#pragma unroll
      for (int rr = 0; rr < 4; ++rr)
        ldvec<VEC>(tn[rr], base + (size_t)(warp * RPW + (b + 1) * 4 + rr) * DK);
    }
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int r = warp * RPW + b * 4 + rr;
#pragma unroll
      for (int c = 0; c < VEC; ++c) t[rr][c] *= D[c];
      for (int j = 0; j < n; ++j) {
        const float uj = U[j * DV + r];
#pragma unroll
        for (int c = 0; c < VEC; ++c) t[rr][c] += uj * Kt[j * DK + lane * VEC + c];
      }
      stvec_cs<VEC>(dst + (size_t)r * DK, t[rr]);
    }
    if (b + 1 < NB) {
#pragma unroll
      for (int rr = 0; rr < 4; ++rr)
#pragma unroll
        for (int c = 0; c < VEC; ++c) t[rr][c] = tn[rr][c];
    }
  }
  if (!a.S_out && h == 0 && tid == 0) {
    a.nlog[it.slot] = 0;
    a.base_of[it.slot] = it.slot;
  }
}

// One CTA per (row, head): copy DV x DK floats of S_in into S̄[slot].
template <int DK, int DV>
__global__ void __launch_bounds__(256) set_state_kernel(const __grid_constant__ SlotListArgs a) {
  const int sh = blockIdx.x, h = sh % a.H, row = sh / a.H;
  const StepItem it = a.items[row];
  const float4* src = reinterpret_cast<const float4*>(a.S_in + (size_t)sh * DV * DK);
  float4* dst = reinterpret_cast<float4*>(a.Sbar + ((size_t)it.slot * a.H + h) * DV * DK);
  constexpr int NV = DV * DK / 4;   // a multiple of 4 x 256 at d = 64 and 128
  static_assert(NV % (4 * 256) == 0, "whole batches of four loads per thread");
  for (int i = threadIdx.x; i < NV; i += 4 * 256) {   // four loads in flight per thread
    const float4 r0 = src[i], r1 = src[i + 256], r2 = src[i + 512], r3 = src[i + 768];
    dst[i] = r0;
    dst[i + 256] = r1;
    dst[i + 512] = r2;
    dst[i + 768] = r3;
  }
  if (h == 0 && threadIdx.x == 0) {
    a.nlog[it.slot] = 0;
    a.base_of[it.slot] = it.slot;
  }
}

// One CTA per (destination, head): copy the source's log rows 0..src_n-1.
template <int OP, int DK, int DV>
__global__ void __launch_bounds__(128) fork_kernel(const __grid_constant__ SlotListArgs a) {
  constexpr int ESA = (OP == RWKV6) ? 2 : 4;
  constexpr int LW = (OP == GDN) ? 1 : DK;    // Λ floats per entry
  const int b = blockIdx.x, h = b % a.H, row = b / a.H;
  const int dst = a.items[row].slot;
  const int n = a.src_n, Mcap = a.Mcap;
  const size_t ls = (size_t)a.src_slot * a.H + h, ld = (size_t)dst * a.H + h;
  {
    const size_t words = (size_t)n * DV * ESA / 16;
    const uint4* s = reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(a.alog) +
                                                    ls * Mcap * DV * ESA);
    uint4* d = reinterpret_cast<uint4*>(static_cast<unsigned char*>(a.alog) + ld * Mcap * DV * ESA);
    for (size_t i = threadIdx.x; i < words; i += 128) d[i] = s[i];
  }
  {
    const size_t words = (size_t)n * DK * 2 / 16;
    const uint4* s = reinterpret_cast<const uint4*>(a.klog + ls * Mcap * DK);
    uint4* d = reinterpret_cast<uint4*>(a.klog + ld * Mcap * DK);
    for (size_t i = threadIdx.x; i < words; i += 128) d[i] = s[i];
  }
  for (int i = threadIdx.x; i < n * LW; i += 128)
    a.Llog[ld * Mcap * LW + i] = a.Llog[ls * Mcap * LW + i];
  if (h == 0 && threadIdx.x == 0) {
    a.nlog[dst] = n;
    a.base_of[dst] = a.src_base;
  }
}

// One CTA per (row, head): the head's slice of each record segment.
template <int OP, int DK, int DV>
__global__ void __launch_bounds__(256) checkpoint_kernel(const __grid_constant__ CkptArgs a) {
  constexpr int ESA = (OP == RWKV6) ? 2 : 4;
  constexpr int LW = (OP == GDN) ? 1 : DK;    // log-decay floats per entry
  const int b = blockIdx.x, h = b % a.H, row = b / a.H;
  const StepItem it = a.items[row];
  const size_t Mcap = a.Mcap;
  unsigned char* rec = a.buf + (size_t)row * a.total;
  const size_t lh = (size_t)it.slot * a.H + h;
  // four 16-byte loads in flight per thread before their stores (one at a
  // time leaves the copy bound by latency); the tail one at a time
  auto copy16 = [&](unsigned char* dst, const unsigned char* src, size_t bytes) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    const size_t nv = bytes / 16;
    size_t i = threadIdx.x;
    for (; i + 3 * 256 < nv; i += 4 * 256) {
      const uint4 r0 = s4[i], r1 = s4[i + 256], r2 = s4[i + 512], r3 = s4[i + 768];
      d4[i] = r0;
      d4[i + 256] = r1;
      d4[i + 512] = r2;
      d4[i + 768] = r3;
    }
    for (; i < nv; i += 256) d4[i] = s4[i];
  };
  const size_t sS = (size_t)DV * DK * 4, sA = Mcap * DV * ESA, sK = Mcap * DK * 2;
  unsigned char* gS = reinterpret_cast<unsigned char*>(a.Sbar) +
                      ((size_t)(a.save ? it.base : it.slot) * a.H + h) * sS;
  unsigned char* gA = static_cast<unsigned char*>(a.alog) + lh * sA;
  unsigned char* gK = reinterpret_cast<unsigned char*>(a.klog) + lh * sK;
  unsigned char* cS = rec + a.offS + h * sS;
  unsigned char* cA = rec + a.offA + h * sA;
  unsigned char* cK = rec + a.offK + h * sK;
  float* gL = a.Llog + lh * Mcap * LW;
  float* cL = reinterpret_cast<float*>(rec + a.offL) + h * Mcap * LW;
  if (a.save) {
    copy16(cS, gS, sS);
    copy16(cA, gA, sA);
    copy16(cK, gK, sK);
    for (size_t i = threadIdx.x; i < Mcap * LW; i += 256) cL[i] = gL[i];
  } else {
    copy16(gS, cS, sS);
    copy16(gA, cA, sA);
    copy16(gK, cK, sK);
    for (size_t i = threadIdx.x; i < Mcap * LW; i += 256) gL[i] = cL[i];
  }
  if (h == 0 && threadIdx.x == 0) {
    int32_t* rn = reinterpret_cast<int32_t*>(rec + a.offN);
    if (a.save) {
      *rn = a.nlog[it.slot];
    } else {
      a.nlog[it.slot] = *rn;
      a.base_of[it.slot] = it.slot;
    }
  }
}

template <int OP, int DK>
static cudaError_t checkpoint_dispatch(const CkptArgs& a, cudaStream_t s) {
  checkpoint_kernel<OP, DK, DK><<<a.rows * a.H, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_checkpoint(int op, int dk, const CkptArgs& a, cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  if (dk == 64) {
    if (op == GDN) return checkpoint_dispatch<GDN, 64>(a, s);
    if (op == KDA) return checkpoint_dispatch<KDA, 64>(a, s);
    return checkpoint_dispatch<RWKV6, 64>(a, s);
  }
  if (op == GDN) return checkpoint_dispatch<GDN, 128>(a, s);
  if (op == KDA) return checkpoint_dispatch<KDA, 128>(a, s);
  return checkpoint_dispatch<RWKV6, 128>(a, s);
}

template <int OP, int DK>
static cudaError_t merge_dispatch(const SlotListArgs& a, cudaStream_t s) {
  int nmax = 0;
  for (int i = 0; i < a.rows; ++i) nmax = a.items[i].n > nmax ? a.items[i].n : nmax;
  const size_t smem = ((size_t)nmax * DK + (size_t)nmax * DK + DK) * sizeof(float);
  merge_kernel<OP, DK, DK><<<a.rows * a.H, 256, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_merge(int op, int dk, const SlotListArgs& a, cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  if (dk == 64) {
    if (op == GDN) return merge_dispatch<GDN, 64>(a, s);
    if (op == KDA) return merge_dispatch<KDA, 64>(a, s);
    return merge_dispatch<RWKV6, 64>(a, s);
  }
  if (op == GDN) return merge_dispatch<GDN, 128>(a, s);
  if (op == KDA) return merge_dispatch<KDA, 128>(a, s);
  return merge_dispatch<RWKV6, 128>(a, s);
}

cudaError_t launch_set_state(int dk, int dv, const SlotListArgs& a, cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  (void)dv;
  if (dk == 64) set_state_kernel<64, 64><<<a.rows * a.H, 256, 0, s>>>(a);
  else set_state_kernel<128, 128><<<a.rows * a.H, 256, 0, s>>>(a);
  return cudaGetLastError();
}

template <int OP, int DK>
static cudaError_t fork_dispatch(const SlotListArgs& a, cudaStream_t s) {
  fork_kernel<OP, DK, DK><<<a.rows * a.H, 128, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_fork(int op, int dk, const SlotListArgs& a, cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  if (dk == 64) {
    if (op == GDN) return fork_dispatch<GDN, 64>(a, s);
    if (op == KDA) return fork_dispatch<KDA, 64>(a, s);
    return fork_dispatch<RWKV6, 64>(a, s);
  }
  if (op == GDN) return fork_dispatch<GDN, 128>(a, s);
  if (op == KDA) return fork_dispatch<KDA, 128>(a, s);
  return fork_dispatch<RWKV6, 128>(a, s);
}

}  // namespace dl
