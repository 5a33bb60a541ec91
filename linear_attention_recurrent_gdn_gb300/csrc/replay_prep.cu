// ReplayPrep: the per slot-head stage of a DeltaLog step.
//
// DeltaLog page ("DeltaLog: Deferred Materialization of Recurrent States for
// Linear Attention Decoding"), section "Kernel implementation": key-side
// factors and log-decay metadata are shared by all value tiles, and one shared
// ReplayPrep stage computes the coefficients once per slot-head before the
// parallel AppendDecode stages.  What it computes here, for the token t of
// slot s whose log holds n entries (k_j, Λ_j), j < n, with Λ cumulative since
// the last merge (Λ_t = Λ_{t-1} + g_t):
//
//   GDN    e^{Λ_t};  ckk_j = e^{Λ_t-Λ_j} (k_j·k_t);  ckq_j = e^{Λ_t-Λ_j} (k_j·q_t);
//          k_t·q_t; beta_t; on a merge step w_j = e^{Λ_t-Λ_j} (w_n = 1)
//   KDA    k̂ = e^{Λ_t}⊙k_t, q̂ = e^{Λ_t}⊙q_t;
//          ckk_j = Σ_i k_ji k_ti e^{Λ_ti-Λ_ji}, ckq_j likewise with q_t;
//          on a merge step D = e^{Λ_t} and K̃_j = k_j ⊙ e^{Λ_t-Λ_j} (K̃_n = k_t)
//   RWKV6  r̂ = e^{Λ_{t-1}}⊙r_t;  crq_j = Σ_i k_ji r_ti e^{Λ_{t-1,i}-Λ_ji};
//          c = Σ_i r_i bonus_i k_i; on a merge step D = e^{Λ_t},
//          K̃_j = k_j ⊙ e^{Λ_t-Λ_j} (K̃_n = k_t)
//
// With these, AppendDecode evaluates α_t S_{t-1} k_t (and S_t q_t) for one
// value row from one pass over the dense base plus the value-side log.  On a
// step that is not a merge step, ReplayPrep also appends k_t and Λ_t (and v_t,
// the value-side factor of RWKV6) to the slot's log, and it advances the
// device slot table.  Only differences of cumulative log-decays are
// exponentiated, so no factor exceeds 1 and nothing underflows through ratios.
//
// Launch: one CTA per slot row of the step, 8 warps, warp w handles heads
// w, w+8, ...; within a head, lanes run over key channels for vectors and over
// log entries for the per-entry coefficients.
#include "dl_device.cuh"
#include "layout.h"
#include "launch.h"

namespace dl {

constexpr int RP_WARPS = 8;

template <int OP, int DK, int DV>
__global__ void __launch_bounds__(RP_WARPS * 32)
replay_prep_kernel(const __grid_constant__ StepArgs a) {
  constexpr int VEC = DK / 32;
  __shared__ __align__(16) float s_x[RP_WARPS][DK];  // k_t (GDN, KDA) or e^{g_t} (RWKV6)
  __shared__ __align__(16) float s_y[RP_WARPS][DK];  // q_t or r_t
  __shared__ __align__(16) float s_L[RP_WARPS][DK];  // Λ_t (KDA) or Λ_{t-1} (RWKV6)

  // Let AppendDecode start its first dense-base loads while this kernel runs.
  pdl_launch_dependents();

  const Layout Lay = make_layout(OP, a.M, DK, DV);
  const int row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const StepItem it = a.items[row];
  const int n = it.n, slot = it.slot;
  const bool merge = (n + 1 == a.M);
  const int Mcap = Lay.Mcap, Mcap4 = Lay.Mcap4;
  const int vecA = HDR + 2 * Mcap4, vecB = vecA + DK;

  for (int h = warp; h < a.H; h += RP_WARPS) {
    const size_t sh = (size_t)row * a.H + h;    // row of the step's inputs
    const size_t lh = (size_t)slot * a.H + h;   // log owner
    float* cf = a.coef + sh * a.CB;
    float kv[VEC], qv[VEC];
    ldvec_bf16<VEC>(kv, a.k + sh * DK + lane * VEC);
    ldvec_bf16<VEC>(qv, a.q + sh * DK + lane * VEC);
    float kq = 0.f;
#pragma unroll
    for (int c = 0; c < VEC; ++c) kq += kv[c] * qv[c];
    kq = warp_sum(kq);

    if constexpr (OP == GDN) {
      const float* Lrow = a.Llog + lh * Mcap;
      const float Lt = (n > 0 ? Lrow[n - 1] : 0.f) + a.g[sh];
#pragma unroll
      for (int c = 0; c < VEC; ++c) {
        s_x[warp][lane * VEC + c] = kv[c];
        s_y[warp][lane * VEC + c] = qv[c];
      }
      __syncwarp();
      for (int j = lane; j < n; j += 32) {
        const float wj = expf(Lt - Lrow[j]);
        const uint16_t* kr = a.klog + (lh * Mcap + j) * DK;
        float dkk = 0.f, dkq = 0.f;
#pragma unroll 4
        for (int i = 0; i < DK; i += 8) {
          const uint4 w = *reinterpret_cast<const uint4*>(kr + i);
          const float e[8] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y),
                              bf16lo(w.z), bf16hi(w.z), bf16lo(w.w), bf16hi(w.w)};
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            dkk += e[c] * s_x[warp][i + c];
            dkq += e[c] * s_y[warp][i + c];
          }
        }
        cf[HDR + j] = wj * dkk;
        cf[HDR + Mcap4 + j] = wj * dkq;
        if (merge) cf[Lay.P0 + j] = wj;
      }
      if (lane == 0) {
        cf[0] = expf(Lt);
        cf[1] = kq;
        cf[2] = a.beta[sh];
        if (merge) cf[Lay.P0 + n] = 1.f;
      }
      if (!merge) {
        // append k_t (bf16 bits copied as they came) and Λ_t
        uint16_t* kd = a.klog + (lh * Mcap + n) * DK + lane * VEC;
        const uint16_t* ks = a.k + sh * DK + lane * VEC;
#pragma unroll
        for (int c = 0; c < VEC; ++c) kd[c] = ks[c];
        if (lane == 0) a.Llog[lh * Mcap + n] = Lt;
      }
    } else {
      // per-key decay: Λ vectors, lanes over key channels
      const float* Lbase = a.Llog + lh * Mcap * DK;
      float Lp[VEC], gt[VEC], Lt[VEC];
      if (n > 0) ldvec<VEC>(Lp, Lbase + (size_t)(n - 1) * DK + lane * VEC);
      else {
#pragma unroll
        for (int c = 0; c < VEC; ++c) Lp[c] = 0.f;
      }
      ldvec<VEC>(gt, a.g + sh * DK + lane * VEC);
#pragma unroll
      for (int c = 0; c < VEC; ++c) Lt[c] = Lp[c] + gt[c];

      if constexpr (OP == KDA) {
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
          const int i = lane * VEC + c;
          const float e = expf(Lt[c]);
          cf[vecA + i] = e * kv[c];
          cf[vecB + i] = e * qv[c];
          s_x[warp][i] = kv[c];
          s_y[warp][i] = qv[c];
          s_L[warp][i] = Lt[c];
          if (merge) {
            cf[Lay.P0 + i] = e;
            cf[Lay.P0 + DK + n * DK + i] = kv[c];
          }
        }
        if (lane == 0) {
          cf[1] = kq;
          cf[2] = a.beta[sh];
        }
      } else {  // RWKV6: q holds r_t
        float bon[VEC];
        ldvec<VEC>(bon, a.bonus + (size_t)h * DK + lane * VEC);
        float cb = 0.f;
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
          const int i = lane * VEC + c;
          cf[vecA + i] = expf(Lp[c]) * qv[c];
          cb += qv[c] * bon[c] * kv[c];
          s_x[warp][i] = expf(gt[c]);   // w_t
          s_y[warp][i] = qv[c];
          s_L[warp][i] = Lp[c];
          if (merge) {
            cf[Lay.P0 + i] = expf(Lt[c]);
            cf[Lay.P0 + DK + n * DK + i] = kv[c];
          }
        }
        cb = warp_sum(cb);
        if (lane == 0) cf[3] = cb;
      }
      __syncwarp();
      for (int j = lane; j < n; j += 32) {
        const uint16_t* kr = a.klog + (lh * Mcap + j) * DK;
        const float* Lr = Lbase + (size_t)j * DK;
        float* Kt = cf + Lay.P0 + DK + j * DK;
        float d1 = 0.f, d2 = 0.f;
#pragma unroll 2
        for (int i = 0; i < DK; i += 8) {
          const uint4 w = *reinterpret_cast<const uint4*>(kr + i);
          const float4 l0 = *reinterpret_cast<const float4*>(Lr + i);
          const float4 l1 = *reinterpret_cast<const float4*>(Lr + i + 4);
          const float e[8] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y),
                              bf16lo(w.z), bf16hi(w.z), bf16lo(w.w), bf16hi(w.w)};
          const float lj[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float kk = e[c] * expf(s_L[warp][i + c] - lj[c]);
            if constexpr (OP == KDA) {
              d1 += kk * s_x[warp][i + c];
              d2 += kk * s_y[warp][i + c];
              if (merge) Kt[i + c] = kk;
            } else {
              d1 += kk * s_y[warp][i + c];
              if (merge) Kt[i + c] = kk * s_x[warp][i + c];
            }
          }
        }
        cf[HDR + j] = d1;
        if constexpr (OP == KDA) cf[HDR + Mcap4 + j] = d2;
      }
      if (!merge) {
        uint16_t* kd = a.klog + (lh * Mcap + n) * DK + lane * VEC;
        const uint16_t* ks = a.k + sh * DK + lane * VEC;
        float* Ld = a.Llog + (lh * Mcap + n) * DK + lane * VEC;
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
          kd[c] = ks[c];
          Ld[c] = Lt[c];
        }
        if constexpr (OP == RWKV6) {
          // the value-side factor of RWKV6 is v_t itself
          uint16_t* vd = static_cast<uint16_t*>(a.alog) + (lh * Mcap + n) * DV;
          const uint16_t* vs = a.v + sh * DV;
          for (int i = lane; i < DV; i += 32) vd[i] = vs[i];
        }
      }
    }
    __syncwarp();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    a.nlog[slot] = merge ? 0 : n + 1;
    a.base_of[slot] = merge ? slot : it.base;
  }
}

template <int OP, int DK>
static cudaError_t launch_rp(const StepArgs& a, cudaStream_t s) {
  replay_prep_kernel<OP, DK, DK><<<a.rows, RP_WARPS * 32, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_replay_prep(int op, int dk, const StepArgs& a, cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  if (dk == 64) {
    if (op == GDN) return launch_rp<GDN, 64>(a, s);
    if (op == KDA) return launch_rp<KDA, 64>(a, s);
    return launch_rp<RWKV6, 64>(a, s);
  }
  if (op == GDN) return launch_rp<GDN, 128>(a, s);
  if (op == KDA) return launch_rp<KDA, 128>(a, s);
  return launch_rp<RWKV6, 128>(a, s);
}

}  // namespace dl
