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
// Launch: one warp per (row, head), 8 warps per CTA.  Lane l holds d_k/32
// consecutive key channels; every log row is read (and every K̃ row written)
// as one coalesced warp access; the per-entry dot products (n <= M-1 <= 31)
// are finished by a transposed butterfly over NE = 8, 16 or 32 entries, which
// leaves entry j on lanes j*32/NE .. (j+1)*32/NE - 1.
#include "dl_device.cuh"
#include "layout.h"
#include "launch.h"

namespace dl {

constexpr int RP_WARPS = 8;

// NE: per-entry partial sums held per lane, the power of two >= M-1 (at least 8).
template <int OP, int DK, int DV, int NE>
__global__ void __launch_bounds__(RP_WARPS * 32)
replay_prep_kernel(const __grid_constant__ StepArgs a) {
  constexpr int VEC = DK / 32;
  constexpr int SHIFT = NE == 32 ? 0 : NE == 16 ? 1 : 2;   // entry of lane l: l >> SHIFT
  const int lane_entry = (threadIdx.x & 31) >> SHIFT;
  const bool entry_writer = ((threadIdx.x & 31) & ((1 << SHIFT) - 1)) == 0;
  // Let AppendDecode start streaming the dense base while this kernel runs.
  pdl_launch_dependents();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sh = blockIdx.x * RP_WARPS + warp;      // (row, head) of the step's inputs
  if (sh >= step_rows(a) * a.H) return;
  const int row = sh / a.H, h = sh - row * a.H;
  const Layout Lay = make_layout(OP, a.M, DK, DV);
  const StepItem it = step_item(a, row);
  const int n = it.n, slot = it.slot;
  const bool merge = (n + 1 == a.M);
  const int Mcap = Lay.Mcap, Mcap4 = Lay.Mcap4;
  const int vecA = HDR + 2 * Mcap4, vecB = vecA + DK;
  const size_t lh = (size_t)slot * a.H + h;          // log owner
  float* cf = a.coef + (size_t)sh * a.CB;
  const int c0 = lane * VEC;

  float kv[VEC], qv[VEC];
  ldvec_bf16<VEC>(kv, a.k + (size_t)sh * DK + c0);
  ldvec_bf16<VEC>(qv, a.q + (size_t)sh * DK + c0);

  float p1[NE], p2[NE];                               // per-entry partial dot products
  if constexpr (OP == GDN) {
    // the scalars a lane needs are loaded before any arithmetic, so their
    // latency overlaps the key-log row loads
    const float* Lrow = a.Llog + lh * Mcap;
    const float g_t = a.g[sh];
    const float beta_t = a.beta[sh];
    const float L_prev = n > 0 ? Lrow[n - 1] : 0.f;
    const bool writer = entry_writer && lane_entry < n;
    const float L_j = writer ? Lrow[lane_entry] : 0.f;
    float kq = 0.f;
#pragma unroll
    for (int c = 0; c < VEC; ++c) kq += kv[c] * qv[c];
    kq = warp_sum(kq);
    const float Lt = L_prev + g_t;
#pragma unroll
    for (int j = 0; j < NE; ++j) {
      float x = 0.f, y = 0.f;
      if (j < n) {
        float kj[VEC];
        ldvec_bf16<VEC>(kj, a.klog + (lh * Mcap + j) * DK + c0);
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
          x += kj[c] * kv[c];
          y += kj[c] * qv[c];
        }
      }
      p1[j] = x;
      p2[j] = y;
    }
    const float dkk = reduce_entries<NE>(p1, lane);
    const float dkq = reduce_entries<NE>(p2, lane);
    if (writer) {
      const float wj = expf(Lt - L_j);
      cf[HDR + lane_entry] = wj * dkk;
      cf[HDR + Mcap4 + lane_entry] = wj * dkq;
      if (merge) cf[Lay.P0 + lane_entry] = wj;
    }
    if (lane == 0) {
      cf[0] = expf(Lt);
      cf[1] = kq;
      cf[2] = beta_t;
      if (merge) cf[Lay.P0 + n] = 1.f;
      if (!merge) a.Llog[lh * Mcap + n] = Lt;
    }
  } else {
    // per-key decay: Λ vectors over this lane's key channels
    const float* Lbase = a.Llog + lh * Mcap * DK;
    float Lp[VEC], gt[VEC], Lt[VEC];
    if (n > 0) {
      ldvec<VEC>(Lp, Lbase + (size_t)(n - 1) * DK + c0);
    } else {
#pragma unroll
      for (int c = 0; c < VEC; ++c) Lp[c] = 0.f;
    }
    ldvec<VEC>(gt, a.g + (size_t)sh * DK + c0);
#pragma unroll
    for (int c = 0; c < VEC; ++c) Lt[c] = Lp[c] + gt[c];
    // Λ used by the coefficients: Λ_t (KDA), Λ_{t-1} (RWKV6: the output reads S_{t-1})
    float Lc[VEC], wt[VEC];
#pragma unroll
    for (int c = 0; c < VEC; ++c) {
      Lc[c] = (OP == KDA) ? Lt[c] : Lp[c];
      wt[c] = (OP == RWKV6) ? expf(gt[c]) : 1.f;
    }
    float* Kt = cf + Lay.P0 + DK;
    if constexpr (OP == KDA) {
      float kq = 0.f;
#pragma unroll
      for (int c = 0; c < VEC; ++c) {
        const float e = expf(Lt[c]);
        cf[vecA + c0 + c] = e * kv[c];
        cf[vecB + c0 + c] = e * qv[c];
        if (merge) {
          cf[Lay.P0 + c0 + c] = e;
          Kt[(size_t)n * DK + c0 + c] = kv[c];
        }
        kq += kv[c] * qv[c];
      }
      kq = warp_sum(kq);
      if (lane == 0) {
        cf[1] = kq;
        cf[2] = a.beta[sh];
      }
    } else {   // RWKV6: q holds r_t
      float bon[VEC];
      ldvec<VEC>(bon, a.bonus + (size_t)h * DK + c0);
      float cb = 0.f;
#pragma unroll
      for (int c = 0; c < VEC; ++c) {
        cf[vecA + c0 + c] = expf(Lp[c]) * qv[c];
        cb += qv[c] * bon[c] * kv[c];
        if (merge) {
          cf[Lay.P0 + c0 + c] = expf(Lt[c]);
          Kt[(size_t)n * DK + c0 + c] = kv[c];
        }
      }
      cb = warp_sum(cb);
      if (lane == 0) cf[3] = cb;
    }
    // entries in groups of 4: the group's key-log and log-decay rows are all
    // requested before any of them is used (a few round trips instead of n)
#pragma unroll
    for (int j0 = 0; j0 < NE; j0 += 4) {
      float kj[4][VEC], lj[4][VEC];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (j0 + u < n) {
          ldvec_bf16<VEC>(kj[u], a.klog + (lh * Mcap + j0 + u) * DK + c0);
          ldvec<VEC>(lj[u], Lbase + (size_t)(j0 + u) * DK + c0);
        } else {
#pragma unroll
          for (int c = 0; c < VEC; ++c) kj[u][c] = lj[u][c] = 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u;
        float x = 0.f, y = 0.f;
        if (j < n) {
          float kk[VEC];
#pragma unroll
          for (int c = 0; c < VEC; ++c) {
            kk[c] = kj[u][c] * __expf(Lc[c] - lj[u][c]);
            if (OP == KDA) {
              x += kk[c] * kv[c];
              y += kk[c] * qv[c];
            } else {
              x += kk[c] * qv[c];
            }
          }
          if (merge) {
            float km[VEC];
#pragma unroll
            for (int c = 0; c < VEC; ++c) km[c] = kk[c] * wt[c];   // K̃_j = k_j ⊙ e^{Λ_t-Λ_j}
            if constexpr (VEC == 4)
              *reinterpret_cast<float4*>(Kt + (size_t)j * DK + c0) = make_float4(km[0], km[1], km[2], km[3]);
            else
              *reinterpret_cast<float2*>(Kt + (size_t)j * DK + c0) = make_float2(km[0], km[1]);
          }
        }
        p1[j] = x;
        p2[j] = y;
      }
    }
    const float d1 = reduce_entries<NE>(p1, lane);
    float d2 = 0.f;
    if constexpr (OP == KDA) d2 = reduce_entries<NE>(p2, lane);
    if (entry_writer && lane_entry < n) {
      cf[HDR + lane_entry] = d1;
      if constexpr (OP == KDA) cf[HDR + Mcap4 + lane_entry] = d2;
    }
    if (!merge) {
      float* Ld = a.Llog + (lh * Mcap + n) * DK + c0;
#pragma unroll
      for (int c = 0; c < VEC; ++c) Ld[c] = Lt[c];
    }
  }

  if (!merge) {
    // append k_t (bf16 bits as they came) to the key log
    uint16_t* kd = a.klog + (lh * Mcap + n) * DK + c0;
    const uint16_t* ks = a.k + (size_t)sh * DK + c0;
#pragma unroll
    for (int c = 0; c < VEC; ++c) kd[c] = ks[c];
    if constexpr (OP == RWKV6) {
      // the value-side factor of RWKV6 is v_t itself
      uint16_t* vd = static_cast<uint16_t*>(a.alog) + (lh * Mcap + n) * DV;
      const uint16_t* vs = a.v + (size_t)sh * DV;
      for (int i = lane; i < DV; i += 32) vd[i] = vs[i];
    }
  }
  if (h == 0 && lane == 0) {
    a.nlog[slot] = merge ? 0 : n + 1;
    a.base_of[slot] = merge ? slot : it.base;
  }
}

template <int OP, int DK>
static cudaError_t launch_rp(const StepArgs& a, cudaStream_t s) {
  const int warps = a.rows * a.H;
  const int blocks = (warps + RP_WARPS - 1) / RP_WARPS;
  if (a.M - 1 <= 8) replay_prep_kernel<OP, DK, DK, 8><<<blocks, RP_WARPS * 32, 0, s>>>(a);
  else if (a.M - 1 <= 16) replay_prep_kernel<OP, DK, DK, 16><<<blocks, RP_WARPS * 32, 0, s>>>(a);
  else replay_prep_kernel<OP, DK, DK, 32><<<blocks, RP_WARPS * 32, 0, s>>>(a);
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
