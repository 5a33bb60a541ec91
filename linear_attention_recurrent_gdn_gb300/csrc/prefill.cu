// Chunked prefill: the state a slot reaches after a context of T tokens, with
// the outputs of those tokens, computed a chunk of C tokens at a time.
//
// Flide page, "Research method step by step", second step: the shared context
// of a request is processed once and its final recurrent state saved, before
// question branches start from it.  This kernel builds that state.  Within a
// chunk it uses the base + log algebra of the DeltaLog page ("Methodology —
// Base + Log"): with S̄ the state at the chunk start and Λ_j the cumulative
// log-decay inside the chunk (GDN: one scalar per token),
//   x_j = α_j S_{j-1} k_j = e^{Λ_j} (S̄ k_j) + Σ_{i<j} e^{Λ_j-Λ_i} (k_i·k_j) u_i
//   u_j = β_j (v_j - x_j)
//   o_j = e^{Λ_j} (S̄ q_j) + Σ_{i<=j} e^{Λ_j-Λ_i} (k_i·q_j) u_i
//   S̄'  = e^{Λ_C} S̄ + Σ_j u_j (e^{Λ_C-Λ_j} k_j)^T
// i.e. the token-by-token recurrence, reorganised so that all C tokens of a
// chunk share one pass over S̄ (S̄K^T, S̄Q^T), the u_j follow by forward
// substitution on each value row, and S̄ is rewritten once per chunk.
//
// One CTA (256 threads) per slot-head, looping over the chunks; S̄ stays in
// shared memory (rows padded to avoid bank conflicts) and goes to HBM at the end.
//
// The per-key ops (KDA, RWKV6) use the same algebra with a log-decay vector per
// key channel: Λ_j = Σ_{i<=j} g_i inside the chunk and, for i <= j,
//   KDA    x_j = S̄ (e^{Λ_j}⊙k_j) + Σ_{i<j} c^{kk}_{ji} u_i,   u_j = β_j (v_j - x_j)
//          o_j = S̄ (e^{Λ_j}⊙q_j) + Σ_{i<=j} c^{kq}_{ji} u_i
//          c^{kk}_{ji} = Σ_c k_i[c] k_j[c] e^{Λ_j[c]-Λ_i[c]}   (likewise c^{kq} with q_j)
//   RWKV6  o_j = S̄ (e^{Λ_{j-1}}⊙r_j) + Σ_{i<j} c^{kr}_{ji} v_i + (Σ_c r_j[c] b[c] k_j[c]) v_j
//          c^{kr}_{ji} = Σ_c k_i[c] r_j[c] e^{Λ_{j-1}[c]-Λ_i[c]}   (Λ_{-1} = 0)
//   S̄' = S̄ Diag(e^{Λ_C}) + Σ_j a_j (k_j ⊙ e^{Λ_C-Λ_j})^T      (a = u, or v for RWKV6)
// Every exponent is a difference Λ_late - Λ_early <= 0, so nothing overflows.
#include "dl_device.cuh"
#include "layout.h"
#include "launch.h"

namespace dl {

constexpr int PF_C = 32;          // tokens per chunk
constexpr int PF_THREADS = 256;

template <int DK, int DV>
struct PfSmem {
  static constexpr int SP = DK + 4;         // padded row stride of S̄, K, Q
  static constexpr int PP = PF_C + 1;       // padded row stride of Pk, Pq, U
  static constexpr int S_OFF = 0;
  static constexpr int K_OFF = S_OFF + DV * SP;
  static constexpr int Q_OFF = K_OFF + PF_C * SP;
  static constexpr int V_OFF = Q_OFF + PF_C * SP;
  static constexpr int PK_OFF = V_OFF + PF_C * DV;
  static constexpr int PQ_OFF = PK_OFF + DV * PP;
  static constexpr int U_OFF = PQ_OFF + DV * PP;
  static constexpr int AKK_OFF = U_OFF + DV * PP;
  static constexpr int AKQ_OFF = AKK_OFF + PF_C * PF_C;
  static constexpr int L_OFF = AKQ_OFF + PF_C * PF_C;
  static constexpr int B_OFF = L_OFF + PF_C;
  static constexpr int FLOATS = B_OFF + PF_C;
  static constexpr size_t BYTES = FLOATS * sizeof(float);
};

template <int DK, int DV>
__global__ void __launch_bounds__(PF_THREADS, 1) prefill_gdn_kernel(const __grid_constant__ SlotListArgs a,
                                                                    const uint16_t* __restrict__ q,
                                                                    const uint16_t* __restrict__ k,
                                                                    const uint16_t* __restrict__ v,
                                                                    const float* __restrict__ g,
                                                                    const float* __restrict__ beta,
                                                                    void* o, int T, int out_bf16,
                                                                    float scale) {
  using L = PfSmem<DK, DV>;
  extern __shared__ __align__(16) float sm[];
  float* Sb = sm + L::S_OFF;
  float* Kc = sm + L::K_OFF;
  float* Qc = sm + L::Q_OFF;
  float* Vc = sm + L::V_OFF;
  float* Pk = sm + L::PK_OFF;
  float* Pq = sm + L::PQ_OFF;
  float* Us = sm + L::U_OFF;
  float* Akk = sm + L::AKK_OFF;
  float* Akq = sm + L::AKQ_OFF;
  float* Lm = sm + L::L_OFF;
  float* Bt = sm + L::B_OFF;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sh = blockIdx.x, row = sh / a.H, h = sh - row * a.H;
  const int slot = a.items[row].slot;
  const size_t nH = (size_t)a.rows * a.H;              // slot-heads per token
  float* gS = a.Sbar + ((size_t)slot * a.H + h) * DV * DK;

  // load S̄ (padded rows)
  for (int idx = tid * 4; idx < DV * DK; idx += PF_THREADS * 4) {
    const int r = idx / DK, c = idx - r * DK;
    *reinterpret_cast<float4*>(Sb + r * L::SP + c) = *reinterpret_cast<const float4*>(gS + idx);
  }

  for (int t0 = 0; t0 < T; t0 += PF_C) {
    const int Cc = (T - t0) < PF_C ? (T - t0) : PF_C;
    __syncthreads();   // S̄ ready / previous chunk done with K, Q, V, U
    // ---- stage the chunk: K, Q, V as fp32, Λ (inclusive scan of g), beta
    for (int idx = tid; idx < PF_C * DK; idx += PF_THREADS) {
      const int j = idx / DK, c = idx - j * DK;
      float kx = 0.f, qx = 0.f;
      if (j < Cc) {
        const size_t base = ((size_t)(t0 + j) * nH + sh) * DK + c;
        kx = bf16f(k[base]);
        qx = bf16f(q[base]);
      }
      Kc[j * L::SP + c] = kx;
      Qc[j * L::SP + c] = qx;
    }
    for (int idx = tid; idx < PF_C * DV; idx += PF_THREADS) {
      const int j = idx / DV, c = idx - j * DV;
      Vc[idx] = j < Cc ? bf16f(v[((size_t)(t0 + j) * nH + sh) * DV + c]) : 0.f;
    }
    if (warp == 0) {
      float gj = lane < Cc ? g[(size_t)(t0 + lane) * nH + sh] : 0.f;
#pragma unroll
      for (int o2 = 1; o2 < 32; o2 <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, gj, o2);
        if (lane >= o2) gj += y;
      }
      Lm[lane] = gj;
      Bt[lane] = lane < Cc ? beta[(size_t)(t0 + lane) * nH + sh] : 0.f;
    }
    __syncthreads();
    // ---- decay-weighted key-key (strictly lower) and query-key (lower) products
    for (int p = tid; p < PF_C * PF_C; p += PF_THREADS) {
      const int j = p / PF_C, i = p - j * PF_C;
      float kk = 0.f, qk = 0.f;
      if (i <= j && j < Cc) {
        const float* kj = Kc + j * L::SP;
        const float* qj = Qc + j * L::SP;
        const float* ki = Kc + i * L::SP;
#pragma unroll 8
        for (int c = 0; c < DK; c += 4) {
          const float4 a4 = *reinterpret_cast<const float4*>(ki + c);
          const float4 b4 = *reinterpret_cast<const float4*>(kj + c);
          const float4 c4 = *reinterpret_cast<const float4*>(qj + c);
          kk += a4.x * b4.x + a4.y * b4.y + a4.z * b4.z + a4.w * b4.w;
          qk += a4.x * c4.x + a4.y * c4.y + a4.z * c4.z + a4.w * c4.w;
        }
        const float w = expf(Lm[j] - Lm[i]);
        kk *= w;
        qk *= w;
        if (i == j) kk = 0.f;
      }
      Akk[p] = kk;
      Akq[p] = qk;
    }
    // ---- S̄ K^T and S̄ Q^T: two threads per value row, 16 tokens each
    if ((tid >> 1) < DV) {
      const int r = tid >> 1, jh = (tid & 1) * (PF_C / 2);
      float pk[PF_C / 2], pq[PF_C / 2];
#pragma unroll
      for (int j = 0; j < PF_C / 2; ++j) pk[j] = pq[j] = 0.f;
      const float* sr = Sb + r * L::SP;
      for (int c = 0; c < DK; c += 4) {
        const float4 s4 = *reinterpret_cast<const float4*>(sr + c);
#pragma unroll
        for (int j = 0; j < PF_C / 2; ++j) {
          const float4 k4 = *reinterpret_cast<const float4*>(Kc + (jh + j) * L::SP + c);
          const float4 q4 = *reinterpret_cast<const float4*>(Qc + (jh + j) * L::SP + c);
          pk[j] += s4.x * k4.x + s4.y * k4.y + s4.z * k4.z + s4.w * k4.w;
          pq[j] += s4.x * q4.x + s4.y * q4.y + s4.z * q4.z + s4.w * q4.w;
        }
      }
#pragma unroll
      for (int j = 0; j < PF_C / 2; ++j) {
        Pk[r * L::PP + jh + j] = pk[j];
        Pq[r * L::PP + jh + j] = pq[j];
      }
    }
    __syncthreads();
    // ---- forward substitution for u, then the outputs: one thread per value row
    if (tid < DV) {
      const int r = tid;
      float u[PF_C];
#pragma unroll
      for (int j = 0; j < PF_C; ++j) {
        float x = expf(Lm[j]) * Pk[r * L::PP + j];
#pragma unroll
        for (int i = 0; i < j; ++i) x += Akk[j * PF_C + i] * u[i];
        u[j] = (j < Cc) ? Bt[j] * (Vc[j * DV + r] - x) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < PF_C; ++j) {
        Us[r * L::PP + j] = u[j];
        if (o != nullptr && j < Cc) {
          float y = expf(Lm[j]) * Pq[r * L::PP + j];
#pragma unroll
          for (int i = 0; i <= j; ++i) y += Akq[j * PF_C + i] * u[i];
          const size_t oi = ((size_t)(t0 + j) * nH + sh) * DV + r;
          if (out_bf16) static_cast<uint16_t*>(o)[oi] = f2bf16(scale * y);
          else static_cast<float*>(o)[oi] = scale * y;
        }
      }
    }
    __syncthreads();
    // ---- S̄ <- e^{Λ_C} S̄ + Σ_j u_j (e^{Λ_C-Λ_j} k_j)^T: two threads per row, half a row each
    if ((tid >> 1) < DV) {
      const int r = tid >> 1, c0 = (tid & 1) * (DK / 2);
      const float LC = Lm[Cc - 1];
      float acc[DK / 2];
      const float eC = expf(LC);
#pragma unroll
      for (int c = 0; c < DK / 2; c += 4) {
        const float4 s4 = *reinterpret_cast<const float4*>(Sb + r * L::SP + c0 + c);
        acc[c] = eC * s4.x; acc[c + 1] = eC * s4.y; acc[c + 2] = eC * s4.z; acc[c + 3] = eC * s4.w;
      }
      for (int j = 0; j < Cc; ++j) {
        const float w = Us[r * L::PP + j] * expf(LC - Lm[j]);
#pragma unroll
        for (int c = 0; c < DK / 2; c += 4) {
          const float4 k4 = *reinterpret_cast<const float4*>(Kc + j * L::SP + c0 + c);
          acc[c] += w * k4.x; acc[c + 1] += w * k4.y; acc[c + 2] += w * k4.z; acc[c + 3] += w * k4.w;
        }
      }
#pragma unroll
      for (int c = 0; c < DK / 2; c += 4)
        *reinterpret_cast<float4*>(Sb + r * L::SP + c0 + c) =
            make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
    }
  }
  __syncthreads();
  for (int idx = tid * 4; idx < DV * DK; idx += PF_THREADS * 4) {
    const int r = idx / DK, c = idx - r * DK;
    *reinterpret_cast<float4*>(gS + idx) = *reinterpret_cast<const float4*>(Sb + r * L::SP + c);
  }
  if (h == 0 && tid == 0) {
    a.nlog[slot] = 0;
    a.base_of[slot] = slot;
  }
}

template <int DK>
static cudaError_t pf_dispatch(const SlotListArgs& a, const void* q, const void* k, const void* v,
                               const float* g, const float* beta, void* o, int T, int out_bf16,
                               float scale, cudaStream_t s) {
  using L = PfSmem<DK, DK>;
  cudaError_t e = cudaFuncSetAttribute(prefill_gdn_kernel<DK, DK>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::BYTES);
  if (e != cudaSuccess) return e;
  prefill_gdn_kernel<DK, DK><<<a.rows * a.H, PF_THREADS, L::BYTES, s>>>(
      a, static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k),
      static_cast<const uint16_t*>(v), g, beta, o, T, out_bf16, scale);
  return cudaGetLastError();
}


// ------------------------------------------------------------ per-key ops --
template <int DK, int DV>
struct PkSmem {
  static constexpr int SP = DK + 4;         // padded row stride of S̄, K, Q, Λ, X
  static constexpr int PP = PF_C + 1;       // padded row stride of Pk, Pq, U
  static constexpr int S_OFF = 0;
  static constexpr int K_OFF = S_OFF + DV * SP;
  static constexpr int Q_OFF = K_OFF + PF_C * SP;    // q (KDA) or r (RWKV6), then its hat
  static constexpr int L_OFF = Q_OFF + PF_C * SP;    // Λ rows
  static constexpr int X_OFF = L_OFF + PF_C * SP;    // e^{Λ_j}⊙k_j, then k_j⊙e^{Λ_C-Λ_j}
  static constexpr int V_OFF = X_OFF + PF_C * SP;
  static constexpr int PK_OFF = V_OFF + PF_C * DV;
  static constexpr int PQ_OFF = PK_OFF + DV * PP;
  static constexpr int U_OFF = PQ_OFF + DV * PP;
  static constexpr int AKK_OFF = U_OFF + DV * PP;
  static constexpr int AKQ_OFF = AKK_OFF + PF_C * PF_C;
  static constexpr int B_OFF = AKQ_OFF + PF_C * PF_C;
  static constexpr int CB_OFF = B_OFF + PF_C;
  static constexpr int E_OFF = CB_OFF + PF_C;
  static constexpr int FLOATS = E_OFF + DK;
  static constexpr size_t BYTES = FLOATS * sizeof(float);
};

template <int OP, int DK, int DV>
__global__ void __launch_bounds__(PF_THREADS, 1) prefill_perkey_kernel(
    const __grid_constant__ SlotListArgs a, const uint16_t* __restrict__ q,
    const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, const float* __restrict__ g,
    const float* __restrict__ beta, const float* __restrict__ bonus, void* o, int T,
    int out_bf16, float scale) {
  using L = PkSmem<DK, DV>;
  constexpr bool DELTA = (OP == KDA);
  extern __shared__ __align__(16) float sm[];
  float* Sb = sm + L::S_OFF;
  float* Kc = sm + L::K_OFF;
  float* Qc = sm + L::Q_OFF;
  float* Lc = sm + L::L_OFF;
  float* Xc = sm + L::X_OFF;
  float* Vc = sm + L::V_OFF;
  float* Pk = sm + L::PK_OFF;
  float* Pq = sm + L::PQ_OFF;
  float* Us = sm + L::U_OFF;
  float* Akk = sm + L::AKK_OFF;
  float* Akq = sm + L::AKQ_OFF;
  float* Bt = sm + L::B_OFF;
  float* Cb = sm + L::CB_OFF;
  float* Ec = sm + L::E_OFF;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sh = blockIdx.x, row = sh / a.H, h = sh - row * a.H;
  const int slot = a.items[row].slot;
  const size_t nH = (size_t)a.rows * a.H;
  float* gS = a.Sbar + ((size_t)slot * a.H + h) * DV * DK;

  for (int idx = tid * 4; idx < DV * DK; idx += PF_THREADS * 4) {
    const int r = idx / DK, c = idx - r * DK;
    *reinterpret_cast<float4*>(Sb + r * L::SP + c) = *reinterpret_cast<const float4*>(gS + idx);
  }

  for (int t0 = 0; t0 < T; t0 += PF_C) {
    const int Cc = (T - t0) < PF_C ? (T - t0) : PF_C;
    __syncthreads();   // S̄ ready / previous chunk done with every buffer
    // ---- stage the chunk (tokens past the end: zero inputs, zero decay)
    for (int idx = tid; idx < PF_C * DK; idx += PF_THREADS) {
      const int j = idx / DK, c = idx - j * DK;
      float kx = 0.f, qx = 0.f, gx = 0.f;
      if (j < Cc) {
        const size_t base = ((size_t)(t0 + j) * nH + sh) * DK + c;
        kx = bf16f(k[base]);
        qx = bf16f(q[base]);
        gx = g[base];
      }
      Kc[j * L::SP + c] = kx;
      Qc[j * L::SP + c] = qx;
      Lc[j * L::SP + c] = gx;
    }
    for (int idx = tid; idx < PF_C * DV; idx += PF_THREADS) {
      const int j = idx / DV, c = idx - j * DV;
      Vc[idx] = j < Cc ? bf16f(v[((size_t)(t0 + j) * nH + sh) * DV + c]) : 0.f;
    }
    if (DELTA && warp == 0) Bt[lane] = lane < Cc ? beta[(size_t)(t0 + lane) * nH + sh] : 0.f;
    __syncthreads();
    // ---- Λ: inclusive scan of g down each key channel; e^{Λ_C}
    if (tid < DK) {
      float acc = 0.f;
      for (int j = 0; j < PF_C; ++j) {
        acc += Lc[j * L::SP + tid];
        Lc[j * L::SP + tid] = acc;
      }
      Ec[tid] = expf(acc);
    }
    if constexpr (!DELTA) {
      // bonus coefficient of each token: Σ_c r_j[c] b[c] k_j[c] (one warp per token)
      for (int j = warp; j < PF_C; j += PF_THREADS / 32) {
        float s = 0.f;
        for (int c = lane; c < DK; c += 32)
          s += Qc[j * L::SP + c] * bonus[(size_t)h * DK + c] * Kc[j * L::SP + c];
        s = warp_sum(s);
        if (lane == 0) Cb[j] = s;
      }
    }
    __syncthreads();
    // ---- decay-weighted pair coefficients (i <= j; the exponents are <= 0)
    for (int p = tid; p < PF_C * PF_C; p += PF_THREADS) {
      const int j = p / PF_C, i = p - j * PF_C;
      float kk = 0.f, qk = 0.f;
      const bool live = DELTA ? (i <= j && j < Cc) : (i < j && j < Cc);
      if (live) {
        const float* ki = Kc + i * L::SP;
        const float* kj = Kc + j * L::SP;
        const float* qj = Qc + j * L::SP;
        const float* li = Lc + i * L::SP;
        const float* lj = Lc + (DELTA ? j : j - 1) * L::SP;   // RWKV6 reads S_{j-1}
#pragma unroll 4
        for (int c = 0; c < DK; ++c) {
          const float w = __expf(lj[c] - li[c]);
          const float kw = ki[c] * w;
          if (DELTA) kk += kw * kj[c];
          qk += kw * qj[c];
        }
        if (DELTA && i == j) kk = 0.f;
      }
      Akk[p] = kk;
      Akq[p] = qk;
    }
    __syncthreads();
    // ---- hats: e^{Λ_j}⊙k_j (KDA) into X; e^{Λ_j}⊙q_j (KDA) or e^{Λ_{j-1}}⊙r_j in place
    for (int idx = tid; idx < PF_C * DK; idx += PF_THREADS) {
      const int j = idx / DK, c = idx - j * DK;
      if (DELTA) {
        const float e = expf(Lc[j * L::SP + c]);
        Xc[j * L::SP + c] = e * Kc[j * L::SP + c];
        Qc[j * L::SP + c] *= e;
      } else {
        Qc[j * L::SP + c] *= (j > 0) ? expf(Lc[(j - 1) * L::SP + c]) : 1.f;
      }
    }
    __syncthreads();
    // ---- S̄ products: two threads per value row, 16 tokens each
    if ((tid >> 1) < DV) {
      const int r = tid >> 1, jh = (tid & 1) * (PF_C / 2);
      float pk[PF_C / 2], pq[PF_C / 2];
#pragma unroll
      for (int j = 0; j < PF_C / 2; ++j) pk[j] = pq[j] = 0.f;
      const float* sr = Sb + r * L::SP;
      for (int c = 0; c < DK; c += 4) {
        const float4 s4 = *reinterpret_cast<const float4*>(sr + c);
#pragma unroll
        for (int j = 0; j < PF_C / 2; ++j) {
          const float4 q4 = *reinterpret_cast<const float4*>(Qc + (jh + j) * L::SP + c);
          pq[j] += s4.x * q4.x + s4.y * q4.y + s4.z * q4.z + s4.w * q4.w;
          if (DELTA) {
            const float4 k4 = *reinterpret_cast<const float4*>(Xc + (jh + j) * L::SP + c);
            pk[j] += s4.x * k4.x + s4.y * k4.y + s4.z * k4.z + s4.w * k4.w;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < PF_C / 2; ++j) {
        Pk[r * L::PP + jh + j] = pk[j];
        Pq[r * L::PP + jh + j] = pq[j];
      }
    }
    __syncthreads();
    // ---- the appended factors and the outputs: one thread per value row
    if (tid < DV) {
      const int r = tid;
      float u[PF_C];
#pragma unroll
      for (int j = 0; j < PF_C; ++j) {
        if (DELTA) {
          float x = Pk[r * L::PP + j];
#pragma unroll
          for (int i = 0; i < j; ++i) x += Akk[j * PF_C + i] * u[i];
          u[j] = (j < Cc) ? Bt[j] * (Vc[j * DV + r] - x) : 0.f;
        } else {
          u[j] = Vc[j * DV + r];
        }
      }
#pragma unroll
      for (int j = 0; j < PF_C; ++j) {
        Us[r * L::PP + j] = u[j];
        if (o != nullptr && j < Cc) {
          float y = Pq[r * L::PP + j];
#pragma unroll
          for (int i = 0; i <= j; ++i) y += Akq[j * PF_C + i] * u[i];   // (RWKV6: zero at i = j)
          if (!DELTA) y += Cb[j] * u[j];
          const size_t oi = ((size_t)(t0 + j) * nH + sh) * DV + r;
          if (out_bf16) static_cast<uint16_t*>(o)[oi] = f2bf16(scale * y);
          else static_cast<float*>(o)[oi] = scale * y;
        }
      }
    }
    // ---- k_j ⊙ e^{Λ_C-Λ_j} into X (X's hats are no longer read)
    for (int idx = tid; idx < PF_C * DK; idx += PF_THREADS) {
      const int j = idx / DK, c = idx - j * DK;
      Xc[j * L::SP + c] =
          Kc[j * L::SP + c] * expf(Lc[(PF_C - 1) * L::SP + c] - Lc[j * L::SP + c]);
    }
    __syncthreads();
    // ---- S̄ <- S̄ Diag(e^{Λ_C}) + Σ_j a_j (k_j ⊙ e^{Λ_C-Λ_j})^T: two threads per row
    if ((tid >> 1) < DV) {
      const int r = tid >> 1, c0 = (tid & 1) * (DK / 2);
      float acc[DK / 2];
#pragma unroll
      for (int c = 0; c < DK / 2; c += 4) {
        const float4 s4 = *reinterpret_cast<const float4*>(Sb + r * L::SP + c0 + c);
        const float4 e4 = *reinterpret_cast<const float4*>(Ec + c0 + c);
        acc[c] = e4.x * s4.x; acc[c + 1] = e4.y * s4.y; acc[c + 2] = e4.z * s4.z; acc[c + 3] = e4.w * s4.w;
      }
      for (int j = 0; j < Cc; ++j) {
        const float w = Us[r * L::PP + j];
#pragma unroll
        for (int c = 0; c < DK / 2; c += 4) {
          const float4 k4 = *reinterpret_cast<const float4*>(Xc + j * L::SP + c0 + c);
          acc[c] += w * k4.x; acc[c + 1] += w * k4.y; acc[c + 2] += w * k4.z; acc[c + 3] += w * k4.w;
        }
      }
#pragma unroll
      for (int c = 0; c < DK / 2; c += 4)
        *reinterpret_cast<float4*>(Sb + r * L::SP + c0 + c) =
            make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
    }
  }
  __syncthreads();
  for (int idx = tid * 4; idx < DV * DK; idx += PF_THREADS * 4) {
    const int r = idx / DK, c = idx - r * DK;
    *reinterpret_cast<float4*>(gS + idx) = *reinterpret_cast<const float4*>(Sb + r * L::SP + c);
  }
  if (h == 0 && tid == 0) {
    a.nlog[slot] = 0;
    a.base_of[slot] = slot;
  }
}

template <int OP, int DK>
static cudaError_t pk_dispatch(const SlotListArgs& a, const void* q, const void* k, const void* v,
                               const float* g, const float* beta, const float* bonus, void* o,
                               int T, int out_bf16, float scale, cudaStream_t s) {
  using L = PkSmem<DK, DK>;
  cudaError_t e = cudaFuncSetAttribute(prefill_perkey_kernel<OP, DK, DK>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::BYTES);
  if (e != cudaSuccess) return e;
  prefill_perkey_kernel<OP, DK, DK><<<a.rows * a.H, PF_THREADS, L::BYTES, s>>>(
      a, static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k),
      static_cast<const uint16_t*>(v), g, beta, bonus, o, T, out_bf16, scale);
  return cudaGetLastError();
}

cudaError_t launch_prefill(int op, int dk, const SlotListArgs& a, const void* q, const void* k,
                           const void* v, const float* g, const float* beta, const float* bonus,
                           void* o, int T, int out_bf16, float scale, cudaStream_t s) {
  if (a.rows <= 0 || T <= 0) return cudaSuccess;
  if (op == GDN) {
    if (dk == 64) return pf_dispatch<64>(a, q, k, v, g, beta, o, T, out_bf16, scale, s);
    return pf_dispatch<128>(a, q, k, v, g, beta, o, T, out_bf16, scale, s);
  }
  if (op == KDA) {
    if (dk == 64) return pk_dispatch<KDA, 64>(a, q, k, v, g, beta, bonus, o, T, out_bf16, scale, s);
    return pk_dispatch<KDA, 128>(a, q, k, v, g, beta, bonus, o, T, out_bf16, scale, s);
  }
  if (dk == 64) return pk_dispatch<RWKV6, 64>(a, q, k, v, g, beta, bonus, o, T, out_bf16, scale, s);
  return pk_dispatch<RWKV6, 128>(a, q, k, v, g, beta, bonus, o, T, out_bf16, scale, s);
}

}  // namespace dl
