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
  static constexpr int AKK_OFF = U_OFF + DV * PP;            // [C][PP]: padded rows
  static constexpr int AKQ_OFF = AKK_OFF + PF_C * PP;
  static constexpr int L_OFF = AKQ_OFF + PF_C * PP;
  static constexpr int B_OFF = L_OFF + PF_C;
  static constexpr int EL_OFF = B_OFF + PF_C;                  // e^{Λ_j}
  static constexpr int EW_OFF = EL_OFF + PF_C;                 // e^{Λ_C - Λ_j}
  static constexpr int FLOATS = EW_OFF + PF_C;
  static constexpr size_t BYTES = FLOATS * sizeof(float);
};

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float dot4(float acc, const float4 a, const float4 b) {
  acc += a.x * b.x;
  acc += a.y * b.y;
  acc += a.z * b.z;
  return acc + a.w * b.w;
}

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
  float* El = sm + L::EL_OFF;
  float* Ew = sm + L::EW_OFF;
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
      const float LC = __shfl_sync(0xffffffffu, gj, Cc - 1);
      Lm[lane] = gj;
      El[lane] = expf(gj);
      Ew[lane] = lane < Cc ? expf(LC - gj) : 0.f;   // padding tokens add nothing
      Bt[lane] = lane < Cc ? beta[(size_t)(t0 + lane) * nH + sh] : 0.f;
    }
    __syncthreads();
    // Register tiles below are laid out so that each warp-wide load of a
    // padded row (stride DK + 4 floats, 4 banks apart) touches distinct banks.
    // ---- decay-weighted key-key (strictly lower) and query-key (lower) products:
    //      a 2x2 block (tokens j = jg, jg + 16; i = ig, ig + 16) per thread
    {
      const int jg = tid >> 4, ig = tid & 15;
      float kk[2][2] = {{0.f, 0.f}, {0.f, 0.f}}, qk[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll 4
      for (int c = 0; c < DK; c += 4) {
        const float4 ki0 = ld4(Kc + ig * L::SP + c), ki1 = ld4(Kc + (ig + 16) * L::SP + c);
        const float4 kj0 = ld4(Kc + jg * L::SP + c), kj1 = ld4(Kc + (jg + 16) * L::SP + c);
        const float4 qj0 = ld4(Qc + jg * L::SP + c), qj1 = ld4(Qc + (jg + 16) * L::SP + c);
        kk[0][0] = dot4(kk[0][0], kj0, ki0);
        kk[0][1] = dot4(kk[0][1], kj0, ki1);
        kk[1][0] = dot4(kk[1][0], kj1, ki0);
        kk[1][1] = dot4(kk[1][1], kj1, ki1);
        qk[0][0] = dot4(qk[0][0], qj0, ki0);
        qk[0][1] = dot4(qk[0][1], qj0, ki1);
        qk[1][0] = dot4(qk[1][0], qj1, ki0);
        qk[1][1] = dot4(qk[1][1], qj1, ki1);
      }
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int y = 0; y < 2; ++y) {
          const int j = jg + 16 * x, i = ig + 16 * y;
          const float w = (i <= j && j < Cc) ? expf(Lm[j] - Lm[i]) : 0.f;   // exponent <= 0
          Akk[j * L::PP + i] = i < j ? kk[x][y] * w : 0.f;
          Akq[j * L::PP + i] = qk[x][y] * w;
        }
    }
    // ---- S̄ K^T and S̄ Q^T: rows rg + 32 m, tokens tg + 8 t per thread
    {
      constexpr int RPT = DV / 32;
      const int rg = tid >> 3, tg = tid & 7;
      float pk[RPT][4], pq[RPT][4];
#pragma unroll
      for (int m = 0; m < RPT; ++m)
#pragma unroll
        for (int t = 0; t < 4; ++t) pk[m][t] = pq[m][t] = 0.f;
#pragma unroll 2
      for (int c = 0; c < DK; c += 4) {
        float4 s4[RPT], k4[4], q4[4];
#pragma unroll
        for (int m = 0; m < RPT; ++m) s4[m] = ld4(Sb + (rg + 32 * m) * L::SP + c);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          k4[t] = ld4(Kc + (tg + 8 * t) * L::SP + c);
          q4[t] = ld4(Qc + (tg + 8 * t) * L::SP + c);
        }
#pragma unroll
        for (int m = 0; m < RPT; ++m)
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            pk[m][t] = dot4(pk[m][t], s4[m], k4[t]);
            pq[m][t] = dot4(pq[m][t], s4[m], q4[t]);
          }
      }
#pragma unroll
      for (int m = 0; m < RPT; ++m)
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          Pk[(rg + 32 * m) * L::PP + tg + 8 * t] = pk[m][t];
          Pq[(rg + 32 * m) * L::PP + tg + 8 * t] = pq[m][t];
        }
    }
    __syncthreads();
    // ---- forward substitution for u, then the outputs: one thread per value
    //      row; each sum runs in four partial sums to shorten its chain
    if (tid < DV) {
      const int r = tid;
      float u[PF_C];
#pragma unroll
      for (int j = 0; j < PF_C; ++j) {
        float x[4] = {El[j] * Pk[r * L::PP + j], 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < j; ++i) x[i & 3] += Akk[j * L::PP + i] * u[i];
        u[j] = Bt[j] * (Vc[j * DV + r] - ((x[0] + x[1]) + (x[2] + x[3])));   // 0 past Cc
      }
#pragma unroll
      for (int j = 0; j < PF_C; ++j) {
        Us[r * L::PP + j] = u[j];
        if (o != nullptr && j < Cc) {
          float y[4] = {El[j] * Pq[r * L::PP + j], 0.f, 0.f, 0.f};
#pragma unroll
          for (int i = 0; i <= j; ++i) y[i & 3] += Akq[j * L::PP + i] * u[i];
          const float yo = (y[0] + y[1]) + (y[2] + y[3]);
          const size_t oi = ((size_t)(t0 + j) * nH + sh) * DV + r;
          if (out_bf16) static_cast<uint16_t*>(o)[oi] = f2bf16(scale * yo);
          else static_cast<float*>(o)[oi] = scale * yo;
        }
      }
    }
    __syncthreads();
    // ---- S̄ <- e^{Λ_C} S̄ + Σ_j u_j (e^{Λ_C-Λ_j} k_j)^T: rows rg + 32 m and
    //      column quads 4 tg + 32 n per thread
    {
      constexpr int RPT = DV / 32, CPT = DK / 32;
      const int rg = tid >> 3, tg = tid & 7;
      const float eC = El[Cc - 1];
      float4 acc[RPT][CPT];
#pragma unroll
      for (int m = 0; m < RPT; ++m)
#pragma unroll
        for (int n4 = 0; n4 < CPT; ++n4) {
          const float4 s4 = ld4(Sb + (rg + 32 * m) * L::SP + 4 * tg + 32 * n4);
          acc[m][n4] = make_float4(eC * s4.x, eC * s4.y, eC * s4.z, eC * s4.w);
        }
      for (int j = 0; j < Cc; ++j) {
        const float ew = Ew[j];
        float w[RPT];
#pragma unroll
        for (int m = 0; m < RPT; ++m) w[m] = Us[(rg + 32 * m) * L::PP + j] * ew;
#pragma unroll
        for (int n4 = 0; n4 < CPT; ++n4) {
          const float4 k4 = ld4(Kc + j * L::SP + 4 * tg + 32 * n4);
#pragma unroll
          for (int m = 0; m < RPT; ++m) {
            acc[m][n4].x += w[m] * k4.x;
            acc[m][n4].y += w[m] * k4.y;
            acc[m][n4].z += w[m] * k4.z;
            acc[m][n4].w += w[m] * k4.w;
          }
        }
      }
#pragma unroll
      for (int m = 0; m < RPT; ++m)
#pragma unroll
        for (int n4 = 0; n4 < CPT; ++n4)
          *reinterpret_cast<float4*>(Sb + (rg + 32 * m) * L::SP + 4 * tg + 32 * n4) = acc[m][n4];
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
