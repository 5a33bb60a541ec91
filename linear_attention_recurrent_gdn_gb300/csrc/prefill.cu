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
// The work is FP32 arithmetic.  Each thread keeps register tiles of the chunk's
// contractions (rows rg + 32m against tokens tg + 8t or column quads), laid out
// so that every warp-wide 16-byte shared-memory load touches distinct banks,
// and the next chunk's inputs load into registers while the current one computes.
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

// One chunk's inputs in registers, between their 16-byte global loads and their
// shared-memory stores: the next chunk's loads are in flight while the current
// chunk computes.  (q, k, v are 16-byte aligned and each token's row of a
// slot-head is d * 2 bytes, so every vector load is aligned.)
template <int D>
struct PfStage {
  static constexpr int VPR = D / 8;                         // 16-byte vectors per row
  static constexpr int NV = PF_C * VPR / PF_THREADS;        // vectors per thread per tensor
  static_assert(NV >= 1 && NV * PF_THREADS == PF_C * VPR, "chunk rows must split evenly");
  uint4 k[NV], q[NV], v[NV];
  float g, b;

  __device__ __forceinline__ void load(const uint16_t* __restrict__ qg,
                                       const uint16_t* __restrict__ kg,
                                       const uint16_t* __restrict__ vg, const float* __restrict__ gg,
                                       const float* __restrict__ bg, int t0, int Cc, size_t nH,
                                       int sh, int tid) {
#pragma unroll
    for (int e = 0; e < NV; ++e) {
      const int idx = tid + e * PF_THREADS, j = idx / VPR, cv = idx - j * VPR;
      if (j < Cc) {
        const size_t base = ((size_t)(t0 + j) * nH + sh) * D + cv * 8;
        k[e] = *reinterpret_cast<const uint4*>(kg + base);
        q[e] = *reinterpret_cast<const uint4*>(qg + base);
        v[e] = *reinterpret_cast<const uint4*>(vg + base);
      } else {
        k[e] = q[e] = v[e] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    if (tid < 32) {
      g = tid < Cc ? gg[(size_t)(t0 + tid) * nH + sh] : 0.f;
      b = tid < Cc ? bg[(size_t)(t0 + tid) * nH + sh] : 0.f;
    }
  }

  // K and Q rows at stride SP (padded), V rows at stride D, as fp32
  __device__ __forceinline__ void store(float* Kc, float* Qc, float* Vc, int SP, int tid) const {
#pragma unroll
    for (int e = 0; e < NV; ++e) {
      const int idx = tid + e * PF_THREADS, j = idx / VPR, cv = idx - j * VPR;
      put8(Kc + j * SP + cv * 8, k[e]);
      put8(Qc + j * SP + cv * 8, q[e]);
      put8(Vc + j * D + cv * 8, v[e]);
    }
  }

  static __device__ __forceinline__ void put8(float* dst, const uint4 w) {
    *reinterpret_cast<float4*>(dst) =
        make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                    __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
    *reinterpret_cast<float4*>(dst + 4) =
        make_float4(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xffff0000u),
                    __uint_as_float(w.w << 16), __uint_as_float(w.w & 0xffff0000u));
  }
};
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

  static_assert(DK == DV, "square state");
  PfStage<DK> st;
  st.load(q, k, v, g, beta, 0, T < PF_C ? T : PF_C, nH, sh, tid);
  for (int t0 = 0; t0 < T; t0 += PF_C) {
    const int Cc = (T - t0) < PF_C ? (T - t0) : PF_C;
    __syncthreads();   // S̄ ready / previous chunk done with K, Q, V, U
    // ---- stage the chunk from registers: K, Q, V as fp32, Λ (inclusive scan
    //      of g), beta; then start loading the next chunk
    st.store(Kc, Qc, Vc, L::SP, tid);
    if (warp == 0) {
      float gj = st.g;
#pragma unroll
      for (int o2 = 1; o2 < 32; o2 <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, gj, o2);
        if (lane >= o2) gj += y;
      }
      const float LC = __shfl_sync(0xffffffffu, gj, Cc - 1);
      Lm[lane] = gj;
      El[lane] = expf(gj);
      Ew[lane] = lane < Cc ? expf(LC - gj) : 0.f;   // padding tokens add nothing
      Bt[lane] = st.b;                               // 0 past Cc
    }
    if (t0 + PF_C < T) {
      const int Cn = (T - t0 - PF_C) < PF_C ? (T - t0 - PF_C) : PF_C;
      st.load(q, k, v, g, beta, t0 + PF_C, Cn, nH, sh, tid);
    }
    __syncthreads();
    // Register tiles below are laid out so that each warp-wide load of a
    // padded row (stride DK + 4 floats, 4 banks apart) touches distinct banks.
    // ---- decay-weighted key-key (strictly lower) and query-key (lower) products:
    //      a 2x2 block (tokens j = jg, jg + 16; i = ig, ig + 16) per thread, whose
    //      corner (jg, ig + 16) lies above the diagonal and is not computed
    {
      const int jg = tid >> 4, ig = tid & 15;
      float kk[2][2] = {{0.f, 0.f}, {0.f, 0.f}}, qk[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll 4
      for (int c = 0; c < DK; c += 4) {
        const float4 ki0 = ld4(Kc + ig * L::SP + c), ki1 = ld4(Kc + (ig + 16) * L::SP + c);
        const float4 kj0 = ld4(Kc + jg * L::SP + c), kj1 = ld4(Kc + (jg + 16) * L::SP + c);
        const float4 qj0 = ld4(Qc + jg * L::SP + c), qj1 = ld4(Qc + (jg + 16) * L::SP + c);
        kk[0][0] = dot4(kk[0][0], kj0, ki0);
        kk[1][0] = dot4(kk[1][0], kj1, ki0);
        kk[1][1] = dot4(kk[1][1], kj1, ki1);
        qk[0][0] = dot4(qk[0][0], qj0, ki0);
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
#pragma unroll 4
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
  static constexpr int PA = PF_C + 4;       // row stride of Akk, Akq (16-byte aligned rows)
  static constexpr int AKK_OFF = U_OFF + DV * PP;            // [C][PA]
  static constexpr int AKQ_OFF = AKK_OFF + PF_C * PA;
  static constexpr int B_OFF = AKQ_OFF + PF_C * PA;
  static constexpr int CB_OFF = B_OFF + PF_C;
  static constexpr int E_OFF = CB_OFF + PF_C;
  static constexpr int FLOATS = E_OFF + DK;
  static constexpr size_t BYTES = FLOATS * sizeof(float);
};

// The per-key ops' chunk inputs in registers: k, q (r), v as in PfStage, and
// the g rows (fp32, one log-decay per key channel; 16-byte aligned rows).
template <int D>
struct PkStage {
  static constexpr int VPR = D / 8, NV = PF_C * VPR / PF_THREADS;
  static constexpr int GPR = D / 4, NG = PF_C * GPR / PF_THREADS;   // float4 of g
  static_assert(NV * PF_THREADS == PF_C * VPR && NG * PF_THREADS == PF_C * GPR, "even split");
  uint4 k[NV], q[NV], v[NV];
  float4 gv[NG];
  float b;

  __device__ __forceinline__ void load(const uint16_t* __restrict__ qg,
                                       const uint16_t* __restrict__ kg,
                                       const uint16_t* __restrict__ vg, const float* __restrict__ gg,
                                       const float* __restrict__ bg, int t0, int Cc, size_t nH,
                                       int sh, int tid) {
#pragma unroll
    for (int e = 0; e < NV; ++e) {
      const int idx = tid + e * PF_THREADS, j = idx / VPR, cv = idx - j * VPR;
      if (j < Cc) {
        const size_t base = ((size_t)(t0 + j) * nH + sh) * D + cv * 8;
        k[e] = *reinterpret_cast<const uint4*>(kg + base);
        q[e] = *reinterpret_cast<const uint4*>(qg + base);
        v[e] = *reinterpret_cast<const uint4*>(vg + base);
      } else {
        k[e] = q[e] = v[e] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int e = 0; e < NG; ++e) {
      const int idx = tid + e * PF_THREADS, j = idx / GPR, c4 = idx - j * GPR;
      gv[e] = j < Cc ? *reinterpret_cast<const float4*>(gg + ((size_t)(t0 + j) * nH + sh) * D + c4 * 4)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (tid < 32) b = (bg != nullptr && tid < Cc) ? bg[(size_t)(t0 + tid) * nH + sh] : 0.f;
  }

  // k, q rows and the g rows at stride SP, v rows at stride D, as fp32
  __device__ __forceinline__ void store(float* Kc, float* Qc, float* Lc, float* Vc, int SP,
                                        int tid) const {
#pragma unroll
    for (int e = 0; e < NV; ++e) {
      const int idx = tid + e * PF_THREADS, j = idx / VPR, cv = idx - j * VPR;
      PfStage<D>::put8(Kc + j * SP + cv * 8, k[e]);
      PfStage<D>::put8(Qc + j * SP + cv * 8, q[e]);
      PfStage<D>::put8(Vc + j * D + cv * 8, v[e]);
    }
#pragma unroll
    for (int e = 0; e < NG; ++e) {
      const int idx = tid + e * PF_THREADS, j = idx / GPR, c4 = idx - j * GPR;
      *reinterpret_cast<float4*>(Lc + j * SP + c4 * 4) = gv[e];
    }
  }
};

// One channel quad of a decay-weighted pair product: w_c = e^{Λ_j[c] - Λ_i[c]}
// (for a pair that is not live the exponent is replaced by 0, so the unused
// result stays finite), kk += k_i[c] w_c k_j[c], qk += k_i[c] w_c q_j[c].
template <bool DELTA>
__device__ __forceinline__ void pair_quad(float& kk, float& qk, const float4 ki, const float4 li,
                                          const float4 lj, const float4 kj, const float4 qj,
                                          bool live) {
  const float a[4] = {ki.x, ki.y, ki.z, ki.w}, l0[4] = {li.x, li.y, li.z, li.w};
  const float l1[4] = {lj.x, lj.y, lj.z, lj.w}, b[4] = {kj.x, kj.y, kj.z, kj.w};
  const float c[4] = {qj.x, qj.y, qj.z, qj.w};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float w = __expf(live ? l1[t] - l0[t] : 0.f);
    const float kw = a[t] * w;
    if (DELTA) kk += kw * b[t];
    qk += kw * c[t];
  }
}

template <int OP, int DK, int DV>
__global__ void __launch_bounds__(PF_THREADS, DK == 64 ? 2 : 1) prefill_perkey_kernel(
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

  static_assert(DK == DV, "square state");
  float bon[DK / 32];   // RWKV6 bonus of this head: channels lane + 32 cc
#pragma unroll
  for (int cc = 0; cc < DK / 32; ++cc) bon[cc] = DELTA ? 0.f : bonus[(size_t)h * DK + lane + 32 * cc];
  PkStage<DK> st;
  st.load(q, k, v, g, DELTA ? beta : nullptr, 0, T < PF_C ? T : PF_C, nH, sh, tid);
  for (int t0 = 0; t0 < T; t0 += PF_C) {
    const int Cc = (T - t0) < PF_C ? (T - t0) : PF_C;
    __syncthreads();   // S̄ ready / previous chunk done with every buffer
    // ---- stage the chunk from registers (tokens past the end: zero inputs,
    //      zero decay), then start loading the next chunk
    st.store(Kc, Qc, Lc, Vc, L::SP, tid);
    if (DELTA && warp == 0) Bt[lane] = st.b;   // 0 past Cc
    if (t0 + PF_C < T) {
      const int Cn = (T - t0 - PF_C) < PF_C ? (T - t0 - PF_C) : PF_C;
      st.load(q, k, v, g, DELTA ? beta : nullptr, t0 + PF_C, Cn, nH, sh, tid);
    }
    __syncthreads();
    // ---- Λ: inclusive scan of g down each key channel, in PF_THREADS / d_k
    //      groups of consecutive tokens per channel (each thread scans its group,
    //      then adds the totals of the groups before it); e^{Λ_C}.  Pk is free
    //      until the S̄ products and holds the group totals.
    {
      constexpr int NGRP = PF_THREADS / DK, TPG = PF_C / NGRP;
      static_assert(NGRP * DK == PF_THREADS && TPG * NGRP == PF_C, "scan groups");
      const int c = tid % DK, grp = tid / DK;
      float acc = 0.f;
#pragma unroll
      for (int j = grp * TPG; j < (grp + 1) * TPG; ++j) {
        acc += Lc[j * L::SP + c];
        Lc[j * L::SP + c] = acc;
      }
      Pk[grp * DK + c] = acc;
      __syncthreads();
      float pre = 0.f;
      for (int q = 0; q < grp; ++q) pre += Pk[q * DK + c];
      if (grp > 0) {
#pragma unroll
        for (int j = grp * TPG; j < (grp + 1) * TPG; ++j) Lc[j * L::SP + c] += pre;
      }
      if (grp == NGRP - 1) Ec[c] = expf(pre + acc);
    }
    if constexpr (!DELTA) {
      // bonus coefficient of each token: Σ_c r_j[c] b[c] k_j[c] (one warp per token)
      for (int j = warp; j < PF_C; j += PF_THREADS / 32) {
        float s = 0.f;
#pragma unroll
        for (int cc = 0; cc < DK / 32; ++cc) {
          const int c = lane + 32 * cc;
          s += Qc[j * L::SP + c] * bon[cc] * Kc[j * L::SP + c];
        }
        s = warp_sum(s);
        if (lane == 0) Cb[j] = s;
      }
    }
    __syncthreads();
    // ---- decay-weighted pair coefficients (live pairs: i <= j for KDA, i < j
    //      for RWKV6, whose exponents Λ_j - Λ_i (RWKV6: Λ_{j-1} - Λ_i) are <= 0).
    //      Each thread takes pairs (jg + 16x, ig + 16y); (x, y) = (0, 1) has i > j
    //      and is never live, (1, 0) always is, the diagonal blocks when ig <= jg
    //      (RWKV6: ig < jg).  Rows ig and jg keep a warp's quad loads conflict-free.
    {
      const int jg = tid >> 4, ig = tid & 15;
      const int j0 = jg, j1 = jg + 16, i0 = ig, i1 = ig + 16;
      const bool dl = DELTA ? ig <= jg : ig < jg;
      const int lr0 = DELTA ? j0 : (j0 > 0 ? j0 - 1 : 0), lr1 = DELTA ? j1 : j1 - 1;
      float kk[3] = {0.f, 0.f, 0.f}, qk[3] = {0.f, 0.f, 0.f};   // pairs (0,0), (1,0), (1,1)
#pragma unroll 2
      for (int c = 0; c < DK; c += 4) {
        const float4 ki0 = ld4(Kc + i0 * L::SP + c), ki1 = ld4(Kc + i1 * L::SP + c);
        const float4 li0 = ld4(Lc + i0 * L::SP + c), li1 = ld4(Lc + i1 * L::SP + c);
        const float4 lj0 = ld4(Lc + lr0 * L::SP + c), lj1 = ld4(Lc + lr1 * L::SP + c);
        const float4 qj0 = ld4(Qc + j0 * L::SP + c), qj1 = ld4(Qc + j1 * L::SP + c);
        float4 kj0 = make_float4(0.f, 0.f, 0.f, 0.f), kj1 = kj0;
        if (DELTA) {
          kj0 = ld4(Kc + j0 * L::SP + c);
          kj1 = ld4(Kc + j1 * L::SP + c);
        }
        pair_quad<DELTA>(kk[0], qk[0], ki0, li0, lj0, kj0, qj0, dl);
        pair_quad<DELTA>(kk[1], qk[1], ki0, li0, lj1, kj1, qj1, true);
        pair_quad<DELTA>(kk[2], qk[2], ki1, li1, lj1, kj1, qj1, dl);
      }
      auto put = [&](int j, int i, float kv, float qv, bool live) {
        const bool ok = live && j < Cc;
        Akk[j * L::PA + i] = (DELTA && ok && i != j) ? kv : 0.f;
        Akq[j * L::PA + i] = ok ? qv : 0.f;
      };
      put(j0, i0, kk[0], qk[0], dl);
      put(j0, i1, 0.f, 0.f, false);
      put(j1, i0, kk[1], qk[1], true);
      put(j1, i1, kk[2], qk[2], dl);
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
        Qc[j * L::SP + c] *= (j > 0) ? __expf(Lc[(j - 1) * L::SP + c]) : 1.f;
      }
    }
    __syncthreads();
    // ---- S̄ products: rows rg + 32 m, tokens tg + 8 t per thread
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
        float4 s4[RPT], x4[4], q4[4];
#pragma unroll
        for (int m = 0; m < RPT; ++m) s4[m] = ld4(Sb + (rg + 32 * m) * L::SP + c);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          q4[t] = ld4(Qc + (tg + 8 * t) * L::SP + c);
          if (DELTA) x4[t] = ld4(Xc + (tg + 8 * t) * L::SP + c);
        }
#pragma unroll
        for (int m = 0; m < RPT; ++m)
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            pq[m][t] = dot4(pq[m][t], s4[m], q4[t]);
            if (DELTA) pk[m][t] = dot4(pk[m][t], s4[m], x4[t]);
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
    // ---- the appended factors and the outputs
    if constexpr (!DELTA) {
      // RWKV6: u_j = v_j, so every output is independent.  Row r = tid % d_v,
      // tokens j ≡ tid / d_v (mod PF_THREADS / d_v).  The pair coefficients
      // of dead pairs (i >= j) are zero, so each sum runs over every i, in
      // four partial sums.
      constexpr int JG = PF_THREADS / DV;
      static_assert(JG * DV == PF_THREADS && PF_C % JG == 0, "output groups");
      const int r = tid % DV, jq = tid / DV;
      float vr[PF_C];
#pragma unroll
      for (int i = 0; i < PF_C; ++i) vr[i] = Vc[i * DV + r];
#pragma unroll
      for (int t = 0; t < PF_C / JG; ++t) {
        const int j = jq + JG * t;
        const float vj = Vc[j * DV + r];
        Us[r * L::PP + j] = vj;
        if (o != nullptr && j < Cc) {
          float y[4] = {Pq[r * L::PP + j], 0.f, 0.f, 0.f};
#pragma unroll
          for (int i = 0; i < PF_C; i += 4) {   // one broadcast 16-byte load per four pairs
            const float4 c4 = ld4(Akq + j * L::PA + i);
            y[0] += c4.x * vr[i];
            y[1] += c4.y * vr[i + 1];
            y[2] += c4.z * vr[i + 2];
            y[3] += c4.w * vr[i + 3];
          }
          const float yo = (y[0] + y[1]) + (y[2] + y[3]) + Cb[j] * vj;
          const size_t oi = ((size_t)(t0 + j) * nH + sh) * DV + r;
          if (out_bf16) static_cast<uint16_t*>(o)[oi] = f2bf16(scale * yo);
          else static_cast<float*>(o)[oi] = scale * yo;
        }
      }
    } else if (tid < DV) {
      // KDA: one thread per value row (u_j needs u_i, i < j); each sum runs in
      // four partial sums to shorten its chain
      const int r = tid;
      float u[PF_C];
#pragma unroll
      for (int j = 0; j < PF_C; ++j) {
        float x[4] = {Pk[r * L::PP + j], 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < j; ++i) x[i & 3] += Akk[j * L::PA + i] * u[i];
        u[j] = Bt[j] * (Vc[j * DV + r] - ((x[0] + x[1]) + (x[2] + x[3])));   // 0 past Cc
      }
#pragma unroll
      for (int j = 0; j < PF_C; ++j) {
        Us[r * L::PP + j] = u[j];
        if (o != nullptr && j < Cc) {
          float y[4] = {Pq[r * L::PP + j], 0.f, 0.f, 0.f};
#pragma unroll
          for (int i = 0; i <= j; ++i) y[i & 3] += Akq[j * L::PA + i] * u[i];
          const float yo = (y[0] + y[1]) + (y[2] + y[3]);
          const size_t oi = ((size_t)(t0 + j) * nH + sh) * DV + r;
          if (out_bf16) static_cast<uint16_t*>(o)[oi] = f2bf16(scale * yo);
          else static_cast<float*>(o)[oi] = scale * yo;
        }
      }
    }
    // ---- k_j ⊙ e^{Λ_C-Λ_j} into X (X's hats are no longer read)
    for (int idx = tid; idx < PF_C * DK; idx += PF_THREADS) {
      const int j = idx / DK, c = idx - j * DK;
      Xc[j * L::SP + c] =
          Kc[j * L::SP + c] * __expf(Lc[(PF_C - 1) * L::SP + c] - Lc[j * L::SP + c]);
    }
    __syncthreads();
    // ---- S̄ <- S̄ Diag(e^{Λ_C}) + Σ_j a_j (k_j ⊙ e^{Λ_C-Λ_j})^T: rows rg + 32 m
    //      and column quads 4 tg + 32 n per thread
    {
      constexpr int RPT = DV / 32, CPT = DK / 32;
      const int rg = tid >> 3, tg = tid & 7;
      float4 acc[RPT][CPT];
#pragma unroll
      for (int n4 = 0; n4 < CPT; ++n4) {
        const float4 e4 = ld4(Ec + 4 * tg + 32 * n4);
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
          const float4 s4 = ld4(Sb + (rg + 32 * m) * L::SP + 4 * tg + 32 * n4);
          acc[m][n4] = make_float4(e4.x * s4.x, e4.y * s4.y, e4.z * s4.z, e4.w * s4.w);
        }
      }
#pragma unroll 4
      for (int j = 0; j < Cc; ++j) {
        float w[RPT];
#pragma unroll
        for (int m = 0; m < RPT; ++m) w[m] = Us[(rg + 32 * m) * L::PP + j];
#pragma unroll
        for (int n4 = 0; n4 < CPT; ++n4) {
          const float4 k4 = ld4(Xc + j * L::SP + 4 * tg + 32 * n4);
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
                           void* o, int T, int out_bf16, float scale, int32_t* status,
                           cudaStream_t s) {
  if (a.rows <= 0 || T <= 0) return cudaSuccess;
  if (op == GDN) {
    if (dk == 64) return pf_dispatch<64>(a, q, k, v, g, beta, o, T, out_bf16, scale, s);
    return launch_prefill_gdn_tc(a, q, k, v, g, beta, o, T, out_bf16, scale, status, s);
  }
  if (op == KDA) {
    if (dk == 64) return pk_dispatch<KDA, 64>(a, q, k, v, g, beta, bonus, o, T, out_bf16, scale, s);
    return launch_prefill_kda_tc(a, q, k, v, g, beta, o, T, out_bf16, scale, status, s);
  }
  if (dk == 64) return launch_prefill_rwkv6_tc(a, q, k, v, g, bonus, o, T, out_bf16, scale, status, s);
  return pk_dispatch<RWKV6, 128>(a, q, k, v, g, beta, bonus, o, T, out_bf16, scale, s);
}

}  // namespace dl
