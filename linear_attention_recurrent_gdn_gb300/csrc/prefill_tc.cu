// Chunked prefill of GDN at d_k = d_v = 128 on the 5th-generation tensor cores.
//
// Same algebra as the CUDA-core kernel in prefill.cu (the DeltaLog page's
// base + log form inside a chunk of C = 32 tokens, the Flide page's first call
// that builds a request's state from its shared context): with S̄ the state at
// the chunk start, Λ_j the cumulative log-decay inside the chunk,
//   x_j = e^{Λ_j} (S̄ k_j) + Σ_{i<j} e^{Λ_j-Λ_i} (k_i·k_j) u_i,  u_j = β_j (v_j - x_j)
//   o_j = e^{Λ_j} (S̄ q_j) + Σ_{i<=j} e^{Λ_j-Λ_i} (k_i·q_j) u_i
//   S̄'  = e^{Λ_C} S̄ + Σ_j (e^{Λ_C-Λ_j} u_j) k_j^T
// The dense contractions of a chunk run as tcgen05 MMAs (bf16 operands, fp32
// accumulators in tensor memory):
//   D0 [128 x 32]  = [K; Q; K; Q] K^T           key-key and query-key products (exact: k, q are bf16)
//   D1 [128 x 64]  = (S̄_hi + S̄_lo) [K; Q]^T     S̄ k_j and S̄ q_j for all 32 tokens
//   D2 [128 x 128] = (W_hi + W_lo) K             the rank-32 rewrite, W = e^{Λ_C-Λ_j} u_j
//   D3 [128 x 32]  = U_hi A_hi + U_lo A_hi + U_hi A_lo   the outputs' log terms,
//                    A[j][i] = e^{Λ_j-Λ_i} (k_i·q_j) for i <= j
// S̄, W, U and A are fp32; each is carried as two bf16 terms (hi = bf16(x),
// lo = bf16(x - hi)), which leaves |x - hi - lo| <= 2^-17 |x|, so the products
// keep the state's 1e-4 tolerance.  The fp32 state itself never leaves the
// registers of the CTA (thread (row r, half h) holds S̄[r][64h .. 64h + 63]); the
// decay e^{Λ_C} and the rank-32 term are added there, and the bf16 terms of the
// new S̄ are written back to shared memory for the next chunk.  The forward
// substitution for u (a chain over the chunk's tokens) runs on the CUDA cores,
// one thread per value row.
//
// One CTA of 256 threads per slot-head.  Warp w reads tensor-memory lanes
// 32 (w % 4) .. +31, i.e. value rows r = 32 (w % 4) + lane.  Thread 0 issues the
// MMAs and waits on their mbarrier (bounded: a wait that runs out records
// DEV_TIMEOUT_MMA in the status word, lets the outstanding MMAs land and frees
// the tensor memory before the CTA returns).
#include "dl_device.cuh"
#include "launch.h"
#include "layout.h"
#include "tc_device.cuh"

namespace dl {

namespace {

constexpr int TC_C = 32;           // tokens per chunk
constexpr int TC_THREADS = 256;
constexpr int TC_D = 128;          // d_k = d_v
constexpr uint32_t TC_COLS = 256;  // TMEM columns: D0 [0, 32), D1 [32, 96), D3 [96, 128), D2 [128, 256)
constexpr uint32_t D0_COL = 0, D1_COL = 32, D3_COL = 96, D2_COL = 128;
// Row strides: v rows padded to 136 bf16 (272 bytes: a warp's staging stores of
// 8 rows x 64 bytes spread over all banks); pair-coefficient rows of 36 floats
// (16-byte aligned, read as float4 broadcasts).
constexpr int VP = TC_D + 8, AP = 36;
constexpr int LPAD = TC_D + 4;   // fp32 rows of k, q, Λ (KDA): quad loads of rows ig, jg spread over banks

// Byte offsets in the dynamic shared memory (operands 16-byte aligned).  The
// per-chunk buffers that the next chunk's preparation fills while the current
// chunk still reads them are doubled (index b = chunk & 1).
struct TcSmem {
  static constexpr uint32_t SHI = 0;                       // S̄ hi, K-major [128 x 128] bf16
  static constexpr uint32_t SLO = SHI + TC_D * TC_D * 2;   // S̄ lo
  static constexpr uint32_t KQ = SLO + TC_D * TC_D * 2;    // rows 0-31 k_j, 32-63 q_j, 64-127 again
  static constexpr uint32_t WHI = KQ + TC_D * TC_D * 2;    // W hi [v (128)] x [j (32)], K-major
  static constexpr uint32_t WLO = WHI + TC_D * TC_C * 2;   // W lo
  static constexpr uint32_t UHI = WLO + TC_D * TC_C * 2;   // U hi [v (128)] x [i (32)], K-major
  static constexpr uint32_t ULO = UHI + TC_D * TC_C * 2;   // U lo
  // doubled: K^T (K as [i (128)] x [j (32)], MN-major), A hi / lo ([j] x [i], K-major),
  // v_j[r] (bf16 rows of VP), A_kk (fp32 [32][AP]), Λ_j, e^{Λ_j}, e^{Λ_C-Λ_j}, β_j ([4][32])
  static constexpr uint32_t KT_SZ = TC_D * TC_C * 2, A_SZ = TC_C * TC_C * 2, VS_SZ = TC_C * VP * 2,
                            AKK_SZ = TC_C * AP * 4, SC_SZ = 4 * TC_C * 4;
  static constexpr uint32_t BUF = KT_SZ + 2 * A_SZ + VS_SZ + AKK_SZ + SC_SZ;   // one set
  static constexpr uint32_t SET0 = ULO + TC_D * TC_C * 2;
  static constexpr uint32_t KT = 0, AHI = KT + KT_SZ, ALO = AHI + A_SZ, VS = ALO + A_SZ,
                            AKK = VS + VS_SZ, SC = AKK + AKK_SZ;   // offsets inside a set
  static constexpr uint32_t BAR = SET0 + 2 * BUF;          // 3 mbarriers, TMEM base, ok flag
  static constexpr uint32_t BYTES = BAR + 32;
  static __host__ __device__ constexpr uint32_t set(int b) { return SET0 + (uint32_t)b * BUF; }
};
static_assert(TcSmem::BYTES <= 227 * 1024, "shared memory");
static_assert(TcSmem::BUF % 16 == 0 && TcSmem::SET0 % 16 == 0, "16-byte aligned buffers");

// Two fp32 values rounded to bf16 as one word (first value in the low half).
__device__ __forceinline__ uint32_t bf16x2(float a, float b) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&p);
}

// 8 consecutive fp32 values -> the bf16 high parts (h) and low parts (l).
__device__ __forceinline__ void split8(const float* x, uint4& h, uint4& l) {
  uint32_t hw[4], lw[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float a = x[2 * e], b = x[2 * e + 1];
    hw[e] = bf16x2(a, b);
    lw[e] = bf16x2(a - __uint_as_float(hw[e] << 16), b - __uint_as_float(hw[e] & 0xffff0000u));
  }
  h = make_uint4(hw[0], hw[1], hw[2], hw[3]);
  l = make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

// Element idx of a chunk's 32 x 16 grid of 16-byte pieces (token j, column
// piece cv): a warp's lanes take 8 consecutive tokens x 4 consecutive pieces,
// so its global loads read 64 contiguous bytes of each of 8 rows and its
// stores into the K-major operands fill whole 128-byte core-matrix rows.
__device__ __forceinline__ void chunk_piece(int idx, int& j, int& cv) {
  const int rest = idx >> 5;
  j = (idx & 7) + 8 * (rest & 3);
  cv = ((idx >> 3) & 3) + 4 * (rest >> 2);
}

// One chunk's k, q, v (bf16) and g, β in the registers of the 128 threads that
// prepare chunks, between their global loads and their shared-memory stores.
struct TcStage {
  uint4 k[4], q[4], v[4];
  float g, b;

  __device__ __forceinline__ void load(const uint16_t* __restrict__ qg, const uint16_t* __restrict__ kg,
                                       const uint16_t* __restrict__ vg, const float* __restrict__ gg,
                                       const float* __restrict__ bg, int t0, int Cc, size_t nH,
                                       int sh, int ptid) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      int j, cv;
      chunk_piece(ptid + e * 128, j, cv);
      if (j < Cc) {
        const size_t base = ((size_t)(t0 + j) * nH + sh) * TC_D + cv * 8;
        k[e] = *reinterpret_cast<const uint4*>(kg + base);
        q[e] = *reinterpret_cast<const uint4*>(qg + base);
        v[e] = *reinterpret_cast<const uint4*>(vg + base);
      } else {
        k[e] = q[e] = v[e] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    if (ptid < 32) {
      g = ptid < Cc ? gg[(size_t)(t0 + ptid) * nH + sh] : 0.f;
      b = ptid < Cc ? bg[(size_t)(t0 + ptid) * nH + sh] : 0.f;
    }
  }

  // k, q into the KQ operand, twice: rows 0-63 and again rows 64-127, so that
  // D0's rows 64-127 repeat its rows 0-63 in the TMEM lanes of warps 6 and 7
  __device__ __forceinline__ void store_kq(unsigned char* sm, int ptid) const {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      int j, cv;
      chunk_piece(ptid + e * 128, j, cv);
#pragma unroll
      for (int rep = 0; rep < 2; ++rep) {
        *reinterpret_cast<uint4*>(sm + TcSmem::KQ + tc::kmaj_off(64 * rep + j, cv * 8, TC_D)) = k[e];
        *reinterpret_cast<uint4*>(sm + TcSmem::KQ + tc::kmaj_off(64 * rep + TC_C + j, cv * 8, TC_D)) = q[e];
      }
    }
  }

  // k into the K^T operand of set `set` (MN-major: k_j[8 cv .. 8 cv + 7] is
  // one 16-byte row of a core matrix), v into its VS
  __device__ __forceinline__ void store_rest(unsigned char* sm, uint32_t set, int ptid) const {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      int j, cv;
      chunk_piece(ptid + e * 128, j, cv);
      *reinterpret_cast<uint4*>(sm + set + TcSmem::VS + (j * VP + cv * 8) * 2) = v[e];
      *reinterpret_cast<uint4*>(sm + set + TcSmem::KT + tc::mnmaj_off(cv * 8, j, TC_C)) = k[e];
    }
  }
};

// Barrier among the 128 threads (warps 4-7) that prepare the next chunk.
__device__ __forceinline__ void prep_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// The per-chunk work that does not depend on S̄, done by warps 4-7 for a chunk
// while warps 0-3 run the previous chunk's forward substitution: stage k, q,
// v, the decays (Λ by a scan over the chunk, e^{Λ_j}, e^{Λ_C-Λ_j}) and β;
// D0 = [K; Q; K; Q] K^T; from it the pair coefficients A_kk (fp32 rows) and A
// (bf16 terms of D3's B operand), each with its decay e^{Λ_j-Λ_i}.
__device__ __forceinline__ void gdn_prepare(unsigned char* sm, const TcStage& st, uint32_t set,
                                            int Cc, int chunk, uint32_t tm, uint32_t sbase,
                                            uint32_t bar0, int32_t* status, int32_t* ok_flag) {
  const int ptid = threadIdx.x - 128, lane = threadIdx.x & 31, pw = ptid >> 5;
  float* Lm = reinterpret_cast<float*>(sm + set + TcSmem::SC);
  float* El = Lm + TC_C;
  float* Ew = El + TC_C;
  float* Bt = Ew + TC_C;
  // k, q first: D0 needs only them, and runs while the rest is staged
  st.store_kq(sm, ptid);
  tc::fence_smem_to_async();   // KQ for the tensor cores
  tc::fence_before_sync();
  prep_sync();
  if (ptid == 0) {
    tc::fence_after_sync();
    constexpr uint32_t id0 = tc::idesc_bf16_f32(128, 32);
#pragma unroll
    for (int kk = 0; kk < TC_D / 16; ++kk)
      tc::mma_bf16(tm, tc::kmaj_desc(sbase + TcSmem::KQ, TC_D, kk),
                   tc::kmaj_desc(sbase + TcSmem::KQ, TC_D, kk), id0, kk > 0);
    tc::mma_commit(bar0);
  }
  st.store_rest(sm, set, ptid);
  if (pw == 0) {
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
  // a wait that gives up records which phase it waited for (-3: parity 0, -4: parity 1)
  if (ptid == 0 && !mbar_wait(bar0, (uint32_t)chunk & 1u, status, DEV_TIMEOUT_MMA))
    *ok_flag = -3 - (chunk & 1);
  prep_sync();
  tc::fence_after_sync();
  // D0 rows 0-31 and 64-95 hold k_j·k_i, rows 32-63 and 96-127 q_j·k_i (row j
  // = lane of the quarter).  Each warp reads its own lane quarter (warp 4 + pw
  // owns lanes 32 pw .. 32 pw + 31): warps 4, 5 columns 0-15, warps 6, 7 columns 16-31.
  {
    const int half = pw >> 1, which = pw & 1, i0 = 16 * half;
    uint32_t x[16];
    tc::tmem_ld16(tm + ((uint32_t)(32 * pw) << 16) + i0, x);
    tc::tmem_wait_ld16(x);
    const int j = lane;
    const float lj = Lm[j];
    float w[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int i = i0 + e;
      const bool live = (which == 0 ? i < j : i <= j) && j < Cc;
      w[e] = live ? __uint_as_float(x[e]) * __expf(lj - Lm[i]) : 0.f;   // exponent <= 0
    }
    if (which == 0) {
      float* Akk = reinterpret_cast<float*>(sm + set + TcSmem::AKK);
#pragma unroll
      for (int e4 = 0; e4 < 4; ++e4)
        *reinterpret_cast<float4*>(Akk + j * AP + i0 + 4 * e4) =
            make_float4(w[4 * e4], w[4 * e4 + 1], w[4 * e4 + 2], w[4 * e4 + 3]);
      if (half == 1) *reinterpret_cast<float4*>(Akk + j * AP + TC_C) = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
#pragma unroll
      for (int c8 = 0; c8 < 2; ++c8) {
        uint4 hv, lv;
        split8(w + 8 * c8, hv, lv);
        const uint32_t off = tc::kmaj_off(j, i0 + 8 * c8, TC_C);
        *reinterpret_cast<uint4*>(sm + set + TcSmem::AHI + off) = hv;
        *reinterpret_cast<uint4*>(sm + set + TcSmem::ALO + off) = lv;
      }
    }
  }
  tc::fence_before_sync();
}

__global__ void __launch_bounds__(TC_THREADS, 1)
prefill_gdn_tc_kernel(const __grid_constant__ SlotListArgs a, const uint16_t* __restrict__ q,
                      const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                      const float* __restrict__ g, const float* __restrict__ beta, void* o, int T,
                      int out_bf16, float scale, int32_t* status) {
  extern __shared__ __align__(1024) unsigned char sm[];
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + TcSmem::BAR + 24);
  int32_t* ok_flag = reinterpret_cast<int32_t*>(sm + TcSmem::BAR + 28);
  const uint32_t sbase = smem_u32(sm);
  const uint32_t bar1 = sbase + TcSmem::BAR, bar2 = bar1 + 8, bar0 = bar1 + 16;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q4 = warp & 3, hw = warp >> 2;      // TMEM lane quarter, column half
  const int r = 32 * q4 + lane;                 // this thread's value row
  const bool prep = warp >= 4;                  // warps 4-7 prepare the next chunk
  const int sh = blockIdx.x, row = sh / a.H, h = sh - row * a.H;
  const int slot = a.items[row].slot;
  const size_t nH = (size_t)a.rows * a.H;
  float* gS = a.Sbar + ((size_t)slot * a.H + h) * TC_D * TC_D;
  const int nch = (T + TC_C - 1) / TC_C;

  if (warp == 0) tc::tmem_alloc(sbase + TcSmem::BAR + 24, TC_COLS);
  if (tid == 0) {
    mbar_init(bar1, 1);
    mbar_init(bar2, 1);
    mbar_init(bar0, 1);
    fence_mbar_init();
    *ok_flag = 1;
  }
  // the fp32 state of this thread's row half, and its bf16 terms for the MMAs
  float S[64];
  {
    const float4* src = reinterpret_cast<const float4*>(gS + (size_t)r * TC_D + 64 * hw);
#pragma unroll
    for (int c4 = 0; c4 < 16; ++c4) {
      const float4 x = src[c4];
      S[4 * c4] = x.x;
      S[4 * c4 + 1] = x.y;
      S[4 * c4 + 2] = x.z;
      S[4 * c4 + 3] = x.w;
    }
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
      uint4 hv, lv;
      split8(S + 8 * c8, hv, lv);
      const uint32_t off = tc::kmaj_off(r, 64 * hw + 8 * c8, TC_D);
      *reinterpret_cast<uint4*>(sm + TcSmem::SHI + off) = hv;
      *reinterpret_cast<uint4*>(sm + TcSmem::SLO + off) = lv;
    }
  }

  TcStage st;
  if (prep) st.load(q, k, v, g, beta, 0, T < TC_C ? T : TC_C, nH, sh, tid - 128);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tm = *tmem_slot;
  const uint32_t tlane = tm + ((uint32_t)(32 * q4) << 16);   // this warp's lane quarter
  // chunk 0 prepared, chunk 1's inputs on their way, then D1 of chunk 0
  if (prep) {
    gdn_prepare(sm, st, TcSmem::set(0), T < TC_C ? T : TC_C, 0, tm + D0_COL, sbase, bar0, status,
                ok_flag);
    if (nch > 1) st.load(q, k, v, g, beta, TC_C, (T - TC_C) < TC_C ? (T - TC_C) : TC_C, nH, sh, tid - 128);
  }
  tc::fence_smem_to_async();
  tc::fence_before_sync();
  __syncthreads();
  bool ok = *ok_flag == 1;
  if (ok && tid == 0) {
    tc::fence_after_sync();
    constexpr uint32_t id1 = tc::idesc_bf16_f32(128, 64);
#pragma unroll
    for (int kk = 0; kk < TC_D / 16; ++kk)
      tc::mma_bf16(tm + D1_COL, tc::kmaj_desc(sbase + TcSmem::SHI, TC_D, kk),
                   tc::kmaj_desc(sbase + TcSmem::KQ, TC_D, kk), id1, kk > 0);
#pragma unroll
    for (int kk = 0; kk < TC_D / 16; ++kk)
      tc::mma_bf16(tm + D1_COL, tc::kmaj_desc(sbase + TcSmem::SLO, TC_D, kk),
                   tc::kmaj_desc(sbase + TcSmem::KQ, TC_D, kk), id1, 1u);
    tc::mma_commit(bar1);
  }
  int chunk = 0;
  for (; chunk < nch && ok; ++chunk) {
    const int t0 = chunk * TC_C;
    const int Cc = (T - t0) < TC_C ? (T - t0) : TC_C;
    const uint32_t par = (uint32_t)chunk & 1u;
    const uint32_t set = TcSmem::set(chunk & 1);
    const float* Lm = reinterpret_cast<const float*>(sm + set + TcSmem::SC);
    const float* El = Lm + TC_C;
    const float* Ew = El + TC_C;
    const float* Bt = Ew + TC_C;
    // ---- D1 = (S̄_hi + S̄_lo) [K; Q]^T of this chunk has landed
    if (tid == 0 && !mbar_wait(bar1, par, status, DEV_TIMEOUT_MMA)) *ok_flag = -1;
    __syncthreads();
    if (*ok_flag != 1) {
      ok = false;
      break;
    }
    tc::fence_after_sync();
    if (!prep) {
      // ---- forward substitution (warps 0-3, one value row each)
      const float* Akk = reinterpret_cast<const float*>(sm + set + TcSmem::AKK);
      const uint16_t* Vs = reinterpret_cast<const uint16_t*>(sm + set + TcSmem::VS);
      float pk[TC_C], u[TC_C];
      {
        uint32_t x[TC_C];
        tc::tmem_ld32(tlane + D1_COL, x);
        tc::tmem_wait_ld(x);
#pragma unroll
        for (int j = 0; j < TC_C; ++j) pk[j] = __uint_as_float(x[j]);
      }
#pragma unroll
      for (int j = 0; j < TC_C; ++j) u[j] = 0.f;   // entries not yet solved multiply zero coefficients
#pragma unroll
      for (int j = 0; j < TC_C; ++j) {
        float x[4] = {El[j] * pk[j], 0.f, 0.f, 0.f};
#pragma unroll
        for (int i4 = 0; i4 < (j + 3) / 4; ++i4) {
          const float4 c = *reinterpret_cast<const float4*>(Akk + j * AP + 4 * i4);
          x[0] += c.x * u[4 * i4];
          x[1] += c.y * u[4 * i4 + 1];
          x[2] += c.z * u[4 * i4 + 2];
          x[3] += c.w * u[4 * i4 + 3];
        }
        u[j] = Bt[j] * (bf16f(Vs[j * VP + r]) - ((x[0] + x[1]) + (x[2] + x[3])));   // 0 past Cc
      }
#pragma unroll
      for (int c8 = 0; c8 < TC_C / 8; ++c8) {
        float w8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) w8[e] = u[8 * c8 + e] * Ew[8 * c8 + e];
        uint4 hv, lv;
        const uint32_t off = tc::kmaj_off(r, 8 * c8, TC_C);
        split8(w8, hv, lv);
        *reinterpret_cast<uint4*>(sm + TcSmem::WHI + off) = hv;
        *reinterpret_cast<uint4*>(sm + TcSmem::WLO + off) = lv;
        split8(u + 8 * c8, hv, lv);
        *reinterpret_cast<uint4*>(sm + TcSmem::UHI + off) = hv;
        *reinterpret_cast<uint4*>(sm + TcSmem::ULO + off) = lv;
      }
    } else if (chunk + 1 < nch) {
      // ---- meanwhile warps 4-7 prepare the next chunk and start loading the one after
      const int Cn = (T - t0 - TC_C) < TC_C ? (T - t0 - TC_C) : TC_C;
      gdn_prepare(sm, st, TcSmem::set((chunk + 1) & 1), Cn, chunk + 1, tm + D0_COL, sbase, bar0,
                  status, ok_flag);
      if (chunk + 2 < nch) {
        const int C2 = (T - t0 - 2 * TC_C) < TC_C ? (T - t0 - 2 * TC_C) : TC_C;
        st.load(q, k, v, g, beta, t0 + 2 * TC_C, C2, nH, sh, tid - 128);
      }
    }
    tc::fence_smem_to_async();   // W, U and the next chunk's operands, for the tensor cores
    tc::fence_before_sync();
    __syncthreads();
    if (*ok_flag != 1) {
      ok = false;
      break;
    }
    // ---- D2 = (W_hi + W_lo) K and D3 = U_hi A_hi^T + U_lo A_hi^T + U_hi A_lo^T
    if (tid == 0) {
      tc::fence_after_sync();
      constexpr uint32_t id2 = tc::idesc_bf16_f32(128, 128, false, true);   // K^T MN-major
      constexpr uint32_t id3 = tc::idesc_bf16_f32(128, 32);
      const uint32_t kt = sbase + set + TcSmem::KT;
      const uint32_t ahi = sbase + set + TcSmem::AHI, alo = sbase + set + TcSmem::ALO;
#pragma unroll
      for (int kk = 0; kk < TC_C / 16; ++kk)
        tc::mma_bf16(tm + D2_COL, tc::kmaj_desc(sbase + TcSmem::WHI, TC_C, kk),
                     tc::kmaj_desc(kt, TC_C, kk), id2, kk > 0);
#pragma unroll
      for (int kk = 0; kk < TC_C / 16; ++kk)
        tc::mma_bf16(tm + D2_COL, tc::kmaj_desc(sbase + TcSmem::WLO, TC_C, kk),
                     tc::kmaj_desc(kt, TC_C, kk), id2, 1u);
#pragma unroll
      for (int kk = 0; kk < TC_C / 16; ++kk)
        tc::mma_bf16(tm + D3_COL, tc::kmaj_desc(sbase + TcSmem::UHI, TC_C, kk),
                     tc::kmaj_desc(ahi, TC_C, kk), id3, kk > 0);
#pragma unroll
      for (int kk = 0; kk < TC_C / 16; ++kk)
        tc::mma_bf16(tm + D3_COL, tc::kmaj_desc(sbase + TcSmem::ULO, TC_C, kk),
                     tc::kmaj_desc(ahi, TC_C, kk), id3, 1u);
#pragma unroll
      for (int kk = 0; kk < TC_C / 16; ++kk)
        tc::mma_bf16(tm + D3_COL, tc::kmaj_desc(sbase + TcSmem::UHI, TC_C, kk),
                     tc::kmaj_desc(alo, TC_C, kk), id3, 1u);
      tc::mma_commit(bar2);
      if (!mbar_wait(bar2, par, status, DEV_TIMEOUT_MMA)) *ok_flag = -2;
    }
    __syncthreads();
    if (*ok_flag != 1) {
      ok = false;
      break;
    }
    tc::fence_after_sync();
    // ---- outputs of tokens 16 h .. 16 h + 15 of row r:
    //      o_j = scale (e^{Λ_j} S̄ q_j + Σ_{i<=j} A[j][i] u_i)
    if (o != nullptr) {
      uint32_t xq[16], x3[16];
      tc::tmem_ld16(tlane + D1_COL + TC_C + 16 * hw, xq);
      tc::tmem_ld16(tlane + D3_COL + 16 * hw, x3);
      tc::tmem_wait_ld16(xq);
      tc::tmem_wait_ld16(x3);
      const size_t ostride = nH * TC_D;
      const size_t obase = ((size_t)(t0 + 16 * hw) * nH + sh) * TC_D + r;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int j = 16 * hw + e;
        if (j < Cc) {
          const float yo = scale * (El[j] * __uint_as_float(xq[e]) + __uint_as_float(x3[e]));
          const size_t oi = obase + (size_t)e * ostride;
          if (out_bf16) static_cast<uint16_t*>(o)[oi] = f2bf16(yo);
          else static_cast<float*>(o)[oi] = yo;
        }
      }
    }
    // ---- S̄ <- e^{Λ_C} S̄ + D2 in registers; its bf16 terms for the next chunk's D1
    {
      const float eC = El[Cc - 1];
      uint32_t x0[32], x1[32];
      tc::tmem_ld32(tlane + D2_COL + 64 * hw, x0);
      tc::tmem_ld32(tlane + D2_COL + 64 * hw + 32, x1);
      tc::tmem_wait_ld(x0);
      tc::tmem_wait_ld(x1);
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        S[c] = eC * S[c] + __uint_as_float(x0[c]);
        S[32 + c] = eC * S[32 + c] + __uint_as_float(x1[c]);
      }
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        uint4 hv, lv;
        split8(S + 8 * c8, hv, lv);
        const uint32_t off = tc::kmaj_off(r, 64 * hw + 8 * c8, TC_D);
        *reinterpret_cast<uint4*>(sm + TcSmem::SHI + off) = hv;
        *reinterpret_cast<uint4*>(sm + TcSmem::SLO + off) = lv;
      }
    }
    tc::fence_smem_to_async();   // the S̄ terms, for the next D1
    tc::fence_before_sync();
    __syncthreads();
    // ---- D1 of the next chunk (its K, Q were staged during the substitution)
    if (chunk + 1 < nch && tid == 0) {
      tc::fence_after_sync();
      constexpr uint32_t id1 = tc::idesc_bf16_f32(128, 64);
#pragma unroll
      for (int kk = 0; kk < TC_D / 16; ++kk)
        tc::mma_bf16(tm + D1_COL, tc::kmaj_desc(sbase + TcSmem::SHI, TC_D, kk),
                     tc::kmaj_desc(sbase + TcSmem::KQ, TC_D, kk), id1, kk > 0);
#pragma unroll
      for (int kk = 0; kk < TC_D / 16; ++kk)
        tc::mma_bf16(tm + D1_COL, tc::kmaj_desc(sbase + TcSmem::SLO, TC_D, kk),
                     tc::kmaj_desc(sbase + TcSmem::KQ, TC_D, kk), id1, 1u);
      tc::mma_commit(bar1);
    }
  }
  if (!ok && tid == 0) {
    // let the MMAs still in flight (those of the wait that gave up) land before
    // the tensor memory is freed; the drain is bounded too
    const int f = *ok_flag;
    if (f == -1) mbar_drain(bar1, (uint32_t)chunk & 1u);
    else if (f == -2) mbar_drain(bar2, (uint32_t)chunk & 1u);
    else if (f == -3 || f == -4) mbar_drain(bar0, (uint32_t)(-3 - f));
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tm, TC_COLS);
  }
  if (!ok) return;
  float4* dst = reinterpret_cast<float4*>(gS + (size_t)r * TC_D + 64 * hw);
#pragma unroll
  for (int c4 = 0; c4 < 16; ++c4)
    dst[c4] = make_float4(S[4 * c4], S[4 * c4 + 1], S[4 * c4 + 2], S[4 * c4 + 3]);
  if (h == 0 && tid == 0) {
    a.nlog[slot] = 0;
    a.base_of[slot] = slot;
  }
}

// ------------------------------------------------------------------- KDA ----
// KDA (per-key decay, delta rule) at d_k = d_v = 128.  With Λ_j the per-channel
// cumulative log-decay inside the chunk (Λ_j[c] = Σ_{i<=j} g_i[c]):
//   x_j = S̄ k̂_j + Σ_{i<j} A_kk[j][i] u_i,  u_j = β_j (v_j - x_j),  k̂_j = e^{Λ_j} ⊙ k_j
//   o_j = S̄ q̂_j + Σ_{i<=j} A[j][i] u_i,                            q̂_j = e^{Λ_j} ⊙ q_j
//   A_kk[j][i] = Σ_c k_i[c] k_j[c] e^{Λ_j[c]-Λ_i[c]},  A[j][i] likewise with q_j
//   S̄' = S̄ Diag(e^{Λ_C}) + Σ_j u_j k̃_j^T,            k̃_j = e^{Λ_C-Λ_j} ⊙ k_j
// The pair weights factor through the chunk start: e^{Λ_j-Λ_i} = e^{Λ_j} e^{-Λ_i},
// so with k̄_i = e^{-Λ_i} ⊙ k_i the pair coefficients are A_kk = k̂ k̄^T and
// A = q̂ k̄^T.  For a live pair (i <= j) every channel's product k̂_j[c] k̄_i[c] =
// k_j[c] k_i[c] e^{Λ_j[c]-Λ_i[c]} is bounded by |k_j[c] k_i[c]|, so nothing
// cancels; the factors themselves stay finite while the chunk's total decay
// stays above -60 in every channel (e^{60} ~ 1e26).  A chunk with stronger
// decay (a block-wide vote after the scan) forms its pair coefficients
// directly on the CUDA cores, one exponential per channel and pair.
// On the tensor cores (fp32 operands as hi + lo bf16 terms, three products each):
//   D0 [128 x 32]  = [k̂; q̂; 0] k̄^T    the pair coefficients (fast chunks)
//   D1 [128 x 64]  = S̄ [k̂; q̂]^T
//   D2 [128 x 128] = U k̃
//   D3 [128 x 32]  = U A^T
struct KdaSmem {
  static constexpr uint32_t SHI = 0;                        // S̄ hi [128 x 128] K-major
  static constexpr uint32_t SLO = SHI + TC_D * TC_D * 2;
  static constexpr uint32_t BHI = SLO + TC_D * TC_D * 2;    // [k̂; q̂; 0] hi [128 x 128] K-major
  static constexpr uint32_t BLO = BHI + TC_D * TC_D * 2;
  static constexpr uint32_t KBHI = BLO + TC_D * TC_D * 2;   // k̄ hi [32 x 128] K-major
  static constexpr uint32_t KBLO = KBHI + TC_C * TC_D * 2;
  static constexpr uint32_t KTHI = KBLO + TC_C * TC_D * 2;  // k̃ hi as [c (128)] x [j (32)], MN-major
  static constexpr uint32_t KTLO = KTHI + TC_D * TC_C * 2;
  static constexpr uint32_t UHI = KTLO + TC_D * TC_C * 2;   // U hi [v (128)] x [i (32)]
  static constexpr uint32_t ULO = UHI + TC_D * TC_C * 2;
  static constexpr uint32_t AHI = ULO + TC_D * TC_C * 2;    // A hi [j (32)] x [i (32)]
  static constexpr uint32_t ALO = AHI + TC_C * TC_C * 2;
  static constexpr uint32_t VS = ALO + TC_C * TC_C * 2;     // v_j[r] bf16, rows of VP
  static constexpr uint32_t LP = VS + TC_C * VP * 2;        // g, then Λ_j[c] fp32, rows of LPAD
  static constexpr uint32_t AKK = LP + TC_C * LPAD * 4;     // A_kk fp32 [32][AP]
  static constexpr uint32_t EC = AKK + TC_C * AP * 4;       // e^{Λ_C[c]} [128]
  static constexpr uint32_t BT = EC + TC_D * 4;             // β_j [32]
  static constexpr uint32_t BAR = BT + TC_C * 4;            // 2 mbarriers, TMEM base, ok flag
  static constexpr uint32_t BYTES = BAR + 32;
};
static_assert(KdaSmem::BYTES <= 227 * 1024, "shared memory");
constexpr float KDA_FACTOR_FLOOR = -60.f;   // lowest chunk log-decay the factored pair products take

// KDA chunk inputs in registers: k, q, v (bf16) as in TcStage, the g rows as
// float4 (4 per thread: row j = idx / 32, channel quad idx % 32), and β.
struct KdaStage {
  uint4 k[2], q[2], v[2];
  float4 gv[4];
  float b;

  __device__ __forceinline__ void load(const uint16_t* __restrict__ qg, const uint16_t* __restrict__ kg,
                                       const uint16_t* __restrict__ vg, const float* __restrict__ gg,
                                       const float* __restrict__ bg, int t0, int Cc, size_t nH,
                                       int sh, int tid) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      int j, cv;
      chunk_piece(tid + e * TC_THREADS, j, cv);
      if (j < Cc) {
        const size_t base = ((size_t)(t0 + j) * nH + sh) * TC_D + cv * 8;
        k[e] = *reinterpret_cast<const uint4*>(kg + base);
        q[e] = *reinterpret_cast<const uint4*>(qg + base);
        v[e] = *reinterpret_cast<const uint4*>(vg + base);
      } else {
        k[e] = q[e] = v[e] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int idx = tid + e * TC_THREADS, j = idx >> 5, c4 = idx & 31;
      gv[e] = j < Cc ? *reinterpret_cast<const float4*>(gg + ((size_t)(t0 + j) * nH + sh) * TC_D + 4 * c4)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (tid < 32) b = tid < Cc ? bg[(size_t)(t0 + tid) * nH + sh] : 0.f;
  }

  // v as bf16 rows, the g rows (scanned in place later), β; k and q stay in
  // registers until the decayed operands are formed
  __device__ __forceinline__ void store(unsigned char* sm, int tid) const {
    float* Lp = reinterpret_cast<float*>(sm + KdaSmem::LP);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      int j, cv;
      chunk_piece(tid + e * TC_THREADS, j, cv);
      *reinterpret_cast<uint4*>(sm + KdaSmem::VS + (j * VP + cv * 8) * 2) = v[e];
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int idx = tid + e * TC_THREADS, j = idx >> 5, c4 = idx & 31;
      *reinterpret_cast<float4*>(Lp + j * LPAD + 4 * c4) = gv[e];
    }
    if (tid < 32) reinterpret_cast<float*>(sm + KdaSmem::BT)[tid] = b;   // 0 past Cc
  }
};

// The 8 bf16 values of a 16-byte piece as fp32.
__device__ __forceinline__ void unpack8(const uint4 w, float (&x)[8]) {
  x[0] = bf16lo(w.x); x[1] = bf16hi(w.x); x[2] = bf16lo(w.y); x[3] = bf16hi(w.y);
  x[4] = bf16lo(w.z); x[5] = bf16hi(w.z); x[6] = bf16lo(w.w); x[7] = bf16hi(w.w);
}

__global__ void __launch_bounds__(TC_THREADS, 1)
prefill_kda_tc_kernel(const __grid_constant__ SlotListArgs a, const uint16_t* __restrict__ q,
                      const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                      const float* __restrict__ g, const float* __restrict__ beta, void* o, int T,
                      int out_bf16, float scale, int32_t* status) {
  extern __shared__ __align__(1024) unsigned char sm[];
  float* Lp = reinterpret_cast<float*>(sm + KdaSmem::LP);
  float* Akk = reinterpret_cast<float*>(sm + KdaSmem::AKK);
  float* Ec = reinterpret_cast<float*>(sm + KdaSmem::EC);
  const float* Bt = reinterpret_cast<const float*>(sm + KdaSmem::BT);
  const uint16_t* Vs = reinterpret_cast<const uint16_t*>(sm + KdaSmem::VS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + KdaSmem::BAR + 16);
  int32_t* ok_flag = reinterpret_cast<int32_t*>(sm + KdaSmem::BAR + 20);
  const uint32_t sbase = smem_u32(sm);
  const uint32_t bar1 = sbase + KdaSmem::BAR, bar2 = sbase + KdaSmem::BAR + 8;
  constexpr uint32_t K_D0 = 0, K_D1 = 32, K_D3 = 96, K_D2 = 128;   // TMEM columns

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q4 = warp & 3, hw = warp >> 2;
  const int r = 32 * q4 + lane;
  const int sh = blockIdx.x, row = sh / a.H, h = sh - row * a.H;
  const int slot = a.items[row].slot;
  const size_t nH = (size_t)a.rows * a.H;
  float* gS = a.Sbar + ((size_t)slot * a.H + h) * TC_D * TC_D;

  if (warp == 0) tc::tmem_alloc(sbase + KdaSmem::BAR + 16, TC_COLS);
  if (tid == 0) {
    mbar_init(bar1, 1);
    mbar_init(bar2, 1);
    fence_mbar_init();
    *ok_flag = 1;
  }
  // rows 64-127 of the [k̂; q̂; 0] operands stay zero; A_kk's row padding too
  for (int idx = tid; idx < 64 * TC_D * 2 / 16; idx += TC_THREADS) {
    reinterpret_cast<uint4*>(sm + KdaSmem::BHI + 64 * TC_D * 2)[idx] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4*>(sm + KdaSmem::BLO + 64 * TC_D * 2)[idx] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (tid < TC_C) *reinterpret_cast<float4*>(Akk + tid * AP + TC_C) = make_float4(0.f, 0.f, 0.f, 0.f);
  float S[64];
  {
    const float4* src = reinterpret_cast<const float4*>(gS + (size_t)r * TC_D + 64 * hw);
#pragma unroll
    for (int c4 = 0; c4 < 16; ++c4) {
      const float4 x = src[c4];
      S[4 * c4] = x.x;
      S[4 * c4 + 1] = x.y;
      S[4 * c4 + 2] = x.z;
      S[4 * c4 + 3] = x.w;
    }
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
      uint4 hv, lv;
      split8(S + 8 * c8, hv, lv);
      const uint32_t off = tc::kmaj_off(r, 64 * hw + 8 * c8, TC_D);
      *reinterpret_cast<uint4*>(sm + KdaSmem::SHI + off) = hv;
      *reinterpret_cast<uint4*>(sm + KdaSmem::SLO + off) = lv;
    }
  }
  KdaStage st;
  st.load(q, k, v, g, beta, 0, T < TC_C ? T : TC_C, nH, sh, tid);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tm = *tmem_slot;
  const uint32_t tlane = tm + ((uint32_t)(32 * q4) << 16);
  bool ok = true;
  int chunk = 0;
  for (int t0 = 0; t0 < T && ok; t0 += TC_C, ++chunk) {
    const int Cc = (T - t0) < TC_C ? (T - t0) : TC_C;
    const uint32_t par = (uint32_t)chunk & 1u;
    // ---- stage; Λ = inclusive scan of g down each channel (padding tokens: g = 0);
    //      the vote: does every channel's chunk log-decay stay above the floor?
    st.store(sm, tid);
    __syncthreads();
    float lc = 0.f;
    if (tid < TC_D) {
#pragma unroll 8
      for (int j = 0; j < TC_C; ++j) {
        lc += Lp[j * LPAD + tid];
        Lp[j * LPAD + tid] = lc;
      }
      Ec[tid] = expf(lc);
    }
    const bool direct = __syncthreads_or(tid < TC_D && !(lc >= KDA_FACTOR_FLOOR)) != 0;
    // ---- decayed operands, 8 channels of one token per piece (k, q from registers):
    //      [k̂_j; q̂_j] and k̄_j (hi, lo), k̃_j (hi, lo; zero past Cc) transposed
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      int j, cv;
      chunk_piece(tid + e * TC_THREADS, j, cv);
      float kx[8], qx[8], kh[8], qh[8], kb[8], kt[8];
      unpack8(st.k[e], kx);
      unpack8(st.q[e], qx);
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int c = cv * 8 + t;
        const float lj = Lp[j * LPAD + c];
        const float el = __expf(lj);                                  // Λ <= 0
        kh[t] = el * kx[t];
        qh[t] = el * qx[t];
        if (direct) {
          kb[t] = 0.f;
          kt[t] = j < Cc ? __expf(Lp[(Cc - 1) * LPAD + c] - lj) * kx[t] : 0.f;   // Λ_C - Λ_j <= 0
        } else {
          const float eb = __expf(-lj);                               // <= e^{60}
          kb[t] = eb * kx[t];
          kt[t] = j < Cc ? fminf(Ec[cv * 8 + t] * eb, 1.f) * kx[t] : 0.f;
        }
      }
      uint4 hv, lv;
      const uint32_t okq = tc::kmaj_off(j, cv * 8, TC_D);
      split8(kh, hv, lv);
      *reinterpret_cast<uint4*>(sm + KdaSmem::BHI + okq) = hv;
      *reinterpret_cast<uint4*>(sm + KdaSmem::BLO + okq) = lv;
      split8(qh, hv, lv);
      *reinterpret_cast<uint4*>(sm + KdaSmem::BHI + tc::kmaj_off(TC_C + j, cv * 8, TC_D)) = hv;
      *reinterpret_cast<uint4*>(sm + KdaSmem::BLO + tc::kmaj_off(TC_C + j, cv * 8, TC_D)) = lv;
      split8(kb, hv, lv);
      *reinterpret_cast<uint4*>(sm + KdaSmem::KBHI + okq) = hv;
      *reinterpret_cast<uint4*>(sm + KdaSmem::KBLO + okq) = lv;
      split8(kt, hv, lv);
      // k̃_j[8 cv .. 8 cv + 7]: one 16-byte row of a core matrix of the MN-major k̃
      const uint32_t otc = tc::mnmaj_off(cv * 8, j, TC_C);
      *reinterpret_cast<uint4*>(sm + KdaSmem::KTHI + otc) = hv;
      *reinterpret_cast<uint4*>(sm + KdaSmem::KTLO + otc) = lv;
    }
    tc::fence_smem_to_async();   // S̄ terms and the decayed operands, for the tensor cores
    tc::fence_before_sync();
    __syncthreads();
    // ---- D0 = [k̂; q̂; 0] k̄^T (fast chunks) and D1 = S̄ [k̂; q̂]^T, three terms each
    if (tid == 0) {
      tc::fence_after_sync();
      constexpr uint32_t id0 = tc::idesc_bf16_f32(128, 32), id1 = tc::idesc_bf16_f32(128, 64);
      const uint32_t sa[3] = {KdaSmem::SHI, KdaSmem::SLO, KdaSmem::SHI};
      const uint32_t ba[3] = {KdaSmem::BHI, KdaSmem::BLO, KdaSmem::BHI};
      const uint32_t bb[3] = {KdaSmem::BHI, KdaSmem::BHI, KdaSmem::BLO};
      const uint32_t kb3[3] = {KdaSmem::KBHI, KdaSmem::KBHI, KdaSmem::KBLO};
#pragma unroll
      for (int term = 0; term < 3; ++term)
#pragma unroll
        for (int kk = 0; kk < TC_D / 16; ++kk) {
          if (!direct)
            tc::mma_bf16(tm + K_D0, tc::kmaj_desc(sbase + ba[term], TC_D, kk),
                         tc::kmaj_desc(sbase + kb3[term], TC_D, kk), id0, (term | kk) != 0);
          tc::mma_bf16(tm + K_D1, tc::kmaj_desc(sbase + sa[term], TC_D, kk),
                       tc::kmaj_desc(sbase + bb[term], TC_D, kk), id1, (term | kk) != 0);
        }
      tc::mma_commit(bar1);
    }
    auto put_a = [&](int j, int i, float av) {   // A[j][i] as the bf16 terms of D3's B operand
      const uint32_t hv = bf16x2(av, 0.f) & 0xffffu;
      const uint32_t lv = bf16x2(av - __uint_as_float(hv << 16), 0.f) & 0xffffu;
      const uint32_t off = tc::kmaj_off(j, i, TC_C);
      *reinterpret_cast<uint16_t*>(sm + KdaSmem::AHI + off) = (uint16_t)hv;
      *reinterpret_cast<uint16_t*>(sm + KdaSmem::ALO + off) = (uint16_t)lv;
    };
    if (direct) {
      // strong decay: every pair (j, i) directly, e^{Λ_j[c]-Λ_i[c]} per channel,
      // with k, q read back from global memory (pairs tid, tid + 256, tid + 512)
      for (int p = tid; p < TC_C * TC_C; p += TC_THREADS) {
        const int j = p >> 5, i = p & 31;
        float kk = 0.f, qk = 0.f;
        if (i <= j && j < Cc) {
          const uint16_t* kj = k + ((size_t)(t0 + j) * nH + sh) * TC_D;
          const uint16_t* qj = q + ((size_t)(t0 + j) * nH + sh) * TC_D;
          const uint16_t* ki = k + ((size_t)(t0 + i) * nH + sh) * TC_D;
          for (int c = 0; c < TC_D; ++c) {
            const float w = __expf(Lp[j * LPAD + c] - Lp[i * LPAD + c]) * bf16f(ki[c]);
            kk += w * bf16f(kj[c]);
            qk += w * bf16f(qj[c]);
          }
        }
        Akk[j * AP + i] = i < j ? kk : 0.f;
        put_a(j, i, qk);
      }
    }
    if (t0 + TC_C < T) {
      const int Cn = (T - t0 - TC_C) < TC_C ? (T - t0 - TC_C) : TC_C;
      st.load(q, k, v, g, beta, t0 + TC_C, Cn, nH, sh, tid);
    }
    if (tid == 0 && !mbar_wait(bar1, par, status, DEV_TIMEOUT_MMA)) *ok_flag = -1;
    __syncthreads();
    if (*ok_flag != 1) {
      ok = false;
      break;
    }
    tc::fence_after_sync();
    // ---- fast chunks: the pair coefficients from D0 (warps 0, 1, 4, 5: rows
    //      0-63, 16 columns each), live below the diagonal (A_kk) or on and below it (A)
    if (!direct && q4 < 2) {
      uint32_t x[16];
      tc::tmem_ld16(tlane + K_D0 + 16 * hw, x);
      tc::tmem_wait_ld16(x);
      const int j = lane, i0 = 16 * hw;
      float w[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int i = i0 + e;
        const bool live = (q4 == 0 ? i < j : i <= j) && j < Cc;
        w[e] = live ? __uint_as_float(x[e]) : 0.f;
      }
      if (q4 == 0) {
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4)
          *reinterpret_cast<float4*>(Akk + j * AP + i0 + 4 * e4) =
              make_float4(w[4 * e4], w[4 * e4 + 1], w[4 * e4 + 2], w[4 * e4 + 3]);
      } else {
#pragma unroll
        for (int c8 = 0; c8 < 2; ++c8) {
          uint4 hv, lv;
          split8(w + 8 * c8, hv, lv);
          const uint32_t off = tc::kmaj_off(j, i0 + 8 * c8, TC_C);
          *reinterpret_cast<uint4*>(sm + KdaSmem::AHI + off) = hv;
          *reinterpret_cast<uint4*>(sm + KdaSmem::ALO + off) = lv;
        }
      }
    }
    __syncthreads();
    // ---- forward substitution (warps 0-3, one value row each)
    if (hw == 0) {
      float pk[TC_C], u[TC_C];
      {
        uint32_t x[TC_C];
        tc::tmem_ld32(tlane + K_D1, x);
        tc::tmem_wait_ld(x);
#pragma unroll
        for (int j = 0; j < TC_C; ++j) pk[j] = __uint_as_float(x[j]);
      }
#pragma unroll
      for (int j = 0; j < TC_C; ++j) u[j] = 0.f;
#pragma unroll
      for (int j = 0; j < TC_C; ++j) {
        float x[4] = {pk[j], 0.f, 0.f, 0.f};
#pragma unroll
        for (int i4 = 0; i4 < (j + 3) / 4; ++i4) {
          const float4 c = *reinterpret_cast<const float4*>(Akk + j * AP + 4 * i4);
          x[0] += c.x * u[4 * i4];
          x[1] += c.y * u[4 * i4 + 1];
          x[2] += c.z * u[4 * i4 + 2];
          x[3] += c.w * u[4 * i4 + 3];
        }
        u[j] = Bt[j] * (bf16f(Vs[j * VP + r]) - ((x[0] + x[1]) + (x[2] + x[3])));   // 0 past Cc
      }
#pragma unroll
      for (int c8 = 0; c8 < TC_C / 8; ++c8) {
        uint4 hv, lv;
        split8(u + 8 * c8, hv, lv);
        const uint32_t off = tc::kmaj_off(r, 8 * c8, TC_C);
        *reinterpret_cast<uint4*>(sm + KdaSmem::UHI + off) = hv;
        *reinterpret_cast<uint4*>(sm + KdaSmem::ULO + off) = lv;
      }
    }
    tc::fence_smem_to_async();   // U and A terms, for the tensor cores
    tc::fence_before_sync();
    __syncthreads();
    // ---- D2 = U k̃ and D3 = U A^T, three terms each
    if (tid == 0) {
      tc::fence_after_sync();
      constexpr uint32_t id2 = tc::idesc_bf16_f32(128, 128, false, true);   // k̃ MN-major
      constexpr uint32_t id3 = tc::idesc_bf16_f32(128, 32);
      const uint32_t ua[3] = {KdaSmem::UHI, KdaSmem::ULO, KdaSmem::UHI};
      const uint32_t kb[3] = {KdaSmem::KTHI, KdaSmem::KTHI, KdaSmem::KTLO};
      const uint32_t ab[3] = {KdaSmem::AHI, KdaSmem::AHI, KdaSmem::ALO};
#pragma unroll
      for (int term = 0; term < 3; ++term)
#pragma unroll
        for (int kk = 0; kk < TC_C / 16; ++kk) {
          tc::mma_bf16(tm + K_D2, tc::kmaj_desc(sbase + ua[term], TC_C, kk),
                       tc::kmaj_desc(sbase + kb[term], TC_C, kk), id2, (term | kk) != 0);
          tc::mma_bf16(tm + K_D3, tc::kmaj_desc(sbase + ua[term], TC_C, kk),
                       tc::kmaj_desc(sbase + ab[term], TC_C, kk), id3, (term | kk) != 0);
        }
      tc::mma_commit(bar2);
    }
    if (tid == 0 && !mbar_wait(bar2, par, status, DEV_TIMEOUT_MMA)) *ok_flag = -2;
    __syncthreads();
    if (*ok_flag != 1) {
      ok = false;
      break;
    }
    tc::fence_after_sync();
    // ---- outputs of tokens 16 h .. 16 h + 15 of row r: o_j = scale (S̄ q̂_j + D3)
    if (o != nullptr) {
      uint32_t xq[16], x3[16];
      tc::tmem_ld16(tlane + K_D1 + TC_C + 16 * hw, xq);
      tc::tmem_ld16(tlane + K_D3 + 16 * hw, x3);
      tc::tmem_wait_ld16(xq);
      tc::tmem_wait_ld16(x3);
      const size_t ostride = nH * TC_D;
      const size_t obase = ((size_t)(t0 + 16 * hw) * nH + sh) * TC_D + r;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        if (16 * hw + e < Cc) {
          const float yo = scale * (__uint_as_float(xq[e]) + __uint_as_float(x3[e]));
          const size_t oi = obase + (size_t)e * ostride;
          if (out_bf16) static_cast<uint16_t*>(o)[oi] = f2bf16(yo);
          else static_cast<float*>(o)[oi] = yo;
        }
      }
    }
    // ---- S̄ <- S̄ Diag(e^{Λ_C}) + D2; its bf16 terms for the next chunk
    {
      uint32_t x0[32], x1[32];
      tc::tmem_ld32(tlane + K_D2 + 64 * hw, x0);
      tc::tmem_ld32(tlane + K_D2 + 64 * hw + 32, x1);
      tc::tmem_wait_ld(x0);
      tc::tmem_wait_ld(x1);
      const float* ec = Ec + 64 * hw;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        S[c] = ec[c] * S[c] + __uint_as_float(x0[c]);
        S[32 + c] = ec[32 + c] * S[32 + c] + __uint_as_float(x1[c]);
      }
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        uint4 hv, lv;
        split8(S + 8 * c8, hv, lv);
        const uint32_t off = tc::kmaj_off(r, 64 * hw + 8 * c8, TC_D);
        *reinterpret_cast<uint4*>(sm + KdaSmem::SHI + off) = hv;
        *reinterpret_cast<uint4*>(sm + KdaSmem::SLO + off) = lv;
      }
    }
    tc::fence_before_sync();
    __syncthreads();
  }
  if (!ok && tid == 0) mbar_drain(*ok_flag == -1 ? bar1 : bar2, (uint32_t)chunk & 1u);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tm, TC_COLS);
  }
  if (!ok) return;
  float4* dst = reinterpret_cast<float4*>(gS + (size_t)r * TC_D + 64 * hw);
#pragma unroll
  for (int c4 = 0; c4 < 16; ++c4)
    dst[c4] = make_float4(S[4 * c4], S[4 * c4 + 1], S[4 * c4 + 2], S[4 * c4 + 3]);
  if (h == 0 && tid == 0) {
    a.nlog[slot] = 0;
    a.base_of[slot] = slot;
  }
}


// ------------------------------------------------------------------ RWKV6 ----
// Chunked prefill of RWKV6 at d_k = d_v = 64 on the tensor cores, two
// slot-heads per CTA (flattened slot-heads 2b and 2b + 1) stacked into the
// 128 rows of an M = 128 MMA.  RWKV6 has no delta rule: with Λ_j the inclusive
// cumulative log-decay inside the chunk (Λ_{-1} = 0), r̂_j = e^{Λ_{j-1}} ⊙ r_j,
// k̄_s = e^{-Λ_s} ⊙ k_s and k̃_s = e^{Λ_C-Λ_s} ⊙ k_s,
//   o_j = scale (S̄ r̂_j + Σ_{s<j} (r̂_j·k̄_s) v_s + c_j v_j),  c_j = Σ_c r_j[c] u[c] k_j[c]
//   S̄'  = S̄ Diag(e^{Λ_C}) + Σ_s v_s k̃_s^T
// (the same algebra as prefill_perkey_kernel in prefill.cu).  Value rows of
// head e sit at rows 64 e + v, its tokens at rows 32 e + j of the token-row
// operands, its key channels at rows 64 e + c of k̃; each product is formed for
// both heads at once and only head e's block of it is read:
//   [D0 | Y] [128 x 192] = [r̂; 0] [k̄; S̄]^T, one N = 192 product:
//       D0, columns 0-63: pair coefficients r̂_j·k̄_s (rows 32 e + j, columns 32 e + s);
//       Y, columns 64-191: (S̄ r̂_j)[v] at row 32 e + j, column 64 + 64 e + v
//   Y += A V^T                        the outputs' log terms, added onto Y
//   D2 [128 x 128] = V k̃              rows 64 e + v, columns 64 e + c
// (rows 64-127 of the first two pad the MMA's M and are not read).  S̄, r̂,
// k̄, k̃ and A are fp32, carried as hi + lo bf16 terms (three products for
// r̂ [k̄; S̄]^T, two with the exact bf16 V).  The factored pair products
// stay finite while the chunk's log-decay stays above -60 in every channel,
// as in KDA's kernel; a chunk below it forms A directly on the CUDA cores.
constexpr int RW_D = 64;
constexpr uint32_t RW_COLS = 512;   // TMEM: [D0 | Y] of even chunks [0, 192), of odd ones [192, 384), D2 [384, 512)
constexpr int RW_LT = TC_C + 1;   // fp32 Λ, channel-major: column 64 e + c at col * RW_LT, token j at + j

struct RwSmem {
  // [k̄; S̄] hi and lo, the B operand of the N = 192 product: k̄ rows 32 e + s,
  // then S̄ rows 64 e + v, each K-major over the 64 key channels
  static constexpr uint32_t KSHI = 0;
  static constexpr uint32_t KSLO = KSHI + (64 + 128) * RW_D * 2;
  static constexpr uint32_t KBHI = KSHI, SHI = KSHI + 64 * RW_D * 2;
  static constexpr uint32_t KBLO = KSLO, SLO = KSLO + 64 * RW_D * 2;
  static constexpr uint32_t RHI = KSLO + (64 + 128) * RW_D * 2;   // [r̂ (64 rows: 32 e + j); 0 (64)] x 64
  static constexpr uint32_t RLO = RHI + 128 * RW_D * 2;
  static constexpr uint32_t KTHI = RLO + 128 * RW_D * 2;      // k̃ [128 rows (64 e + c)] x [32 tokens], MN-major
  static constexpr uint32_t KTLO = KTHI + 128 * TC_C * 2;
  static constexpr uint32_t VO = KTLO + 128 * TC_C * 2;       // V [128 rows (64 e + v)] x [32 tokens], MN-major,
  static constexpr uint32_t VO_SZ = 128 * TC_C * 2;           //   two (even and odd chunks)
  static constexpr uint32_t AHI = VO + 2 * VO_SZ;             // A [64 rows (32 e + j)] x [32 (s)]
  static constexpr uint32_t ALO = AHI + 64 * TC_C * 2;
  static constexpr uint32_t LP = ALO + 64 * TC_C * 2;         // Λ_j of direct chunks, fp32 [128][RW_LT]
  static constexpr uint32_t ER = LP + 128 * RW_LT * 4;        // e^{Λ_{j-1}}, same layout
  static constexpr uint32_t EB = ER + 128 * RW_LT * 4;        // e^{-Λ_j}, same layout
  static constexpr uint32_t HT = EB + 128 * RW_LT * 4;        // Λ_15 of each column [128]
  static constexpr uint32_t EC = HT + 128 * 4;                // e^{Λ_C} [128]
  static constexpr uint32_t UB = EC + 128 * 4;                // bonus u of both heads [128]
  static constexpr uint32_t CBP = UB + 128 * 4;               // c_j partials [2][32][8]
  static constexpr uint32_t CB = CBP + 2 * TC_C * 8 * 4;      // c_j [2][32], two (even and odd chunks)
  static constexpr uint32_t BAR = CB + 2 * 2 * TC_C * 4;      // 2 mbarriers, TMEM base, ok flag
  static constexpr uint32_t BYTES = BAR + 32;
};
static_assert(RwSmem::BYTES <= 227 * 1024, "shared memory");
static_assert(RwSmem::LP % 16 == 0 && RwSmem::BAR % 16 == 0, "16-byte aligned buffers");
// The pair-coefficient product reads A as an M = 128 operand: its rows 64-127
// are the next 4 KB (ALO, then the start of LP), whatever they hold; the
// product's rows 64-127 are never read.
static_assert(RwSmem::ALO == RwSmem::AHI + 64 * TC_C * 2 && RwSmem::LP == RwSmem::ALO + 64 * TC_C * 2 &&
              RwSmem::LP + 64 * TC_C * 2 <= RwSmem::BYTES, "A's padding rows stay inside the block");

// One chunk's r, k, v (bf16) and g of the CTA's two slot-heads, in registers
// between the global loads and their use.  The two slot-heads' rows of a token
// are adjacent in the token-major inputs, so a token's 128 values (64 e + c)
// are one contiguous run; a second slot-head past the batch (`two` false)
// loads zeros.  r, k, v come as pieces (8 channels of one token); g comes in
// the scan's layout: thread (half hf, column cl = 64 e + c) holds g of tokens
// 16 hf .. 16 hf + 15 of its column (for one token the 128 columns' loads are
// one contiguous 512-byte run).
struct RwStage {
  uint4 r[2], k[2], v[2];
  float gs[16];

  __device__ __forceinline__ void load(const uint16_t* __restrict__ rg, const uint16_t* __restrict__ kg,
                                       const uint16_t* __restrict__ vg, const float* __restrict__ gg,
                                       int t0, int Cc, size_t nH, int sh0, bool two, int tid) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      int j, cv;
      chunk_piece(tid + e * TC_THREADS, j, cv);   // cv / 8: slot-head, (cv % 8) * 8: channel
      if (j < Cc && (two || cv < 8)) {
        const size_t base = ((size_t)(t0 + j) * nH + sh0) * RW_D + cv * 8;
        r[e] = *reinterpret_cast<const uint4*>(rg + base);
        k[e] = *reinterpret_cast<const uint4*>(kg + base);
        v[e] = *reinterpret_cast<const uint4*>(vg + base);
      } else {
        r[e] = k[e] = v[e] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    const int cl = tid & 127, hf = tid >> 7;
    const bool col_ok = two || cl < RW_D;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int jj = 16 * hf + j;
      gs[j] = (jj < Cc && col_ok) ? gg[((size_t)(t0 + jj) * nH + sh0) * RW_D + cl] : 0.f;
    }
  }
};

__global__ void __launch_bounds__(TC_THREADS, 1)
prefill_rwkv6_tc_kernel(const __grid_constant__ SlotListArgs a, const uint16_t* __restrict__ r_in,
                        const uint16_t* __restrict__ k_in, const uint16_t* __restrict__ v_in,
                        const float* __restrict__ g, const float* __restrict__ bonus, void* o, int T,
                        int out_bf16, float scale, int32_t* status) {
  extern __shared__ __align__(1024) unsigned char sm[];
  float* Lp = reinterpret_cast<float*>(sm + RwSmem::LP);
  float* Er = reinterpret_cast<float*>(sm + RwSmem::ER);
  float* Eb = reinterpret_cast<float*>(sm + RwSmem::EB);
  float* Ht = reinterpret_cast<float*>(sm + RwSmem::HT);
  float* Ec = reinterpret_cast<float*>(sm + RwSmem::EC);
  float* Ub = reinterpret_cast<float*>(sm + RwSmem::UB);
  float* Cbp = reinterpret_cast<float*>(sm + RwSmem::CBP);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + RwSmem::BAR + 16);
  int32_t* ok_flag = reinterpret_cast<int32_t*>(sm + RwSmem::BAR + 20);
  const uint32_t sbase = smem_u32(sm);
  const uint32_t bar1 = sbase + RwSmem::BAR, bar2 = sbase + RwSmem::BAR + 8;
  constexpr uint32_t K_D0 = 0, K_Y = 64, K_SET = 192, K_D2 = 384;   // TMEM columns

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q4 = warp & 3, hw = warp >> 2;
  const int r = 32 * q4 + lane;          // row: slot-head e = r / 64, value row r % 64
  const int he = r >> 6, vrow = r & 63;  // (he is uniform over a warp)
  const int nH = a.rows * a.H;
  const int sh0 = 2 * (int)blockIdx.x;
  const bool two = sh0 + 1 < nH;
  const int she = sh0 + he;
  const bool mine = he == 0 || two;      // this thread's row belongs to a slot-head of the batch
  auto state_of = [&](int sh) {
    const int row = sh / a.H, h = sh - row * a.H;
    return a.Sbar + ((size_t)a.items[row].slot * a.H + h) * RW_D * RW_D;
  };

  if (warp == 0) tc::tmem_alloc(sbase + RwSmem::BAR + 16, RW_COLS);
  if (tid == 0) {
    mbar_init(bar1, 1);
    mbar_init(bar2, 1);
    fence_mbar_init();
    *ok_flag = 1;
  }
  // rows 64-127 of the [r̂; 0] operand stay zero
  for (int idx = tid; idx < 64 * RW_D * 2 / 16; idx += TC_THREADS) {
    reinterpret_cast<uint4*>(sm + RwSmem::RHI + 64 * RW_D * 2)[idx] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4*>(sm + RwSmem::RLO + 64 * RW_D * 2)[idx] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (tid < 128) {   // bonus u of slot-head tid / 64, channel tid % 64
    const int sh = sh0 + (tid >> 6);
    Ub[tid] = sh < nH ? bonus[(size_t)(sh % a.H) * RW_D + (tid & 63)] : 0.f;
  }
  // this thread's state: S̄ of slot-head he, value row vrow, channels 32 hw .. 32 hw + 31
  float S[32];
  {
    if (mine) {
      const float4* src = reinterpret_cast<const float4*>(state_of(she) + (size_t)vrow * RW_D + 32 * hw);
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 x = src[c4];
        S[4 * c4] = x.x;
        S[4 * c4 + 1] = x.y;
        S[4 * c4 + 2] = x.z;
        S[4 * c4 + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int c = 0; c < 32; ++c) S[c] = 0.f;
    }
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) {
      uint4 hv, lv;
      split8(S + 8 * c8, hv, lv);
      const uint32_t off = tc::kmaj_off(r, 32 * hw + 8 * c8, RW_D);
      *reinterpret_cast<uint4*>(sm + RwSmem::SHI + off) = hv;
      *reinterpret_cast<uint4*>(sm + RwSmem::SLO + off) = lv;
    }
  }
  RwStage st;
  st.load(r_in, k_in, v_in, g, 0, T < TC_C ? T : TC_C, (size_t)nH, sh0, two, tid);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tm = *tmem_slot;
  const uint32_t tlane = tm + ((uint32_t)(32 * q4) << 16);
  const bool ovec = (reinterpret_cast<uintptr_t>(o) & 15u) == 0;
  // The outputs o_j = scale (Y_j + c_j v_j) of a finished chunk (the TMEM, V
  // and c_j sets bo) for token j = lane of slot-head e = q4 (warps q4 < 2),
  // values 32 hw .. 32 hw + 31, from Y's row 32 e + j; 16-byte stores when o is
  // 16-byte aligned (a token's 32 values are contiguous).  Chunk c - 1's run
  // while chunk c's first MMA group does.
  auto emit = [&](int bo, int t0o, int Cco) {
    if (q4 < 2 && o != nullptr && (q4 == 0 || two)) {   // uniform over the warp
      const int j = lane;
      uint32_t y[32];
      tc::tmem_ld32(tlane + K_SET * bo + K_Y + 64 * q4 + 32 * hw, y);
      float vj[32];   // v_j of values 32 hw .. 32 hw + 31: value rows 64 e + v of V
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        float t8[8];
        unpack8(*reinterpret_cast<const uint4*>(sm + RwSmem::VO + RwSmem::VO_SZ * bo +
                                                tc::mnmaj_off(64 * q4 + 32 * hw + 8 * c8, j, TC_C)),
                t8);
#pragma unroll
        for (int e = 0; e < 8; ++e) vj[8 * c8 + e] = t8[e];
      }
      const float cb = reinterpret_cast<const float*>(sm + RwSmem::CB)[2 * TC_C * bo + TC_C * q4 + j];
      tc::tmem_wait_ld(y);
      if (j < Cco) {
        float yo[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) yo[i] = scale * (__uint_as_float(y[i]) + cb * vj[i]);
        const size_t oi = ((size_t)(t0o + j) * nH + sh0 + q4) * RW_D + 32 * hw;
        if (out_bf16) {
          uint16_t* ob = static_cast<uint16_t*>(o) + oi;
          if (ovec) {
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8)
              reinterpret_cast<uint4*>(ob)[c8] =
                  make_uint4(bf16x2(yo[8 * c8], yo[8 * c8 + 1]), bf16x2(yo[8 * c8 + 2], yo[8 * c8 + 3]),
                             bf16x2(yo[8 * c8 + 4], yo[8 * c8 + 5]), bf16x2(yo[8 * c8 + 6], yo[8 * c8 + 7]));
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) ob[i] = f2bf16(yo[i]);
          }
        } else {
          float* of = static_cast<float*>(o) + oi;
          if (ovec) {
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4)
              reinterpret_cast<float4*>(of)[c4] =
                  make_float4(yo[4 * c4], yo[4 * c4 + 1], yo[4 * c4 + 2], yo[4 * c4 + 3]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) of[i] = yo[i];
          }
        }
      }
    }
  };
  // Thread 64 (a warp without outputs) issues the MMAs and waits for them.
  constexpr int MMA_TID = 64;
  bool ok = true;
  int chunk = 0;
  for (int t0 = 0; t0 < T && ok; t0 += TC_C, ++chunk) {
    const int Cc = (T - t0) < TC_C ? (T - t0) : TC_C;
    const uint32_t par = (uint32_t)chunk & 1u;
    const int b = chunk & 1;
    const uint32_t vo = RwSmem::VO + RwSmem::VO_SZ * b, tb = K_SET * b;
    // ---- Λ = inclusive scan of g down each of the 128 columns (64 e + c; padding
    //      tokens and a missing second slot-head have g = 0); the vote: does every
    //      column's chunk log-decay stay above the floor?  Thread (half hf, column
    //      cl) scans tokens 16 hf .. 16 hf + 15 of its column from its registers,
    //      the second half then adds the first half's total, and each thread forms
    //      its tokens' decay factors e^{Λ_{j-1}} (for r̂) and e^{-Λ_j} (for k̄ and
    //      k̃; only used while the vote passes).
    float lc = 0.f;
    const int cl = tid & 127, hf = tid >> 7;
    float* col = Lp + cl * RW_LT + 16 * hf;
    float lam[16];
    float pre;
    {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        lc += st.gs[j];
        lam[j] = lc;
      }
      if (hf == 0) Ht[cl] = lc;
      __syncthreads();
      pre = hf ? Ht[cl] : 0.f;   // Λ at the half's first token minus one
      float* er = Er + cl * RW_LT + 16 * hf;
      float* eb = Eb + cl * RW_LT + 16 * hf;
      float prev = pre;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float l = pre + lam[j];
        er[j] = __expf(prev);   // Λ_{j-1} <= 0
        eb[j] = __expf(-l);     // <= e^{60} while the vote passes
        prev = l;
      }
      lc = pre + lc;            // Λ_C for the second half's threads
      if (hf) Ec[cl] = expf(lc);
    }
    const bool direct = __syncthreads_or(tid >= 128 && !(lc >= KDA_FACTOR_FLOOR)) != 0;
    if (direct) {   // Λ itself, over the staged g, for the direct path's exponents
#pragma unroll
      for (int j = 0; j < 16; ++j) col[j] = pre + lam[j];
      __syncthreads();
    }
    // ---- operands, 8 channels of one token of one slot-head per piece (r, k, v
    //      from registers), one 16-byte store each: r̂ and k̄ (hi, lo) K-major as
    //      token rows; k̃ (hi, lo) and V MN-major, whose core-matrix rows are a
    //      token's eight channels (eight lanes of a warp fill one core matrix);
    //      the bonus sums' partials.
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      int j, cv;
      chunk_piece(tid + e * TC_THREADS, j, cv);
      const int hd = cv >> 3, c0 = (cv & 7) * 8, col0 = 8 * cv;   // col0 = 64 hd + c0
      float rx[8], kx[8], rh[8], kb[8], kt[8];
      unpack8(st.r[e], rx);
      unpack8(st.k[e], kx);
      // e^{Λ_C} and the bonus u of the piece's 8 columns (two 16-byte loads each)
      const float4 e0 = *reinterpret_cast<const float4*>(Ec + col0);
      const float4 e1 = *reinterpret_cast<const float4*>(Ec + col0 + 4);
      const float4 u0 = *reinterpret_cast<const float4*>(Ub + col0);
      const float4 u1 = *reinterpret_cast<const float4*>(Ub + col0 + 4);
      const float ec8[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
      const float ub8[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
      float cb = 0.f;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int col = col0 + t;
        const int cj = col * RW_LT + j;
        rh[t] = Er[cj] * rx[t];
        if (direct) {
          kb[t] = 0.f;
          kt[t] = j < Cc ? __expf(Lp[col * RW_LT + TC_C - 1] - Lp[cj]) * kx[t] : 0.f;   // <= 0
        } else {
          const float eb = Eb[cj];                                     // <= e^{60}
          kb[t] = eb * kx[t];
          kt[t] = j < Cc ? fminf(ec8[t] * eb, 1.f) * kx[t] : 0.f;
        }
        cb += rx[t] * ub8[t] * kx[t];
      }
      Cbp[(hd * TC_C + j) * 8 + (cv & 7)] = cb;
      uint4 hv, lv;
      const uint32_t otok = tc::kmaj_off(TC_C * hd + j, c0, RW_D);
      split8(rh, hv, lv);
      *reinterpret_cast<uint4*>(sm + RwSmem::RHI + otok) = hv;
      *reinterpret_cast<uint4*>(sm + RwSmem::RLO + otok) = lv;
      split8(kb, hv, lv);
      *reinterpret_cast<uint4*>(sm + RwSmem::KBHI + otok) = hv;
      *reinterpret_cast<uint4*>(sm + RwSmem::KBLO + otok) = lv;
      split8(kt, hv, lv);
      const uint32_t ocol = tc::mnmaj_off(col0, j, TC_C);   // rows col0 .. col0 + 7 of token j
      *reinterpret_cast<uint4*>(sm + RwSmem::KTHI + ocol) = hv;
      *reinterpret_cast<uint4*>(sm + RwSmem::KTLO + ocol) = lv;
      *reinterpret_cast<uint4*>(sm + vo + ocol) = st.v[e];
    }
    tc::fence_smem_to_async();   // S̄ terms and the chunk's operands, for the tensor cores
    tc::fence_before_sync();
    __syncthreads();
    // ---- [D0 | Y] = [r̂; 0] [k̄; S̄]^T, three terms (a direct chunk's k̄ is zero)
    if (tid == MMA_TID) {
      tc::fence_after_sync();
      constexpr uint32_t id192 = tc::idesc_bf16_f32(128, 192);
      const uint32_t ra[3] = {RwSmem::RHI, RwSmem::RLO, RwSmem::RHI};
      const uint32_t kb3[3] = {RwSmem::KSHI, RwSmem::KSHI, RwSmem::KSLO};
#pragma unroll
      for (int term = 0; term < 3; ++term)
#pragma unroll
        for (int kk = 0; kk < RW_D / 16; ++kk)
          tc::mma_bf16(tm + tb + K_D0, tc::kmaj_desc(sbase + ra[term], RW_D, kk),
                       tc::kmaj_desc(sbase + kb3[term], RW_D, kk), id192, (term | kk) != 0);
      tc::mma_commit(bar1);
    }
    if (chunk > 0) emit(b ^ 1, t0 - TC_C, TC_C);   // (only the last chunk is ragged)
    // the bonus sums c_j (warps 3 and 7), in a fixed order
    if (warp == 3 || warp == 7) {
      const int i = (warp == 3 ? 0 : TC_C) + lane;
      const float* p = Cbp + i * 8;
      reinterpret_cast<float*>(sm + RwSmem::CB)[2 * TC_C * b + i] =
          ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]));
    }
    auto put_a = [&](int row, int s, float av) {   // A's bf16 terms, row 32 e + j, column s
      const uint32_t hv = bf16x2(av, 0.f) & 0xffffu;
      const uint32_t lv = bf16x2(av - __uint_as_float(hv << 16), 0.f) & 0xffffu;
      const uint32_t off = tc::kmaj_off(row, s, TC_C);
      *reinterpret_cast<uint16_t*>(sm + RwSmem::AHI + off) = (uint16_t)hv;
      *reinterpret_cast<uint16_t*>(sm + RwSmem::ALO + off) = (uint16_t)lv;
    };
    if (direct) {
      // strong decay: every pair (j, s < j) of both slot-heads directly,
      // e^{Λ_{j-1}[c]-Λ_s[c]} per channel, with r and k read back from global
      // memory (pairs tid + 256 p)
      for (int pr = tid; pr < 2 * TC_C * TC_C; pr += TC_THREADS) {
        const int hd = pr >> 10, j = (pr >> 5) & 31, s = pr & 31;
        float av = 0.f;
        if (s < j && j < Cc && (hd == 0 || two)) {
          const uint16_t* rj = r_in + ((size_t)(t0 + j) * nH + sh0 + hd) * RW_D;
          const uint16_t* ks = k_in + ((size_t)(t0 + s) * nH + sh0 + hd) * RW_D;
          for (int c = 0; c < RW_D; ++c) {
            const int col = RW_D * hd + c;
            av += bf16f(rj[c]) * bf16f(ks[c]) * __expf(Lp[col * RW_LT + j - 1] - Lp[col * RW_LT + s]);
          }
        }
        put_a(TC_C * hd + j, s, av);
      }
    }
    if (t0 + TC_C < T) {
      const int Cn = (T - t0 - TC_C) < TC_C ? (T - t0 - TC_C) : TC_C;
      st.load(r_in, k_in, v_in, g, t0 + TC_C, Cn, (size_t)nH, sh0, two, tid);
    }
    if (tid == MMA_TID && !mbar_wait(bar1, par, status, DEV_TIMEOUT_MMA)) *ok_flag = -1;
    __syncthreads();
    if (*ok_flag != 1) {
      ok = false;
      break;
    }
    tc::fence_after_sync();
    // ---- fast chunks: A from D0 (warps with q4 = e < 2 read rows 32 e + j, the
    //      columns 32 e + 16 hw .. +15 of their slot-head's block), live below
    //      the diagonal
    if (!direct && q4 < 2) {
      uint32_t x[16];
      tc::tmem_ld16(tlane + tb + K_D0 + 32 * q4 + 16 * hw, x);
      tc::tmem_wait_ld16(x);
      const int j = lane, s0 = 16 * hw;
      float w[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) w[e] = (s0 + e < j && j < Cc) ? __uint_as_float(x[e]) : 0.f;
#pragma unroll
      for (int c8 = 0; c8 < 2; ++c8) {
        uint4 hv, lv;
        split8(w + 8 * c8, hv, lv);
        const uint32_t off = tc::kmaj_off(TC_C * q4 + j, s0 + 8 * c8, TC_C);
        *reinterpret_cast<uint4*>(sm + RwSmem::AHI + off) = hv;
        *reinterpret_cast<uint4*>(sm + RwSmem::ALO + off) = lv;
      }
    }
    tc::fence_smem_to_async();   // A terms, for the tensor cores
    tc::fence_before_sync();
    __syncthreads();
    // ---- Y += [A; *] V^T and D2 = V k̃, two terms each (V is exact in bf16)
    if (tid == MMA_TID) {
      tc::fence_after_sync();
      constexpr uint32_t idy = tc::idesc_bf16_f32(128, 128, false, true);   // V MN-major
      constexpr uint32_t id2 = tc::idesc_bf16_f32(128, 128, true, true);    // V, k̃ MN-major
      const uint32_t ab[2] = {RwSmem::AHI, RwSmem::ALO};
      const uint32_t kb2[2] = {RwSmem::KTHI, RwSmem::KTLO};
#pragma unroll
      for (int term = 0; term < 2; ++term)
#pragma unroll
        for (int kk = 0; kk < TC_C / 16; ++kk) {
          tc::mma_bf16(tm + tb + K_Y, tc::kmaj_desc(sbase + ab[term], TC_C, kk),
                       tc::kmaj_desc(sbase + vo, TC_C, kk), idy, 1u);
          tc::mma_bf16(tm + K_D2, tc::kmaj_desc(sbase + vo, TC_C, kk),
                       tc::kmaj_desc(sbase + kb2[term], TC_C, kk), id2, (term | kk) != 0);
        }
      tc::mma_commit(bar2);
    }
    if (tid == MMA_TID && !mbar_wait(bar2, par, status, DEV_TIMEOUT_MMA)) *ok_flag = -2;
    __syncthreads();
    if (*ok_flag != 1) {
      ok = false;
      break;
    }
    tc::fence_after_sync();
    // ---- S̄ <- S̄ Diag(e^{Λ_C}) + D2 (slot-head he's columns 64 he + c) and its
    //      bf16 terms for the next chunk, every thread for its row r (the
    //      outputs follow under the next chunk's first MMA group)
    {
      uint32_t x[32];
      tc::tmem_ld32(tlane + K_D2 + 64 * he + 32 * hw, x);
      tc::tmem_wait_ld(x);
      const float* ec = Ec + 64 * he + 32 * hw;
#pragma unroll
      for (int c = 0; c < 32; ++c) S[c] = ec[c] * S[c] + __uint_as_float(x[c]);
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        uint4 hv, lv;
        split8(S + 8 * c8, hv, lv);
        const uint32_t off = tc::kmaj_off(r, 32 * hw + 8 * c8, RW_D);
        *reinterpret_cast<uint4*>(sm + RwSmem::SHI + off) = hv;
        *reinterpret_cast<uint4*>(sm + RwSmem::SLO + off) = lv;
      }
    }
    tc::fence_before_sync();
    __syncthreads();
  }
  if (ok) {   // the last chunk's outputs
    const int last = (T - 1) / TC_C;
    emit(last & 1, TC_C * last, T - TC_C * last);
  }
  if (!ok && tid == MMA_TID) mbar_drain(*ok_flag == -1 ? bar1 : bar2, (uint32_t)chunk & 1u);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tm, RW_COLS);
  }
  if (!ok || !mine) return;
  float4* dst = reinterpret_cast<float4*>(state_of(she) + (size_t)vrow * RW_D + 32 * hw);
#pragma unroll
  for (int c4 = 0; c4 < 8; ++c4)
    dst[c4] = make_float4(S[4 * c4], S[4 * c4 + 1], S[4 * c4 + 2], S[4 * c4 + 3]);
  if (tid == 0 || (tid == 64 && two)) {   // each slot's table entry, from its head 0
    const int row = she / a.H;
    if (she - row * a.H == 0) {
      const int slot = a.items[row].slot;
      a.nlog[slot] = 0;
      a.base_of[slot] = slot;
    }
  }
}

}  // namespace

cudaError_t launch_prefill_gdn_tc(const SlotListArgs& a, const void* q, const void* k,
                                  const void* v, const float* g, const float* beta, void* o, int T,
                                  int out_bf16, float scale, int32_t* status, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(prefill_gdn_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)TcSmem::BYTES);
  if (e != cudaSuccess) return e;
  prefill_gdn_tc_kernel<<<a.rows * a.H, TC_THREADS, TcSmem::BYTES, s>>>(
      a, static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k),
      static_cast<const uint16_t*>(v), g, beta, o, T, out_bf16, scale, status);
  return cudaGetLastError();
}

cudaError_t launch_prefill_kda_tc(const SlotListArgs& a, const void* q, const void* k,
                                  const void* v, const float* g, const float* beta, void* o, int T,
                                  int out_bf16, float scale, int32_t* status, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(prefill_kda_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)KdaSmem::BYTES);
  if (e != cudaSuccess) return e;
  prefill_kda_tc_kernel<<<a.rows * a.H, TC_THREADS, KdaSmem::BYTES, s>>>(
      a, static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k),
      static_cast<const uint16_t*>(v), g, beta, o, T, out_bf16, scale, status);
  return cudaGetLastError();
}

cudaError_t launch_prefill_rwkv6_tc(const SlotListArgs& a, const void* r, const void* k,
                                    const void* v, const float* g, const float* bonus, void* o,
                                    int T, int out_bf16, float scale, int32_t* status,
                                    cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(prefill_rwkv6_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)RwSmem::BYTES);
  if (e != cudaSuccess) return e;
  const int nH = a.rows * a.H;
  prefill_rwkv6_tc_kernel<<<(nH + 1) / 2, TC_THREADS, RwSmem::BYTES, s>>>(
      a, static_cast<const uint16_t*>(r), static_cast<const uint16_t*>(k),
      static_cast<const uint16_t*>(v), g, bonus, o, T, out_bf16, scale, status);
  return cudaGetLastError();
}

}  // namespace dl
