// Device-side building blocks shared by the DeltaLog kernels (sm_103a).
//
// * mbarrier + cp.async.bulk (the 1-D TMA engine) wrappers in inline PTX;
// * bounded waits: every spin on an mbarrier gives up after a time limit,
//   records an error code in the context's device status word and lets the
//   kernel return, so that a bug cannot hang the GPU;
// * bf16 bit helpers and the launch-argument structs.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace dl {

enum Op : int { GDN = 0, KDA = 1, RWKV6 = 2 };

constexpr int BV = 32;            // value rows per tile (one warp owns one tile)
constexpr int MAX_NCW = 8;        // consumer warps per AppendDecode / EagerStep CTA (at most)
constexpr int MAX_NPW = 2;        // prep warps per fused AppendDecode CTA (at most)
constexpr int PIPE_THREADS_MAX = (MAX_NCW + 1 + MAX_NPW) * 32;   // consumers + producer + prep
constexpr int MAX_ROWS = 1024;    // slot rows per launch (more are split into chunks)
constexpr int HDR = 8;            // scalar header of a coefficient block (floats)
constexpr int BAR_BYTES = 1024;   // mbarrier area at the start of the pipelined kernels' shared memory

// Device status codes (written with atomicCAS into the context's status word).
constexpr int32_t DEV_TIMEOUT_TILE = 1;
constexpr int32_t DEV_TIMEOUT_AUX = 2;
constexpr int32_t DEV_TIMEOUT_EMPTY = 3;
constexpr int32_t DEV_BAD_ITEM = 4;
constexpr int32_t DEV_TEST_STALL = 5;   // the test-only stall below ran out (nothing else sets it)
constexpr int32_t DEV_TIMEOUT_MMA = 6;  // a wait for tensor-core MMAs to complete gave up
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;  // 2 s (default per-launch limit)

// One-line meaning of a device status code (host side).
inline const char* device_status_str(int32_t code) {
  switch (code) {
    case DEV_TIMEOUT_TILE: return "a wait for a state tile gave up";
    case DEV_TIMEOUT_AUX: return "a wait for a unit's inputs or coefficients gave up";
    case DEV_TIMEOUT_EMPTY: return "a wait for a stage or input slot to be released gave up";
    case DEV_BAD_ITEM: return "a plan row was out of range";
    case DEV_TEST_STALL: return "the test-only stall's bounded wait gave up";
    case DEV_TIMEOUT_MMA: return "a wait for tensor-core MMAs to complete gave up";
    default: return "unknown device status";
  }
}

struct StepItem {
  int32_t slot;   // slot stepped (log owner, and the storage a merge writes)
  int32_t base;   // storage slot whose dense base S̄ is read this step
  int32_t n;      // log length before the step (0 <= n < M)
};

// Per-step launch arguments (passed by value as a __grid_constant__ parameter).
struct StepArgs {
  const uint16_t* q;     // [rows, H, DK] bf16 (r for RWKV6)
  const uint16_t* k;     // [rows, H, DK] bf16
  const uint16_t* v;     // [rows, H, DV] bf16
  const float* g;        // [rows, H] or [rows, H, DK]
  const float* beta;     // [rows, H] (delta-rule ops)
  void* o;               // [rows, H, DV] bf16 or fp32
  float* Sbar;           // [slots, H, DV, DK]
  void* alog;            // [slots, H, Mcap, DV] fp32 (bf16 for RWKV6)
  uint16_t* klog;        // [slots, H, Mcap, DK] bf16
  float* Llog;           // [slots, H, Mcap] or [slots, H, Mcap, DK]
  float* coef;           // [rows, H, CB] scratch written by ReplayPrep
  const float* bonus;    // [H, DK] (RWKV6)
  int32_t* nlog;         // [slots] device slot table
  int32_t* base_of;      // [slots]
  int32_t* status;       // device status word
  int32_t rows, H, M, Mcap, Mcap4, CB, P0;   // P0: coefficient floats needed on append steps
  int32_t G, NG;         // value tiles per work unit, units per slot-head
  int32_t ns, na;        // pipeline stages (tiles), aux slots
  int32_t ncw;           // consumer warps per CTA (block = ncw + 1 (+ npw) warps)
  int32_t npw;           // prep warps of the fused form (divides na)
  int32_t tps;           // value tiles per stage (one bulk copy): 1, or 2 for d_k = 64
  int32_t l2_stream;     // 1: read S̄ with an L2 evict-first policy (state larger than L2 can keep)
  int32_t pdl_prefetch;  // 1: the previous launch on the stream was a step of this context, so
                         //    tiles of rows with n > 0 may stream before griddepcontrol.wait
  int32_t aux_bytes;     // bytes of one aux slot
  int32_t arows;         // log rows an aux slot holds in this launch (0: M); every row's
                         // log length n is at most arows, and below it where the step
                         // uses the current token's row n (RWKV6, merge steps)
  int32_t out_bf16;
  float scale;
  // How long a bounded wait spins before it records an error and gives up
  // (WAIT_LIMIT_NS unless a test asks for less).
  unsigned long long wait_ns;
  // Test only (0 in normal use): the first consumer warp of CTA 0 also waits
  // (for wait_ns / 2) on a barrier that nothing arrives on, so that its
  // bounded wait runs out, records DEV_TEST_STALL and the kernel takes its
  // error exit.
  int32_t test_stall;
  // Device-resident plan (ragged decode windows): when set, the launch reads
  // its rows from plan_dev and processes min(*rows_dev, rows) of them; `rows`
  // is then the capacity the grid was sized for.  Otherwise the rows are
  // items[0 .. rows).
  const StepItem* plan_dev;
  const int32_t* rows_dev;
  StepItem items[MAX_ROWS];
};

// The plan row `row` of a launch, from the parameters or the device plan.
__device__ __forceinline__ StepItem step_item(const StepArgs& a, int row) {
  return a.plan_dev ? a.plan_dev[row] : a.items[row];
}
// Rows this launch processes (a device-resident count is clamped to the capacity).
__device__ __forceinline__ int step_rows(const StepArgs& a) {
  if (!a.rows_dev) return a.rows;
  const int r = *a.rows_dev;
  return r < 0 ? 0 : (r < a.rows ? r : a.rows);
}

// Arguments of the standalone merge / read-state kernel and of the set-state
// and fork copy kernels.
struct SlotListArgs {
  float* Sbar;
  void* alog;
  uint16_t* klog;
  float* Llog;
  int32_t* nlog;
  int32_t* base_of;
  const float* S_in;     // set-state source [rows, H, DV, DK]
  float* S_out;          // read-state destination [rows, H, DV, DK] (nullptr: write S̄)
  int32_t rows, H, Mcap;
  int32_t src_slot, src_n, src_base;   // fork
  StepItem items[MAX_ROWS];
};

// ---------------------------------------------------------------- bf16 ------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float(uint32_t(h) << 16); }
__device__ __forceinline__ uint16_t f2bf16(float x) {
  __nv_bfloat16 b = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&b);
}

// ---------------------------------------------------------------- PTX -------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Wait until the phase with the given parity has completed.  Gives up after
// limit_ns, or early once another warp has recorded an error, and then
// returns false (after recording `code` if nobody did before).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t* status,
                                          int32_t code,
                                          unsigned long long limit_ns = WAIT_LIMIT_NS) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*reinterpret_cast<volatile int32_t*>(status) != 0) return false;
      if (globaltimer() - t0 > limit_ns) {
        atomicCAS(status, 0, code);
        return false;
      }
    }
  }
}

// Same, but only time-bounded (used to drain copies already in flight).
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > WAIT_LIMIT_NS) return;
  }
}

// 1-D bulk copy global -> shared (TMA engine), completion counted in bytes on
// `bar`, with an L2 eviction-priority policy: evict_first for a state that is
// streamed through once per step, evict_normal for one small enough to stay in
// L2.  dst, src 16-byte aligned; bytes a non-zero multiple of 16.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
      "[%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// 16-byte asynchronous copy global -> shared through the load/store unit (not
// the TMA engine), and an mbarrier arrival that fires when all of this thread's
// earlier such copies have landed (counted as one of the barrier's expected
// arrivals).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Programmatic dependent launch controls.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Streaming global stores / loads.
__device__ __forceinline__ void st_cs_f4(float* p, float4 v) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_cs_f2(float* p, float2 v) {
  asm volatile("st.global.cs.v2.f32 [%0], {%1, %2};" ::"l"(p), "f"(v.x), "f"(v.y) : "memory");
}

// ---------------------------------------------------------- reductions -------
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Transposed reduction: v[r] holds this lane's partial sum for row r (32
// rows).  Returns, on lane l, the full sum over the 32 lanes for row l.  Five
// halving exchanges: 16 + 8 + 4 + 2 + 1 = 31 shuffles for 32 rows.
template <int N>
__device__ __forceinline__ void rs_stage(float (&v)[32], int lane) {
  constexpr int HALF = N / 2;
  const bool up = (lane & HALF) != 0;
#pragma unroll
  for (int j = 0; j < HALF; ++j) {
    const float send = up ? v[j] : v[j + HALF];
    const float keep = up ? v[j + HALF] : v[j];
    v[j] = keep + __shfl_xor_sync(0xffffffffu, send, HALF);
  }
}
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane) {
  rs_stage<32>(v, lane);
  rs_stage<16>(v, lane);
  rs_stage<8>(v, lane);
  rs_stage<4>(v, lane);
  rs_stage<2>(v, lane);
  return v[0];
}

// Transposed reduction of NE = 2^E per-entry partial sums (NE <= 32): E halving
// exchanges over lane bits 4, 3, ... leave one entry per lane group, then the
// remaining 5-E lane bits are summed.  Returns, on every lane, the full sum of
// entry (lane >> (5 - E)).
template <int NE>
__device__ __forceinline__ float reduce_entries(float (&v)[NE], int lane) {
  constexpr int E = NE == 32 ? 5 : NE == 16 ? 4 : NE == 8 ? 3 : NE == 4 ? 2 : 1;
  static_assert((1 << E) == NE, "NE must be a power of two <= 32");
#pragma unroll
  for (int s = 0; s < E; ++s) {
    const int off = 16 >> s;
    const int half = NE >> (s + 1);
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int j = 0; j < half; ++j) {
      const float send = up ? v[j] : v[j + half];
      const float keep = up ? v[j + half] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  float r = v[0];
#pragma unroll
  for (int off = 16 >> E; off > 0; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
  return r;
}

// Load VEC consecutive floats (VEC = 2 or 4) from shared or global memory.
template <int VEC>
__device__ __forceinline__ void ldvec(float (&d)[VEC], const float* p) {
  if constexpr (VEC == 4) {
    const float4 t = *reinterpret_cast<const float4*>(p);
    d[0] = t.x; d[1] = t.y; d[2] = t.z; d[3] = t.w;
  } else {
    const float2 t = *reinterpret_cast<const float2*>(p);
    d[0] = t.x; d[1] = t.y;
  }
}
// VEC consecutive bf16 -> float.
template <int VEC>
__device__ __forceinline__ void ldvec_bf16(float (&d)[VEC], const uint16_t* p) {
  if constexpr (VEC == 4) {
    const uint2 t = *reinterpret_cast<const uint2*>(p);
    d[0] = bf16lo(t.x); d[1] = bf16hi(t.x); d[2] = bf16lo(t.y); d[3] = bf16hi(t.y);
  } else {
    const uint32_t t = *reinterpret_cast<const uint32_t*>(p);
    d[0] = bf16lo(t); d[1] = bf16hi(t);
  }
}
template <int VEC>
__device__ __forceinline__ void stvec_cs(float* p, const float (&d)[VEC]) {
  if constexpr (VEC == 4) st_cs_f4(p, make_float4(d[0], d[1], d[2], d[3]));
  else st_cs_f2(p, make_float2(d[0], d[1]));
}

}  // namespace dl
