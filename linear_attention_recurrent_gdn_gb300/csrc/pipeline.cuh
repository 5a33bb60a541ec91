// Pipelined value-tile kernels: AppendDecode (DeltaLog step with the merge
// fused) and EagerStep (dense read-modify-write step).
//
// DeltaLog page, section "Kernel implementation": the state is split along the
// value dimension d_v and each work item handles one slice of the dense base
// together with the matching shard of the value-side log, while the key-side
// factors and log-decay metadata (here: the ReplayPrep coefficient block) are
// shared by all value tiles of a slot-head.
//
// Structure on sm_103a (persistent over work units; two to four CTAs per SM):
//   * work unit = (slot-head, group of G value tiles); tile = 32 value rows of
//     the dense base (32 x d_k fp32, contiguous in HBM: 16 KiB at d_k = 128);
//   * warps 0 .. ncw-1 are consumers, warp ncw the producer, and any further
//     warps (fused form) prep warps;
//   * producer: one lane issues one 1-D bulk copy (TMA engine) per stage (one
//     tile, or two at d_k = 64) into the stage ring, completion counted in
//     bytes on an mbarrier, with an L2 evict-first policy when the state does
//     not fit in L2.  The unit's small inputs (k/q/v, log rows, log-decays,
//     g, beta, bonus; the coefficient block in the two-kernel form) are copied
//     by all 32 lanes with 16-byte cp.async into a ring of `na` aux slots: a
//     bulk copy has a fixed issue cost per copy on this GPU, so it is kept for
//     the tiles.  The producer is on the critical path of every refill, so its
//     per-tile bookkeeping is incremental (no divisions);
//   * consumers: warp w owns stages w*R .. w*R+R-1 and processes tiles w,
//     w+ncw, ...  Lane l holds d_k/32 consecutive key channels; a pass over
//     the 32 rows accumulates per-row partial dot products, a transposed
//     butterfly (31 shuffles for 32 rows) leaves row l's sums on lane l, which
//     then finishes that row: log replay, output, the appended factor; on a
//     merge step the warp then re-reads the tile from shared memory and writes
//     the updated rows;
//   * every wait is bounded (see mbar_wait).  On an append step a consumer
//     releases its stage right after the tile pass, so the refill overlaps its
//     epilogue.
// Forms of the ReplayPrep stage:
//   * FUSED (default): the coefficients are computed inside this kernel from
//     the unit's inputs in its aux slot (prep_unit) -- by `npw` prep warps that
//     signal the consumers on a per-slot barrier (cready) when a unit spans
//     several stages, or by the unit's own consumer warp when it is a single
//     stage.  No second launch and no coefficient round trip through HBM.
//     Inside a captured decode window each step is a programmatic dependent of
//     the previous one (see the producer);
//   * APPEND: ReplayPrep is its own kernel (replay_prep.cu) and AppendDecode
//     launches as its programmatic dependent: the producer streams the first
//     ns tiles before it waits for the coefficient blocks.
#pragma once
#include "dl_device.cuh"
#include "layout.h"

namespace dl {

enum Mode : int { APPEND = 0, EAGER = 1, FUSED = 2 };

constexpr int MAX_NS = 24, MAX_NA = 24;   // (barrier area: 8 bytes each)

static_assert(BAR_BYTES == 8 * BAR_SLOTS, "barrier area and planner agree");

struct Bars {
  uint32_t b0;
  int ns, na;
  __device__ uint32_t full(int s) const { return b0 + 8u * s; }
  __device__ uint32_t empty(int s) const { return b0 + 8u * (ns + s); }
  __device__ uint32_t afull(int x) const { return b0 + 8u * (2 * ns + x); }
  __device__ uint32_t aempty(int x) const { return b0 + 8u * (2 * ns + na + x); }
  __device__ uint32_t cready(int x) const { return b0 + 8u * (2 * ns + 2 * na + x); }
  // fused form with prep warps: the unit's key-side vectors are written (the
  // consumers' pass over the tile may start; cready follows with the rest)
  __device__ uint32_t vready(int x) const { return b0 + 8u * (2 * ns + 3 * na + x); }
  // The last barrier of the area (the planner keeps the others below it):
  // initialised and never arrived on (the test-only stall waits on it).
  __device__ uint32_t never() const { return b0 + (uint32_t)BAR_BYTES - 8u; }
};

// Stage ownership: tile i (CTA-local order) belongs to consumer warp i % ncw,
// and each warp owns R = ns / ncw consecutive stages that it cycles through.
// A warp therefore waits on a stage only after it released that stage's
// previous phase itself, so no barrier is ever awaited more than one phase
// ahead (mbarrier parity waits cannot tell phases two apart).
__device__ __forceinline__ int stage_of(int i, int R, int ncw) {
  return (i % ncw) * R + (i / ncw) % R;
}
__device__ __forceinline__ uint32_t stage_parity(int i, int R, int ncw) {
  return (uint32_t)((i / ncw) / R) & 1u;
}

struct UnitPos {
  int sh, row, h, grp;
};

__device__ __forceinline__ UnitPos unit_pos(const StepArgs& a, int u) {
  UnitPos p;
  p.sh = u / a.NG;
  p.grp = u - p.sh * a.NG;
  p.row = p.sh / a.H;
  p.h = p.sh - p.row * a.H;
  return p;
}

// Walks a CTA's units u, u + grid, u + 2*grid, ... without dividing: the
// position advances by the precomputed quotients and remainders of the grid
// stride (by NG, then by H).
struct UnitWalk {
  UnitPos p;
  int NG, H, sq, sr, hq0, hr0, hq1, hr1;
  __device__ __forceinline__ void init(const StepArgs& a, int u0) {
    NG = a.NG;
    H = a.H;
    p = unit_pos(a, u0);
    const int grid = (int)gridDim.x;
    sq = grid / NG;
    sr = grid - sq * NG;
    hq0 = sq / H;
    hr0 = sq - hq0 * H;
    hq1 = (sq + 1) / H;
    hr1 = (sq + 1) - hq1 * H;
  }
  __device__ __forceinline__ void next() {
    int dq, dr;
    p.grp += sr;
    if (p.grp >= NG) {
      p.grp -= NG;
      p.sh += sq + 1;
      dq = hq1;
      dr = hr1;
    } else {
      p.sh += sq;
      dq = hq0;
      dr = hr0;
    }
    p.h += dr;
    p.row += dq;
    if (p.h >= H) {
      p.h -= H;
      p.row += 1;
    }
  }
};

__device__ __forceinline__ void store_out(const StepArgs& a, size_t idx, float val) {
  if (a.out_bf16) static_cast<uint16_t*>(a.o)[idx] = f2bf16(val);
  else static_cast<float*>(a.o)[idx] = val;
}

// ---------------------------------------------------------------- producer --
// A unit's small inputs (coefficient block, k/q/v, value-side log rows, key
// log rows on a GDN merge) are copied by all 32 lanes of the producer warp with
// 16-byte cp.async (load/store unit path: the TMA engine's per-copy cost is
// kept for the 16 KiB tiles).  Each lane then arrives once on the unit's aux
// barrier (expected count 32) when its own copies have landed.
__device__ __forceinline__ void copy_seg(uint32_t dst, const void* src, uint32_t bytes, int lane) {
  const unsigned char* s = static_cast<const unsigned char*>(src);
  for (uint32_t off = (uint32_t)lane * 16u; off < bytes; off += 32u * 16u) cp_async16(dst + off, s + off);
}

// Fused form: `part` 1 copies the unit's inputs (the step's own tensors, the
// bonus), 2 its log rows (which the previous step may still be writing), 3
// both.  The other forms copy everything.
template <int OP, int DK, int DV, int MODE>
__device__ __forceinline__ void issue_aux(const StepArgs& a, const Layout& Lay, const UnitPos& p,
                                          unsigned char* ax, int lane, int part = 3) {
  constexpr bool DELTA = OP != RWKV6;
  const StepItem it = step_item(a, p.row);
  const size_t sh = p.sh;
  const uint32_t base = smem_u32(ax);
  if constexpr (MODE == APPEND) {
    constexpr int ESA = DELTA ? 4 : 2;
    const int n = it.n;
    const bool merge = (n + 1 == a.M);
    const size_t lh = (size_t)it.slot * a.H + p.h;
    if (OP == GDN) {
      copy_seg(base + Lay.aux_kq, a.k + sh * DK, DK * 2, lane);
      copy_seg(base + Lay.aux_kq + DK * 2, a.q + sh * DK, DK * 2, lane);
    }
    if (DELTA) copy_seg(base + Lay.aux_v, a.v + sh * DV, DV * 2, lane);
    if (n > 0)
      copy_seg(base + Lay.aux_U, static_cast<const unsigned char*>(a.alog) + lh * Lay.Mcap * DV * ESA,
               (uint32_t)n * DV * ESA, lane);
    if (OP == RWKV6) copy_seg(base + Lay.aux_U + n * DV * 2, a.v + sh * DV, DV * 2, lane);
    if (OP == GDN && merge) {
      if (n > 0) copy_seg(base + Lay.aux_kl, a.klog + lh * Lay.Mcap * DK, (uint32_t)n * DK * 2, lane);
      copy_seg(base + Lay.aux_kl + n * DK * 2, a.k + sh * DK, DK * 2, lane);
    }
  } else if constexpr (MODE == FUSED) {
    // everything the fused ReplayPrep stage and the consumers read
    constexpr int ESA = DELTA ? 4 : 2;
    const int n = it.n;
    const bool merge = (n + 1 == a.M);
    const size_t lh = (size_t)it.slot * a.H + p.h;
    if (part & 1) {   // the step's inputs
      copy_seg(base + Lay.f_kq, a.k + sh * DK, DK * 2, lane);
      copy_seg(base + Lay.f_kq + DK * 2, a.q + sh * DK, DK * 2, lane);
      if (DELTA) copy_seg(base + Lay.f_v, a.v + sh * DV, DV * 2, lane);
      if (OP == RWKV6) copy_seg(base + Lay.f_U + n * DV * 2, a.v + sh * DV, DV * 2, lane);
      if (OP == GDN && merge) copy_seg(base + Lay.f_kl + n * DK * 2, a.k + sh * DK, DK * 2, lane);
      if constexpr (OP == GDN) {
        if (lane == 0) cp_async4(base + Lay.f_g, a.g + sh);
      } else {
        copy_seg(base + Lay.f_g, a.g + sh * DK, DK * 4, lane);
      }
      if (DELTA && lane == 0) cp_async4(base + Lay.f_beta, a.beta + sh);
      if (OP == RWKV6) copy_seg(base + Lay.f_bonus, a.bonus + (size_t)p.h * DK, DK * 4, lane);
    }
    if ((part & 2) && n > 0) {   // the slot's log rows
      copy_seg(base + Lay.f_U, static_cast<const unsigned char*>(a.alog) + lh * Lay.Mcap * DV * ESA,
               (uint32_t)n * DV * ESA, lane);
      copy_seg(base + Lay.f_kl, a.klog + lh * Lay.Mcap * DK, (uint32_t)n * DK * 2, lane);
      if constexpr (OP == GDN) {
        // scalar log-decays (rows are not 16-byte aligned): 4-byte copies
        if (lane < n) cp_async4(base + Lay.f_L + lane * 4, a.Llog + lh * Lay.Mcap + lane);
      } else {
        copy_seg(base + Lay.f_L, a.Llog + lh * Lay.Mcap * DK, (uint32_t)n * DK * 4, lane);
      }
    }
  } else {
    copy_seg(base + Lay.e_kq, a.k + sh * DK, DK * 2, lane);
    copy_seg(base + Lay.e_kq + DK * 2, a.q + sh * DK, DK * 2, lane);
    copy_seg(base + Lay.e_v, a.v + sh * DV, DV * 2, lane);
    if (OP != GDN) copy_seg(base + Lay.e_g, a.g + sh * DK, DK * 4, lane);
  }
}

// The coefficient block (written by ReplayPrep), then this lane's arrival.
template <int OP, int DK, int DV>
__device__ __forceinline__ void issue_coef_and_arrive(const StepArgs& a, const Layout& Lay,
                                                      const UnitPos& p, unsigned char* ax,
                                                      uint32_t bar, int lane) {
  const StepItem it = step_item(a, p.row);
  const bool merge = (it.n + 1 == a.M);
  copy_seg(smem_u32(ax + Lay.aux_coef), a.coef + (size_t)p.sh * a.CB,
           (merge ? Lay.CB : Lay.P0) * 4u, lane);
  cp_async_arrive_noinc(bar);
}

// ------------------------------------------------- ReplayPrep stage (fused) --
// The per slot-head coefficients of the DeltaLog page's ReplayPrep stage
// ("Kernel implementation — Staged execution"), computed by one warp of the
// AppendDecode CTA from the unit's inputs already in shared memory, and
// written into the unit's aux slot for its value-tile consumers.  The same
// formulas as the ReplayPrep kernel (replay_prep.cu, which states them); this
// stage sums each entry's lane partials in groups of four entries, that kernel
// in one butterfly over all entries, so the two agree to rounding.  Every
// fused launch runs this stage, whatever its batch, so a slot-head's bits do
// not depend on the batch.  On an append step the owner unit (value-tile
// group 0) of the slot-head also appends k_t, Λ_t (and v_t for RWKV6) to the
// slot's log in HBM, and the (head 0, group 0) unit advances the device slot
// table.
// `vbar` (prep warps only, else 0): arrived on once the consumers' pass over
// the tile has what it reads (GDN: at once, it reads k_t, q_t from the aux
// slot; KDA and RWKV6: once k̂, q̂ or r̂ are written).
template <int OP, int DK, int DV, int NE>
__device__ __forceinline__ void prep_unit(const StepArgs& a, const Layout& Lay, const UnitPos& p,
                                          unsigned char* ax, int lane, uint32_t vbar = 0) {
  constexpr int VEC = DK / 32;
  const StepItem it = step_item(a, p.row);
  const int n = it.n, slot = it.slot;
  const bool merge = (n + 1 == a.M);
  const bool owner = (p.grp == 0);
  const int Mcap = Lay.Mcap, Mcap4 = Lay.Mcap4;
  const int vecA = HDR + 2 * Mcap4, vecB = vecA + DK;
  const size_t lh = (size_t)slot * a.H + p.h;
  float* cf = reinterpret_cast<float*>(ax + Lay.f_coef);
  const uint16_t* kq16 = reinterpret_cast<const uint16_t*>(ax + Lay.f_kq);
  const uint16_t* kl = reinterpret_cast<const uint16_t*>(ax + Lay.f_kl);
  float* Ls = reinterpret_cast<float*>(ax + Lay.f_L);
  const float* gs = reinterpret_cast<const float*>(ax + Lay.f_g);
  const int c0 = lane * VEC;
  float kv[VEC], qv[VEC];
  ldvec_bf16<VEC>(kv, kq16 + c0);
  ldvec_bf16<VEC>(qv, kq16 + DK + c0);
  if constexpr (OP == GDN) {
    if (vbar && lane == 0) mbar_arrive(vbar);
    const float beta_t = reinterpret_cast<const float*>(ax + Lay.f_beta)[0];
    const float Lt = (n > 0 ? Ls[n - 1] : 0.f) + gs[0];
    float kq = 0.f;
#pragma unroll
    for (int c = 0; c < VEC; ++c) kq += kv[c] * qv[c];
    kq = warp_sum(kq);
    // entries in groups of four in a rolled loop (as KDA's below)
#pragma unroll 1
    for (int j0 = 0; j0 < n; j0 += 4) {
      float q1[4], q2[4];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int j = j0 + jj;
        float x = 0.f, y = 0.f;
        if (j < n) {
          float kj[VEC];
          ldvec_bf16<VEC>(kj, kl + j * DK + c0);
#pragma unroll
          for (int c = 0; c < VEC; ++c) {
            x += kj[c] * kv[c];
            y += kj[c] * qv[c];
          }
        }
        q1[jj] = x;
        q2[jj] = y;
      }
      const float dkk = reduce_entries<4>(q1, lane);   // entry j0 + lane / 8
      const float dkq = reduce_entries<4>(q2, lane);
      const int e = j0 + (lane >> 3);
      if ((lane & 7) == 0 && e < n) {
        const float wj = expf(Lt - Ls[e]);
        cf[HDR + e] = wj * dkk;
        cf[HDR + Mcap4 + e] = wj * dkq;
        if (merge) cf[Lay.P0 + e] = wj;
      }
    }
    if (lane == 0) {
      cf[0] = expf(Lt);
      cf[1] = kq;
      cf[2] = beta_t;
      if (merge) cf[Lay.P0 + n] = 1.f;
      if (!merge && owner) a.Llog[lh * Mcap + n] = Lt;
    }
  } else {
    float Lp[VEC], gt[VEC], Lt[VEC], Lc[VEC], wt[VEC];
    if (n > 0) {
      ldvec<VEC>(Lp, Ls + (size_t)(n - 1) * DK + c0);
    } else {
#pragma unroll
      for (int c = 0; c < VEC; ++c) Lp[c] = 0.f;
    }
    ldvec<VEC>(gt, gs + c0);
#pragma unroll
    for (int c = 0; c < VEC; ++c) {
      Lt[c] = Lp[c] + gt[c];
      Lc[c] = (OP == KDA) ? Lt[c] : Lp[c];
      wt[c] = (OP == RWKV6) ? expf(gt[c]) : 1.f;
    }
    __syncwarp();   // every lane has read row n-1 before K̃ rows overwrite the log-decay rows
    if constexpr (OP == KDA) {
      float kq = 0.f;
#pragma unroll
      for (int c = 0; c < VEC; ++c) {
        // the fast exponential for this step's k̂, q̂ (the prep warp is on the
        // consumers' path: measured on GB300, 77.6 -> 78.3 M tokens·heads/s);
        // the merge's decay, which scales the base from here on, stays exact
        const float e = __expf(Lt[c]);
        cf[vecA + c0 + c] = e * kv[c];
        cf[vecB + c0 + c] = e * qv[c];
        if (merge) cf[Lay.P0 + c0 + c] = expf(Lt[c]);
        kq += kv[c] * qv[c];
      }
      kq = warp_sum(kq);
      if (lane == 0) {
        cf[1] = kq;
        cf[2] = reinterpret_cast<const float*>(ax + Lay.f_beta)[0];
      }
    } else {
      float bon[VEC];
      ldvec<VEC>(bon, reinterpret_cast<const float*>(ax + Lay.f_bonus) + c0);
      float cb = 0.f;
#pragma unroll
      for (int c = 0; c < VEC; ++c) {
        cf[vecA + c0 + c] = expf(Lp[c]) * qv[c];
        cb += qv[c] * bon[c] * kv[c];
        if (merge) cf[Lay.P0 + c0 + c] = expf(Lt[c]);
      }
      cb = warp_sum(cb);
      if (lane == 0) cf[3] = cb;
    }
    if (vbar) {   // k̂, q̂ (KDA) or r̂ (RWKV6) are in place
      __syncwarp();
      if (lane == 0) mbar_arrive(vbar);
    }
    if constexpr (OP == KDA) {
      // Entries in groups of four, one transposed reduction per group and
      // product, in a rolled loop: the prep's code stays small enough for the
      // instruction cache next to the consumers', and short logs stop early.
      // Measured on GB300: the fully unrolled loop left KDA launches at a 77 %
      // instruction-cache hit rate (91 % now); M = 16 windows 849 -> 787 us,
      // M = 32 2731 -> 2086 us.
#pragma unroll 1
      for (int j0 = 0; j0 < n; j0 += 4) {
        float q1[4], q2[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = j0 + jj;
          float x = 0.f, y = 0.f;
          if (j < n) {
            float kj[VEC], lj[VEC], kk[VEC];
            ldvec_bf16<VEC>(kj, kl + j * DK + c0);
            ldvec<VEC>(lj, Ls + (size_t)j * DK + c0);
#pragma unroll
            for (int c = 0; c < VEC; ++c) {
              kk[c] = kj[c] * __expf(Lc[c] - lj[c]);
              x += kk[c] * kv[c];
              y += kk[c] * qv[c];
            }
            if (merge) {   // K̃_j = k_j ⊙ e^{Λ_t-Λ_j} over this lane's columns of row j
#pragma unroll
              for (int c = 0; c < VEC; ++c) Ls[(size_t)j * DK + c0 + c] = kk[c];
            }
          }
          q1[jj] = x;
          q2[jj] = y;
        }
        const float d1 = reduce_entries<4>(q1, lane);   // entry j0 + lane / 8
        const float d2 = reduce_entries<4>(q2, lane);
        const int e = j0 + (lane >> 3);
        if ((lane & 7) == 0 && e < n) {
          cf[HDR + e] = d1;
          cf[HDR + Mcap4 + e] = d2;
        }
      }
      if (merge) {
#pragma unroll
        for (int c = 0; c < VEC; ++c) Ls[(size_t)n * DK + c0 + c] = kv[c];   // K̃_n = k_t
      }
    } else {   // RWKV6: the same grouping
#pragma unroll 1
      for (int j0 = 0; j0 < n; j0 += 4) {
        float q1[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = j0 + jj;
          float x = 0.f;
          if (j < n) {
            float kj[VEC], lj[VEC], kk[VEC];
            ldvec_bf16<VEC>(kj, kl + j * DK + c0);
            ldvec<VEC>(lj, Ls + (size_t)j * DK + c0);
#pragma unroll
            for (int c = 0; c < VEC; ++c) {
              kk[c] = kj[c] * __expf(Lc[c] - lj[c]);
              x += kk[c] * qv[c];
            }
            if (merge) {   // K̃_j = k_j ⊙ e^{Λ_t-Λ_j} over this lane's columns of row j
#pragma unroll
              for (int c = 0; c < VEC; ++c) Ls[(size_t)j * DK + c0 + c] = kk[c] * wt[c];
            }
          }
          q1[jj] = x;
        }
        const float d1 = reduce_entries<4>(q1, lane);   // entry j0 + lane / 8
        const int e = j0 + (lane >> 3);
        if ((lane & 7) == 0 && e < n) cf[HDR + e] = d1;
      }
      if (merge) {
#pragma unroll
        for (int c = 0; c < VEC; ++c) Ls[(size_t)n * DK + c0 + c] = kv[c];   // K̃_n = k_t
      }
    }
    if (!merge && owner) {
      float* Ld = a.Llog + (lh * Mcap + n) * DK + c0;
#pragma unroll
      for (int c = 0; c < VEC; ++c) Ld[c] = Lt[c];
    }
  }
  if (!merge && owner) {
    uint16_t* kd = a.klog + (lh * Mcap + n) * DK + c0;
#pragma unroll
    for (int c = 0; c < VEC; ++c) kd[c] = kq16[c0 + c];
    if constexpr (OP == RWKV6) {
      uint16_t* vd = static_cast<uint16_t*>(a.alog) + (lh * Mcap + n) * DV;
      const uint16_t* vs = reinterpret_cast<const uint16_t*>(ax + Lay.f_U) + n * DV;
      for (int i = lane; i < DV; i += 32) vd[i] = vs[i];
    }
  }
  if (owner && p.h == 0 && lane == 0) {
    a.nlog[slot] = merge ? 0 : n + 1;
    a.base_of[slot] = merge ? slot : it.base;
  }
}

// ---------------------------------------------------------- AppendDecode ----
// Where a unit's inputs sit in its aux slot (they differ between the two-kernel
// and the fused form).
struct AuxView {
  const float* cf;        // coefficient block
  const uint16_t* kq;     // k_t, q_t (bf16)
  const uint16_t* v;      // v_t (bf16, delta-rule ops)
  unsigned char* U;       // value-side log rows (+ row n)
  const uint16_t* kl;     // key log rows, row n = k_t (GDN merge)
  const float* Kt;        // K̃ rows (per-key merge)
};

template <int OP, int DK, int MODE>
__device__ __forceinline__ AuxView aux_view(const Layout& Lay, unsigned char* ax) {
  AuxView v;
  if constexpr (MODE == FUSED) {
    v.cf = reinterpret_cast<const float*>(ax + Lay.f_coef);
    v.kq = reinterpret_cast<const uint16_t*>(ax + Lay.f_kq);
    v.v = reinterpret_cast<const uint16_t*>(ax + Lay.f_v);
    v.U = ax + Lay.f_U;
    v.kl = reinterpret_cast<const uint16_t*>(ax + Lay.f_kl);
    v.Kt = reinterpret_cast<const float*>(ax + Lay.f_L);
  } else {
    v.cf = reinterpret_cast<const float*>(ax + Lay.aux_coef);
    v.kq = reinterpret_cast<const uint16_t*>(ax + Lay.aux_kq);
    v.v = reinterpret_cast<const uint16_t*>(ax + Lay.aux_v);
    v.U = ax + Lay.aux_U;
    v.kl = reinterpret_cast<const uint16_t*>(ax + Lay.aux_kl);
    v.Kt = v.cf + Lay.P0 + DK;
  }
  return v;
}

// RWKV6's row sum S̄[row]·r̂ for row `lane` of a 32-row tile T (d_k floats a
// row), computed by that lane alone: it reads the row and r̂ in 16-byte
// chunks, starting at chunk lane mod (d_k / 4), so that the eight lanes of a
// quarter-warp read eight different chunks, which sit in distinct banks
// although the rows are a multiple of 128 bytes apart.  Four partial sums.
// The one-tile pass and the two-tile pass both use it, so a row's sum has
// the same bits whatever the unit size (batch invariance).
template <int DK>
__device__ __forceinline__ void rwkv6_row_chunk(float (&s)[4], const float* Trow, const float* R,
                                                int kc, int lane) {
  const int ch = ((kc + lane) & (DK / 4 - 1)) * 4;
  const float4 r = *reinterpret_cast<const float4*>(R + ch);
  const float4 x = *reinterpret_cast<const float4*>(Trow + ch);
  s[0] += x.x * r.x; s[1] += x.y * r.y; s[2] += x.z * r.z; s[3] += x.w * r.w;
}
__device__ __forceinline__ float sum4(const float (&s)[4]) { return (s[0] + s[1]) + (s[2] + s[3]); }

// Returns true if it already released the tile stage (append steps release it
// right after the pass over the tile, so the refill overlaps the epilogue;
// GDN and RWKV6 merge steps once the update has read the tile's last rows).
// With `coef_bar` set (fused form with prep warps) the pass over the tile
// runs as soon as its vectors are in place, and the coefficients are awaited
// on coef_bar (phase parity coef_par) before the epilogue; if that wait gives
// up, *failed is set and nothing more is written.
template <int OP, int DK, int DV>
__device__ __forceinline__ bool consume_append(const StepArgs& a, const Layout& Lay,
                                               const UnitPos& p, int vt, const float* T,
                                               const AuxView& av, int lane, uint32_t empty_bar,
                                               bool may_release, uint32_t coef_bar = 0,
                                               uint32_t coef_par = 0, bool* failed = nullptr) {
  constexpr int VEC = DK / 32;
  constexpr bool DELTA = OP != RWKV6;
  const StepItem it = step_item(a, p.row);
  const int n = it.n;
  const bool merge = (n + 1 == a.M);
  const float* cf = av.cf;
  const int vecA = HDR + 2 * Lay.Mcap4;

  float A = 0.f, B = 0.f;
  if constexpr (DELTA) {
    // pass 1: per-row partial dot products over this lane's key channels (k̂
    // and q̂ stay in registers), then a transposed reduction leaves row l's
    // sums on lane l
    float kv[VEC], qv[VEC];
    if constexpr (OP == GDN) {
      ldvec_bf16<VEC>(kv, av.kq + lane * VEC);
      ldvec_bf16<VEC>(qv, av.kq + DK + lane * VEC);
    } else {
      ldvec<VEC>(kv, cf + vecA + lane * VEC);
      ldvec<VEC>(qv, cf + vecA + DK + lane * VEC);
    }
    float pa[32], pb[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      float t[VEC];
      ldvec<VEC>(t, T + r * DK + lane * VEC);
      float x = 0.f, y = 0.f;
#pragma unroll
      for (int c = 0; c < VEC; ++c) {
        x += t[c] * kv[c];
        y += t[c] * qv[c];
      }
      pa[r] = x;
      pb[r] = y;
    }
    if (!merge && may_release) {
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);
    }
    A = reduce_scatter32(pa, lane);
    B = reduce_scatter32(pb, lane);
  } else {
    // pass 1, RWKV6: lane l computes row l alone (rwkv6_row_chunk)
    float s0[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kc = 0; kc < DK / 4; ++kc) rwkv6_row_chunk<DK>(s0, T + lane * DK, cf + vecA, kc, lane);
    if (!merge && may_release) {
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);
    }
    A = sum4(s0);
  }

  if (coef_bar &&
      !__all_sync(0xffffffffu, mbar_wait(coef_bar, coef_par, a.status, DEV_TIMEOUT_AUX, a.wait_ns))) {
    *failed = true;
    return !merge && may_release;
  }

  // row epilogue on lane = row
  const int col = vt * BV + lane;
  const size_t oidx = (size_t)p.sh * DV + col;
  if constexpr (DELTA) {
    const float* U = reinterpret_cast<const float*>(av.U);
    float x = (OP == GDN) ? cf[0] * A : A;
    float ob = (OP == GDN) ? cf[0] * B : B;
#pragma unroll 4
    for (int j = 0; j < n; ++j) {
      const float uj = U[j * DV + col];
      x += cf[HDR + j] * uj;
      ob += cf[HDR + Lay.Mcap4 + j] * uj;
    }
    const float vv = bf16f(av.v[col]);
    const float u = cf[2] * (vv - x);
    store_out(a, oidx, a.scale * (ob + cf[1] * u));
    if (!merge) {
      const size_t lh = (size_t)it.slot * a.H + p.h;
      static_cast<float*>(a.alog)[(lh * Lay.Mcap + n) * DV + col] = u;
    } else {
      reinterpret_cast<float*>(av.U)[n * DV + col] = u;
      __syncwarp();
    }
  } else {
    const uint16_t* V = reinterpret_cast<const uint16_t*>(av.U);
    float o = A;
#pragma unroll 4
    for (int j = 0; j < n; ++j) o += cf[HDR + j] * bf16f(V[j * DV + col]);
    o += cf[3] * bf16f(V[n * DV + col]);
    store_out(a, oidx, a.scale * o);
  }
  if (!merge) return may_release;

  // merge: S̄[slot] rows = D ⊙ S̄[base] rows + Σ_{j<=n} a_j[row] K̃_j
  // The tile is read only for D ⊙ S̄: once the last of its rows are in
  // registers, the stage goes back to the producer (if this call may release
  // it), so that the next unit's tile lands while the update runs.
  auto release_stage = [&]() {
    if (may_release) {
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar);
    }
  };
  if constexpr (OP == RWKV6 && DK == 64) {
    // Half-warp h takes rows 16h..16h+15 of the tile and lane l of it columns
    // 4l..4l+3, so that one load of a value row feeds sixteen rows, and each
    // packed FMA updates two adjacent rows of a column from one bf16 word.
    // Per element: the same product D·S̄, then the same fused multiply-adds in
    // the same order of j as the general loop below.
    const int hr = (lane >> 4) * 16, c4 = (lane & 15) * 4;
    const float4 Dv = *reinterpret_cast<const float4*>(cf + Lay.P0 + c4);
    float2 acc[8][4];   // [row pair m][column]: rows hr + 2m, hr + 2m + 1
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const float4 t0 = *reinterpret_cast<const float4*>(T + (hr + 2 * m) * DK + c4);
      const float4 t1 = *reinterpret_cast<const float4*>(T + (hr + 2 * m + 1) * DK + c4);
      acc[m][0] = make_float2(Dv.x * t0.x, Dv.x * t1.x);
      acc[m][1] = make_float2(Dv.y * t0.y, Dv.y * t1.y);
      acc[m][2] = make_float2(Dv.z * t0.z, Dv.z * t1.z);
      acc[m][3] = make_float2(Dv.w * t0.w, Dv.w * t1.w);
    }
    release_stage();
    const uint16_t* Vb = reinterpret_cast<const uint16_t*>(av.U) + vt * BV + hr;
#pragma unroll 1
    for (int j = 0; j <= n; ++j) {
      const float4 K = *reinterpret_cast<const float4*>(av.Kt + j * DK + c4);
      const uint4 w0 = *reinterpret_cast<const uint4*>(Vb + j * DV);
      const uint4 w1 = *reinterpret_cast<const uint4*>(Vb + j * DV + 8);
      const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      const float2 k0 = make_float2(K.x, K.x), k1 = make_float2(K.y, K.y);
      const float2 k2 = make_float2(K.z, K.z), k3 = make_float2(K.w, K.w);
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const float2 vp = make_float2(bf16lo(w[m]), bf16hi(w[m]));
        acc[m][0] = __ffma2_rn(vp, k0, acc[m][0]);
        acc[m][1] = __ffma2_rn(vp, k1, acc[m][1]);
        acc[m][2] = __ffma2_rn(vp, k2, acc[m][2]);
        acc[m][3] = __ffma2_rn(vp, k3, acc[m][3]);
      }
    }
    float* dst = a.Sbar + (((size_t)it.slot * a.H + p.h) * DV + vt * BV + hr) * DK + c4;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const float r0[4] = {acc[m][0].x, acc[m][1].x, acc[m][2].x, acc[m][3].x};
      const float r1[4] = {acc[m][0].y, acc[m][1].y, acc[m][2].y, acc[m][3].y};
      stvec_cs<4>(dst + (size_t)(2 * m) * DK, r0);
      stvec_cs<4>(dst + (size_t)(2 * m + 1) * DK, r1);
    }
    return may_release;
  }
  float D[VEC];
  if constexpr (OP == GDN) {
#pragma unroll
    for (int c = 0; c < VEC; ++c) D[c] = cf[0];
  } else {
    ldvec<VEC>(D, cf + Lay.P0 + lane * VEC);
  }
  float* dst = a.Sbar + (((size_t)it.slot * a.H + p.h) * DV + vt * BV) * DK + lane * VEC;
  if constexpr (OP == GDN && DK == 128) {
    // Sixteen rows at a time, each packed FMA updating two adjacent rows of a
    // column: one load of a u row's sixteen values feeds 64 accumulators.
    // Per element the same operations in the same order as the loop below.
    // (Measured on GB300: GDN M = 16 windows 1.1 % faster; KDA, whose K̃ rows
    // are fp32, 0.4 % slower at M = 16 and 1.7 % at M = 32, so it keeps the
    // loop below.)
#pragma unroll 1
    for (int rb = 0; rb < 2; ++rb) {
      float2 acc[8][VEC];   // [row pair m][column]: rows 16 rb + 2m, 16 rb + 2m + 1
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        float t0[VEC], t1[VEC];
        ldvec<VEC>(t0, T + (rb * 16 + 2 * m) * DK + lane * VEC);
        ldvec<VEC>(t1, T + (rb * 16 + 2 * m + 1) * DK + lane * VEC);
#pragma unroll
        for (int c = 0; c < VEC; ++c) acc[m][c] = make_float2(D[c] * t0[c], D[c] * t1[c]);
      }
      if (rb == 1) release_stage();
#pragma unroll 1
      for (int j = 0; j <= n; ++j) {
        float K[VEC];
        ldvec_bf16<VEC>(K, av.kl + j * DK + lane * VEC);
        const float w = cf[Lay.P0 + j];
#pragma unroll
        for (int c = 0; c < VEC; ++c) K[c] *= w;
        const float* Urow = reinterpret_cast<const float*>(av.U) + j * DV + vt * BV + rb * 16;
        const float4* U = reinterpret_cast<const float4*>(Urow);
        float2 up[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 u = U[q];
          up[2 * q] = make_float2(u.x, u.y);
          up[2 * q + 1] = make_float2(u.z, u.w);
        }
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
          const float2 kk = make_float2(K[c], K[c]);
#pragma unroll
          for (int m = 0; m < 8; ++m) acc[m][c] = __ffma2_rn(up[m], kk, acc[m][c]);
        }
      }
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        float r0[VEC], r1[VEC];
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
          r0[c] = acc[m][c].x;
          r1[c] = acc[m][c].y;
        }
        stvec_cs<VEC>(dst + (size_t)(rb * 16 + 2 * m) * DK, r0);
        stvec_cs<VEC>(dst + (size_t)(rb * 16 + 2 * m + 1) * DK, r1);
      }
    }
    return may_release;
  } else {
#pragma unroll 1
    for (int rb = 0; rb < 4; ++rb) {
      float acc[8][VEC];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float t[VEC];
        ldvec<VEC>(t, T + (rb * 8 + i) * DK + lane * VEC);
#pragma unroll
        for (int c = 0; c < VEC; ++c) acc[i][c] = D[c] * t[c];
      }
#pragma unroll 2
      for (int j = 0; j <= n; ++j) {
        float K[VEC];
        if constexpr (OP == GDN) {
          ldvec_bf16<VEC>(K, av.kl + j * DK + lane * VEC);
          const float w = cf[Lay.P0 + j];
#pragma unroll
          for (int c = 0; c < VEC; ++c) K[c] *= w;
        } else {
          ldvec<VEC>(K, av.Kt + j * DK + lane * VEC);
        }
        float uu[8];
        if constexpr (DELTA) {
          const float* U = reinterpret_cast<const float*>(av.U) + j * DV + vt * BV + rb * 8;
          const float4 u0 = *reinterpret_cast<const float4*>(U);
          const float4 u1 = *reinterpret_cast<const float4*>(U + 4);
          uu[0] = u0.x; uu[1] = u0.y; uu[2] = u0.z; uu[3] = u0.w;
          uu[4] = u1.x; uu[5] = u1.y; uu[6] = u1.z; uu[7] = u1.w;
        } else {
          const uint4 w = *reinterpret_cast<const uint4*>(
              reinterpret_cast<const uint16_t*>(av.U) + j * DV + vt * BV + rb * 8);
          uu[0] = bf16lo(w.x); uu[1] = bf16hi(w.x); uu[2] = bf16lo(w.y); uu[3] = bf16hi(w.y);
          uu[4] = bf16lo(w.z); uu[5] = bf16hi(w.z); uu[6] = bf16lo(w.w); uu[7] = bf16hi(w.w);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int c = 0; c < VEC; ++c) acc[i][c] += uu[i] * K[c];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) stvec_cs<VEC>(dst + (size_t)(rb * 8 + i) * DK, acc[i]);
    }
    // The general loop (KDA, and every op at other head sizes) keeps the stage
    // to the end: releasing it before the last quarter's update measured 0.6 %
    // slower for KDA at M = 32 on GB300, and no faster at M = 16.
    return false;
  }
}

// RWKV6 append step at d_k = 64, where one stage holds both 32-row tiles of the
// slot-head.  RWKV6 needs one dot product per row, so each lane computes its
// row of both tiles alone, and the two replay chains run interleaved.  The
// arithmetic and its order are consume_append's.
template <int DK, int DV>
__device__ __forceinline__ void consume_rwkv6_pair(const StepArgs& a, const Layout& Lay,
                                                   const UnitPos& p, int vt0, const float* T,
                                                   const AuxView& av, int lane,
                                                   uint32_t empty_bar, int n) {
  static_assert(DK == 64, "one 16 KiB stage holds both tiles at d_k = 64");
  const float* cf = av.cf;
  // Lane l takes row l of each tile whole (rwkv6_row_chunk), both rows in one
  // loop; the two tiles' chunks of r̂ are the same loads.
  const float* R = cf + HDR + 2 * Lay.Mcap4;   // r̂
  float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int kc = 0; kc < DK / 4; ++kc) {
    rwkv6_row_chunk<DK>(s0, T + lane * DK, R, kc, lane);
    rwkv6_row_chunk<DK>(s1, T + BV * DK + lane * DK, R, kc, lane);
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(empty_bar);
  const float A0 = sum4(s0);
  const float A1 = sum4(s1);
  const uint16_t* V = reinterpret_cast<const uint16_t*>(av.U);
  const int col0 = vt0 * BV + lane, col1 = col0 + BV;
  float o0 = A0, o1 = A1;
#pragma unroll 4
  for (int j = 0; j < n; ++j) {
    const float c = cf[HDR + j];
    o0 += c * bf16f(V[j * DV + col0]);
    o1 += c * bf16f(V[j * DV + col1]);
  }
  o0 += cf[3] * bf16f(V[n * DV + col0]);
  o1 += cf[3] * bf16f(V[n * DV + col1]);
  store_out(a, (size_t)p.sh * DV + col0, a.scale * o0);
  store_out(a, (size_t)p.sh * DV + col1, a.scale * o1);
}

// ------------------------------------------------------------- EagerStep ----
template <int OP, int DK, int DV>
__device__ __forceinline__ void consume_eager(const StepArgs& a, const Layout& Lay,
                                              const UnitPos& p, int vt, const float* T,
                                              unsigned char* ax, int lane, float g_s, float beta_s) {
  constexpr int VEC = DK / 32;
  const StepItem it = step_item(a, p.row);
  float kv[VEC], qv[VEC], D[VEC], kh[VEC], qh[VEC];
  const uint16_t* kq16 = reinterpret_cast<const uint16_t*>(ax + Lay.e_kq);
  ldvec_bf16<VEC>(kv, kq16 + lane * VEC);
  ldvec_bf16<VEC>(qv, kq16 + DK + lane * VEC);
  float sc = 0.f;   // k·q (delta ops) or Σ r bonus k (RWKV6)
  if constexpr (OP == GDN) {
    const float al = expf(g_s);
#pragma unroll
    for (int c = 0; c < VEC; ++c) {
      D[c] = al; kh[c] = kv[c]; qh[c] = qv[c];
      sc += kv[c] * qv[c];
    }
  } else {
    float gv[VEC];
    ldvec<VEC>(gv, reinterpret_cast<const float*>(ax + Lay.e_g) + lane * VEC);
    if constexpr (OP == KDA) {
#pragma unroll
      for (int c = 0; c < VEC; ++c) {
        D[c] = expf(gv[c]);
        kh[c] = D[c] * kv[c];
        qh[c] = D[c] * qv[c];
        sc += kv[c] * qv[c];
      }
    } else {
      float bon[VEC];
      ldvec<VEC>(bon, a.bonus + (size_t)p.h * DK + lane * VEC);
#pragma unroll
      for (int c = 0; c < VEC; ++c) {
        D[c] = expf(gv[c]);
        kh[c] = qv[c];
        qh[c] = 0.f;
        sc += qv[c] * bon[c] * kv[c];
      }
    }
  }
  sc = warp_sum(sc);

  float pa[32], pb[32];
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    float t[VEC];
    ldvec<VEC>(t, T + r * DK + lane * VEC);
    float x = 0.f, y = 0.f;
#pragma unroll
    for (int c = 0; c < VEC; ++c) {
      x += t[c] * kh[c];
      if (OP != RWKV6) y += t[c] * qh[c];
    }
    pa[r] = x;
    pb[r] = y;
  }
  const float A = reduce_scatter32(pa, lane);
  float B = 0.f;
  if constexpr (OP != RWKV6) B = reduce_scatter32(pb, lane);
  const int col = vt * BV + lane;
  const float vv = bf16f(reinterpret_cast<const uint16_t*>(ax + Lay.e_v)[col]);
  float u;
  if constexpr (OP == GDN) {
    u = beta_s * (vv - D[0] * A);
    store_out(a, (size_t)p.sh * DV + col, a.scale * (D[0] * B + sc * u));
  } else if constexpr (OP == KDA) {
    u = beta_s * (vv - A);
    store_out(a, (size_t)p.sh * DV + col, a.scale * (B + sc * u));
  } else {
    u = vv;
    store_out(a, (size_t)p.sh * DV + col, a.scale * (A + sc * vv));
  }
  float* dst = a.Sbar + (((size_t)it.slot * a.H + p.h) * DV + vt * BV) * DK + lane * VEC;
#pragma unroll 4
  for (int r = 0; r < 32; ++r) {
    const float ur = __shfl_sync(0xffffffffu, u, r);
    float t[VEC];
    ldvec<VEC>(t, T + r * DK + lane * VEC);
#pragma unroll
    for (int c = 0; c < VEC; ++c) t[c] = D[c] * t[c] + ur * kv[c];
    stvec_cs<VEC>(dst + (size_t)r * DK, t);
  }
}

// ----------------------------------------------------------------- kernel ---
// NE: the fused form's bound on log entries (8, 16 or 32: M - 1 <= NE), one
// instance each so that a launch carries only the code its M needs; 0 for the
// two-kernel and eager forms.
template <int OP, int DK, int DV, int MODE, int NE = 0>
__global__ void __maxnreg__(128) pipe_kernel(const __grid_constant__ StepArgs a) {
  static_assert(MODE != FUSED || NE == 8 || NE == 16 || NE == 32, "fused form needs NE");
  // Per-key ops' prep warps signal a unit's vectors before its coefficients,
  // and consumers run their pass over the tile in between, for logs of up to
  // 32 entries (measured on GB300, KDA M = 32: 48.0 against 45.5 M
  // tokens·heads/s).  With 16 at most the prep is short and waiting for all of
  // it first is faster (KDA M = 16: 77.1 against 75.6); GDN's prep is short at
  // any M (M = 32: 75.1 against 75.3).
  constexpr bool SPLIT_PREP = MODE == FUSED && NE == 32 && OP != GDN;
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr uint32_t TILE_BYTES = BV * DK * 4;
  const Layout Lay = make_layout(OP, a.M, DK, DV, a.arows);
  const int NS = a.ns, NA = a.na, G = a.G, NCWr = a.ncw, TPS = a.tps;
  const int IPU = G / TPS;                       // stage items per unit
  const uint32_t STAGE_BYTES = TILE_BYTES * TPS; // one bulk copy per stage item
  const int R = NS / NCWr;   // stages per consumer warp (ns is a multiple of ncw)
  const uint32_t aux_bytes =
      (MODE == APPEND) ? Lay.aux_bytes : (MODE == FUSED) ? Lay.f_bytes : Lay.e_bytes;
  const Bars bars{smem_u32(smem), NS, NA};
  float* tiles = reinterpret_cast<float*>(smem + BAR_BYTES);
  unsigned char* auxm = smem + BAR_BYTES + (size_t)NS * STAGE_BYTES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(bars.full(s), 1);
      mbar_init(bars.empty(s), 1);
    }
    for (int x = 0; x < NA; ++x) {
      mbar_init(bars.afull(x), 32);   // one arrival per producer lane
      mbar_init(bars.aempty(x), IPU);
      mbar_init(bars.cready(x), 1);   // fused form: the prep warp's arrival
      if (SPLIT_PREP && a.npw > 0) mbar_init(bars.vready(x), 1);
    }
    mbar_init(bars.never(), 1);
    fence_mbar_init();
  }
  __syncthreads();

  const int n_units = step_rows(a) * a.H * a.NG;
  const int my_units =
      (int)blockIdx.x < n_units ? (n_units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int my_tiles = my_units * IPU;   // stage items of this CTA

  if (warp == NCWr) {
    // ------------------------------------------------------------ producer
    // The whole warp runs this loop (uniform control flow); lane 0 also
    // issues the tile bulk copies.
    const uint64_t pol = a.l2_stream ? policy_evict_first() : policy_evict_normal();
    // APPEND and FUSED launch as programmatic dependents (of ReplayPrep, of the
    // previous step).  Before griddepcontrol.wait the producer only claims aux
    // slots, copies inputs and streams tiles: APPEND copies the inputs that
    // ReplayPrep does not write; FUSED copies the step's own tensors (not the
    // log rows, which the previous step appends to), and streams only tiles of
    // rows whose log is non-empty (a.pdl_prefetch), whose dense base the
    // previous step did not write (only merge rows write it, and they restart
    // at n = 0).
    bool primary_done = (MODE == EAGER);
    int pending_from = 0;   // units [pending_from, ka) still need their deferred copies
    int ti = 0, ka = 0;
    bool ok = true;
    auto issue_pending = [&]() {
      for (int u = pending_from; u < ka; ++u) {
        const UnitPos p = unit_pos(a, (int)blockIdx.x + u * (int)gridDim.x);
        unsigned char* ax = auxm + (size_t)(u % NA) * aux_bytes;
        if constexpr (MODE == APPEND) {
          issue_coef_and_arrive<OP, DK, DV>(a, Lay, p, ax, bars.afull(u % NA), lane);
        } else {   // FUSED: the inputs went out when the slot was claimed
          issue_aux<OP, DK, DV, MODE>(a, Lay, p, ax, lane, 2);
          cp_async_arrive_noinc(bars.afull(u % NA));
        }
      }
      pending_from = ka;
    };
    // Per-tile bookkeeping is incremental (no divisions on the issue path):
    // unit kt and item j of tile ti, the owning warp w, its stage round r and
    // phase parity; the unit's tile source is computed once per unit.
    int kt = 0, j = 0, w = 0, r = 0;
    uint32_t par = 0;
    int ax_x = 0;                 // aux slot of unit ka
    uint32_t ax_par = 0;          // phase parity of that slot for unit ka
    const float* src_unit = nullptr;
    UnitWalk walk;                // position of unit ka
    walk.init(a, (int)blockIdx.x);
    while (ti < my_tiles) {
      if (!primary_done) {
        // the next wait needs consumers to make progress, and they need inputs
        bool need = ti >= NS || (kt == ka && ka >= NA);
        if constexpr (MODE == FUSED) {
          if (!need && !a.pdl_prefetch) need = true;
          if (!need && step_item(a, unit_pos(a, (int)blockIdx.x + kt * (int)gridDim.x).row).n == 0)
            need = true;
        }
        if (need) {
          pdl_wait_primary();
          primary_done = true;
          if constexpr (MODE == FUSED) {
            if (lane == 0) pdl_launch_dependents();   // the next step may start its prologue
          }
          issue_pending();
        }
      }
      if (kt == ka) {
        const int x = ax_x;
        if (!__all_sync(0xffffffffu,
                        mbar_wait(bars.aempty(x), ax_par ^ 1u, a.status, DEV_TIMEOUT_EMPTY, a.wait_ns))) {
          ok = false;
          break;
        }
        const UnitPos p = walk.p;
        unsigned char* ax = auxm + (size_t)x * aux_bytes;
        if constexpr (MODE == APPEND) {
          issue_aux<OP, DK, DV, MODE>(a, Lay, p, ax, lane);
          if (primary_done) {
            issue_coef_and_arrive<OP, DK, DV>(a, Lay, p, ax, bars.afull(x), lane);
            pending_from = ka + 1;
          }
        } else if constexpr (MODE == FUSED) {
          if (primary_done) {
            issue_aux<OP, DK, DV, MODE>(a, Lay, p, ax, lane);
            cp_async_arrive_noinc(bars.afull(x));
            pending_from = ka + 1;
          } else {
            // before the previous step has completed: only the step's own
            // inputs (the log rows follow after the wait, then the arrival)
            issue_aux<OP, DK, DV, MODE>(a, Lay, p, ax, lane, 1);
          }
        } else {
          issue_aux<OP, DK, DV, MODE>(a, Lay, p, ax, lane);
          cp_async_arrive_noinc(bars.afull(x));
        }
        // DeltaLog steps read the base the slot indexes (a fork source's until
        // the first merge); the eager step reads the slot's own state
        const StepItem it = step_item(a, p.row);
        const int base = (MODE == EAGER) ? it.slot : it.base;
        src_unit = a.Sbar + (((size_t)base * a.H + p.h) * DV + (size_t)p.grp * G * BV) * DK;
        ++ka;
        walk.next();
        if (++ax_x == NA) {
          ax_x = 0;
          ax_par ^= 1u;
        }
      }
      const int s = w * R + r;   // = stage_of(ti, R, NCWr)
      if (!__all_sync(0xffffffffu, mbar_wait(bars.empty(s), par ^ 1u, a.status, DEV_TIMEOUT_EMPTY, a.wait_ns))) {
        ok = false;
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(bars.full(s), STAGE_BYTES);
        bulk_g2s_hint(smem_u32(tiles + (size_t)s * TPS * BV * DK),
                      src_unit + (size_t)j * TPS * BV * DK, STAGE_BYTES, bars.full(s), pol);
      }
      __syncwarp();
      ++ti;
      if (++j == IPU) {
        j = 0;
        ++kt;
      }
      if (++w == NCWr) {
        w = 0;
        if (++r == R) {
          r = 0;
          par ^= 1u;
        }
      }
    }
    if (ok && !primary_done) {
      pdl_wait_primary();
      primary_done = true;
      if constexpr (MODE == FUSED) {
        if (lane == 0) pdl_launch_dependents();
      }
      issue_pending();
    }
    if (!ok) {
      // an error was recorded: let the copies already in flight land before exiting
      if (!primary_done) pdl_wait_primary();
      if (lane == 0)
        for (int t = ti - NS > 0 ? ti - NS : 0; t < ti; ++t)
          mbar_drain(bars.full(stage_of(t, R, NCWr)), stage_parity(t, R, NCWr));
    }
    cp_async_wait_all();
    return;
  }

  // Everything below reads or writes global memory only after the previous
  // step (the primary grid) has completed.
  if constexpr (MODE == FUSED) pdl_wait_primary();

  if constexpr (MODE == FUSED && DK != 64) {   // (d_k = 64 units are one stage: no prep warps)
  if (warp > NCWr) {
    // ------------------------------------------------- fused ReplayPrep stage
    // Prep warp pw owns the aux slots x with x % npw == pw and takes their
    // units in order, so it waits on every phase of those slots' barriers.
    const int pw = warp - NCWr - 1, NPW = a.npw;
    UnitWalk walk;
    walk.init(a, (int)blockIdx.x);
    for (int kk = 0; kk < my_units; ++kk, walk.next()) {
      const int x = kk % NA;
      if (x % NPW != pw) continue;
      if (!__all_sync(0xffffffffu, mbar_wait(bars.afull(x), (kk / NA) & 1, a.status, DEV_TIMEOUT_AUX, a.wait_ns)))
        break;
      const UnitPos p = walk.p;
      unsigned char* ax = auxm + (size_t)x * aux_bytes;
      prep_unit<OP, DK, DV, NE>(a, Lay, p, ax, lane, SPLIT_PREP ? bars.vready(x) : 0u);
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.cready(x));
    }
    return;
  }
  }

  // -------------------------------------------------------------- consumers
  // Incremental bookkeeping (tile i of this warp: unit kk, item j within the
  // unit, aux slot x with phase parity xpar, stage round r with parity spar);
  // the unit's position is recomputed only when the unit changes.
  int kk = warp / IPU, j = warp - (warp / IPU) * IPU;
  int x = kk % NA;
  uint32_t xpar = (uint32_t)(kk / NA) & 1u;
  int r = 0;
  uint32_t spar = 0;
  UnitWalk walk;                // position of unit kk
  walk.init(a, (int)blockIdx.x + kk * (int)gridDim.x);
  for (int i = warp; i < my_tiles; i += NCWr) {
    if (i != warp) {   // advance from the previous tile of this warp
      j += NCWr;
      while (j >= IPU) {
        j -= IPU;
        ++kk;
        walk.next();
        if (++x == NA) {
          x = 0;
          xpar ^= 1u;
        }
      }
      if (++r == R) {
        r = 0;
        spar ^= 1u;
      }
    }
    const UnitPos p = walk.p;
    const int vt0 = p.grp * G + j * TPS;
    const int s = warp * R + r;   // = stage_of(i, R, NCWr)
    float g_s = 0.f, beta_s = 0.f;
    if constexpr (MODE == EAGER) {
      if (OP == GDN) g_s = a.g[p.sh];
      if (OP != RWKV6) beta_s = a.beta[p.sh];
    }
    unsigned char* ax = auxm + (size_t)x * aux_bytes;
    bool ok;
    bool cprep = false;
    if constexpr (MODE == FUSED) cprep = (DK == 64 || a.npw == 0);
    if (cprep) {
      // One-stage units, no prep warps: this warp owns aux slot x (na is a
      // multiple of ncw, so every unit of the slot is this warp's) and has
      // seen each earlier phase of its barrier itself, so it can wait for the
      // unit's inputs first and compute the coefficients while the tile is
      // still landing.
      ok = mbar_wait(bars.afull(x), xpar, a.status, DEV_TIMEOUT_AUX, a.wait_ns);
      if (!__all_sync(0xffffffffu, ok)) break;
      if constexpr (MODE == FUSED) prep_unit<OP, DK, DV, NE>(a, Lay, p, ax, lane);
      __syncwarp();
      ok = mbar_wait(bars.full(s), spar, a.status, DEV_TIMEOUT_TILE, a.wait_ns);
    } else {
      // The tile first: it is issued after its unit's aux copies, so once it
      // has landed the aux barrier is in this unit's phase and the parity test
      // below is unambiguous.
      ok = mbar_wait(bars.full(s), spar, a.status, DEV_TIMEOUT_TILE, a.wait_ns);
      // fused form: the whole prep (cready), or, with SPLIT_PREP, only the
      // unit's vectors (vready): consume_append then awaits the coefficients
      // after its pass over the tile
      ok = ok && mbar_wait(MODE == FUSED ? (SPLIT_PREP ? bars.vready(x) : bars.cready(x))
                                         : bars.afull(x),
                           xpar, a.status, DEV_TIMEOUT_AUX, a.wait_ns);
    }
    // Test only: wait on a barrier that nothing arrives on, with half the
    // limit, so that this wait runs out before the waits that depend on this
    // warp (the producer's, for the stage it holds) and its code is recorded.
    if (a.test_stall && blockIdx.x == 0 && i == 0)
      ok = ok && mbar_wait(bars.never(), 0u, a.status, DEV_TEST_STALL, a.wait_ns / 2);
    if (!__all_sync(0xffffffffu, ok)) break;
    bool released = false;
    bool paired = false;
    if constexpr (MODE != EAGER && OP == RWKV6 && DK == 64) {
      const int n = step_item(a, p.row).n;
      if (TPS == 2 && n + 1 != a.M) {   // append step: both tiles of the stage at once
        consume_rwkv6_pair<DK, DV>(a, Lay, p, vt0, tiles + (size_t)s * TPS * BV * DK,
                                   aux_view<OP, DK, MODE>(Lay, ax), lane, bars.empty(s), n);
        released = paired = true;
      }
    }
    bool failed = false;
    for (int t = 0; t < TPS && !paired && !failed; ++t) {
      const float* T = tiles + ((size_t)s * TPS + t) * BV * DK;
      if constexpr (MODE == EAGER) {
        consume_eager<OP, DK, DV>(a, Lay, p, vt0 + t, T, ax, lane, g_s, beta_s);
      } else {
        const AuxView av = aux_view<OP, DK, MODE>(Lay, ax);
        const bool split = SPLIT_PREP && !cprep;   // prep warps: coefficients come later
        released = consume_append<OP, DK, DV>(a, Lay, p, vt0 + t, T, av, lane, bars.empty(s),
                                              t == TPS - 1, split ? bars.cready(x) : 0u, xpar,
                                              &failed);
      }
    }
    if (failed) break;
    // No proxy fence here: consumers never write shared memory that a bulk
    // copy refills (tiles are read-only; the aux slots they write are refilled
    // by cp.async, which is in the generic proxy), so the mbarrier release and
    // the producer's acquiring wait order everything.
    __syncwarp();
    if (lane == 0) {
      if (!released) mbar_arrive(bars.empty(s));
      mbar_arrive(bars.aempty(x));
    }
  }
}

}  // namespace dl
