// Memory layouts shared by the host runtime and the kernels.
//
// Coefficient block (fp32, one per (row, head) of a step, written by
// ReplayPrep, read by AppendDecode through a bulk copy):
//   [0, HDR)                 header: 0 e^{Λ_t} (GDN), 1 k_t·q_t, 2 beta_t, 3 bonus
//                            coefficient sum_i r_i bonus_i k_i (RWKV6)
//   [HDR, HDR+Mcap4)         ckk_j: decay-weighted k_j·k_t (RWKV6: k_j·r_t)
//   [HDR+Mcap4, HDR+2Mcap4)  ckq_j: decay-weighted k_j·q_t
//   per-key ops only         vecA [d_k]: e^{Λ_t}⊙k_t (KDA), e^{Λ_{t-1}}⊙r_t (RWKV6)
//                            vecB [d_k]: e^{Λ_t}⊙q_t (KDA)
//   -- P0 floats: what an append step needs; the rest only on merge steps --
//   GDN                      w_j = e^{Λ_t - Λ_j} [M4] (w_n = 1: the current token)
//   per-key ops              D = e^{Λ_t} [d_k], then K̃_j = k_j ⊙ e^{Λ_t - Λ_j} [M][d_k]
//
// Aux slot (shared memory of AppendDecode, one per work unit in flight; byte
// offsets, each 16-byte aligned):
//   coef   the coefficient block (CB floats)
//   kq     GDN: k_t, q_t as bf16 [2][d_k]
//   v      delta-rule ops: v_t bf16 [d_v]
//   U      value-side log rows 0..n-1 (fp32 u_j; bf16 v_j for RWKV6) and one
//          more row: u_t written by the consumer at a merge, or v_t (RWKV6)
//   kl     GDN merge: key log rows 0..n-1 and k_t as row n, bf16 [M][d_k]
// The log-row sections hold `arows` rows: M by default, or, when the launcher
// knows every row's n, the largest log length n of a launch's rows, plus one
// where a step uses the current token's row (RWKV6's v_t, a merge step's u_t
// and k_t), so that short logs leave room for more units in flight.
#pragma once

#ifdef __CUDACC__
#define DL_HD __host__ __device__
#else
#define DL_HD
#endif

namespace dl {

struct Layout {
  int Mcap, Mcap4, M4;       // log capacity, rounded to multiples of 4
  int P0, CB;                // coefficient floats for append steps / block stride
  int aux_coef, aux_kq, aux_v, aux_U, aux_kl, aux_bytes;   // AppendDecode aux slot
  int e_kq, e_v, e_g, e_bytes;                              // EagerStep aux slot
  // AppendDecode with the ReplayPrep stage fused in as a warp role: the aux
  // slot also holds what that warp reads (key log, log-decays, g, beta, bonus)
  // and it writes the coefficients into f_coef (the K̃ rows of a per-key merge
  // go over the log-decay rows, in f_L).
  int f_coef, f_kq, f_v, f_U, f_kl, f_L, f_g, f_beta, f_bonus, f_bytes;
};

DL_HD inline int round4(int x) { return (x + 3) & ~3; }
DL_HD inline int round16(int x) { return (x + 15) & ~15; }

DL_HD inline Layout make_layout(int op, int M, int dk, int dv, int arows = 0) {
  Layout L{};
  const bool perkey = (op != 0);
  const bool delta = (op != 2);
  const int R = (arows > 0 && arows < M) ? arows : M;   // log rows of an aux slot
  L.Mcap = M > 1 ? M - 1 : 1;
  L.Mcap4 = round4(L.Mcap);
  L.M4 = round4(M);
  L.P0 = 8 + 2 * L.Mcap4 + (perkey ? 2 * dk : 0);
  L.CB = L.P0 + (perkey ? dk + M * dk : L.M4);
  int off = 0;
  L.aux_coef = off; off += round16(L.CB * 4);
  L.aux_kq = off;   off += (op == 0) ? 2 * dk * 2 : 0;
  L.aux_v = off;    off += delta ? round16(dv * 2) : 0;
  L.aux_U = off;    off += R * dv * (delta ? 4 : 2);
  L.aux_kl = off;   off += (op == 0) ? R * dk * 2 : 0;
  L.aux_bytes = round16(off);
  off = 0;
  L.e_kq = off;     off += 2 * dk * 2;
  L.e_v = off;      off += round16(dv * 2);
  L.e_g = off;      off += perkey ? dk * 4 : 0;
  L.e_bytes = round16(off);
  off = 0;
  L.f_coef = off;   off += round16((L.P0 + (perkey ? dk : L.M4)) * 4);
  L.f_kq = off;     off += 2 * dk * 2;
  L.f_v = off;      off += delta ? round16(dv * 2) : 0;
  L.f_U = off;      off += R * dv * (delta ? 4 : 2);
  L.f_kl = off;     off += R * dk * 2;
  L.f_L = off;      off += perkey ? R * dk * 4 : round4(R) * 4;
  L.f_g = off;      off += perkey ? dk * 4 : 16;
  L.f_beta = off;   off += delta ? 16 : 0;
  L.f_bonus = off;  off += (op == 2) ? dk * 4 : 0;
  L.f_bytes = round16(off);
  return L;
}

// Shape of the pipelined kernels for one launch: `cps` CTAs per SM, each with
// `ncw` consumer warps owning `ns / ncw` tile stages apiece and `na` aux slots
// (at least 2, so the next unit's inputs load while the current one is used).
// The fused form adds `npw` prep warps; prep warp w owns the aux slots x with
// x % npw == w, so na is a multiple of npw.  With npw = 0 (one-stage units)
// each consumer warp computes its units' coefficients itself and owns the aux
// slots x with x % ncw == w, so na is a multiple of ncw.  Returns ns = 0 when
// nothing fits.
constexpr int BAR_SLOTS = 128;   // 8-byte mbarriers in the pipelined kernels' barrier area

struct PipePlan {
  int cps, ncw, ns, na, npw;
  int smem;   // dynamic shared memory per CTA (bytes): the CTA's share of the SM
};

// Fit one candidate shape (cps CTAs per SM, ncw consumer warps, R stages per
// warp) into the shared-memory budget; ns = 0 if it does not fit.  `npw` is
// the number of prep warps (-1: none, the two-kernel and eager forms).
inline PipePlan fit_pipeline(int cps, int ncw, int R, int dk, int aux_bytes, int G, int smem_optin,
                             int smem_per_sm, int tps = 1, int npw = -1, int regs = 0,
                             int max_na = 16) {
  const PipePlan none{0, 0, 0, 0, 0, 0};
  if (ncw < 1 || ncw > 8 || R < 1 || npw > 2) return none;
  // one-stage units are prepared by their consumer warp, larger ones by prep warps
  if (npw >= 0 && (npw == 0) != (G / tps == 1)) return none;
  // registers: cps CTAs of (ncw + 1 + npw) warps must be resident together.
  // Each of the SM's 4 sub-partitions holds 16 Ki registers, allocated per
  // warp in multiples of 8 per thread; a warp lives on one sub-partition.
  const int warps = ncw + 1 + (npw > 0 ? npw : 0);
  if (regs > 0) {
    const int per_sub = 16384 / (32 * ((regs + 7) / 8 * 8));
    if (cps * warps > 4 * per_sub) return none;
  }
  const int tile = 32 * dk * 4 * tps;   // bytes of one stage
  const int per_cta = smem_per_sm / cps - 1024;     // 1 KiB per CTA is reserved
  const int budget = (per_cta < smem_optin ? per_cta : smem_optin) - 1024 - 1024;
  const int ns = ncw * R;
  // aux slots: all the shared memory the stages leave, up to max_na (each slot
  // lets the producer fetch one more unit's inputs ahead of the consumers)
  const int mult = npw > 0 ? npw : npw == 0 ? ncw : 1;
  const int na_min = mult > 2 ? mult : 2;
  const long left = (long)budget - (long)ns * tile;
  int na = left > 0 ? (int)(left / aux_bytes) : 0;
  if (na > max_na) na = max_na;
  // the mbarrier area holds BAR_SLOTS barriers: full and empty per stage,
  // three per aux slot (four with prep warps: their early "vectors ready"),
  // and one spare
  const int per_slot = npw > 0 ? 4 : 3;
  if (2 * ns + per_slot * na + 1 > BAR_SLOTS) na = (BAR_SLOTS - 1 - 2 * ns) / per_slot;
  na = na / mult * mult;
  const long need = (long)ns * tile + (long)na * aux_bytes;
  if (na < na_min || ns > 24 || na > 24 || need > budget) return none;
  // Each CTA claims its whole share of the SM's shared memory, not just what
  // its stages and slots need: consecutive launches of a decode loop then ask
  // for the same amount whenever they run the same number of CTAs per SM,
  // whatever their log lengths.  Measured on GB300 (RWKV6 decode, aux slots
  // sized by the launch's log length): launches whose dynamic shared memory
  // changed from one to the next ran M = 4 windows at 221.6 M tokens·heads/s,
  // against 280.2 M once each claimed its full share.
  const int claim = (per_cta < smem_optin ? per_cta : smem_optin) & ~127;
  return PipePlan{cps, ncw, ns, na, npw > 0 ? npw : 0, claim};
}

// Stages hold one 16 KiB bulk copy: one value tile at d_k = 128, two at d_k = 64
// (when the unit has both tiles), because each bulk copy has a fixed issue cost.
inline int tiles_per_stage(int dk, int G) { return (dk == 64 && G % 2 == 0) ? 2 : 1; }

inline PipePlan plan_pipeline(int dk, int aux_bytes, int G, int smem_optin, int smem_per_sm,
                              const int* force = nullptr, int npw = -1, int regs = 0,
                              bool merge_launch = false) {
  const int tps = tiles_per_stage(dk, G);
  if (force) {   // tuning override: {cps, ncw, R, npw (-1: default), max_na (0: default)}
    const PipePlan p = fit_pipeline(force[0], force[1], force[2], dk, aux_bytes, G, smem_optin,
                                    smem_per_sm, tps, force[3] >= 0 ? force[3] : npw, regs,
                                    force[4] > 0 ? force[4] : 16);
    if (p.ns > 0) return p;
  }
  // Candidates in order of preference (cps, ncw, R), from measurements of
  // these shapes on GB300.  Two CTAs per SM with one 16 KiB stage per consumer
  // warp stream best for the two-kernel and eager forms, and for the fused
  // form's units of several stages (their prep warps): measured with aux slots
  // sized by the launch's log length, (2,4,1) beat (4,2,1), (3,2,1), (2,3,1)
  // and (1,8,1) for GDN and KDA at every M of 4 to 32 where it fits (GDN
  // M = 32: 75.1 against 68.6 M tokens·heads/s for (4,2,1); M = 4: 78.2
  // against 67.2).  The fused form's one-stage units (d_k = 64) do better
  // with four CTAs of two consumer warps where their aux slots fit (more
  // producers, and more units whose coefficients are computed at once).
  // 8 KiB stages (d_k = 64 with one tile per unit) need more stages per warp.
  // Each list ends with small shapes that only large aux slots fall back to
  // (per-key ops at M near 32), so that every supported configuration has one.
  static const int c16k[][3] = {{2, 4, 1}, {2, 3, 1}, {1, 8, 1}, {1, 6, 1}, {1, 4, 1},
                                {2, 2, 1}, {1, 2, 1}, {2, 1, 1}, {1, 1, 1}};
  static const int c16k_fused[][3] = {{4, 2, 1}, {2, 4, 1}, {3, 2, 1}, {2, 3, 1}, {1, 8, 1},
                                      {1, 4, 1}, {2, 2, 1}, {1, 2, 1}, {2, 1, 1}, {1, 1, 1}};
  static const int c16k_prep[][3] = {{2, 4, 1}, {3, 2, 1}, {2, 3, 1}, {4, 2, 1}, {1, 8, 1},
                                     {1, 4, 1}, {2, 2, 1}, {1, 2, 1}, {2, 1, 1}, {1, 1, 1}};
  static const int c8k[][3] = {{2, 4, 3}, {2, 4, 2}, {2, 3, 2}, {1, 8, 2}, {1, 8, 1}, {1, 4, 1},
                               {2, 2, 1}, {1, 2, 1}, {2, 1, 1}, {1, 1, 1}};
  const bool big = 32 * dk * 4 * tps >= 16384;
  const bool fused = npw >= 0;
  const int (*cand)[3] = !big ? c8k : !fused ? c16k : npw == 0 ? c16k_fused : c16k_prep;
  const int ncand = !big ? 10 : fused ? 10 : 9;
  const int npref = ncand - 4;   // the shapes before the fallbacks
  if (npw == 0 && merge_launch && dk == 64) {
    // One-stage d_k = 64 units on a launch where every row merges: each unit's
    // rank-M update holds its stage for most of the unit's time, so more
    // consumer warps per CTA pay more than deep input slots (measured on GB300
    // for 5120 RWKV6 slot-heads at M = 16: 60.4 us a launch at (2,4,1), 62.5 at
    // (4,2,1), 69.6 at the append steps' (3,2,1)).  Callers ask for it only for
    // M >= 8: at M = 4 the update is short and the append shape stays faster.
    static const int cm[][3] = {{2, 4, 1}, {4, 2, 1}};
    for (const auto& m : cm) {
      const PipePlan p = fit_pipeline(m[0], m[1], m[2], dk, aux_bytes, G, smem_optin, smem_per_sm,
                                      tps, npw, regs);
      if (p.ns > 0) return p;
    }
  }
  if (npw == 0) {
    // One-stage units, each prepared by its own consumer warp: a warp's aux
    // slots are how far ahead its units' inputs load (measured on GB300: one
    // slot per warp leaves ~1.3 us of input latency exposed per unit), so take
    // the shape with the most slots per consumer warp, counting up to 3, and
    // among those the earliest in the list (more CTAs per SM).  Shapes with
    // one CTA per SM (one producer) only come in when no other fits.
    PipePlan best{0, 0, 0, 0, 0, 0};
    int best_depth = 0;
    for (int ci = 0; ci < npref; ++ci) {
      if (cand[ci][0] < 2) continue;
      const PipePlan p = fit_pipeline(cand[ci][0], cand[ci][1], cand[ci][2], dk, aux_bytes, G,
                                      smem_optin, smem_per_sm, tps, npw, regs);
      if (p.ns == 0) continue;
      int depth = p.na / p.ncw;
      if (depth > 3) depth = 3;
      if (depth > best_depth) {
        best = p;
        best_depth = depth;
      }
    }
    if (best.ns > 0) return best;
  }
  for (int ci = 0; ci < ncand; ++ci) {
    const PipePlan p = fit_pipeline(cand[ci][0], cand[ci][1], cand[ci][2], dk, aux_bytes, G,
                                    smem_optin, smem_per_sm, tps, npw, regs);
    if (p.ns > 0) return p;
  }
  return PipePlan{0, 0, 0, 0, 0, 0};
}

}  // namespace dl
