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
};

DL_HD inline int round4(int x) { return (x + 3) & ~3; }
DL_HD inline int round16(int x) { return (x + 15) & ~15; }

DL_HD inline Layout make_layout(int op, int M, int dk, int dv) {
  Layout L{};
  const bool perkey = (op != 0);
  const bool delta = (op != 2);
  L.Mcap = M > 1 ? M - 1 : 1;
  L.Mcap4 = round4(L.Mcap);
  L.M4 = round4(M);
  L.P0 = 8 + 2 * L.Mcap4 + (perkey ? 2 * dk : 0);
  L.CB = L.P0 + (perkey ? dk + M * dk : L.M4);
  int off = 0;
  L.aux_coef = off; off += round16(L.CB * 4);
  L.aux_kq = off;   off += (op == 0) ? 2 * dk * 2 : 0;
  L.aux_v = off;    off += delta ? round16(dv * 2) : 0;
  L.aux_U = off;    off += M * dv * (delta ? 4 : 2);
  L.aux_kl = off;   off += (op == 0) ? M * dk * 2 : 0;
  L.aux_bytes = round16(off);
  off = 0;
  L.e_kq = off;     off += 2 * dk * 2;
  L.e_v = off;      off += round16(dv * 2);
  L.e_g = off;      off += perkey ? dk * 4 : 0;
  L.e_bytes = round16(off);
  return L;
}

}  // namespace dl
