"""Host-side pipeline planner (`csrc/layout.h`), compiled with the host compiler.

Every shape the step launcher can ask for (three ops, d = 64 / 128, M = 1..32,
whole-slot-head or one-tile units, each kernel form, append or merge launches,
instances of 0 / 96 / 128 registers) must:
- exist, and fit the GB300 budgets: 227 KiB of shared memory per CTA and
  228 KiB per SM with 1 KiB reserved per CTA; 16 Ki registers in each of the
  SM's four sub-partitions, allocated per warp in steps of 8 per thread;
- keep the ownership rules that the barrier protocol model
  (test_pipeline_protocol.py) shows safe: each consumer warp owns ns / ncw >= 1
  stages; prep warps own na / npw aux slots; one-stage units are prepared by
  their own consumer warp, which then owns na / ncw aux slots;
- give merge launches of one-stage d_k = 64 units with M >= 8 the wider shape.
Aux slots sized by a launch's longest log (`arows` = n_max + 1 log rows) must
hold every section a row with n < arows uses, and plan like full slots.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "linear_attention_recurrent_gdn_gb300", "csrc")
OPTIN, PER_SM = 232448, 233472

DRIVER = r"""
#include <cstdio>
#include "layout.h"
// prep warps of the fused form, as the step launcher picks them
static int prep_warps(int op, int dk, int G, int M) {
  if (G / dl::tiles_per_stage(dk, G) == 1) return 0;
  if (op == 0) return 1;
  return M <= 16 ? 1 : 2;
}
int main() {
  const int optin = 232448, per_sm = 233472;
  const int dks[2] = {64, 128}, regss[3] = {0, 96, 128};
  for (int op = 0; op < 3; ++op)
    for (int di = 0; di < 2; ++di)
      for (int M = 1; M <= 32; ++M)
        for (int whole = 0; whole < 2; ++whole)
          for (int kind = 0; kind < 3; ++kind)      // 0 two-kernel, 1 fused, 2 eager
            for (int merge = 0; merge < 2; ++merge)
              for (int ar = 0; ar <= (kind == 2 ? 0 : M); ++ar)   // aux log rows (0: M)
              for (int ri = 0; ri < 3; ++ri) {
                if (merge && ar != 0 && ar != M) continue;   // a merge row has n = M - 1
                const int dk = dks[di], G = whole ? dk / 32 : 1;
                const dl::Layout L = dl::make_layout(op, M, dk, dk, ar);
                const int aux = kind == 0 ? L.aux_bytes : kind == 1 ? L.f_bytes : L.e_bytes;
                const int npw = kind == 1 ? prep_warps(op, dk, G, M) : -1;
                const bool ml = kind == 1 && merge && M >= 8;
                const dl::PipePlan p = dl::plan_pipeline(dk, aux, G, optin, per_sm, nullptr, npw,
                                                         regss[ri], ml);
                std::printf("%d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d\n", op, dk, M, G,
                            kind, (int)ml, regss[ri], npw, aux, dl::tiles_per_stage(dk, G),
                            p.cps, p.ncw, p.ns, p.na, p.npw, p.smem, ar);
              }
  return 0;
}
"""

FIELDS = ("op dk M G kind merge regs npw_req aux tps cps ncw ns na npw smem arows").split()


def _expected_rows():
    n = 0
    for M in range(1, 33):
        for kind in range(3):
            for merge in range(2):
                ars = [0] if kind == 2 else [a for a in range(M + 1) if not merge or a in (0, M)]
                n += len(ars)
    return n * 3 * 2 * 2 * 3   # ops, d, unit kinds, register counts


@pytest.fixture(scope="module")
def plans(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if not cxx:
        pytest.skip("no host C++ compiler")
    d = tmp_path_factory.mktemp("planner")
    src, exe = d / "plan.cpp", d / "plan"
    src.write_text(DRIVER)
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    rows = [dict(zip(FIELDS, map(int, line.split()))) for line in out.splitlines()]
    assert len(rows) == _expected_rows()
    return rows


def test_every_plan_exists_and_fits_the_budgets(plans):
    for p in plans:
        assert p["ns"] > 0, p
        assert p["smem"] <= OPTIN, p
        assert p["cps"] * (p["smem"] + 1024) <= PER_SM, p
        stage = 32 * p["dk"] * 4 * p["tps"]
        assert p["smem"] >= p["ns"] * stage + p["na"] * p["aux"], p
        # the mbarrier area (128): full and empty per stage, three per aux slot
        # (four with prep warps), one spare
        per_slot = 4 if p["npw"] > 0 else 3
        assert 2 * p["ns"] + per_slot * p["na"] + 1 <= 128, p
        if p["regs"]:
            warps = p["ncw"] + 1 + p["npw"]
            alloc = 32 * ((p["regs"] + 7) // 8 * 8)
            assert p["cps"] * warps <= 4 * (16384 // alloc), p


def test_every_plan_keeps_the_ownership_rules(plans):
    for p in plans:
        assert p["ns"] % p["ncw"] == 0 and p["ns"] >= p["ncw"], p   # whole stages per warp
        assert p["na"] >= 2, p
        if p["kind"] != 1:
            assert p["npw"] == 0, p
            continue
        one_stage = p["G"] // p["tps"] == 1
        assert p["npw"] == p["npw_req"], p
        if one_stage:
            assert p["npw"] == 0 and p["na"] % p["ncw"] == 0, p   # aux-first waits on own slots
        else:
            assert p["npw"] in (1, 2) and p["na"] % p["npw"] == 0, p


def test_merge_launches_of_one_stage_d64_units_widen(plans):
    seen = 0
    for p in plans:
        if not (p["kind"] == 1 and p["merge"] and p["dk"] == 64 and p["npw"] == 0):
            continue
        twin = next(q for q in plans if all(q[k] == p[k] for k in FIELDS[:7] if k != "merge")
                    and q["merge"] == 0 and q["kind"] == 1 and q["arows"] == p["arows"])
        if (p["cps"], p["ncw"]) != (twin["cps"], twin["ncw"]):
            assert (p["cps"], p["ncw"], p["ns"]) in ((2, 4, 4), (4, 2, 2)), p
            seen += 1
    assert seen > 0


def test_shapes_of_the_three_workloads(plans):
    """The shapes the M = 16 decode workloads run with whole-slot-head units:
    GDN and KDA (2,4,1) with one prep warp; RWKV6 append launches (3,2,1) with
    two aux slots per consumer warp, its merge launches (2,4,1)."""
    def pick(op, dk, M, merge, regs=128):
        return next(p for p in plans if p["op"] == op and p["dk"] == dk and p["M"] == M
                    and p["G"] == dk // 32 and p["kind"] == 1 and p["merge"] == merge
                    and p["regs"] == regs and p["arows"] == 0)
    gdn, kda = pick(0, 128, 16, 0), pick(1, 128, 16, 0)
    assert (gdn["cps"], gdn["ncw"], gdn["ns"], gdn["npw"]) == (2, 4, 4, 1)
    assert (kda["cps"], kda["ncw"], kda["ns"], kda["npw"]) == (2, 4, 4, 1)
    rw, rwm = pick(2, 64, 16, 0), pick(2, 64, 16, 1)
    assert (rw["cps"], rw["ncw"], rw["ns"], rw["na"], rw["npw"]) == (3, 2, 2, 4, 0)
    assert (rwm["cps"], rwm["ncw"], rwm["ns"], rwm["npw"]) == (2, 4, 4, 0)


def test_sized_slots_shrink_with_the_log_and_prep_units_keep_two_by_four(plans):
    """A slot sized for fewer log rows is never larger; units of several
    stages (GDN, KDA at d = 128, with prep warps) keep (2,4,1) at M <= 16
    whatever the log length, the shape measured fastest for them at every
    M of 4 to 32 where it fits."""
    by = {}
    for p in plans:
        if p["kind"] in (0, 1) and p["merge"] == 0 and p["regs"] == 128:
            by.setdefault((p["op"], p["dk"], p["M"], p["G"], p["kind"]), []).append(p)
    for key, ps in by.items():
        sized = sorted((p for p in ps if p["arows"] > 0), key=lambda p: p["arows"])
        full = next(p for p in ps if p["arows"] == 0)
        assert sized[-1]["aux"] == full["aux"], key     # arows = M is the full slot
        for a, b in zip(sized, sized[1:]):
            assert a["aux"] <= b["aux"], key
    for p in plans:
        if (p["kind"] == 1 and p["dk"] == 128 and p["G"] == 4 and p["op"] in (0, 1)
                and p["M"] in (4, 8, 16) and p["regs"] == 128):
            assert (p["cps"], p["ncw"], p["ns"]) == (2, 4, 4), p


LAYOUT_DRIVER = r"""
#include <cstdio>
#include "layout.h"
int main() {
  for (int op = 0; op < 3; ++op)
    for (int dk = 64; dk <= 128; dk += 64)
      for (int M = 1; M <= 32; ++M)
        for (int ar = 0; ar <= M; ++ar) {
          const dl::Layout L = dl::make_layout(op, M, dk, dk, ar);
          std::printf("%d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d\n", op, dk, M, ar,
                      L.aux_coef, L.aux_kq, L.aux_v, L.aux_U, L.aux_kl, L.aux_bytes,
                      L.f_coef, L.f_kq, L.f_v, L.f_U, L.f_kl, L.f_L, L.f_g, L.f_beta, L.f_bonus,
                      L.f_bytes, L.CB, L.P0);
        }
  return 0;
}
"""


def test_sized_slot_sections_hold_every_row_a_launch_uses(tmp_path):
    """With `arows` = n_max + 1, each log section of an aux slot holds the n
    log rows of any row with n < arows plus the current token's row (u_t or
    v_t at row n, k_t at row n on a GDN merge, the K-tilde rows 0..n of a
    per-key merge), the sections are 16-byte aligned and do not overlap, and
    the coefficient block does not depend on arows."""
    cxx = shutil.which("g++") or shutil.which("c++")
    if not cxx:
        pytest.skip("no host C++ compiler")
    src, exe = tmp_path / "lay.cpp", tmp_path / "lay"
    src.write_text(LAYOUT_DRIVER)
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    names = ("op dk M ar aux_coef aux_kq aux_v aux_U aux_kl aux_bytes f_coef f_kq f_v f_U f_kl "
             "f_L f_g f_beta f_bonus f_bytes CB P0").split()
    rows = [dict(zip(names, map(int, line.split()))) for line in out.splitlines()]
    full = {(r["op"], r["dk"], r["M"]): r for r in rows if r["ar"] == 0}
    for r in rows:
        op, d, M = r["op"], r["dk"], r["M"]
        R = r["ar"] if 0 < r["ar"] < M else M
        delta, perkey = op != 2, op != 0
        esz = 4 if delta else 2
        f = full[(op, d, M)]
        assert (r["CB"], r["P0"], r["f_coef"], r["f_kq"]) == (f["CB"], f["P0"], f["f_coef"], f["f_kq"])
        offs = [r[k] for k in ("f_coef", "f_kq", "f_v", "f_U", "f_kl", "f_L", "f_g", "f_beta",
                                "f_bonus", "f_bytes")]
        assert all(o % 16 == 0 for o in offs[:5]) and offs == sorted(offs), r
        assert r["f_kl"] - r["f_U"] >= R * d * esz, r           # rows 0..n of U
        assert r["f_L"] - r["f_kl"] >= R * d * 2, r             # key rows 0..n
        assert r["f_g"] - r["f_L"] >= (R * d * 4 if perkey else R * 4), r
        assert r["aux_kl"] - r["aux_U"] >= R * d * esz, r
        assert r["aux_bytes"] - r["aux_kl"] >= (R * d * 2 if op == 0 else 0), r
