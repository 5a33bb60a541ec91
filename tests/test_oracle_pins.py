"""Pins of the fp64 oracle to facts other than itself (CPU only).

Each check is chosen so that a plausible mistake in the oracle (a dropped
decay or beta, a sign, a transposed state, a key/query swap, an off-by-one
token, a wrong factor order) fails at least one of them:

  golden     hand-worked 2x2 examples (tests/golden/hand_worked_2x2.json)
  P1         closed-form unrolled products for the delta rules (explicit
             d_k x d_k transitions, non-recursive sums), GDN and KDA
  P2         closed form of RWKV6 (non-recursive), and the key-major form as
             written against the value-major one
  P3         special cases: beta = 0, one step from zero, one-hot keys (the
             delta rule's overwrite), RWKV6 with w = 1 and no bonus
  P4         the base + log + merge-every-M model equals eager at every step,
             for every M in 1..T+1 (DeltaLog's claim that only the schedule
             changes, not the function); forced merges at random tokens and
             slots, of plain and of forked slots, keep it equal to eager, empty
             the log and privatise the base (planted mistakes fail it)
  P5         fork by base index equals copy-then-run, and equals eager from
             the source's materialised state
  P6         the integer bookkeeping model on hand-written traces and invariants
"""
import json
import os
import random

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_2x2.json")
rng = np.random.default_rng(20261202)


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _tiny(op, T, BH, dk, dv, seed=0):
    r = np.random.default_rng(seed)
    S0 = r.normal(0, 0.5, (BH, dv, dk))
    if op == oracle.RWKV6:
        q = r.normal(size=(T, BH, dk))
        k = r.normal(size=(T, BH, dk))
        g = -np.exp(r.normal(-0.5, 0.5, (T, BH, dk)))
        extra = r.normal(0, 0.1, (BH, dk))  # bonus
    else:
        q = _unit(r.normal(size=(T, BH, dk)))
        k = _unit(r.normal(size=(T, BH, dk)))
        gshape = (T, BH) if op == oracle.GDN else (T, BH, dk)
        g = -0.1 * np.log1p(np.exp(r.normal(size=gshape)))
        extra = 1 / (1 + np.exp(-r.normal(size=(T, BH))))  # beta
    v = r.normal(size=(T, BH, dv))
    return S0, q, k, v, g, extra


def _eager(op, S0, q, k, v, g, extra, snap=None):
    fn = {oracle.GDN: oracle.gdn_eager, oracle.KDA: oracle.kda_eager,
          oracle.RWKV6: oracle.rwkv6_eager}[op]
    return fn(S0, q, k, v, g, extra, snap=snap)


# ---------------------------------------------------------------- golden -----
def test_golden_gdn():
    G = json.load(open(GOLD))["gdn"]
    S0 = np.array(G["S0"], float)[None]
    st = G["steps"]
    q = np.array([[s["q"]] for s in st], float)
    k = np.array([[s["k"]] for s in st], float)
    v = np.array([[s["v"]] for s in st], float)
    g = np.log(np.array([[s["alpha"]] for s in st], float))
    beta = np.array([[s["beta"]] for s in st], float)
    o, S, snaps = oracle.gdn_eager(S0, q, k, v, g, beta, snap=[0, 1])
    for t, s in enumerate(st):
        np.testing.assert_allclose(o[t, 0], s["o"], atol=1e-14)
        np.testing.assert_allclose(snaps[t, 0], s["S"], atol=1e-14)


def test_golden_kda():
    G = json.load(open(GOLD))["kda"]
    s = G["steps"][0]
    S0 = np.array(G["S0"], float)[None]
    o, S, _ = oracle.kda_eager(S0, np.array([[s["q"]]]), np.array([[s["k"]]]),
                               np.array([[s["v"]]]), np.log(np.array([[s["alpha"]]])),
                               np.array([[s["beta"]]]))
    np.testing.assert_allclose(o[0, 0], s["o"], atol=1e-14)
    np.testing.assert_allclose(S[0], s["S"], atol=1e-14)
    assert not np.allclose(S[0], G["wrong_order_S_I_minus_kkT_then_Diag_alpha"])


def test_golden_rwkv6_both_layouts():
    G = json.load(open(GOLD))["rwkv6"]
    s = G["steps"][0]
    S0 = np.array(G["S0"], float)[None]
    args = (S0, np.array([[s["r"]]], float), np.array([[s["k"]]], float),
            np.array([[s["v"]]], float), np.log(np.array([[s["w"]]])),
            np.array([G["bonus"]], float))
    o, S, _ = oracle.rwkv6_eager(*args)
    np.testing.assert_allclose(o[0, 0], s["o"], atol=1e-14)
    np.testing.assert_allclose(S[0], s["S"], atol=1e-14)
    o2, S2 = oracle.rwkv6_eager_keymajor(*args)
    np.testing.assert_allclose(o2[0, 0], s["o"], atol=1e-14)
    np.testing.assert_allclose(S2[0], s["S"], atol=1e-14)


# ---------------------------------------------------------------- P1 ---------
def _transition(op, k, g, beta):
    dk = k.shape[-1]
    alpha = np.exp(g) * np.ones(dk)          # scalar (GDN) or per key (KDA)
    return np.diag(alpha) @ (np.eye(dk) - beta * np.outer(k, k))


@pytest.mark.parametrize("op", [oracle.GDN, oracle.KDA])
def test_p1_closed_form_products(op):
    T, BH, dk, dv = 9, 3, 5, 4
    S0, q, k, v, g, beta = _tiny(op, T, BH, dk, dv, seed=1)
    o, S_final, snaps = _eager(op, S0, q, k, v, g, beta, snap=list(range(T)))
    for bh in range(BH):
        P = [_transition(op, k[t, bh], g[t, bh], beta[t, bh]) for t in range(T)]
        for t in range(T):
            # S_t = S_0 P_1...P_t + sum_j beta_j v_j k_j^T P_{j+1}...P_t  (each product from scratch)
            prod = np.eye(dk)
            for i in range(t + 1):
                prod = prod @ P[i]
            S_t = S0[bh] @ prod
            for j in range(t + 1):
                tail = np.eye(dk)
                for i in range(j + 1, t + 1):
                    tail = tail @ P[i]
                S_t = S_t + beta[j, bh] * np.outer(v[j, bh], k[j, bh]) @ tail
            assert _rel(snaps[t, bh], S_t) < 1e-12
            assert _rel(o[t, bh], S_t @ q[t, bh]) < 1e-12


# ---------------------------------------------------------------- P2 ---------
def test_p2_rwkv6_closed_form_and_keymajor():
    T, BH, dk, dv = 8, 3, 6, 5
    S0, r, k, v, g, bonus = _tiny(oracle.RWKV6, T, BH, dk, dv, seed=2)
    o, S_final, snaps = oracle.rwkv6_eager(S0, r, k, v, g, bonus, snap=list(range(T)))
    w = np.exp(g)
    for bh in range(BH):
        def closed(t):  # state after tokens 0..t-1 (t tokens), non-recursive
            S = S0[bh] * np.prod(w[:t, bh], axis=0)[None, :]
            for j in range(t):
                S = S + np.outer(v[j, bh], k[j, bh] * np.prod(w[j + 1:t, bh], axis=0))
            return S
        for t in range(T):
            assert _rel(snaps[t, bh], closed(t + 1)) < 1e-12
            cb = np.sum(r[t, bh] * bonus[bh] * k[t, bh])
            assert _rel(o[t, bh], closed(t) @ r[t, bh] + cb * v[t, bh]) < 1e-12
    o2, S2 = oracle.rwkv6_eager_keymajor(S0, r, k, v, g, bonus)
    assert _rel(o2, o) < 1e-13 and _rel(S2, S_final) < 1e-13


# ---------------------------------------------------------------- P3 ---------
@pytest.mark.parametrize("op", [oracle.GDN, oracle.KDA])
def test_p3_beta_zero_is_pure_decay(op):
    T, BH, dk, dv = 7, 2, 4, 3
    S0, q, k, v, g, beta = _tiny(op, T, BH, dk, dv, seed=3)
    beta = np.zeros_like(beta)
    o, S, _ = _eager(op, S0, q, k, v, g, beta)
    if op == oracle.GDN:
        expect = S0 * np.exp(g.sum(0))[:, None, None]
    else:
        expect = S0 * np.exp(g.sum(0))[:, None, :]
    assert _rel(S, expect) < 1e-14


@pytest.mark.parametrize("op", [oracle.GDN, oracle.KDA])
def test_p3_one_step_from_zero(op):
    T, BH, dk, dv = 1, 3, 6, 5
    S0, q, k, v, g, beta = _tiny(op, T, BH, dk, dv, seed=4)
    S0 = np.zeros_like(S0)
    o, S, _ = _eager(op, S0, q, k, v, g, beta)
    for bh in range(BH):
        np.testing.assert_allclose(S[bh], beta[0, bh] * np.outer(v[0, bh], k[0, bh]), atol=1e-15)
        np.testing.assert_allclose(o[0, bh], beta[0, bh] * (k[0, bh] @ q[0, bh]) * v[0, bh], atol=1e-15)


@pytest.mark.parametrize("op", [oracle.GDN, oracle.KDA])
def test_p3_one_hot_key_overwrites_column(op):
    T, BH, dk, dv = 6, 2, 5, 4
    S0, q, k, v, g, beta = _tiny(op, T, BH, dk, dv, seed=5)
    idx = [0, 3, 3, 1, 4, 0]
    k = np.zeros_like(k)
    for t, i in enumerate(idx):
        k[t, :, i] = 1.0
    g = np.zeros_like(g)
    beta = np.ones_like(beta)
    o, S, snaps = _eager(op, S0, q, k, v, g, beta, snap=list(range(T)))
    prev = S0
    for t, i in enumerate(idx):
        # the written column equals v_t up to one rounding of S + (v - S);
        # every other column is carried over from the previous state bit for bit
        np.testing.assert_allclose(snaps[t][:, :, i], v[t], rtol=0, atol=4e-15)
        others = [c for c in range(dk) if c != i]
        assert np.array_equal(snaps[t][:, :, others], prev[:, :, others])
        prev = snaps[t]


def test_p3_rwkv6_no_decay_no_bonus():
    T, BH, dk, dv = 6, 2, 4, 3
    S0, r, k, v, g, bonus = _tiny(oracle.RWKV6, T, BH, dk, dv, seed=6)
    o, S, _ = oracle.rwkv6_eager(S0, r, k, v, np.zeros_like(g), np.zeros_like(bonus))
    assert _rel(S, S0 + np.einsum("tbv,tbk->bvk", v, k)) < 1e-14
    assert _rel(o[0], np.einsum("bvk,bk->bv", S0, r[0])) < 1e-14


# ---------------------------------------------------------------- P4 ---------
def _model_run(op, M, S0, q, k, v, g, extra, H):
    """Run the DeltaLog model on BH = B*H slot-heads (B slots of H heads)."""
    T, BH, dk = q.shape
    dv = v.shape[-1]
    B = BH // H
    model = oracle.DeltaLogModel(op, B, H, dk, dv, M,
                                 bonus=extra.reshape(B, H, dk)[0] if op == oracle.RWKV6 else None)
    model.set_state(list(range(B)), S0.reshape(B, H, dv, dk))
    outs, states = [], []
    for t in range(T):
        rs = lambda x: x[t].reshape((B, H) + x.shape[2:])
        beta = None if op == oracle.RWKV6 else extra[t].reshape(B, H)
        outs.append(model.step(list(range(B)), rs(q), rs(k), rs(v), rs(g), beta).reshape(BH, dv))
        states.append(model.read_state(list(range(B))).reshape(BH, dv, dk))
    return np.stack(outs), np.stack(states), model


@pytest.mark.parametrize("op", [oracle.GDN, oracle.KDA, oracle.RWKV6])
def test_p4_base_plus_log_equals_eager_every_M(op):
    T, B, H, dk, dv = 11, 2, 2, 5, 4
    S0, q, k, v, g, extra = _tiny(op, T, B * H, dk, dv, seed=7)
    if op == oracle.RWKV6:
        extra = np.tile(extra[:H], (B, 1))  # bonus is per head
    o_ref, _, snaps = _eager(op, S0, q, k, v, g, extra, snap=list(range(T)))
    for M in range(1, T + 2):
        o, states, model = _model_run(op, M, S0, q, k, v, g, extra, H)
        assert _rel(o, o_ref) < 1e-12, M
        assert _rel(states, snaps) < 1e-12, M
        n, _ = model.meta()
        assert all(x == T % M for x in n), (M, n)


def _check_forced_merges(model_cls, op, M, seed):
    """Forced merges (DeltaLog page, "Methodology — Base + Log", merge phase,
    taken early): after merging a slot, its materialised state is still eager's
    state at that token, its log is empty and it owns its base; the outputs of
    every later token still equal eager's.  Part A: plain slots.  Part B: a
    source forked into two branches by base index; merging a branch must write
    the branch's own storage and leave the source's base untouched."""
    T, B, H, dk, dv = 12, 3, 2, 5, 4
    r = np.random.default_rng(seed)
    S0, q, k, v, g, extra = _tiny(op, T, B * H, dk, dv, seed=seed)
    if op == oracle.RWKV6:
        extra = np.tile(extra[:H], (B, 1))
    o_ref, _, snaps = _eager(op, S0, q, k, v, g, extra, snap=list(range(T)))
    slots = list(range(B))
    model = model_cls(op, B, H, dk, dv, M, bonus=extra[:H] if op == oracle.RWKV6 else None)
    model.set_state(slots, S0.reshape(B, H, dv, dk))
    rs = lambda x, t: x[t].reshape((B, H) + x.shape[2:])
    merged_any = False
    for t in range(T):
        beta = None if op == oracle.RWKV6 else extra[t].reshape(B, H)
        o = model.step(slots, rs(q, t), rs(k, t), rs(v, t), rs(g, t), beta)
        assert _rel(o.reshape(B * H, dv), o_ref[t]) < 1e-12, ("output", t)
        if r.random() < 0.5:
            sel = sorted(int(s) for s in r.choice(B, size=int(r.integers(1, B + 1)), replace=False))
            model.merge(sel)
            merged_any = True
            n, base_of = model.meta()
            for s in sel:
                assert n[s] == 0 and base_of[s] == s and model.log[s] == [], ("bookkeeping", t, s)
        state = model.read_state(slots).reshape(B * H, dv, dk)
        assert _rel(state, snaps[t]) < 1e-12, ("state", t)
    assert merged_any

    # Part B: fork, then merge a branch before and between its own steps
    Tctx, Tq = 5, 7
    S0, q, k, v, g, extra = _tiny(op, Tctx + Tq, 3 * H, dk, dv, seed=seed + 1)
    bonus = extra[:H] if op == oracle.RWKV6 else None
    model = model_cls(op, 3, H, dk, dv, M, bonus=bonus)
    model.set_state([0], S0.reshape(3, H, dv, dk)[:1])
    row = lambda x, t, s: x[t].reshape((3, H) + x.shape[2:])[s:s + 1]
    beta = lambda t, s: None if op == oracle.RWKV6 else extra[t].reshape(3, H)[s:s + 1]
    for t in range(Tctx):
        model.step([0], row(q, t, 0), row(k, t, 0), row(v, t, 0), row(g, t, 0), beta(t, 0))
    src_state = model.read_state([0])[0].copy()
    src_store = model.store[0].copy()
    model.fork(0, [1, 2])
    model.merge([1])                                   # privatise branch 1 before it steps
    n, base_of = model.meta()
    assert base_of[1] == 1 and n[1] == 0 and model.log[1] == [], "fork-merge bookkeeping"
    assert np.array_equal(model.store[0], src_store), "source base changed by a branch merge"
    assert _rel(model.read_state([1])[0], src_state) < 1e-12, "branch state after merge"
    assert _rel(model.read_state([0])[0], src_state) < 1e-12, "source state after branch merge"
    for s in (1, 2):
        sel = lambda x: x[Tctx:].reshape((Tq, 3, H) + x.shape[2:])[:, s]
        ex = bonus if op == oracle.RWKV6 else sel(extra)
        o_e, _, snap_e = _eager(op, src_state, sel(q), sel(k), sel(v), sel(g), ex,
                                snap=list(range(Tq)))
        for j, t in enumerate(range(Tctx, Tctx + Tq)):
            o = model.step([s], row(q, t, s), row(k, t, s), row(v, t, s), row(g, t, s), beta(t, s))
            assert _rel(o[0], o_e[j]) < 1e-12, ("branch output", s, j)
            if j % 3 == 1:
                model.merge([s])
                assert model.meta()[1][s] == s and model.log[s] == []
            assert _rel(model.read_state([s])[0], snap_e[j]) < 1e-12, ("branch state", s, j)
            assert np.array_equal(model.store[0], src_store), "source base changed"


class _MergeKeepsLog(oracle.DeltaLogModel):
    """Planted mistake: the forced merge writes the base but leaves the log."""

    def merge(self, slots):
        logs = {s: list(self.log[s]) for s in slots}
        super().merge(slots)
        for s in slots:
            self.log[s] = logs[s]


class _MergeStoresIntoReadBase(oracle.DeltaLogModel):
    """Planted mistake: the merged state goes to the storage the slot read
    (a fork source's base) instead of the slot's own."""

    def merge(self, slots):
        mats = [self._materialise(s, self.table.base_of[s], self._L_prev(s)) for s in slots]
        targets = [self.table.base_of[s] for s in slots]
        assert self.table.merge(list(slots)) == oracle.OK
        for s, tgt, S in zip(slots, targets, mats):
            self.store[tgt] = S
            self.log[s] = []


class _MergeDropsDecay(oracle.DeltaLogModel):
    """Planted mistake: the materialisation forgets the base's decay D."""

    def merge(self, slots):
        mats = []
        for s in slots:
            L0 = self._L_prev(s)
            S = self._materialise(s, self.table.base_of[s], L0)
            Sb = self.store[self.table.base_of[s]]
            D = np.exp(L0)[:, None, None] if self.op == oracle.GDN else np.exp(L0)[:, None, :]
            mats.append(S - D * Sb + Sb)
        assert self.table.merge(list(slots)) == oracle.OK
        for s, S in zip(slots, mats):
            self.store[s] = S
            self.log[s] = []


@pytest.mark.parametrize("op", [oracle.GDN, oracle.KDA, oracle.RWKV6])
@pytest.mark.parametrize("M", [1, 2, 3, 5, 13])
def test_p4_forced_merges_keep_eager(op, M):
    _check_forced_merges(oracle.DeltaLogModel, op, M, seed=100 + 10 * op + M)


@pytest.mark.parametrize("op", [oracle.GDN, oracle.KDA, oracle.RWKV6])
@pytest.mark.parametrize("mutant", [_MergeKeepsLog, _MergeStoresIntoReadBase, _MergeDropsDecay])
def test_p4_forced_merge_check_catches_planted_mistakes(op, mutant):
    with pytest.raises(AssertionError):
        _check_forced_merges(mutant, op, 5, seed=100 + 10 * op + 5)


# ---------------------------------------------------------------- P5 ---------
@pytest.mark.parametrize("op", [oracle.GDN, oracle.KDA, oracle.RWKV6])
def test_p5_fork_by_index_equals_copy_and_eager(op):
    Tctx, Tq, H, dk, dv, M, nb = 10, 9, 2, 4, 3, 4, 3
    S0, q, k, v, g, extra = _tiny(op, Tctx + Tq, H * (1 + 2 * nb), dk, dv, seed=8)
    bonus = extra[:H] if op == oracle.RWKV6 else None
    rs = lambda x, t, rows: x[t].reshape((-1, H) + x.shape[2:])[rows]
    beta = lambda t, rows: None if op == oracle.RWKV6 else extra[t].reshape(-1, H)[rows]
    # slot 0: request; slots 1..nb: branches by index; nb+1..2nb: branches by copy
    model = oracle.DeltaLogModel(op, 1 + 2 * nb, H, dk, dv, M, bonus=bonus)
    model.set_state([0], S0.reshape(-1, H, dv, dk)[:1])
    for t in range(Tctx):  # ends mid-window (10 % 4 = 2): the fork copies a live log
        model.step([0], rs(q, t, [0]), rs(k, t, [0]), rs(v, t, [0]), rs(g, t, [0]), beta(t, [0]))
    src_state = model.read_state([0])[0]
    by_index = list(range(1, nb + 1))
    by_copy = list(range(nb + 1, 2 * nb + 1))
    model.fork(0, by_index)
    n, base_of = model.meta()
    assert [base_of[s] for s in by_index] == [0] * nb and [n[s] for s in by_index] == [Tctx % M] * nb
    model.set_state(by_copy, np.stack([model.store[0]] * nb))
    for s in by_copy:
        model.log[s] = [(a.copy(), kk.copy(), L.copy()) for a, kk, L in model.log[0]]
        model.table.n[s] = model.table.n[0]
    rows = list(range(1, nb + 1))  # same inputs for the i-th branch of each kind
    for t in range(Tctx, Tctx + Tq):
        oi = model.step(by_index, rs(q, t, rows), rs(k, t, rows), rs(v, t, rows), rs(g, t, rows), beta(t, rows))
        oc = model.step(by_copy, rs(q, t, rows), rs(k, t, rows), rs(v, t, rows), rs(g, t, rows), beta(t, rows))
        assert np.array_equal(oi, oc)
    # every branch merged at least once, so each now owns its base
    n, base_of = model.meta()
    assert [base_of[s] for s in by_index] == by_index
    # eager from the source's materialised state gives the same outputs
    for i, s in enumerate(by_index):
        sel = lambda x: x[Tctx:].reshape((Tq, -1, H) + x.shape[2:])[:, s].reshape((Tq, H) + x.shape[2:])
        ex = bonus if op == oracle.RWKV6 else sel(extra)
        o_e, S_e, _ = _eager(op, src_state, sel(q), sel(k), sel(v), sel(g), ex)
        assert _rel(model.read_state([s])[0], S_e) < 1e-12
    assert model.table.refs[0] == 0


# ---------------------------------------------------------------- P6 ---------
def test_p6_bookkeeping_trace_by_hand():
    t = oracle.SlotTableModel(4, 3)
    assert t.step([0, 1])[0] == oracle.OK
    assert t.snapshot()[0] == [1, 1, 0, 0]
    rc, plan = t.step([0])
    assert plan == [(0, 0, 1, False)] and t.n[0] == 2
    rc, plan = t.step([0, 1])
    assert plan == [(0, 0, 2, True), (1, 1, 1, False)] and t.n[:2] == [0, 2]
    assert t.fork(1, [2, 3]) == oracle.OK
    assert t.base_of == [0, 1, 1, 1] and t.n == [0, 2, 2, 2] and t.refs[1] == 2
    assert t.step([1]) == (oracle.EBUSY, [])          # frozen: branches index it
    assert t.set_state([1]) == oracle.EBUSY
    assert t.step([2, 2])[0] == oracle.EINVAL           # duplicate
    assert t.step([4])[0] == oracle.EINVAL              # out of range
    assert t.fork(2, [2]) == oracle.EINVAL              # src among dsts
    rc, plan = t.step([2, 3])                           # n 2 -> merge: privatise
    assert plan == [(2, 1, 2, True), (3, 1, 2, True)]
    assert t.base_of == [0, 1, 2, 3] and t.refs[1] == 0 and t.n == [0, 2, 0, 0]
    assert t.step([1]) == (oracle.OK, [(1, 1, 2, True)])  # unfrozen; n 2 -> merge
    assert t.step([3]) == (oracle.OK, [(3, 3, 0, False)])
    assert t.step_eager([0, 1]) == oracle.OK             # empty logs, own bases
    assert t.step_eager([3]) == oracle.EINVAL            # pending log entry


def test_p6_bookkeeping_invariants_random():
    random.seed(11)
    for M in (1, 2, 5):
        t = oracle.SlotTableModel(7, M)
        for _ in range(400):
            opk = random.choice(["step", "step", "fork", "set", "merge"])
            sl = random.sample(range(7), random.randint(1, 4))
            if opk == "step":
                t.step(sl)
            elif opk == "fork":
                t.fork(random.randrange(7), sl)
            elif opk == "set":
                t.set_state(sl)
            else:
                t.merge(sl)
            n, base_of, refs = t.snapshot()
            assert all(0 <= x < M for x in n)
            for s in range(7):
                b = base_of[s]
                assert base_of[b] == b                  # bases are roots
                assert refs[s] == sum(1 for x in range(7) if x != s and base_of[x] == s)
