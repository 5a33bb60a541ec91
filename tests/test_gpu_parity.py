"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bars: output max relative error <= 5e-3 with bf16 output (1e-4 with fp32
output), state max relative error <= 1e-4 (fp32 state), bookkeeping (log
lengths, base indices) bit-exact against the oracle's integer model, and
fork-by-index bit-identical to copy-then-run on the GPU.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (OUT_TOL_BF16, OUT_TOL_F32, STATE_TOL, gpu_run, make_case,
                         max_step_rel, oracle_run, rel_err)
from linear_attention_recurrent_gdn_gb300 import build
from linear_attention_recurrent_gdn_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

OPS = [gen.GDN, gen.KDA, gen.RWKV6]
STAGINGS = [0, 1]   # ReplayPrep fused as a warp role / as its own kernel


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()


def _flat_o(o):
    T, B, H, dv = o.shape
    return o.reshape(T, B * H, dv).numpy()


def _flat_S(S):
    B, H, dv, dk = S.shape
    return S.reshape(B * H, dv, dk).numpy()


# ------------------------------------------------------------------ config 0 --
@pytest.mark.parametrize("M", [8, 1])
def test_config0_gdn_full(M):
    """GDN decode, B=1, H=4, d=64, 64 tokens (config 0), every output and the
    state after every 8th token."""
    x, S0, _ = make_case(gen.GDN, 1, 4, 64, 64, seed=1000)
    snap = list(range(3, 64, 8))
    o_ref, S_ref, S_snap = oracle_run(gen.GDN, x, S0, None, snap=snap)
    for out_bf16, tol in ((True, OUT_TOL_BF16), (False, OUT_TOL_F32)):
        o, states, ctx = gpu_run(gen.GDN, x, S0, None, M, out_bf16=out_bf16, snap=snap)
        assert max_step_rel(_flat_o(o), o_ref) <= tol
        for i, t in enumerate(snap):
            assert rel_err(_flat_S(states[t]), S_snap[i]) <= STATE_TOL, t
        n, base_of = ctx.get_meta()
        assert list(n) == [64 % M] and list(base_of) == [0]


# ------------------------------------------------- all ops, sizes, merge intervals
@pytest.mark.parametrize("staging", STAGINGS)
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("M", [1, 3, 8, 9, 16, 17, 32])
def test_ops_small_ragged(op, d, M, staging):
    """B=3 slots x H=5 heads (15 slot-heads, several value tiles each), T = 2M+3
    tokens: two merges and a partial window; fp32 output, state at every step.
    M = 9 and 17 fill every entry slot of their coefficient bound (8, 16) on the
    merge step. M = 32 gives KDA at d=128 aux slots of 41.5 KB, which only the
    planner's fallback shapes fit with one-tile units."""
    B, H, T = 3, 5, 2 * M + 3
    x, S0, bonus = make_case(op, B, H, d, T, seed=17 + 3 * op + d + M)
    snap = list(range(T))
    o_ref, S_ref, S_snap = oracle_run(op, x, S0, bonus, snap=snap)
    o, states, ctx = gpu_run(op, x, S0, bonus, M, out_bf16=False, snap=snap, staging=staging)
    assert max_step_rel(_flat_o(o), o_ref) <= OUT_TOL_F32
    for t in snap:
        assert rel_err(_flat_S(states[t]), S_snap[t]) <= STATE_TOL, t
    n, base_of = ctx.get_meta()
    assert list(n) == [T % M] * B and list(base_of) == list(range(B))


@pytest.mark.parametrize("staging", STAGINGS)
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("M", [4, 16])
def test_ops_bf16_output_many_units(op, d, M, staging):
    """320 slot-heads (enough work units for whole-slot-head units, so d=128
    runs with prep warps), 20 tokens, bf16 output, compared on every
    slot-head. M=16 takes the log to 15 entries before its merge."""
    B, H, T = 40, 8, 20
    x, S0, bonus = make_case(op, B, H, d, T, seed=300 + op + d)
    o_ref, S_ref, _ = oracle_run(op, x, S0, bonus)
    o, _, ctx = gpu_run(op, x, S0, bonus, M, out_bf16=True, staging=staging)
    assert max_step_rel(_flat_o(o), o_ref) <= OUT_TOL_BF16
    S = ctx.read_state(list(range(B))).cpu()
    assert rel_err(_flat_S(S), S_ref) <= STATE_TOL


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("M", [16, 32])
def test_staggered_logs_in_one_launch(op, d, M):
    """Slots that joined at different tokens share every launch, so one launch
    carries rows from an empty log to a merge (its aux slots are sized for the
    longest log among them). Each slot's outputs (fp32) and final state match
    the oracle run over that slot's own tokens."""
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    H = 3
    lead = [0, 5, 11, 17, M - 3, M - 1]                 # tokens each slot runs before the last joins
    B, T2 = len(lead), M + 3
    Ttot = max(lead) + T2
    x, S0, bonus = make_case(op, B, H, d, Ttot, seed=980 + 7 * op + d + M)
    start = [max(lead) - L for L in lead]               # the global token at which slot s joins
    ctx = dl.DeltaLog(op, B, H, d, d, M, out_bf16=False)
    ctx.set_state(list(range(B)), S0.cuda())
    if bonus is not None:
        ctx.set_bonus(bonus.cuda())
    dev = {k_: (v_.cuda() if v_ is not None else None) for k_, v_ in x.items()}
    outs = {s: [] for s in range(B)}
    for t in range(Ttot):
        act = [s for s in range(B) if start[s] <= t]
        idx = torch.tensor(act, device="cuda")
        sel = lambda key: dev[key][t].index_select(0, idx).contiguous() if dev[key] is not None else None
        o = ctx.step(act, sel("q"), sel("k"), sel("v"), sel("g"), sel("beta")).cpu()
        for i, s in enumerate(act):
            outs[s].append(o[i])
    S_gpu = ctx.read_state(list(range(B))).cpu()
    for s in range(B):
        xs = {k_: (v_[start[s]:, s:s + 1] if v_ is not None else None) for k_, v_ in x.items()}
        o_ref, S_ref, _ = oracle_run(op, xs, S0[s:s + 1], bonus)
        o_s = torch.stack(outs[s]).reshape(len(outs[s]), H, d).numpy()
        assert max_step_rel(o_s, o_ref) <= OUT_TOL_F32, s
        assert rel_err(S_gpu[s].numpy(), S_ref) <= STATE_TOL, s
    n, _ = ctx.get_meta()
    assert list(n) == [(Ttot - start[s]) % M for s in range(B)]


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("d", [64, 128])
def test_extreme_decays_and_gates(op, d):
    """Degenerate and extreme gates inside merge windows: no decay (g = 0) next
    to decays of e^-30 a token (a window's cumulative log-decay reaches -450,
    far below fp32's range for e^Λ), β = 0 (the delta rule writes nothing) and
    β = 1, and zero value vectors. Outputs (fp32) and states match the oracle,
    with nothing infinite or NaN."""
    B, H, M = 3, 4, 16
    T = 2 * M + 5
    x, S0, bonus = make_case(op, B, H, d, T, seed=1200 + 5 * op + d)
    g = x["g"].clone()
    gen_ = torch.Generator().manual_seed(77 + op)
    pick = torch.randint(0, 3, g.shape, generator=gen_)
    g = torch.where(pick == 0, torch.zeros_like(g), torch.where(pick == 1, torch.full_like(g, -30.0), g))
    x["g"] = g.contiguous()
    if x["beta"] is not None:
        pb = torch.randint(0, 3, x["beta"].shape, generator=gen_)
        beta = torch.where(pb == 0, torch.zeros_like(x["beta"]),
                           torch.where(pb == 1, torch.ones_like(x["beta"]), x["beta"]))
        x["beta"] = beta.contiguous()
    v = x["v"].clone()
    v[3] = 0
    v[M - 1, 1] = 0
    x["v"] = v.contiguous()
    o_ref, S_ref, _ = oracle_run(op, x, S0, bonus)
    o, states, ctx = gpu_run(op, x, S0, bonus, M, out_bf16=False, snap=(T - 1,))
    assert torch.isfinite(o).all()
    assert max_step_rel(_flat_o(o), o_ref) <= OUT_TOL_F32
    assert rel_err(_flat_S(states[T - 1]), S_ref) <= STATE_TOL


# ------------------------------------------------------------------- eager ----
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("d", [64, 128])
def test_eager_kernel(op, d):
    B, H, T = 4, 3, 9
    x, S0, bonus = make_case(op, B, H, d, T, seed=50 + op + d)
    o_ref, S_ref, _ = oracle_run(op, x, S0, bonus)
    o, _, ctx = gpu_run(op, x, S0, bonus, 1, out_bf16=False, eager=True)
    assert max_step_rel(_flat_o(o), o_ref) <= OUT_TOL_F32
    S = ctx.read_state(list(range(B))).cpu()
    assert rel_err(_flat_S(S), S_ref) <= STATE_TOL
    # DeltaLog with M = 1 computes the same rounding-level result
    o1, _, ctx1 = gpu_run(op, x, S0, bonus, 1, out_bf16=False)
    assert rel_err(o1.numpy(), o.numpy()) <= 1e-5


def test_eager_requires_empty_log():
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    x, S0, _ = make_case(gen.GDN, 2, 2, 64, 1, seed=5)
    ctx = dl.DeltaLog(gen.GDN, 2, 2, 64, 64, 4)
    ctx.set_state([0, 1], S0.cuda())
    dev = {k: v.cuda() for k, v in x.items()}
    ctx.step([0, 1], dev["q"][0], dev["k"][0], dev["v"][0], dev["g"][0], dev["beta"][0])
    with pytest.raises(dl.DeltaLogError) as e:
        ctx.step_eager([0], dev["q"][0][:1], dev["k"][0][:1], dev["v"][0][:1], dev["g"][0][:1],
                       dev["beta"][0][:1])
    assert e.value.status == dl.EINVAL


# --------------------------------------------------------- merge / read-state --
@pytest.mark.parametrize("op", OPS)
def test_forced_merge_mid_window(op):
    B, H, d, M, T = 2, 3, 64, 8, 13
    x, S0, bonus = make_case(op, B, H, d, T, seed=70 + op)
    o_ref, S_ref, _ = oracle_run(op, x, S0, bonus)
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    ctx = dl.DeltaLog(op, B, H, d, d, M, out_bf16=False)
    ctx.set_state([0, 1], S0.cuda())
    if bonus is not None:
        ctx.set_bonus(bonus.cuda())
    dev = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    outs = []
    for t in range(T):
        if t in (5, 6):
            ctx.merge([1] if t == 5 else [0, 1])     # forced merges on partial logs
        b = dev["beta"][t] if dev["beta"] is not None else None
        outs.append(ctx.step([0, 1], dev["q"][t], dev["k"][t], dev["v"][t], dev["g"][t], b).float())
    o = torch.stack(outs).cpu()
    assert max_step_rel(_flat_o(o), o_ref) <= OUT_TOL_F32
    S = ctx.read_state([0, 1]).cpu()
    assert rel_err(_flat_S(S), S_ref) <= STATE_TOL
    n, _ = ctx.get_meta()
    # slot 0: merged at t=6 (n=0), then 7 steps -> 7; slot 1: merged at 6 -> 7
    assert list(n) == [7 % M, 7 % M]


# ------------------------------------------------------------------- fork -----
@pytest.mark.parametrize("staging", STAGINGS)
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("ctx_len", [16, 18])
def test_fork_by_index(op, ctx_len, staging):
    """2 requests build a base over ctx_len tokens (M=8: 16 ends on a merge, 18
    leaves 2 log entries), each forks 3 branches by index; branches run ragged
    lengths; outputs and states match the oracle run from the request's state,
    bookkeeping matches the oracle model at every step."""
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    H, d, M, R, NB = 3, 64, 8, 2, 3
    lens = [5, 12, 20, 9, 17, 3]       # per branch (request-major)
    Tq = max(lens)
    S = R + R * NB
    xc, S0, bonus = make_case(op, R, H, d, ctx_len, seed=90 + op)
    xq, _, _ = make_case(op, R * NB, H, d, Tq, seed=91 + op)
    ctx = dl.DeltaLog(op, S, H, d, d, M, out_bf16=False, staging=staging)
    model = oracle.SlotTableModel(S, M)
    ctx.set_state(list(range(R)), S0.cuda())
    model.set_state(list(range(R)))
    if bonus is not None:
        ctx.set_bonus(bonus.cuda())
    dc = {k: (v.cuda() if v is not None else None) for k, v in xc.items()}
    for t in range(ctx_len):
        b = dc["beta"][t] if dc["beta"] is not None else None
        ctx.step(list(range(R)), dc["q"][t], dc["k"][t], dc["v"][t], dc["g"][t], b)
        model.step(list(range(R)))
    branches = [[R + r * NB + i for i in range(NB)] for r in range(R)]
    for r in range(R):
        ctx.fork(r, branches[r])
        assert model.fork(r, branches[r]) == oracle.OK
    with pytest.raises(dl.DeltaLogError) as e:   # a request indexed by branches is frozen
        ctx.step([0], dc["q"][0][:1], dc["k"][0][:1], dc["v"][0][:1], dc["g"][0][:1],
                 dc["beta"][0][:1] if dc["beta"] is not None else None)
    assert e.value.status == dl.EBUSY
    flat = [s for bl in branches for s in bl]
    dq = {k: (v.cuda() if v is not None else None) for k, v in xq.items()}
    outs = {s: [] for s in flat}
    for t in range(Tq):
        act = [i for i, s in enumerate(flat) if lens[i] > t]
        sl = [flat[i] for i in act]
        idx = torch.tensor(act, device="cuda")
        sel = lambda key: dq[key][t].index_select(0, idx).contiguous() if dq[key] is not None else None
        o = ctx.step(sl, sel("q"), sel("k"), sel("v"), sel("g"), sel("beta"))
        model.step(sl)
        for j, s in enumerate(sl):
            outs[s].append(o[j].float().cpu())
        n, base_of = ctx.get_meta()
        mn, mb, _ = model.snapshot()
        assert list(n) == mn and list(base_of) == mb, t
    final = ctx.read_state(flat).cpu()
    for i, s in enumerate(flat):
        r = i // NB
        L = lens[i]
        # oracle: the request's context tokens followed by this branch's tokens, from S_0
        sub = {k: (torch.cat([xc[k][:, r:r + 1], xq[k][:L, i:i + 1]]) if xq[k] is not None else None)
               for k in xq}
        o_ref, S_ref, _ = oracle_run(op, sub, S0[r:r + 1], bonus)
        o = torch.stack(outs[s]).numpy()                     # [L, H, dv]
        assert max_step_rel(o, o_ref[ctx_len:]) <= OUT_TOL_F32, s
        assert rel_err(final[i].numpy(), S_ref) <= STATE_TOL, s


@pytest.mark.parametrize("op", OPS)
def test_fork_equals_copy_then_run_bitwise(op):
    """Branches that index a base (n = 0 at the fork) and branches that start
    from a copy of that base run the same kernels on the same bits."""
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    H, d, M, T = 2, 128, 4, 11
    xc, S0, bonus = make_case(op, 1, H, d, 8, seed=120 + op)
    xq, _, _ = make_case(op, 2, H, d, T, seed=121 + op)
    ctx = dl.DeltaLog(op, 5, H, d, d, M)
    ctx.set_state([0], S0.cuda())
    if bonus is not None:
        ctx.set_bonus(bonus.cuda())
    dc = {k: (v.cuda() if v is not None else None) for k, v in xc.items()}
    for t in range(8):   # 8 = 2 windows: the log is empty afterwards
        b = dc["beta"][t] if dc["beta"] is not None else None
        ctx.step([0], dc["q"][t], dc["k"][t], dc["v"][t], dc["g"][t], b)
    ctx.fork(0, [1, 2])
    base = ctx.read_state([0])
    ctx.set_state([3, 4], torch.cat([base, base]).contiguous())
    dq = {k: (v.cuda() if v is not None else None) for k, v in xq.items()}
    for t in range(T):
        cat = lambda key: torch.cat([dq[key][t], dq[key][t]]).contiguous() if dq[key] is not None else None
        o = ctx.step([1, 2, 3, 4], cat("q"), cat("k"), cat("v"), cat("g"), cat("beta"))
        assert torch.equal(o[:2], o[2:]), t
    S = ctx.read_state([1, 2, 3, 4])
    assert torch.equal(S[:2], S[2:])


# -------------------------------------------------------------- error paths --
def test_argument_errors():
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    ctx = dl.DeltaLog(gen.GDN, 4, 2, 64, 64, 4)
    x, S0, _ = make_case(gen.GDN, 2, 2, 64, 1, seed=3)
    dev = {k: v.cuda() for k, v in x.items()}
    args = (dev["q"][0], dev["k"][0], dev["v"][0], dev["g"][0], dev["beta"][0])
    for bad in ([0, 0], [0, 4], [-1, 1]):
        with pytest.raises(dl.DeltaLogError) as e:
            ctx.step(bad, *args)
        assert e.value.status == dl.EINVAL
    with pytest.raises(dl.DeltaLogError) as e:
        ctx.fork(1, [1, 2])
    assert e.value.status == dl.EINVAL
    # misaligned q (bulk-copied: needs 16 bytes), through the raw C entry point
    qb = torch.empty(2 * 2 * 64 + 8, dtype=torch.bfloat16, device="cuda")
    q_mis = qb[1:1 + 2 * 2 * 64].view(2, 2, 64)
    o = torch.empty(2, 2, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dl.DeltaLogError) as e:
        dl.dl_step(ctx.handle, [0, 1], q_mis, *args[1:], o)
    assert e.value.status == dl.EINVAL
    ob = torch.empty(2 * 2 * 64 + 8, dtype=torch.uint8, device="cuda")
    with pytest.raises(dl.DeltaLogError) as e:     # o must be aligned to its element size
        dl.dl_step(ctx.handle, [0, 1], *args, ob[1:])
    assert e.value.status == dl.EINVAL
    # the context is still usable and nothing was stepped
    n, _ = ctx.get_meta()
    assert list(n) == [0, 0, 0, 0]
    ctx.step([0, 1], *args)
    n, _ = ctx.get_meta()
    assert list(n) == [1, 1, 0, 0]
    # unsupported shapes are refused at creation
    for bad_cfg in (dict(d_k=96), dict(merge_interval=33), dict(d_v=64, d_k=128)):
        kw = dict(op=gen.GDN, num_slots=2, num_heads=2, d_k=64, d_v=None, merge_interval=4)
        kw.update(bad_cfg)
        with pytest.raises(dl.DeltaLogError) as e:
            dl.DeltaLog(**kw)
        assert e.value.status in (dl.EUNSUPPORTED, dl.EINVAL)


def test_rwkv6_requires_bonus():
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    ctx = dl.DeltaLog(gen.RWKV6, 2, 2, 64, 64, 4)
    x, S0, _ = make_case(gen.RWKV6, 2, 2, 64, 1, seed=3)
    dev = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    with pytest.raises(dl.DeltaLogError) as e:
        ctx.step([0, 1], dev["q"][0], dev["k"][0], dev["v"][0], dev["g"][0], None)
    assert e.value.status == dl.EINVAL


def test_allocation_failure_is_reported(monkeypatch):
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    monkeypatch.setenv("DL_TEST_FAIL_ALLOC", "3")
    with pytest.raises(dl.DeltaLogError) as e:
        dl.DeltaLog(gen.GDN, 4, 2, 64, 64, 4)
    assert e.value.status == dl.ENOMEM
    monkeypatch.delenv("DL_TEST_FAIL_ALLOC")
    dl.DeltaLog(gen.GDN, 4, 2, 64, 64, 4).close()


def test_step_host_matches_device_path():
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    B, H, d, T, M = 6, 4, 128, 10, 4
    x, S0, _ = make_case(gen.GDN, B, H, d, T, seed=11)
    o_dev, _, _ = gpu_run(gen.GDN, x, S0, None, M)
    ctx = dl.DeltaLog(gen.GDN, B, H, d, d, M)
    ctx.set_state(list(range(B)), S0.cuda())
    pin = {k: v.pin_memory() for k, v in x.items()}
    outs = [ctx.step_host(list(range(B)), pin["q"][t], pin["k"][t], pin["v"][t], pin["g"][t],
                          pin["beta"][t]).float() for t in range(T)]
    assert torch.equal(torch.stack(outs), o_dev)


@pytest.mark.parametrize("staging", STAGINGS)
@pytest.mark.parametrize("op", OPS)
def test_decode_host_matches_device_path(op, staging):
    """dl_decode_host (host buffers, copies overlapping the computation) gives
    the bits of dl_step on device buffers, over two merges and a partial window."""
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    B, H, d, M = 6, 4, 128 if op != gen.RWKV6 else 64, 4
    T = 2 * M + 3
    x, S0, bonus = make_case(op, B, H, d, T, seed=900 + op)
    o_dev, states, ref = gpu_run(op, x, S0, bonus, M, snap=(T - 1,), staging=staging)
    ctx = dl.DeltaLog(op, B, H, d, d, M, staging=staging)
    ctx.set_state(list(range(B)), S0.cuda())
    if bonus is not None:
        ctx.set_bonus(bonus.cuda())
    pin = {k_: (v_.contiguous().pin_memory() if v_ is not None else None) for k_, v_ in x.items()}
    o = ctx.decode_host(list(range(B)), pin["q"], pin["k"], pin["v"], pin["g"], pin["beta"])
    assert torch.equal(o.float(), o_dev)
    assert torch.equal(ctx.read_state(list(range(B))).cpu(), states[T - 1])
    assert list(ctx.get_meta()[0]) == [T % M] * B


@pytest.mark.parametrize("op", OPS)
def test_decode_host_wraps_the_staging_ring(op):
    """Enough token groups (eight tokens a group at this batch) that each of
    the four staging sets is reused twice, with a ragged last group: the
    outputs, the state and the log lengths are the bits of dl_step on device
    buffers."""
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    B, H, d, M = 6, 4, 128 if op != gen.RWKV6 else 64, 4
    T = 8 * 9 + 3
    x, S0, bonus = make_case(op, B, H, d, T, seed=960 + op)
    o_dev, states, ref = gpu_run(op, x, S0, bonus, M, snap=(T - 1,))
    ctx = dl.DeltaLog(op, B, H, d, d, M)
    ctx.set_state(list(range(B)), S0.cuda())
    if bonus is not None:
        ctx.set_bonus(bonus.cuda())
    pin = {k_: (v_.contiguous().pin_memory() if v_ is not None else None) for k_, v_ in x.items()}
    o = ctx.decode_host(list(range(B)), pin["q"], pin["k"], pin["v"], pin["g"], pin["beta"])
    assert torch.equal(o.float(), o_dev)
    assert torch.equal(ctx.read_state(list(range(B))).cpu(), states[T - 1])
    assert list(ctx.get_meta()[0]) == [T % M] * B


@pytest.mark.parametrize("out_bf16", [True, False])
@pytest.mark.parametrize("op", OPS)
def test_decode_host_whole_windows_bitwise(op, out_bf16):
    """Slots that start on their own bases with empty logs, and T a multiple of
    M, go through captured decode windows, one per staging set: nine windows
    wrap the four sets twice. A second batch captures new windows. A call of
    T = M + 3 (not whole windows), and the next call (its slots then start
    mid-window), take the per-token path. Every output, the states and the log
    lengths are the bits of dl_step on device buffers."""
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    B, H, M = 6, 4, 4
    d = 64 if op == gen.RWKV6 else 128
    calls = [(list(range(B)), 0, 9 * M),        # whole windows, sets wrap
             ([0, 2, 4], 9 * M, 11 * M),        # another batch: new windows
             ([1, 3, 5], 9 * M, 10 * M + 3),    # not whole windows: per token
             ([1, 3, 5], 10 * M + 3, 12 * M + 3)]   # mid-window start: per token
    Ttot = max(c[2] for c in calls)
    x, S0, bonus = make_case(op, B, H, d, Ttot, seed=970 + op)
    ref = dl.DeltaLog(op, B, H, d, d, M, out_bf16=out_bf16)
    hst = dl.DeltaLog(op, B, H, d, d, M, out_bf16=out_bf16)
    for c in (ref, hst):
        c.set_state(list(range(B)), S0.cuda())
        if bonus is not None:
            c.set_bonus(bonus.cuda())
    dev = {k_: (v_.cuda() if v_ is not None else None) for k_, v_ in x.items()}
    for slots, t0, t1 in calls:
        idx = torch.tensor(slots)
        outs = []
        for t in range(t0, t1):
            sel = lambda key: (dev[key][t].index_select(0, idx.cuda()).contiguous()
                               if dev[key] is not None else None)
            outs.append(ref.step(slots, sel("q"), sel("k"), sel("v"), sel("g"), sel("beta")))
        o_ref = torch.stack(outs).cpu()
        pin = {k_: (v_[t0:t1].index_select(1, idx).contiguous().pin_memory() if v_ is not None else None)
               for k_, v_ in x.items()}
        o = hst.decode_host(slots, pin["q"], pin["k"], pin["v"], pin["g"], pin["beta"])
        assert torch.equal(o, o_ref), (slots, t0, t1)
    assert torch.equal(hst.read_state(list(range(B))), ref.read_state(list(range(B))))
    assert [list(m) for m in hst.get_meta()] == [list(m) for m in ref.get_meta()]


def test_decode_host_frozen_slot_is_refused():
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    B, H, d, M, T = 3, 2, 64, 4, 5
    x, S0, _ = make_case(gen.GDN, B, H, d, T, seed=950)
    ctx = dl.DeltaLog(gen.GDN, B + 1, H, d, d, M)
    ctx.set_state(list(range(B)), S0.cuda())
    ctx.fork(0, [B])                       # slot 0 is now a fork source: frozen
    pin = {k_: (v_.contiguous().pin_memory() if v_ is not None else None) for k_, v_ in x.items()}
    with pytest.raises(dl.DeltaLogError) as e:
        ctx.decode_host([0, 1, 2], pin["q"], pin["k"], pin["v"], pin["g"], pin["beta"])
    assert e.value.status == dl.EBUSY
    o = ctx.decode_host([1, 2], pin["q"][:, 1:].contiguous(), pin["k"][:, 1:].contiguous(),
                        pin["v"][:, 1:].contiguous(), pin["g"][:, 1:].contiguous(),
                        pin["beta"][:, 1:].contiguous())
    assert o.shape == (T, 2, H, d) and torch.isfinite(o.float()).all()
