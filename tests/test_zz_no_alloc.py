"""dl_step_noalloc: the decode step for callers that cannot let the library
allocate device memory (engines that reserve the GPU's memory for their own
pools at start-up, code whose buffers must all come from its own allocator,
loops that cannot take the synchronisation an allocation may cause).

The caller owns the state, the logs and the device slot table (plain torch
tensors here, laid out as dl_create lays them out) and plans each step with a
host slot table; the library keeps only the per-step coefficient scratch and a
status word, in static device arrays.  Checked here:
  * against the fp64 oracle, for every operator, d in {64, 128} and
    M in {4, 16, 32} over 2M+3 tokens, so that the replay runs over full logs
    and two merges happen: every output, the dense base right after each merge,
    and the device slot table;
  * a fork (a source's base indexed by two branches, the log copied by the
    caller), against eager runs from the source's state;
  * two calls in a row against dl_step on a context;
  * the status word: a clean run reads back 0; a test-only stall makes one
    bounded wait run out, dl_noalloc_sync reports it once and clears it, and
    the next steps are correct again.
This file is collected last on purpose, and it depends on nothing an earlier
test left behind.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import OUT_TOL_BF16, STATE_TOL, make_case, oracle_run, rel_err
from linear_attention_recurrent_gdn_gb300 import build
from linear_attention_recurrent_gdn_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()


def _caller_buffers(op, B, H, d, M, S0, bonus):
    Mcap = max(M - 1, 1)
    lw = (Mcap,) if op == gen.GDN else (Mcap, d)
    return {
        "Sbar": S0.clone().contiguous(),
        "alog": torch.zeros(B, H, Mcap, d, device="cuda",
                            dtype=torch.bfloat16 if op == gen.RWKV6 else torch.float32),
        "klog": torch.zeros(B, H, Mcap, d, device="cuda", dtype=torch.bfloat16),
        "Llog": torch.zeros((B, H) + lw, device="cuda", dtype=torch.float32),
        "n_log": torch.zeros(B, device="cuda", dtype=torch.int32),
        "base_of": torch.arange(B, device="cuda", dtype=torch.int32),
        "bonus": bonus,
    }


def _step(dl, cfg, buf, table, slots, x, t, rows=None, stream=None):
    """One token through dl_step_noalloc for `slots`; row i of the inputs is rows[i]."""
    rows = list(range(len(slots))) if rows is None else rows
    rc, plan = table.step(slots)
    assert rc == dl.OK
    pick = lambda key: x[key][t][rows].contiguous() if x[key] is not None else None
    o = torch.empty((len(slots),) + tuple(x["v"].shape[2:]), device="cuda", dtype=torch.bfloat16)
    dl.dl_step_noalloc(cfg, buf, plan, pick("q"), pick("k"), pick("v"), pick("g"), pick("beta"),
                       o, stream)
    return o


@pytest.mark.parametrize("M", [4, 16, 32])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("op", [gen.GDN, gen.KDA, gen.RWKV6])
def test_noalloc_matches_oracle(op, d, M):
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    B, H = 3, 2
    T = 2 * M + 3
    x, S0, bonus = make_case(op, B, H, d, T, seed=900 + 7 * op + M + d, device="cpu")
    o_ref, _, snaps = oracle_run(op, x, S0, bonus, snap=[M - 1, 2 * M - 1])
    xd = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    buf = _caller_buffers(op, B, H, d, M, S0.cuda(), bonus.cuda() if bonus is not None else None)
    table = dl.SlotTable(B, M)
    cfg = dl.dl_config(op, B, H, d, d, M, 1, 1.0)
    slots = list(range(B))
    outs, merged = [], {}
    for t in range(T):
        outs.append(_step(dl, cfg, buf, table, slots, xd, t).float())
        if t in (M - 1, 2 * M - 1):
            merged[t] = buf["Sbar"].clone()
    assert dl.dl_noalloc_sync() == (dl.OK, 0, "")
    o = torch.stack(outs).cpu().numpy().reshape(T, B * H, d)
    for t in range(T):
        assert rel_err(o[t], o_ref[t]) <= OUT_TOL_BF16, t
    for i, t in enumerate((M - 1, 2 * M - 1)):   # the base is the state right after a merge
        assert rel_err(merged[t].cpu().numpy().reshape(B * H, d, d), snaps[i]) <= STATE_TOL, t
    n_tab, b_tab = table.get()[:2]
    assert list(buf["n_log"].cpu().numpy()) == list(n_tab) == [T % M] * B
    assert list(buf["base_of"].cpu().numpy()) == list(b_tab) == slots


@pytest.mark.parametrize("op", [gen.GDN, gen.KDA, gen.RWKV6])
def test_noalloc_fork_by_index_matches_oracle(op):
    """Slot 0 decodes a context and ends mid-window; slots 1 and 2 fork from it
    (base indexed, log copied by the caller, as dl_fork does on a context);
    every branch output and each branch's first private base match eager runs
    from the source's state, and the source's base stays untouched."""
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    B, H, d, M, Tctx, Tq = 3, 2, 64, 8, 11, 12
    x, S0, bonus = make_case(op, B, H, d, Tctx + Tq, seed=950 + op, device="cpu")
    xd = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    buf = _caller_buffers(op, B, H, d, M, S0.cuda(), bonus.cuda() if bonus is not None else None)
    table = dl.SlotTable(B, M)
    cfg = dl.dl_config(op, B, H, d, d, M, 1, 1.0)
    for t in range(Tctx):
        _step(dl, cfg, buf, table, [0], xd, t, rows=[0])
    ctx_x = {k: (v[:Tctx, :1] if v is not None else None) for k, v in x.items()}
    _, S_src, _ = oracle_run(op, ctx_x, S0[:1], bonus)
    base0 = buf["Sbar"][0].clone()
    assert table.fork(0, [1, 2]) == dl.OK
    n_tab, b_tab = table.get()[:2]
    for s in (1, 2):   # the device side of the fork, done by the caller: log rows and table
        for key in ("alog", "klog", "Llog"):
            buf[key][s].copy_(buf[key][0])
    buf["n_log"].copy_(torch.tensor(n_tab, dtype=torch.int32))
    buf["base_of"].copy_(torch.tensor(b_tab, dtype=torch.int32))
    outs = []
    for t in range(Tctx, Tctx + Tq):
        outs.append(_step(dl, cfg, buf, table, [1, 2], xd, t, rows=[1, 2]).float())
        assert torch.equal(buf["Sbar"][0], base0), t
    assert dl.dl_noalloc_sync() == (dl.OK, 0, "")
    o = torch.stack(outs).cpu().numpy()
    S_src = torch.from_numpy(S_src).reshape(1, H, d, d).float()
    for i, s in enumerate((1, 2)):
        bx = {k: (v[Tctx:, s:s + 1] if v is not None else None) for k, v in x.items()}
        o_e, _, snap = oracle_run(op, bx, S_src, bonus, snap=[M - Tctx % M - 1])
        assert rel_err(o[:, i].reshape(Tq, H, d), o_e.reshape(Tq, H, d)) <= OUT_TOL_BF16, s
        # the branch's first merge wrote its private base
        assert rel_err(buf["Sbar"][s].cpu().numpy(), snap[0].reshape(H, d, d)) <= STATE_TOL
    n_tab, b_tab = table.get()[:2]
    assert list(buf["n_log"].cpu().numpy()) == list(n_tab)
    assert list(buf["base_of"].cpu().numpy()) == list(b_tab) == [0, 1, 2]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("op", [gen.GDN, gen.KDA, gen.RWKV6])
def test_noalloc_step_matches_dl_step_two_calls(op, d):
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    B, H, M, T = 5, 4, 2, 2
    x, S0, bonus = make_case(op, B, H, d, T, seed=800 + op + d, device="cuda")
    slots = list(range(B))
    ref = dl.DeltaLog(op, B, H, d, d, M)
    ref.set_state(slots, S0)
    if bonus is not None:
        ref.set_bonus(bonus)
    buf = _caller_buffers(op, B, H, d, M, S0, bonus)
    table = dl.SlotTable(B, M)
    cfg = dl.dl_config(op, B, H, d, d, M, 1, 1.0)
    stream = torch.cuda.current_stream().cuda_stream
    for t in range(T):
        beta = x["beta"][t] if x["beta"] is not None else None
        o_ref = ref.step(slots, x["q"][t], x["k"][t], x["v"][t], x["g"][t], beta)
        o = _step(dl, cfg, buf, table, slots, x, t, stream=stream)
        assert rel_err(o.float().cpu().numpy(), o_ref.float().cpu().numpy()) <= OUT_TOL_BF16, t
    S_ref = ref.read_state(slots)
    assert dl.dl_noalloc_sync(stream) == (dl.OK, 0, "")
    assert rel_err(buf["Sbar"].cpu().numpy(), S_ref.cpu().numpy()) <= STATE_TOL
    n_ref, b_ref = ref.get_meta()
    assert list(buf["n_log"].cpu().numpy()) == list(n_ref)
    assert list(buf["base_of"].cpu().numpy()) == list(b_ref)
    ref.close()


def test_noalloc_device_error_is_reported_once(monkeypatch):
    """DL_TEST_STALL makes one consumer warp wait on a barrier nothing arrives
    on; with a 50 ms limit the wait runs out, the kernels take their error exit
    and the code lands in the static status word.  No fault is involved."""
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    op, B, H, d, M, T = gen.GDN, 4, 4, 128, 4, 6
    x, S0, bonus = make_case(op, B, H, d, T, seed=990, device="cpu")
    xd = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    buf = _caller_buffers(op, B, H, d, M, S0.cuda(), None)
    table = dl.SlotTable(B, M)
    cfg = dl.dl_config(op, B, H, d, d, M, 1, 1.0)
    slots = list(range(B))
    assert dl.dl_noalloc_sync()[0] == dl.OK          # nothing pending from earlier calls
    monkeypatch.setenv("DL_TEST_WAIT_MS", "50")
    monkeypatch.setenv("DL_TEST_STALL", "1")
    _step(dl, cfg, buf, table, slots, xd, 0)
    monkeypatch.delenv("DL_TEST_STALL")
    monkeypatch.delenv("DL_TEST_WAIT_MS")
    rc, code, msg = dl.dl_noalloc_sync()
    assert rc == dl.EDEVICE and code == dl.DEV_TEST_STALL, (rc, code, msg)
    assert "status %d" % dl.DEV_TEST_STALL in msg
    assert dl.dl_noalloc_sync() == (dl.OK, 0, "")  # reported once, then cleared
    # the failed token left garbage: start again from S0 and check parity
    buf = _caller_buffers(op, B, H, d, M, S0.cuda(), None)
    table = dl.SlotTable(B, M)
    o_ref, _, _ = oracle_run(op, x, S0, bonus)
    outs = [_step(dl, cfg, buf, table, slots, xd, t).float() for t in range(T)]
    assert dl.dl_noalloc_sync() == (dl.OK, 0, "")
    o = torch.stack(outs).cpu().numpy().reshape(T, B * H, d)
    assert max(rel_err(o[t], o_ref[t]) for t in range(T)) <= OUT_TOL_BF16


def test_noalloc_rejects_steps_beyond_the_static_scratch():
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    op, B, H, d, M = gen.KDA, 1024, 4, 128, 32          # needs 1024*4*4552 floats > 4 Mi
    cfg = dl.dl_config(op, B, H, d, d, M, 1, 1.0)
    t = lambda *s, dt=torch.float32: torch.zeros(*s, device="cuda", dtype=dt)
    buf = {"Sbar": t(4), "alog": t(4), "klog": t(8, dt=torch.bfloat16), "Llog": t(4),
           "n_log": t(4, dt=torch.int32), "base_of": t(4, dt=torch.int32), "bonus": None}
    plan = np.zeros((B, 4), np.int32)
    plan[:, 0] = plan[:, 1] = np.arange(B)
    x = t(16)
    with pytest.raises(dl.DeltaLogError) as e:
        dl.dl_step_noalloc(cfg, buf, plan, x, x, x, x, x, x)
    assert e.value.status == dl.EINVAL
    assert "DL_NOALLOC_SCRATCH_FLOATS" in str(e.value)
