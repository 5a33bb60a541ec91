"""GPU checks of properties beyond element-wise parity.

* Batch invariance (Flide page, fourth step: a batch-invariant mode fixes the
  summation order and per-question boundaries so that load changes do not
  change bits): every slot-head's arithmetic here is independent of the batch
  it runs in — the same reduction order whatever the batch size, the value-tile
  grouping or the launch chunking — so a slot stepped alone and the same slot
  stepped inside a large batch give bit-identical outputs and states.
* Prefix checkpoints (Flide page, fourth step: resume from a checkpoint saved
  at a matching prefix): a restored slot continues bit for bit as the saved
  slot, also in another context, and both match the oracle.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import OUT_TOL_F32, STATE_TOL, make_case, max_step_rel, oracle_run, rel_err
from linear_attention_recurrent_gdn_gb300 import build
from linear_attention_recurrent_gdn_gb300 import inputs as gen

pytestmark = pytest.mark.gpu
OPS = [gen.GDN, gen.KDA, gen.RWKV6]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("M", [4, 16, 32])
def test_batch_invariance_bitwise(op, d, M):
    """A slot stepped alone (one-tile units) gives the bits it gets inside a
    1280 slot-head batch (whole-slot-head units: at d = 64 both tiles in one
    stage, RWKV6's append steps through the two-tile pass; at d = 128 prep
    warps, with split waits for per-key logs of up to 32 entries), over two
    merges, for each log-entry bound (8, 16, 32).  Outputs in fp32, so that a
    change of summation order cannot hide behind bf16 rounding."""
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    B, H, T = 320, 4, 2 * M + 1                # 1280 slot-heads: whole-slot-head units
    x, S0, bonus = make_case(op, B, H, d, T, seed=400 + op, device="cuda")
    probe = [0, 77, 319]
    big = dl.DeltaLog(op, B, H, d, d, M, out_bf16=False)
    big.set_state(list(range(B)), S0)
    small = dl.DeltaLog(op, B, H, d, d, M, out_bf16=False)   # same slots, stepped one at a time
    small.set_state(list(range(B)), S0)
    if bonus is not None:
        big.set_bonus(bonus)
        small.set_bonus(bonus)
    for t in range(T):
        b = x["beta"][t] if x["beta"] is not None else None
        o_big = big.step(list(range(B)), x["q"][t], x["k"][t], x["v"][t], x["g"][t], b)
        for s in probe:
            sl = slice(s, s + 1)
            o_one = small.step([s], x["q"][t][sl], x["k"][t][sl], x["v"][t][sl], x["g"][t][sl],
                               b[sl] if b is not None else None)
            assert torch.equal(o_one[0], o_big[s]), (t, s)
    assert torch.equal(big.read_state(probe), small.read_state(probe))


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("t_save", [8, 11])
def test_checkpoint_resume_bitwise(op, t_save):
    """Save mid-window (t_save=11, M=8: 3 log entries) and on a window edge."""
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    B, H, d, M, T = 2, 3, 64, 8, 25
    x, S0, bonus = make_case(op, B, H, d, T, seed=500 + op)
    dev = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    ctx = dl.DeltaLog(op, 4, H, d, d, M, out_bf16=False)
    other = dl.DeltaLog(op, 3, H, d, d, M, out_bf16=False)
    ctx.set_state([0, 1], S0.cuda())
    for c in (ctx, other):
        if bonus is not None:
            c.set_bonus(bonus.cuda())
    beta = lambda t, sl: dev["beta"][t][sl] if dev["beta"] is not None else None
    outs = []
    for t in range(T):
        if t == t_save:
            buf = ctx.checkpoint_save([1])
            ctx.checkpoint_load([3], buf)       # same context, another slot
            other.checkpoint_load([2], buf)     # another context
            n, base_of = ctx.get_meta()
            assert n[3] == t_save % M and base_of[3] == 3
        outs.append(ctx.step([0, 1], dev["q"][t], dev["k"][t], dev["v"][t], dev["g"][t],
                             beta(t, slice(0, 2))).float())
        if t >= t_save:
            sl = slice(1, 2)
            o3 = ctx.step([3], dev["q"][t][sl], dev["k"][t][sl], dev["v"][t][sl],
                          dev["g"][t][sl], beta(t, sl))
            o2 = other.step([2], dev["q"][t][sl], dev["k"][t][sl], dev["v"][t][sl],
                            dev["g"][t][sl], beta(t, sl))
            assert torch.equal(o3[0], outs[-1][1]) and torch.equal(o2[0], outs[-1][1]), t
    assert torch.equal(ctx.read_state([1])[0], ctx.read_state([3])[0])
    assert torch.equal(ctx.read_state([1])[0], other.read_state([2])[0])
    o_ref, S_ref, _ = oracle_run(op, x, S0, bonus)
    o = torch.stack(outs).cpu().reshape(T, B * H, d).numpy()
    assert max_step_rel(o, o_ref) <= OUT_TOL_F32
    assert rel_err(ctx.read_state([0, 1]).cpu().reshape(B * H, d, d).numpy(), S_ref) <= STATE_TOL


@pytest.mark.parametrize("op", OPS)
def test_checkpoint_many_slots_with_fork_branch(op):
    """One save of three slots, one of them a fork branch that still reads its
    source's base and holds a log entry of its own, restored under other slot
    ids in another context: both then step bit for bit alike. M=3 leaves GDN's
    log-decay rows at 12 bytes a head."""
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    H, d, M, T0, T1 = 5, 128, 3, 4, 5
    T = T0 + 1 + T1
    x, S0, bonus = make_case(op, 3, H, d, T, seed=520 + op, device="cuda")
    ctx = dl.DeltaLog(op, 6, H, d, d, M, out_bf16=False)
    other = dl.DeltaLog(op, 4, H, d, d, M, out_bf16=False)
    ctx.set_state([0, 1, 2], S0)
    for c in (ctx, other):
        if bonus is not None:
            c.set_bonus(bonus)
    beta = lambda t: x["beta"][t] if x["beta"] is not None else None
    for t in range(T0):
        ctx.step([0, 1, 2], x["q"][t], x["k"][t], x["v"][t], x["g"][t], beta(t))
    ctx.fork(0, [3])
    ctx.step([1, 2, 3], x["q"][T0], x["k"][T0], x["v"][T0], x["g"][T0], beta(T0))
    n, base_of = ctx.get_meta()
    assert base_of[3] == 0 and n[3] == T0 % M + 1     # still on the source's base
    buf = ctx.checkpoint_save([1, 3, 2])
    other.checkpoint_load([0, 1, 2], buf)
    n2, base2 = other.get_meta()
    assert list(n2[:3]) == [n[1], n[3], n[2]] and list(base2[:3]) == [0, 1, 2]
    for t in range(T0 + 1, T):
        oa = ctx.step([1, 3, 2], x["q"][t], x["k"][t], x["v"][t], x["g"][t], beta(t))
        ob = other.step([0, 1, 2], x["q"][t], x["k"][t], x["v"][t], x["g"][t], beta(t))
        assert torch.equal(oa, ob), t
    assert torch.equal(ctx.read_state([1, 3, 2]), other.read_state([0, 1, 2]))


@pytest.mark.parametrize("op", OPS)
def test_graph_window_matches_stepping_bitwise(op):
    """A captured merge window replayed 3 times gives the bits of 3*M plain
    steps; the inputs are refilled between launches."""
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    B, H, d, M, W = 8, 4, 64, 4, 3
    T = M * W
    x, S0, bonus = make_case(op, B, H, d, T, seed=600 + op, device="cuda")
    a = dl.DeltaLog(op, B, H, d, d, M)
    b = dl.DeltaLog(op, B, H, d, d, M)
    for c in (a, b):
        c.set_state(list(range(B)), S0)
        if bonus is not None:
            c.set_bonus(bonus)
    ref = []
    for t in range(T):
        beta = x["beta"][t] if x["beta"] is not None else None
        ref.append(a.step(list(range(B)), x["q"][t], x["k"][t], x["v"][t], x["g"][t], beta).clone())
    buf = {k: (v[:M].clone() if v is not None else None) for k, v in x.items()}
    win = b.window(list(range(B)), buf["q"], buf["k"], buf["v"], buf["g"], buf["beta"])
    for w in range(W):
        for k_, v_ in x.items():
            if v_ is not None:
                buf[k_].copy_(v_[w * M:(w + 1) * M])
        out = win.launch()
        for j in range(M):
            assert torch.equal(out[j], ref[w * M + j]), (w, j)
    assert torch.equal(a.read_state(list(range(B))), b.read_state(list(range(B))))
    na, ba = a.get_meta()
    nb, bb = b.get_meta()
    assert list(na) == list(nb) and list(ba) == list(bb)
    # a slot with a pending log cannot enter a window
    sl = slice(0, 1)
    beta = x["beta"][0][sl] if x["beta"] is not None else None
    b.step([0], x["q"][0][sl], x["k"][0][sl], x["v"][0][sl], x["g"][0][sl], beta)
    with pytest.raises(dl.DeltaLogError) as e:
        win.launch()
    assert e.value.status == dl.EINVAL
    win.close()


@pytest.mark.parametrize("op,B,H,d", [(gen.GDN, 96, 32, 128), (gen.KDA, 64, 32, 128),
                                      (gen.RWKV6, 128, 40, 64)])
def test_graph_window_many_units_bitwise(op, B, H, d):
    """Windows at a size where every CTA streams many work units: from the
    second token of a window on, each step launches as a programmatic
    dependent of the previous one and streams dense-base tiles before it waits
    for it.  Two windows back to back must give the bits of plain stepping."""
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    M, W = 8, 2
    T = M * W
    x, S0, bonus = make_case(op, B, H, d, T, seed=650 + op, device="cuda")
    slots = list(range(B))
    a = dl.DeltaLog(op, B, H, d, d, M)
    b = dl.DeltaLog(op, B, H, d, d, M)
    for c in (a, b):
        c.set_state(slots, S0)
        if bonus is not None:
            c.set_bonus(bonus)
    ref = torch.empty((T, B, H, d), dtype=torch.bfloat16, device="cuda")
    for t in range(T):
        beta = x["beta"][t] if x["beta"] is not None else None
        a.step(slots, x["q"][t], x["k"][t], x["v"][t], x["g"][t], beta, ref[t])
    out = torch.empty_like(ref)
    sl = lambda key, j: x[key][j * M:(j + 1) * M] if x[key] is not None else None
    wins = [b.window(slots, sl("q", j), sl("k", j), sl("v", j), sl("g", j), sl("beta", j),
                     out[j * M:(j + 1) * M]) for j in range(W)]
    for w in wins:
        w.launch()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert torch.equal(a.read_state(slots), b.read_state(slots))
    for w in wins:
        w.close()


@pytest.mark.parametrize("op,d", [(gen.GDN, 128), (gen.KDA, 128), (gen.RWKV6, 64)])
def test_ragged_window_matches_stepping_bitwise(op, d):
    """A ragged window (device-resident per-token slot lists and counts, tail
    padding) replayed over changing active sets gives the bits of plain steps
    with the same rows: random subsets per token, an empty token, a full token,
    and branches that index a fork source's base with non-empty logs."""
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    import random
    S_, H, M, W = 10, 4, 4, 3
    T = M * W
    n_max = S_ - 1                      # slot 0 becomes a fork source (frozen)
    x, S0, bonus = make_case(op, n_max, H, d, T + 2, seed=660 + op, device="cuda")
    _, S0a, _ = make_case(op, S_, H, d, 1, seed=661 + op, device="cuda")
    ctxs = [dl.DeltaLog(op, S_, H, d, d, M) for _ in range(2)]
    for c in ctxs:
        c.set_state(list(range(S_)), S0a)
        if bonus is not None:
            c.set_bonus(bonus)
        for t in (T, T + 1):           # two tokens on slot 0, then fork it into 8 and 9
            sl = slice(0, 1)
            b = x["beta"][t][sl] if x["beta"] is not None else None
            c.step([0], x["q"][t][sl], x["k"][t][sl], x["v"][t][sl], x["g"][t][sl], b)
        c.fork(0, [8, 9])
    a, r = ctxs
    rng = random.Random(5 + op)
    lists = []
    for t in range(T):
        if t == 2:
            lst = []
        elif t == 5:
            lst = list(range(1, S_))
        else:
            lst = rng.sample(range(1, S_), rng.randint(1, n_max))
        lists.append(lst)
    ref = torch.zeros((T, n_max, H, d), dtype=torch.bfloat16, device="cuda")
    for t, lst in enumerate(lists):
        k_ = len(lst)
        if k_:
            b = x["beta"][t][:k_] if x["beta"] is not None else None
            a.step(lst, x["q"][t][:k_], x["k"][t][:k_], x["v"][t][:k_], x["g"][t][:k_], b,
                   ref[t][:k_])
    buf = {k_: (v_[:M].clone() if v_ is not None else None) for k_, v_ in x.items()}
    win = r.window_ragged(n_max, buf["q"], buf["k"], buf["v"], buf["g"], buf["beta"])
    for w in range(W):
        for k_, v_ in x.items():
            if v_ is not None:
                buf[k_].copy_(v_[w * M:(w + 1) * M])
        out = win.launch(lists[w * M:(w + 1) * M])
        torch.cuda.synchronize()
        for j in range(M):
            k_ = len(lists[w * M + j])
            assert torch.equal(out[j][:k_], ref[w * M + j][:k_]), (w, j)
    assert torch.equal(a.read_state(list(range(S_))), r.read_state(list(range(S_))))
    assert [list(m) for m in a.get_meta()] == [list(m) for m in r.get_meta()]
    win.close()


def test_ragged_window_refusals():
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    S_, H, d, M = 6, 2, 64, 4
    x, S0, _ = make_case(gen.GDN, S_, H, d, M, seed=670, device="cuda")
    c = dl.DeltaLog(gen.GDN, S_, H, d, d, M)
    c.set_state(list(range(S_)), S0)
    c.fork(0, [5])
    win = c.window_ragged(4, x["q"][:, :4].contiguous(), x["k"][:, :4].contiguous(),
                          x["v"][:, :4].contiguous(), x["g"][:, :4].contiguous(),
                          x["beta"][:, :4].contiguous())
    meta = [list(m) for m in c.get_meta()]
    with pytest.raises(dl.DeltaLogError) as e:          # fork source in token 2
        win.launch([[1], [2], [0, 3], []])
    assert e.value.status == dl.EBUSY
    with pytest.raises(dl.DeltaLogError) as e:          # duplicate in a token
        win.launch([[1, 1], [], [], []])
    assert e.value.status == dl.EINVAL
    with pytest.raises(dl.DeltaLogError) as e:          # id out of range
        win.launch([[], [], [], [S_]])
    assert e.value.status == dl.EINVAL
    assert [list(m) for m in c.get_meta()] == meta       # nothing was applied
    with pytest.raises(dl.DeltaLogError) as e:          # fixed-window launch of a ragged window
        dl.dl_window_launch(c.handle, win._h)
    assert e.value.status == dl.EINVAL
    win.launch([[1, 2], [5], [3, 4, 1], [2]])
    torch.cuda.synchronize()
    assert list(c.get_meta()[0])[1:5] == [2, 2, 1, 1]
    win.close()


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("T", [75, 32, 1])
def test_chunked_prefill_then_decode(op, d, T):
    """dl_prefill over T context tokens (ragged last chunk for T=75), then 10
    decode steps: every output and the final state match the oracle run over
    the whole sequence."""
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    B, H, M, Td = 3, 4, 8, 10
    x, S0, bonus = make_case(op, B, H, d, T + Td, seed=700 + d + T + 31 * op)
    o_ref, S_ref, S_snap = oracle_run(op, x, S0, bonus, snap=[T - 1])
    ctx = dl.DeltaLog(op, B, H, d, d, M, out_bf16=False)
    ctx.set_state(list(range(B)), S0.cuda())
    if bonus is not None:
        ctx.set_bonus(bonus.cuda())
    dev = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    sl = lambda key: dev[key][:T].contiguous() if dev[key] is not None else None
    o_pf = ctx.prefill(list(range(B)), sl("q"), sl("k"), sl("v"), sl("g"), sl("beta"))
    S_pf = ctx.read_state(list(range(B))).cpu().reshape(B * H, d, d).numpy()
    assert rel_err(S_pf, S_snap[0]) <= STATE_TOL
    assert max_step_rel(o_pf.cpu().reshape(T, B * H, d).numpy(), o_ref[:T]) <= OUT_TOL_F32
    outs = []
    for t in range(T, T + Td):
        beta = dev["beta"][t] if dev["beta"] is not None else None
        outs.append(ctx.step(list(range(B)), dev["q"][t], dev["k"][t], dev["v"][t], dev["g"][t],
                             beta).float())
    o = torch.stack(outs).cpu().reshape(Td, B * H, d).numpy()
    assert max_step_rel(o, o_ref[T:]) <= OUT_TOL_F32
    S = ctx.read_state(list(range(B))).cpu().reshape(B * H, d, d).numpy()
    assert rel_err(S, S_ref) <= STATE_TOL


def test_prefill_rules():
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    x, S0, _ = make_case(gen.RWKV6, 1, 2, 64, 4, seed=9)
    ctx = dl.DeltaLog(gen.RWKV6, 1, 2, 64, 64, 4)
    with pytest.raises(dl.DeltaLogError) as e:     # RWKV6 needs its bonus first
        ctx.prefill([0], x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["g"].cuda(), None)
    assert e.value.status == dl.EINVAL
    x, S0, _ = make_case(gen.GDN, 1, 2, 64, 4, seed=9)
    ctx = dl.DeltaLog(gen.GDN, 1, 2, 64, 64, 4)
    dev = {k: v.cuda() for k, v in x.items()}
    ctx.step([0], dev["q"][0], dev["k"][0], dev["v"][0], dev["g"][0], dev["beta"][0])
    with pytest.raises(dl.DeltaLogError) as e:      # pending log entry
        ctx.prefill([0], dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"])
    assert e.value.status == dl.EINVAL
