"""Chunked prefill over long contexts against the fp64 oracle.

The Flide page's first call builds a request's base from its whole shared
context ("Research method step by step", second step); the fork workload does
this over 2048 tokens, and the prefill bench lines run 512-token contexts.
Here dl_prefill runs those lengths for every operator at its decode workload's
head size, with bf16 outputs, and a sample of slot-heads is checked against the
eager fp64 oracle: every token's output (max relative error <= 5e-3, the
DeltaLog page's "Results" bound) and the final state (<= 1e-4).  RWKV6's
per-key decays reach cumulative log-decays of about -100 inside a window, so
a long context is where fp32 drift in the chunked form would show.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import OUT_TOL_BF16, STATE_TOL, make_case, max_step_rel, oracle_run, rel_err
from linear_attention_recurrent_gdn_gb300 import build
from linear_attention_recurrent_gdn_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()


@pytest.mark.parametrize("T", [512, 2048])
@pytest.mark.parametrize("op,d", [(gen.GDN, 128), (gen.KDA, 128), (gen.RWKV6, 64)])
def test_long_prefill_matches_oracle(op, d, T):
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    B, H, M = 8, 4, 16
    x, S0, bonus = make_case(op, B, H, d, T, seed=5100 + op + T)
    rng = np.random.default_rng(T + op)
    n_sel = 4 if T > 1024 else 8
    flat = rng.choice(B * H, size=n_sel, replace=False)
    sel = [(int(i) // H, int(i) % H) for i in flat]
    o_ref, S_ref, _ = oracle_run(op, x, S0, bonus, sel=sel)
    ctx = dl.DeltaLog(op, B, H, d, d, M, out_bf16=True)
    slots = list(range(B))
    ctx.set_state(slots, S0.cuda())
    if bonus is not None:
        ctx.set_bonus(bonus.cuda())
    dev = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    o = ctx.prefill(slots, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"])
    S = ctx.read_state(slots).cpu()
    n, base_of = ctx.get_meta()
    ctx.close()
    bi = torch.tensor([s[0] for s in sel])
    hi = torch.tensor([s[1] for s in sel])
    o_sel = o.float().cpu()[:, bi, hi].numpy()
    assert max_step_rel(o_sel, o_ref) <= OUT_TOL_BF16
    assert rel_err(S[bi, hi].numpy(), S_ref) <= STATE_TOL
    assert list(n) == [0] * B and list(base_of) == slots


@pytest.mark.parametrize("strong", ["all", "mixed"])
@pytest.mark.parametrize("op,d,gain", [(gen.KDA, 128, 40.0), (gen.RWKV6, 64, 4.0)])
def test_prefill_strong_decay_matches_oracle(op, d, gain, strong):
    """The tensor-core kernels of the per-key ops factor their pair
    coefficients through the chunk start while a chunk's total log-decay stays
    above -60 in every channel; a chunk with stronger decay takes the direct
    path (one exponential per channel and pair).  Here the log-decays are
    scaled up (to about -2.8 a token: -90 over a chunk) for every token, or for
    the tokens of every other chunk only, so that both paths run and
    alternate; the result must still match the oracle."""
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    B, H, M, T = 2, 4, 16, 160
    x, S0, bonus = make_case(op, B, H, d, T, seed=5300 + len(strong) + 11 * op)
    g = x["g"].clone()
    if strong == "all":
        g *= gain
    else:
        for c0 in range(0, T, 64):
            g[c0:c0 + 32] *= gain
    x["g"] = g.contiguous()
    o_ref, S_ref, _ = oracle_run(op, x, S0, bonus)
    ctx = dl.DeltaLog(op, B, H, d, d, M, out_bf16=False)
    slots = list(range(B))
    ctx.set_state(slots, S0.cuda())
    if bonus is not None:
        ctx.set_bonus(bonus.cuda())
    dev = {k_: (v_.cuda() if v_ is not None else None) for k_, v_ in x.items()}
    o = ctx.prefill(slots, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"])
    S = ctx.read_state(slots).cpu().reshape(B * H, d, d).numpy()
    ctx.close()
    assert max_step_rel(o.float().cpu().reshape(T, B * H, d).numpy(), o_ref) <= 1e-4
    assert rel_err(S, S_ref) <= STATE_TOL


@pytest.mark.parametrize("T", [33, 97])
@pytest.mark.parametrize("B,H", [(3, 3), (1, 1), (2, 4)])
def test_rwkv6_tensor_core_prefill_slot_head_pairs(B, H, T):
    """RWKV6's tensor-core prefill takes two slot-heads per CTA (flattened
    slot-heads 2b and 2b + 1, which may belong to different slots); with an odd
    count the last CTA holds one.  Ragged and full chunk counts, fp32 outputs,
    then decode steps from the prefilled state: every output and the state
    match the oracle, and each slot's table entry is reset."""
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    d, M, Td = 64, 8, 5
    x, S0, bonus = make_case(gen.RWKV6, B, H, d, T + Td, seed=5500 + 13 * B + 7 * H + T)
    o_ref, S_ref, S_snap = oracle_run(gen.RWKV6, x, S0, bonus, snap=[T - 1])
    ctx = dl.DeltaLog(gen.RWKV6, B, H, d, d, M, out_bf16=False)
    slots = list(range(B))
    ctx.set_state(slots, S0.cuda())
    ctx.set_bonus(bonus.cuda())
    dev = {k_: (v_.cuda() if v_ is not None else None) for k_, v_ in x.items()}
    sl = lambda key: dev[key][:T].contiguous() if dev[key] is not None else None
    o_pf = ctx.prefill(slots, sl("q"), sl("k"), sl("v"), sl("g"), None)
    S_pf = ctx.read_state(slots).cpu().reshape(B * H, d, d).numpy()
    assert rel_err(S_pf, S_snap[0]) <= STATE_TOL
    assert max_step_rel(o_pf.cpu().reshape(T, B * H, d).numpy(), o_ref[:T]) <= 1e-4
    n, base_of = ctx.get_meta()
    assert list(n) == [0] * B and list(base_of) == slots
    outs = []
    for t in range(T, T + Td):
        outs.append(ctx.step(slots, dev["q"][t], dev["k"][t], dev["v"][t], dev["g"][t], None).float())
    o = torch.stack(outs).cpu().reshape(Td, B * H, d).numpy()
    assert max_step_rel(o, o_ref[T:]) <= 1e-4
    S = ctx.read_state(slots).cpu().reshape(B * H, d, d).numpy()
    assert rel_err(S, S_ref) <= STATE_TOL
    ctx.close()


@pytest.mark.parametrize("out_bf16", [False, True])
def test_rwkv6_tensor_core_prefill_unaligned_output(out_bf16):
    """RWKV6's tensor-core prefill writes a token's 32 values per thread as
    16-byte vectors when o is 16-byte aligned, and element by element when it
    is only element-aligned (the boundary's rule).  An output buffer one
    element past a 16-byte boundary gives bitwise the same outputs and state as
    an aligned one, and both match the oracle."""
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    B, H, d, M, T = 2, 3, 64, 8, 70
    x, S0, bonus = make_case(gen.RWKV6, B, H, d, T, seed=5600 + int(out_bf16))
    o_ref, _, S_snap = oracle_run(gen.RWKV6, x, S0, bonus, snap=[T - 1])
    dev = {k_: (v_.cuda() if v_ is not None else None) for k_, v_ in x.items()}
    slots = list(range(B))
    dt = torch.bfloat16 if out_bf16 else torch.float32
    numel = T * B * H * d
    res = []
    for shift in (0, 1):
        ctx = dl.DeltaLog(gen.RWKV6, B, H, d, d, M, out_bf16=out_bf16)
        ctx.set_state(slots, S0.cuda())
        ctx.set_bonus(bonus.cuda())
        buf = torch.full((numel + 16,), float("nan"), dtype=dt, device="cuda")
        out = buf[shift:shift + numel].view(T, B, H, d)
        assert (out.data_ptr() % 16 == 0) == (shift == 0)
        ctx.prefill(slots, dev["q"], dev["k"], dev["v"], dev["g"], None, out=out)
        S = ctx.read_state(slots).cpu().reshape(B * H, d, d).numpy()
        res.append((out.float().cpu(), S))
        assert torch.isnan(buf[:shift]).all() and torch.isnan(buf[shift + numel:]).all()
        ctx.close()
    assert torch.equal(res[0][0], res[1][0])
    assert (res[0][1] == res[1][1]).all()
    assert rel_err(res[1][1], S_snap[0]) <= STATE_TOL
    tol = OUT_TOL_BF16 if out_bf16 else 1e-4
    assert max_step_rel(res[1][0].reshape(T, B * H, d).numpy(), o_ref[:T]) <= tol


@pytest.mark.parametrize("T", [33, 64, 97, 130])
@pytest.mark.parametrize("op", [gen.GDN, gen.KDA])
def test_tensor_core_prefill_chunk_counts(op, T):
    """The tensor-core kernels at d = 128 pipeline their chunks: the next
    chunk's operands go to the other half of doubled buffers while the current
    chunk is solved, and inputs two chunks ahead are prefetched.  Chunk counts
    2, 2, 4 and 5 (T = 33, 64, 97, 130: ragged and full last chunks), fp32
    outputs, then decode steps from the prefilled state: every output and the
    state match the oracle."""
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    B, H, d, M, Td = 3, 4, 128, 8, 5
    x, S0, bonus = make_case(op, B, H, d, T + Td, seed=5400 + op * 7 + T)
    o_ref, S_ref, S_snap = oracle_run(op, x, S0, bonus, snap=[T - 1])
    ctx = dl.DeltaLog(op, B, H, d, d, M, out_bf16=False)
    slots = list(range(B))
    ctx.set_state(slots, S0.cuda())
    dev = {k_: (v_.cuda() if v_ is not None else None) for k_, v_ in x.items()}
    sl = lambda key: dev[key][:T].contiguous() if dev[key] is not None else None
    o_pf = ctx.prefill(slots, sl("q"), sl("k"), sl("v"), sl("g"), sl("beta"))
    S_pf = ctx.read_state(slots).cpu().reshape(B * H, d, d).numpy()
    assert rel_err(S_pf, S_snap[0]) <= STATE_TOL
    assert max_step_rel(o_pf.cpu().reshape(T, B * H, d).numpy(), o_ref[:T]) <= 1e-4
    outs = []
    for t in range(T, T + Td):
        beta = dev["beta"][t] if dev["beta"] is not None else None
        outs.append(ctx.step(slots, dev["q"][t], dev["k"][t], dev["v"][t], dev["g"][t], beta).float())
    o = torch.stack(outs).cpu().reshape(Td, B * H, d).numpy()
    assert max_step_rel(o, o_ref[T:]) <= 1e-4
    S = ctx.read_state(slots).cpu().reshape(B * H, d, d).numpy()
    assert rel_err(S, S_ref) <= STATE_TOL
    ctx.close()
