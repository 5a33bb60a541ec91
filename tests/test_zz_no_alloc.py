"""dl_step_noalloc: the decode step for callers that cannot let the library
allocate device memory (engines that reserve the GPU's memory for their own
pools at start-up, code whose buffers must all come from its own allocator,
loops that cannot take the synchronisation an allocation may cause).

The caller owns the state, the logs and the device slot table (plain torch
tensors here, laid out as dl_create lays them out) and plans each step with a
host slot table; the library keeps only the per-step coefficient scratch, in
a static device array.  Two calls in a row (an append step, then the merge
step for M = 2) must give what dl_step gives on a context, within the tests'
tolerances, and leave the same state and slot table.  This file is collected
last on purpose, and it depends on nothing an earlier test left behind.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import OUT_TOL_BF16, STATE_TOL, make_case, rel_err
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


@pytest.mark.parametrize("op", [gen.GDN, gen.KDA, gen.RWKV6])
def test_noalloc_step_matches_dl_step_two_calls(op):
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    B, H, d, M, T = 5, 4, 128, 2, 2
    x, S0, bonus = make_case(op, B, H, d, T, seed=800 + op, device="cuda")
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
        rc, plan = table.step(slots)
        assert rc == dl.OK
        o = torch.empty_like(o_ref)
        dl.dl_step_noalloc(cfg, buf, plan, x["q"][t], x["k"][t], x["v"][t], x["g"][t], beta, o,
                           stream)
        assert rel_err(o.float().cpu().numpy(), o_ref.float().cpu().numpy()) <= OUT_TOL_BF16, t
    S_ref = ref.read_state(slots)
    torch.cuda.synchronize()
    assert rel_err(buf["Sbar"].cpu().numpy(), S_ref.cpu().numpy()) <= STATE_TOL
    n_ref, b_ref = ref.get_meta()
    assert list(buf["n_log"].cpu().numpy()) == list(n_ref)
    assert list(buf["base_of"].cpu().numpy()) == list(b_ref)


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
