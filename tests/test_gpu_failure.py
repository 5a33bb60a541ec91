"""Device-side failure detection, without a GPU fault.

Every wait in the pipelined kernels is bounded: when it runs out, the kernel
records a code in the context's device status word, lets its copies in flight
land and returns.  Here a test-only stall (DL_TEST_STALL=1, read by dl_create)
makes one consumer warp wait on an mbarrier that nothing ever arrives on, with
the limit shortened to 50 ms (DL_TEST_WAIT_MS).  Checked: the step itself
returns DL_OK (the work is asynchronous); dl_sync returns DL_EDEVICE naming
the stall's code; the context stays failed (sticky) for later calls; and a
fresh context on the same device then passes a parity step against the
oracle, so the GPU context is still usable.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import OUT_TOL_BF16, STATE_TOL, gpu_run, make_case, max_step_rel, oracle_run, rel_err
from linear_attention_recurrent_gdn_gb300 import build
from linear_attention_recurrent_gdn_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()


# (op, B, H, d, M, staging, eager): prep warps with multi-stage units (GDN d=128
# at 320 slot-heads), one-stage units (RWKV6 d=64), the two-kernel form, eager
CASES = [
    (gen.GDN, 80, 4, 128, 8, 0, False),
    (gen.RWKV6, 6, 4, 64, 4, 0, False),
    (gen.KDA, 4, 4, 128, 4, 1, False),
    (gen.GDN, 4, 4, 64, 1, 0, True),
]


@pytest.mark.parametrize("op,B,H,d,M,staging,eager", CASES)
def test_bounded_wait_runs_out_and_is_reported(monkeypatch, op, B, H, d, M, staging, eager):
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    T = 3
    x, S0, bonus = make_case(op, B, H, d, T, seed=4040 + op, device="cuda")
    slots = list(range(B))
    monkeypatch.setenv("DL_TEST_WAIT_MS", "50")
    monkeypatch.setenv("DL_TEST_STALL", "1")
    ctx = dl.DeltaLog(op, B, H, d, d, M, staging=staging)
    monkeypatch.delenv("DL_TEST_STALL")
    monkeypatch.delenv("DL_TEST_WAIT_MS")
    ctx.set_state(slots, S0)
    if bonus is not None:
        ctx.set_bonus(bonus)
    beta = x["beta"][0] if x["beta"] is not None else None
    step = ctx.step_eager if eager else ctx.step
    step(slots, x["q"][0], x["k"][0], x["v"][0], x["g"][0], beta)   # enqueued: DL_OK
    with pytest.raises(dl.DeltaLogError) as e:
        ctx.sync()
    assert e.value.status == dl.EDEVICE
    assert "device status %d" % dl.DEV_TEST_STALL in str(e.value), str(e.value)
    with pytest.raises(dl.DeltaLogError) as e:                       # sticky
        step(slots, x["q"][1], x["k"][1], x["v"][1], x["g"][1], beta)
    assert e.value.status == dl.EDEVICE
    ctx.close()
    # the GPU context is intact: a fresh context decodes correctly
    xc = {k: (v.cpu() if v is not None else None) for k, v in x.items()}
    S0c, bc = S0.cpu(), bonus.cpu() if bonus is not None else None
    o, states, ctx2 = gpu_run(op, xc, S0c, bc, M, eager=eager, snap=(T - 1,), staging=staging)
    o_ref, S_ref, _ = oracle_run(op, xc, S0c, bc)
    assert max_step_rel(o.numpy().reshape(T, B * H, d), o_ref) <= OUT_TOL_BF16
    assert rel_err(states[T - 1].numpy().reshape(B * H, d, d), S_ref) <= STATE_TOL
    ctx2.close()
