"""Host-side argument checks of dl_step_noalloc (no GPU needed).

Every call below is invalid in exactly one way, so the library must return
DL_EINVAL from its host checks before it makes any CUDA call; the pointers are
fake device addresses that are never dereferenced.  The baseline arguments are
valid in every other respect (aligned addresses, a plan that dl_table_step
would produce).
"""
import numpy as np
import pytest

from linear_attention_recurrent_gdn_gb300 import build

BASE = 0x7f0000000000


@pytest.fixture(scope="module")
def dl():
    build.build()
    from linear_attention_recurrent_gdn_gb300 import deltalog
    return deltalog


def _args(dl, op, M=4, B=4):
    """Aligned fake tensors, one per argument, 1 MiB apart."""
    addr = iter(range(BASE, BASE + 64 * (1 << 20), 1 << 20))
    state = {f: next(addr) for f in ("Sbar", "alog", "klog", "Llog", "n_log", "base_of")}
    state["bonus"] = next(addr) if op == dl.RWKV6 else None
    x = {f: next(addr) for f in ("q", "k", "v", "g", "beta", "o")}
    if op == dl.RWKV6:
        x["beta"] = None
    plan = np.array([[s, s, 0, 1 if M == 1 else 0] for s in range(B)], np.int32)
    return dl.dl_config(op, B, 2, 64, 64, M, 1, 1.0), state, plan, x


def _call(dl, cfg, state, plan, x):
    with pytest.raises(dl.DeltaLogError) as e:
        dl.dl_step_noalloc(cfg, state, plan, x["q"], x["k"], x["v"], x["g"], x["beta"], x["o"])
    assert e.value.status == dl.EINVAL, str(e.value)
    return str(e.value)


@pytest.mark.parametrize("field,offset,op", [
    ("o", 1, 0),          # bf16 output on an odd address
    ("beta", 2, 0),       # fp32 per-head beta
    ("g", 2, 0),          # fp32 per-head log-decay (GDN)
    ("g", 4, 1),          # per-key log-decay rows move as 16-byte vectors (KDA)
    ("q", 8, 2),
    ("v", 4, 1),
])
def test_misaligned_tensor_is_refused(dl, field, offset, op):
    cfg, state, plan, x = _args(dl, op)
    x[field] += offset
    assert "misaligned tensor" in _call(dl, cfg, state, plan, x)


@pytest.mark.parametrize("field,offset,op", [
    ("Sbar", 8, 0), ("alog", 4, 1), ("klog", 2, 2), ("Llog", 4, 1), ("Llog", 2, 0),
    ("n_log", 2, 0), ("base_of", 1, 1), ("bonus", 4, 2),
])
def test_misaligned_state_is_refused(dl, field, offset, op):
    cfg, state, plan, x = _args(dl, op)
    state[field] += offset
    assert "misaligned state" in _call(dl, cfg, state, plan, x)


def test_duplicate_slot_is_refused(dl):
    cfg, state, plan, x = _args(dl, 0)
    plan[2, 0] = plan[2, 1] = 1
    assert "appears twice" in _call(dl, cfg, state, plan, x)


def test_merge_flag_must_match_log_length(dl):
    cfg, state, plan, x = _args(dl, 0, M=4)
    plan[1, 3] = 1                      # n = 0 is not the merge step of M = 4
    assert "inconsistent" in _call(dl, cfg, state, plan, x)
    cfg, state, plan, x = _args(dl, 0, M=4)
    plan[1, 2], plan[1, 3] = 3, 0      # n = 3 is
    assert "inconsistent" in _call(dl, cfg, state, plan, x)


def test_reading_a_base_that_merges_in_the_same_call_is_refused(dl):
    cfg, state, plan, x = _args(dl, 0, M=4)
    plan[0] = [0, 0, 3, 1]              # slot 0 merges: it rewrites its base
    plan[1] = [1, 0, 2, 0]              # slot 1 (a branch of 0) reads that base
    assert "merges in the same call" in _call(dl, cfg, state, plan, x)


def test_out_of_range_plan_rows_are_refused(dl):
    for row in ([4, 4, 0, 0], [0, -1, 0, 0], [0, 0, 4, 0]):
        cfg, state, plan, x = _args(dl, 1, M=4)
        plan[0] = row
        assert "out of range" in _call(dl, cfg, state, plan, x)
