"""GPU parity on seeded random configurations against the fp64 oracle.

The fixed cases pick a few merge intervals, batches and head sizes; these draw
op, head size (64 / 128), merge interval (1..32), batch (1..40 slots x 1..12
heads, so both one-tile and whole-slot-head units), the ReplayPrep staging and
the output precision at random, so that planner shapes and launch paths the
fixed cases do not reach run too.  Each case steps T = M + 2 + U{0..M} tokens
and checks every output, the final state and the log lengths.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import (OUT_TOL_BF16, OUT_TOL_F32, STATE_TOL, gpu_run, make_case,
                         max_step_rel, oracle_run, rel_err)
from linear_attention_recurrent_gdn_gb300 import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()


def draw(case):
    rng = np.random.default_rng(9000 + case)
    return dict(op=int(rng.integers(3)), d=int(rng.choice([64, 128])), M=int(rng.integers(1, 33)),
                B=int(rng.integers(1, 41)), H=int(rng.integers(1, 13)),
                staging=int(rng.integers(2)), out_bf16=bool(rng.integers(2)),
                extra=int(rng.integers(0, 33)))


@pytest.mark.parametrize("case", range(24))
def test_random_configuration(case):
    c = draw(case)
    op, d, M, B, H = c["op"], c["d"], c["M"], c["B"], c["H"]
    T = M + 2 + c["extra"] % (M + 1)
    x, S0, bonus = make_case(op, B, H, d, T, seed=700 + case)
    o_ref, S_ref, _ = oracle_run(op, x, S0, bonus)
    o, _, ctx = gpu_run(op, x, S0, bonus, M, out_bf16=c["out_bf16"], staging=c["staging"])
    tol = OUT_TOL_BF16 if c["out_bf16"] else OUT_TOL_F32
    assert max_step_rel(o.reshape(T, B * H, d).numpy(), o_ref) <= tol, c
    S = ctx.read_state(list(range(B))).cpu().reshape(B * H, d, d).numpy()
    assert rel_err(S, S_ref) <= STATE_TOL, c
    n, base_of = ctx.get_meta()
    assert list(n[:B]) == [T % M] * B and list(base_of[:B]) == list(range(B)), c
