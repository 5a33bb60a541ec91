"""The roofline numerators of bench.py, pinned on the CPU.

- Algorithmic bytes per token·head (`fused_bytes`, `eager_bytes`), averaged
  over a merge window, against the byte table derived from the step's
  definition (one dense base read a step, one write a window, (M-1)/2 log rows
  read on average, M-1 appended rows, the inputs and the bf16 output).
- The chunked prefill's FLOP count (`prefill_flops`) against an explicit
  enumeration of the multiply-adds of its contractions, chunk by chunk.
"""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def window_average(op, d, M):
    return sum(bench.fused_bytes(op, d, M, n)[0] for n in range(M)) / M


@pytest.mark.parametrize("op,d,M,total", [
    (0, 128, 4, 84_689), (0, 128, 8, 78_138), (0, 128, 16, 77_178), (0, 128, 32, 81_330),
    (1, 128, 16, 81_972), (2, 64, 16, 22_496)])
def test_window_bytes_match_the_table(op, d, M, total):
    assert abs(window_average(op, d, M) - total) <= 1


@pytest.mark.parametrize("op,d,total,writes", [(0, 128, 132_104, 65_792), (1, 128, 132_612, 65_792),
                                               (2, 64, 33_536, 16_512)])
def test_eager_bytes_match_the_table(op, d, total, writes):
    assert bench.eager_bytes(op, d) == (total, writes)   # (total, of which writes)


def enumerate_prefill_fmas(op, d, C):
    """Multiply-adds of one chunk of C tokens, loop by loop, divided by C."""
    fma = 0
    dv = dk = d
    delta = op != 2
    for j in range(C):                         # products with S̄
        fma += dv * dk * (2 if delta else 1)
    for j in range(C):                         # pair products, lower triangle
        for i in range(C):
            if delta:
                fma += dk * (i < j) + dk * (i <= j)
            else:
                fma += dk * (i < j)
    for r in range(dv):                        # substitution and outputs
        for j in range(C):
            if delta:
                fma += j                       # Σ_{i<j} A_kk[j,i] u_i
                fma += j + 1                   # Σ_{i<=j} A_kq[j,i] u_i
            else:
                fma += j + 1                   # Σ_{i<j} A_kr[j,i] v_i, plus the bonus term
    fma += dv * dk                             # chunk-end scaling of S̄
    for j in range(C):                         # rank-C rewrite
        fma += dv * dk
    return fma / C


@pytest.mark.parametrize("op", [0, 1, 2])
@pytest.mark.parametrize("d,C", [(8, 4), (16, 8), (64, 32), (128, 32)])
def test_prefill_flops_match_the_enumeration(op, d, C):
    assert bench.prefill_flops(op, d, C) == pytest.approx(2 * enumerate_prefill_fmas(op, d, C))
