"""Boundary checks that need no GPU.

* The C-ABI library loads and exports every function include/deltalog.h declares.
* The library's host slot table (the bookkeeping every context uses to plan a
  step) follows the oracle's integer model exactly: same return codes, same
  per-step plans, same log lengths / base indices / reference counts, on
  hand-written and random operation sequences, including error cases
  (out-of-range and duplicate ids, frozen slots, forks onto the source).
"""
import ctypes
import os
import random
import re

import numpy as np
import pytest

import oracle
from linear_attention_recurrent_gdn_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dl():
    build.build()
    from linear_attention_recurrent_gdn_gb300 import deltalog
    return deltalog


def test_header_symbols_exported(dl):
    hdr = open(os.path.join(ROOT, "include", "deltalog.h")).read()
    declared = set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(dl_\w+)\s*\(", hdr, re.M))
    assert len(declared) >= 20
    lib = ctypes.CDLL(dl.LIB_PATH)
    missing = [s for s in sorted(declared) if not hasattr(lib, s)]
    assert not missing, missing
    assert declared == set(dl.EXPORTS)
    assert dl.dl_abi_version() == 2


def test_status_strings(dl):
    for code, name in enumerate(dl.STATUS_NAMES):
        assert dl.library().dl_status_str(code).decode() == name


def test_table_create_rejects_bad_args(dl):
    h = ctypes.c_void_p()
    assert dl.library().dl_table_create(0, 4, ctypes.byref(h)) == dl.EINVAL
    assert dl.library().dl_table_create(4, 0, ctypes.byref(h)) == dl.EINVAL
    assert not h.value


def _compare(tab, model):
    n, b, r = tab.get()
    mn, mb, mr = model.snapshot()
    assert list(n) == mn and list(b) == mb and list(r) == mr


def test_table_matches_model_by_hand(dl):
    tab, model = dl.SlotTable(5, 3), oracle.SlotTableModel(5, 3)
    seq = [("step", [0, 1]), ("step", [0]), ("fork", 0, [2, 3]), ("step", [0]),
           ("step", [2, 2]), ("step", [5]), ("fork", 2, [2]), ("step", [2, 3, 1]),
           ("reset", [0]), ("step", [0]), ("fork", 1, [4]), ("step", [1]), ("step", [4]),
           ("step", [4]), ("step", [1])]
    for op in seq:
        if op[0] == "step":
            rc, plan = tab.step(op[1])
            mrc, mplan = model.step(op[1])
            assert rc == mrc, op
            if rc == 0:
                assert [tuple(int(x) for x in p[:3]) + (bool(p[3]),) for p in plan] == mplan
        elif op[0] == "fork":
            assert tab.fork(op[1], op[2]) == model.fork(op[1], op[2]), op
        else:
            assert tab.reset(op[1]) == model.set_state(op[1]), op
        _compare(tab, model)


@pytest.mark.parametrize("M", [1, 2, 4, 16])
def test_table_matches_model_random(dl, M):
    rng = random.Random(1000 + M)
    S = 9
    tab, model = dl.SlotTable(S, M), oracle.SlotTableModel(S, M)
    for _ in range(2000):
        kind = rng.choice(["step", "step", "step", "fork", "reset", "merge", "eager", "check"])
        k = rng.randint(0, 4)
        sl = [rng.randrange(-1, S + 1) for _ in range(k)] if rng.random() < 0.15 else \
            rng.sample(range(S), k)
        if kind == "step":
            rc, plan = tab.step(sl)
            mrc, mplan = model.step(sl)
            assert rc == mrc
            if rc == 0:
                assert [tuple(int(x) for x in p[:3]) + (bool(p[3]),) for p in plan] == mplan
        elif kind == "fork":
            src = rng.randrange(-1, S + 1)
            assert tab.fork(src, sl) == model.fork(src, sl)
        elif kind == "reset":
            assert tab.reset(sl) == model.set_state(sl)
        elif kind == "merge":
            assert tab.reset(sl) == model.merge(sl)
        elif kind == "eager":
            assert tab.step_eager(sl) == model.step_eager(sl)
        else:
            assert tab.check(sl) == model.read_state(sl)
        _compare(tab, model)


def test_step_plan_empty_list(dl):
    tab = dl.SlotTable(3, 2)
    rc, plan = tab.step([])
    assert rc == 0 and plan.shape == (0, 4)
