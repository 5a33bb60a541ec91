"""ctypes front end of the fp64 eager recurrences in ``recurrence.c``.

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
CPU-baseline leg of the benchmark, never by the product library.

Shapes (any float dtype is accepted and converted to float64):
    S0            [BH, dv, dk]    value-major state, row = value index
    q, k (r)      [T, BH, dk]
    v             [T, BH, dv]
    g             [T, BH] (GDN) or [T, BH, dk] (KDA, RWKV6): log-decay
    beta          [T, BH]
    bonus         [BH, dk] (RWKV6)
Returns ``(o [T, BH, dv], S_final [BH, dv, dk], S_snap [n_snap, BH, dv, dk])``.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "recurrence.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lib = None


def build(force=False):
    """Compile recurrence.c with gcc (OpenMP, no fast-math, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC",
               "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64, I32, F64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        common = [I64, I64, I32, I32, F64, P, P, P, P, P, P, P, P]
        for name in ("oracle_gdn", "oracle_kda", "oracle_rwkv6"):
            fn = getattr(lib, name)
            fn.argtypes = common + [I32, P, P]
            fn.restype = None
        lib.oracle_rwkv6_keymajor.argtypes = common
        lib.oracle_rwkv6_keymajor.restype = None
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def num_threads():
    """Host threads the oracle's OpenMP loop over (batch, head) pairs uses."""
    return int(_load().oracle_num_threads())


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _run(name, S0, a, k, v, g, last, scale, snap):
    S0, a, k, v, g, last = (_f64(x) for x in (S0, a, k, v, g, last))
    BH, dv, dk = S0.shape
    T = a.shape[0]
    assert a.shape == (T, BH, dk) and k.shape == (T, BH, dk) and v.shape == (T, BH, dv)
    o = np.empty((T, BH, dv))
    S_final = np.empty((BH, dv, dk))
    snap_t = np.ascontiguousarray(np.asarray(snap if snap is not None else [], dtype=np.int64))
    S_snap = np.empty((len(snap_t), BH, dv, dk))
    getattr(_load(), name)(BH, T, dk, dv, float(scale), _ptr(S0), _ptr(a), _ptr(k), _ptr(v),
                           _ptr(g), _ptr(last), _ptr(o), _ptr(S_final),
                           len(snap_t), _ptr(snap_t), _ptr(S_snap))
    return o, S_final, S_snap


def gdn_eager(S0, q, k, v, g, beta, scale=1.0, snap=None):
    """Gated DeltaNet, eager (head-scalar decay, delta rule); g is [T, BH]."""
    assert np.asarray(g).ndim == 2
    return _run("oracle_gdn", S0, q, k, v, g, beta, scale, snap)


def kda_eager(S0, q, k, v, g, beta, scale=1.0, snap=None):
    """Kimi Delta Attention, eager, with the explicit d_k x d_k transition; g is [T, BH, dk]."""
    assert np.asarray(g).ndim == 3
    return _run("oracle_kda", S0, q, k, v, g, beta, scale, snap)


def rwkv6_eager(S0, r, k, v, g, bonus, scale=1.0, snap=None):
    """RWKV6, eager, value-major state; g = log w is [T, BH, dk]; bonus is [BH, dk]."""
    assert np.asarray(g).ndim == 3
    return _run("oracle_rwkv6", S0, r, k, v, g, bonus, scale, snap)


def rwkv6_eager_keymajor(S0, r, k, v, g, bonus, scale=1.0):
    """RWKV6 as written on a key-major state (transposed internally); returns (o, S_final)."""
    S0, r, k, v, g, bonus = (_f64(x) for x in (S0, r, k, v, g, bonus))
    BH, dv, dk = S0.shape
    T = r.shape[0]
    o = np.empty((T, BH, dv))
    S_final = np.empty((BH, dv, dk))
    _load().oracle_rwkv6_keymajor(BH, T, dk, dv, float(scale), _ptr(S0), _ptr(r), _ptr(k),
                                  _ptr(v), _ptr(g), _ptr(bonus), _ptr(o), _ptr(S_final))
    return o, S_final
