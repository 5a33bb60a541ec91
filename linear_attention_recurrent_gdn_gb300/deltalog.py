"""ctypes binding of libdeltalog (C ABI in include/deltalog.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of the library.  PyTorch supplies device memory and streams.  If the
library has not been built this module raises at import time; there is no
fallback path.

The module-level functions carry the C names (dl_create, dl_step, ...); the
``DeltaLog`` class and ``SlotTable`` class wrap them for convenience.
"""
import ctypes
import os

import numpy as np

from . import build as _build

GDN, KDA, RWKV6 = 0, 1, 2
OK, EINVAL, ENOMEM, ECUDA, EBUSY, EDEVICE, EUNSUPPORTED = range(7)
# Codes a kernel writes into a device status word (the library reports them as
# EDEVICE): a bounded wait for a state tile, for a unit's inputs or
# coefficients, or for a stage / input slot to be released gave up; a plan row
# was out of range; the test-only stall ran out; a wait for tensor-core MMAs
# (chunked prefill) gave up.
DEV_TIMEOUT_TILE, DEV_TIMEOUT_AUX, DEV_TIMEOUT_EMPTY, DEV_BAD_ITEM, DEV_TEST_STALL = 1, 2, 3, 4, 5
DEV_TIMEOUT_MMA = 6
STATUS_NAMES = ["DL_OK", "DL_EINVAL", "DL_ENOMEM", "DL_ECUDA", "DL_EBUSY", "DL_EDEVICE",
                "DL_EUNSUPPORTED"]
LIB_PATH = _build.LIB

# Every symbol the header declares (checked by the CPU test suite).
EXPORTS = [
    "dl_table_create", "dl_table_destroy", "dl_table_step", "dl_table_step_eager",
    "dl_table_fork", "dl_table_reset", "dl_table_check", "dl_table_get",
    "dl_create", "dl_destroy", "dl_set_stream", "dl_set_state", "dl_set_bonus", "dl_fork",
    "dl_step", "dl_step_host", "dl_decode_host", "dl_step_eager", "dl_merge", "dl_read_state", "dl_get_meta",
    "dl_sync", "dl_set_timing", "dl_get_timing", "dl_last_error", "dl_status_str",
    "dl_abi_version", "dl_checkpoint_bytes", "dl_checkpoint_save", "dl_checkpoint_load",
    "dl_window_create", "dl_window_launch", "dl_window_destroy", "dl_window_create_ragged",
    "dl_window_launch_ragged", "dl_prefill",
    "dl_step_noalloc", "dl_noalloc_sync",
]


class DeltaLogError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__("%s: %s" % (STATUS_NAMES[status] if 0 <= status < 7 else status, msg))
        self.status = status


class dl_config(ctypes.Structure):
    _fields_ = [("op", ctypes.c_int32), ("num_slots", ctypes.c_int32),
                ("num_heads", ctypes.c_int32), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("merge_interval", ctypes.c_int32),
                ("out_bf16", ctypes.c_int32), ("scale", ctypes.c_float),
                ("staging", ctypes.c_int32)]

STAGE_FUSED, STAGE_KERNELS = 0, 1


class dl_state_view(ctypes.Structure):
    _fields_ = [("Sbar", ctypes.c_void_p), ("alog", ctypes.c_void_p), ("klog", ctypes.c_void_p),
                ("Llog", ctypes.c_void_p), ("n_log", ctypes.c_void_p),
                ("base_of", ctypes.c_void_p), ("bonus", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libdeltalog is not built (%s); run "
                          "linear_attention_recurrent_gdn_gb300.build.build()" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    PP = ctypes.POINTER(ctypes.c_void_p)
    sig = {
        "dl_table_create": ([I32, I32, PP], I32),
        "dl_table_destroy": ([P], None),
        "dl_table_step": ([P, P, I32, P], I32),
        "dl_table_step_eager": ([P, P, I32], I32),
        "dl_table_fork": ([P, I32, P, I32], I32),
        "dl_table_reset": ([P, P, I32], I32),
        "dl_table_check": ([P, P, I32], I32),
        "dl_table_get": ([P, P, P, P], I32),
        "dl_create": ([ctypes.POINTER(dl_config), P, PP], I32),
        "dl_destroy": ([P], I32),
        "dl_set_stream": ([P, P], I32),
        "dl_set_state": ([P, P, I32, P], I32),
        "dl_set_bonus": ([P, P], I32),
        "dl_fork": ([P, I32, P, I32], I32),
        "dl_step": ([P, P, I32, P, P, P, P, P, P], I32),
        "dl_step_host": ([P, P, I32, P, P, P, P, P, P], I32),
        "dl_decode_host": ([P, P, I32, I32, P, P, P, P, P, P], I32),
        "dl_step_eager": ([P, P, I32, P, P, P, P, P, P], I32),
        "dl_merge": ([P, P, I32], I32),
        "dl_read_state": ([P, P, I32, P], I32),
        "dl_get_meta": ([P, P, P], I32),
        "dl_sync": ([P], I32),
        "dl_set_timing": ([P, I32], I32),
        "dl_get_timing": ([P, P, P], I32),
        "dl_last_error": ([P], ctypes.c_char_p),
        "dl_status_str": ([I32], ctypes.c_char_p),
        "dl_abi_version": ([], I32),
        "dl_checkpoint_bytes": ([P], I64),
        "dl_checkpoint_save": ([P, P, I32, P], I32),
        "dl_checkpoint_load": ([P, P, I32, P], I32),
        "dl_window_create": ([P, P, I32, P, P, P, P, P, P, PP], I32),
        "dl_window_launch": ([P], I32),
        "dl_window_destroy": ([P], I32),
        "dl_window_create_ragged": ([P, I32, P, P, P, P, P, P, PP], I32),
        "dl_window_launch_ragged": ([P, P, P], I32),
        "dl_prefill": ([P, P, I32, I32, P, P, P, P, P, P], I32),
        "dl_step_noalloc": ([ctypes.POINTER(dl_config), ctypes.POINTER(dl_state_view), P, I32,
                             P, P, P, P, P, P, P, ctypes.c_char_p, I32], I32),
        "dl_noalloc_sync": ([P, ctypes.POINTER(I32), ctypes.c_char_p, I32], I32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()


def library():
    return _lib


def _slots(slots):
    a = np.ascontiguousarray(np.asarray(slots, dtype=np.int32).reshape(-1))
    return a, a.ctypes.data_as(ctypes.c_void_p), int(a.size)


def _check(rc, ctx=None):
    if rc != OK:
        msg = _lib.dl_last_error(ctx).decode() if ctx else STATUS_NAMES[rc]
        raise DeltaLogError(rc, msg)


# ------------------------------------------------------------- C-named API --
def dl_table_create(num_slots, merge_interval):
    h = ctypes.c_void_p()
    _check(_lib.dl_table_create(num_slots, merge_interval, ctypes.byref(h)))
    return h


def dl_table_destroy(t):
    _lib.dl_table_destroy(t)


def dl_table_step(t, slots):
    """Returns (status, plan [n, 4]) without raising."""
    a, p, n = _slots(slots)
    plan = np.zeros((max(n, 1), 4), np.int32)
    rc = _lib.dl_table_step(t, p, n, plan.ctypes.data_as(ctypes.c_void_p))
    return rc, plan[:n]


def dl_table_step_eager(t, slots):
    a, p, n = _slots(slots)
    return _lib.dl_table_step_eager(t, p, n)


def dl_table_fork(t, src, dsts):
    a, p, n = _slots(dsts)
    return _lib.dl_table_fork(t, int(src), p, n)


def dl_table_reset(t, slots):
    a, p, n = _slots(slots)
    return _lib.dl_table_reset(t, p, n)


def dl_table_check(t, slots):
    a, p, n = _slots(slots)
    return _lib.dl_table_check(t, p, n)


def dl_table_get(t, num_slots):
    n = np.zeros(num_slots, np.int32)
    b = np.zeros(num_slots, np.int32)
    r = np.zeros(num_slots, np.int32)
    vp = lambda x: x.ctypes.data_as(ctypes.c_void_p)
    _check(_lib.dl_table_get(t, vp(n), vp(b), vp(r)))
    return n, b, r


def _ptr(t):
    """Device address of a tensor (an int passes through as an address)."""
    if t is None:
        return ctypes.c_void_p(0)
    return ctypes.c_void_p(t if isinstance(t, int) else t.data_ptr())


def dl_create(cfg, stream=None):
    h = ctypes.c_void_p()
    st = ctypes.c_void_p(0 if stream is None else int(stream))
    rc = _lib.dl_create(ctypes.byref(cfg), st, ctypes.byref(h))
    _check(rc)
    return h


def dl_destroy(ctx):
    return _lib.dl_destroy(ctx)


def dl_set_stream(ctx, stream):
    _check(_lib.dl_set_stream(ctx, ctypes.c_void_p(int(stream))), ctx)


def dl_set_state(ctx, slots, S):
    a, p, n = _slots(slots)
    _check(_lib.dl_set_state(ctx, p, n, _ptr(S)), ctx)


def dl_set_bonus(ctx, bonus):
    _check(_lib.dl_set_bonus(ctx, _ptr(bonus)), ctx)


def dl_fork(ctx, src, dsts):
    a, p, n = _slots(dsts)
    _check(_lib.dl_fork(ctx, int(src), p, n), ctx)


def dl_step(ctx, slots, q, k, v, g, beta, o):
    a, p, n = _slots(slots)
    _check(_lib.dl_step(ctx, p, n, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(o)), ctx)


def dl_step_eager(ctx, slots, q, k, v, g, beta, o):
    a, p, n = _slots(slots)
    _check(_lib.dl_step_eager(ctx, p, n, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                              _ptr(o)), ctx)


def dl_step_host(ctx, slots, q, k, v, g, beta, o):
    """Host (CPU, ideally pinned) torch tensors in, host tensor o out; synchronous."""
    a, p, n = _slots(slots)
    _check(_lib.dl_step_host(ctx, p, n, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                             _ptr(o)), ctx)


def dl_decode_host(ctx, slots, q, k, v, g, beta, o):
    """T tokens of host (pinned) torch tensors [T, n, ...] in, host o [T, n, H, d_v] out;
    copies overlap the computation; synchronous."""
    a, p, n = _slots(slots)
    T = int(q.shape[0])
    _check(_lib.dl_decode_host(ctx, p, n, T, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                               _ptr(o)), ctx)


def dl_merge(ctx, slots):
    a, p, n = _slots(slots)
    _check(_lib.dl_merge(ctx, p, n), ctx)


def dl_read_state(ctx, slots, S_out):
    a, p, n = _slots(slots)
    _check(_lib.dl_read_state(ctx, p, n, _ptr(S_out)), ctx)


def dl_get_meta(ctx, num_slots):
    nl = np.zeros(num_slots, np.int32)
    bo = np.zeros(num_slots, np.int32)
    _check(_lib.dl_get_meta(ctx, nl.ctypes.data_as(ctypes.c_void_p),
                            bo.ctypes.data_as(ctypes.c_void_p)), ctx)
    return nl, bo


def dl_sync(ctx):
    _check(_lib.dl_sync(ctx), ctx)


def dl_set_timing(ctx, enable):
    _check(_lib.dl_set_timing(ctx, 1 if enable else 0), ctx)


def dl_get_timing(ctx):
    ms = np.zeros(4, np.float64)
    cnt = np.zeros(4, np.int64)
    _check(_lib.dl_get_timing(ctx, ms.ctypes.data_as(ctypes.c_void_p),
                              cnt.ctypes.data_as(ctypes.c_void_p)), ctx)
    return ms, cnt


def dl_checkpoint_bytes(ctx):
    return int(_lib.dl_checkpoint_bytes(ctx))


def dl_checkpoint_save(ctx, slots, buf):
    a, p, n = _slots(slots)
    _check(_lib.dl_checkpoint_save(ctx, p, n, _ptr(buf)), ctx)


def dl_checkpoint_load(ctx, slots, buf):
    a, p, n = _slots(slots)
    _check(_lib.dl_checkpoint_load(ctx, p, n, _ptr(buf)), ctx)


def dl_prefill(ctx, slots, q, k, v, g, beta, o):
    a, p, n = _slots(slots)
    T = int(q.shape[0])
    _check(_lib.dl_prefill(ctx, p, n, T, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(o)),
           ctx)


def dl_window_create(ctx, slots, q, k, v, g, beta, o):
    a, p, n = _slots(slots)
    h = ctypes.c_void_p()
    _check(_lib.dl_window_create(ctx, p, n, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                 _ptr(o), ctypes.byref(h)), ctx)
    return h


def dl_window_launch(ctx, w):
    _check(_lib.dl_window_launch(w), ctx)


def dl_window_destroy(w):
    _lib.dl_window_destroy(w)


def dl_window_create_ragged(ctx, n_max, q, k, v, g, beta, o):
    h = ctypes.c_void_p()
    _check(_lib.dl_window_create_ragged(ctx, int(n_max), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                        _ptr(beta), _ptr(o), ctypes.byref(h)), ctx)
    return h


def dl_window_launch_ragged(ctx, w, slots, counts):
    """slots: int32 host array [M, n_max]; counts: int32 host array [M]."""
    s = np.ascontiguousarray(slots, dtype=np.int32)
    c = np.ascontiguousarray(counts, dtype=np.int32)
    _check(_lib.dl_window_launch_ragged(w, s.ctypes.data_as(ctypes.c_void_p),
                                        c.ctypes.data_as(ctypes.c_void_p)), ctx)


def dl_step_noalloc(cfg, state, plan, q, k, v, g, beta, o, stream=None):
    """One step on caller-owned buffers with no allocation inside the library.
    `state` maps dl_state_view field names to torch tensors (bonus may be None);
    `plan` is the [n, 4] int32 array from dl_table_step."""
    pl = np.ascontiguousarray(np.asarray(plan, dtype=np.int32).reshape(-1, 4))
    sv = dl_state_view(*[_ptr(state.get(f)).value for f, _ in dl_state_view._fields_])
    err = ctypes.create_string_buffer(256)
    st = ctypes.c_void_p(0 if stream is None else int(stream))
    rc = _lib.dl_step_noalloc(ctypes.byref(cfg), ctypes.byref(sv),
                              pl.ctypes.data_as(ctypes.c_void_p), int(pl.shape[0]), _ptr(q),
                              _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(o), st, err, 256)
    if rc != OK:
        raise DeltaLogError(rc, err.value.decode())


def dl_noalloc_sync(stream=None):
    """Synchronise the stream and read the static device status word of the
    allocation-free step.  Returns (status, device code, message); the word is
    cleared when it held an error."""
    err = ctypes.create_string_buffer(256)
    code = ctypes.c_int32(0)
    st = ctypes.c_void_p(0 if stream is None else int(stream))
    rc = _lib.dl_noalloc_sync(st, ctypes.byref(code), err, 256)
    return int(rc), int(code.value), err.value.decode()


def dl_last_error(ctx):
    return _lib.dl_last_error(ctx).decode()


def dl_abi_version():
    return int(_lib.dl_abi_version())


# ------------------------------------------------------------------ classes --
class SlotTable:
    """Host bookkeeping of a context (no GPU needed)."""

    def __init__(self, num_slots, merge_interval):
        self.num_slots = num_slots
        self._h = dl_table_create(num_slots, merge_interval)

    def __del__(self):
        if getattr(self, "_h", None):
            dl_table_destroy(self._h)
            self._h = None

    def step(self, slots):
        return dl_table_step(self._h, slots)

    def step_eager(self, slots):
        return dl_table_step_eager(self._h, slots)

    def fork(self, src, dsts):
        return dl_table_fork(self._h, src, dsts)

    def reset(self, slots):
        return dl_table_reset(self._h, slots)

    def check(self, slots):
        return dl_table_check(self._h, slots)

    def get(self):
        return dl_table_get(self._h, self.num_slots)


class DecodeWindow:
    """A captured merge window; launch() replays it on the context's stream."""

    def __init__(self, ctx, slots, q, k, v, g, beta, out):
        n = len(list(slots))
        if out is None:
            out = ctx.torch.empty((ctx.M, n, ctx.H, ctx.d_v), dtype=ctx.out_dtype, device="cuda")
        self.ctx, self.out = ctx, out
        self._keep = (q, k, v, g, beta)
        self._h = dl_window_create(ctx.handle, slots, q, k, v, g, beta, out)

    def launch(self):
        dl_window_launch(self.ctx.handle, self._h)
        return self.out

    def close(self):
        if getattr(self, "_h", None):
            dl_window_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class RaggedWindow:
    """A captured merge window whose per-token active slots change from launch
    to launch; launch(slot_lists) replays it on the context's stream."""

    def __init__(self, ctx, n_max, q, k, v, g, beta, out):
        if out is None:
            out = ctx.torch.empty((ctx.M, n_max, ctx.H, ctx.d_v), dtype=ctx.out_dtype,
                                  device="cuda")
        self.ctx, self.out, self.n_max = ctx, out, int(n_max)
        self._keep = (q, k, v, g, beta)
        self._h = dl_window_create_ragged(ctx.handle, n_max, q, k, v, g, beta, out)

    def launch(self, slot_lists):
        """slot_lists: M lists of slot ids (token j's active rows, in input-row order)."""
        M = self.ctx.M
        if len(slot_lists) != M:
            raise ValueError("a window takes %d slot lists" % M)
        slots = np.full((M, self.n_max), -1, dtype=np.int32)
        counts = np.zeros(M, dtype=np.int32)
        for j, lst in enumerate(slot_lists):
            lst = list(lst)
            if len(lst) > self.n_max:
                raise ValueError("token %d has more than n_max rows" % j)
            slots[j, :len(lst)] = lst
            counts[j] = len(lst)
        dl_window_launch_ragged(self.ctx.handle, self._h, slots, counts)
        return self.out

    def close(self):
        if getattr(self, "_h", None):
            dl_window_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class DeltaLog:
    """A DeltaLog decode context on the current CUDA device.

    Tensors are torch CUDA tensors (C-contiguous): q, k [n, H, d_k] bf16;
    v [n, H, d_v] bf16; g [n, H] (GDN) or [n, H, d_k] (KDA, RWKV6) fp32;
    beta [n, H] fp32; states [n, H, d_v, d_k] fp32.  Slot lists are host ints.
    """

    def __init__(self, op, num_slots, num_heads, d_k, d_v=None, merge_interval=16,
                 out_bf16=True, scale=1.0, stream=None, staging=STAGE_FUSED):
        import torch
        self.torch = torch
        d_v = d_k if d_v is None else d_v
        self.cfg = dl_config(int(op), int(num_slots), int(num_heads), int(d_k), int(d_v),
                             int(merge_interval), 1 if out_bf16 else 0, float(scale), int(staging))
        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        self.stream = int(stream)
        self._h = dl_create(self.cfg, self.stream)
        self.op, self.num_slots, self.H, self.d_k, self.d_v = op, num_slots, num_heads, d_k, d_v
        self.M = merge_interval
        self.out_dtype = torch.bfloat16 if out_bf16 else torch.float32

    # -- lifecycle
    def close(self):
        if getattr(self, "_h", None):
            dl_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    # -- checks (marshalling)
    def _need(self, t, shape, dtype, name):
        torch = self.torch
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError("%s must be a CUDA tensor" % name)
        if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
            raise ValueError("%s: expected contiguous %s %s, got %s %s"
                             % (name, dtype, tuple(shape), t.dtype, tuple(t.shape)))

    def _check_step(self, n, q, k, v, g, beta):
        torch = self.torch
        self._need(q, (n, self.H, self.d_k), torch.bfloat16, "q")
        self._need(k, (n, self.H, self.d_k), torch.bfloat16, "k")
        self._need(v, (n, self.H, self.d_v), torch.bfloat16, "v")
        gshape = (n, self.H) if self.op == GDN else (n, self.H, self.d_k)
        self._need(g, gshape, torch.float32, "g")
        if self.op != RWKV6:
            self._need(beta, (n, self.H), torch.float32, "beta")

    # -- operations
    def set_state(self, slots, S):
        a, _, n = _slots(slots)
        self._need(S, (n, self.H, self.d_v, self.d_k), self.torch.float32, "S")
        dl_set_state(self._h, a, S)

    def set_bonus(self, bonus):
        self._need(bonus, (self.H, self.d_k), self.torch.float32, "bonus")
        dl_set_bonus(self._h, bonus)

    def fork(self, src, dsts):
        dl_fork(self._h, src, dsts)

    def step(self, slots, q, k, v, g, beta=None, out=None):
        a, _, n = _slots(slots)
        self._check_step(n, q, k, v, g, beta)
        if out is None:
            out = self.torch.empty((n, self.H, self.d_v), dtype=self.out_dtype, device=q.device)
        else:
            self._need(out, (n, self.H, self.d_v), self.out_dtype, "out")
        dl_step(self._h, a, q, k, v, g, beta, out)
        return out

    def step_eager(self, slots, q, k, v, g, beta=None, out=None):
        a, _, n = _slots(slots)
        self._check_step(n, q, k, v, g, beta)
        if out is None:
            out = self.torch.empty((n, self.H, self.d_v), dtype=self.out_dtype, device=q.device)
        dl_step_eager(self._h, a, q, k, v, g, beta, out)
        return out

    def step_host(self, slots, q, k, v, g, beta=None, out=None):
        a, _, n = _slots(slots)
        if out is None:
            out = self.torch.empty((n, self.H, self.d_v), dtype=self.out_dtype, pin_memory=True)
        for t in (q, k, v, g, beta, out):
            if t is not None and (t.is_cuda or not t.is_contiguous()):
                raise ValueError("step_host takes contiguous host tensors")
        dl_step_host(self._h, a, q, k, v, g, beta, out)
        return out

    def decode_host(self, slots, q, k, v, g, beta=None, out=None):
        """T tokens from host tensors q, k, v, g, beta [T, n, ...]; returns o [T, n, H, d_v]."""
        a, _, n = _slots(slots)
        T = int(q.shape[0])
        if out is None:
            out = self.torch.empty((T, n, self.H, self.d_v), dtype=self.out_dtype, pin_memory=True)
        for t in (q, k, v, g, beta, out):
            if t is not None and (t.is_cuda or not t.is_contiguous() or int(t.shape[0]) != T):
                raise ValueError("decode_host takes contiguous host tensors with T leading rows")
        dl_decode_host(self._h, a, q, k, v, g, beta, out)
        return out

    def merge(self, slots):
        dl_merge(self._h, slots)

    def read_state(self, slots, out=None):
        a, _, n = _slots(slots)
        if out is None:
            out = self.torch.empty((n, self.H, self.d_v, self.d_k), dtype=self.torch.float32,
                                   device="cuda")
        dl_read_state(self._h, a, out)
        return out

    def get_meta(self):
        return dl_get_meta(self._h, self.num_slots)

    def checkpoint_save(self, slots, buf=None):
        """Save the exact representation of each slot; returns a uint8 device buffer."""
        a, _, n = _slots(slots)
        per = dl_checkpoint_bytes(self._h)
        if buf is None:
            buf = self.torch.empty(n * per, dtype=self.torch.uint8, device="cuda")
        dl_checkpoint_save(self._h, a, buf)
        return buf

    def prefill(self, slots, q, k, v, g, beta, out=None, want_out=True):
        """Feed T context tokens ([T, n, ...] tensors) to each slot in one call."""
        a, _, n = _slots(slots)
        T = int(q.shape[0])
        for name, t, d in (("q", q, self.d_k), ("k", k, self.d_k), ("v", v, self.d_v)):
            self._need(t, (T, n, self.H, d), self.torch.bfloat16, name)
        gshape = (T, n, self.H) if self.op == GDN else (T, n, self.H, self.d_k)
        self._need(g, gshape, self.torch.float32, "g")
        if self.op != RWKV6:
            self._need(beta, (T, n, self.H), self.torch.float32, "beta")
        else:
            beta = None
        if out is None and want_out:
            out = self.torch.empty((T, n, self.H, self.d_v), dtype=self.out_dtype, device="cuda")
        dl_prefill(self._h, a, q, k, v, g, beta, out)
        return out

    def window_ragged(self, n_max, q, k, v, g, beta=None, out=None):
        """Capture one merge window for up to n_max rows per token whose active
        slots are given at each launch; tensors are [M, n_max, ...] device buffers."""
        return RaggedWindow(self, n_max, q, k, v, g, beta, out)

    def window(self, slots, q, k, v, g, beta=None, out=None):
        """Capture one merge window (M tokens) of `slots` into a CUDA graph; the
        tensors are [M, n, ...] device buffers that the graph reads at each launch."""
        return DecodeWindow(self, slots, q, k, v, g, beta, out)

    def checkpoint_load(self, slots, buf):
        dl_checkpoint_load(self._h, slots, buf)

    def sync(self):
        dl_sync(self._h)

    def set_timing(self, enable):
        dl_set_timing(self._h, enable)

    def get_timing(self):
        return dl_get_timing(self._h)
