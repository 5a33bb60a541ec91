"""DeltaLog recurrent-state decoding for linear attention (GDN, KDA, RWKV6) on GB300.

``build.build()`` compiles the CUDA library in-tree; ``deltalog`` is its ctypes
binding (C names dl_* and the ``DeltaLog`` / ``SlotTable`` classes);
``inputs`` draws seeded synthetic decode inputs.  The binding is imported on
first use so that ``build`` works before the library exists.
"""
from . import build  # noqa: F401

GDN, KDA, RWKV6 = 0, 1, 2


def __getattr__(name):
    if name in ("DeltaLog", "SlotTable", "DeltaLogError"):
        import importlib
        return getattr(importlib.import_module(__name__ + ".deltalog"), name)
    raise AttributeError(name)
