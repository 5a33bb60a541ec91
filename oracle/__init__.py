"""Plain, slow, fp64 CPU oracle for DeltaLog recurrent-state decoding.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
benchmark's CPU-baseline / reference leg may import anything from here; the
product library (``linear_attention_recurrent_gdn_gb300`` and its CUDA code)
never does, and the two share no code.  Inputs reach both from the seeded
generator module, which holds none of the method's arithmetic.

Contents
  eager                eager GDN / KDA / RWKV6 recurrences in C (fp64, OpenMP
                       over (batch, head) pairs, serial over tokens); the
                       definition every result is compared against
  deltalog_model       base + bounded log + merge-every-M model (numpy fp64)
  slot_table_model     integer bookkeeping: log lengths, base indices, forks
Pins: tests/test_oracle_pins.py checks these against closed forms, special
cases, hand-worked values (tests/golden/) and invariants.
"""
from .eager import (build, num_threads, gdn_eager, kda_eager, rwkv6_eager,
                    rwkv6_eager_keymajor)
from .deltalog_model import DeltaLogModel, GDN, KDA, RWKV6
from .slot_table_model import SlotTableModel, OK, EINVAL, EBUSY

__all__ = ["build", "num_threads", "gdn_eager", "kda_eager", "rwkv6_eager",
           "rwkv6_eager_keymajor", "DeltaLogModel", "SlotTableModel",
           "GDN", "KDA", "RWKV6", "OK", "EINVAL", "EBUSY"]
