"""The fact that lets a decode step start streaming dense-base tiles before the
previous launch has finished (programmatic dependent launch inside a captured
decode window): a row whose log is non-empty never reads a dense base that the
launch just before it wrote.  A step writes a base only when a row merges (its
own storage, after which its log is empty), a forced merge or a set-state
leaves the slot with an empty log, and a fork source is frozen while any branch
indexes it.  Checked on the oracle's integer model of the slot table over
random sequences of steps, forks, forced merges and set-states; the negative
control shows that rows with an empty log do read just-written bases, so the
n > 0 condition is needed."""
import random

from oracle.slot_table_model import OK, SlotTableModel


def run(seed):
    rng = random.Random(seed)
    S, M = rng.randint(2, 12), rng.randint(1, 6)
    m = SlotTableModel(S, M)
    written = set()          # storage slots whose dense base the previous launch wrote
    hits_empty_log = 0
    for _ in range(80):
        r = rng.random()
        if r < 0.7:
            rc, plan = m.step(rng.sample(range(S), rng.randint(1, S)))
            if rc != OK:
                continue
            for slot, base, n, merge in plan:
                if n > 0:
                    assert base not in written, (seed, slot, base, n)
                elif base in written:
                    hits_empty_log += 1
            written = {slot for slot, base, n, merge in plan if merge}
        elif r < 0.8:
            src = rng.randrange(S)
            dsts = [d for d in rng.sample(range(S), rng.randint(1, S - 1)) if d != src]
            if dsts and m.fork(src, dsts) == OK:
                written = set()            # a fork copies log rows, no dense base
        elif r < 0.9:
            slots = rng.sample(range(S), rng.randint(1, S))
            if m.merge(slots) == OK:
                written = set(slots)
        else:
            slots = rng.sample(range(S), rng.randint(1, S))
            if m.set_state(slots) == OK:
                written = set(slots)
    return hits_empty_log


def test_rows_with_a_log_never_read_a_base_the_previous_launch_wrote():
    hits = sum(run(seed) for seed in range(300))
    assert hits > 0       # negative control: merged rows (n = 0) do read fresh bases
