"""Integer model of DeltaLog's per-slot bookkeeping, with Flide-style forking.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

What it follows.
* DeltaLog page, "Methodology — Base + Log" and the two-phase cycle: a slot
  keeps a dense base and a bounded log; for M-1 steps a step only appends to
  the log, and on every M-th step the base and the replayed log are merged back
  into the dense base and the log is cleared.  Reading adopted: the log holds
  at most M-1 entries between calls, the step that would make it M long is the
  merge step, and M = 1 makes every step a merge (eager decoding).
* Flide page, "Research method step by step", second step: the shared context
  is run once and its final recurrent state saved; each question branch then
  starts from its own request's saved state by indexing it, not by copying it.
  Reading adopted: ``fork`` points the branch's base index at the source's
  base, copies the source's log and log length, and the branch writes a
  private dense state at its first merge.  While any branch still indexes a
  slot's storage, that slot is frozen: stepping, merging or re-seeding it is
  refused (it would change the state the branch reads).

Every operation validates all of its arguments first and changes nothing when
it returns an error code.  Codes match the library's: OK=0, EINVAL=1, EBUSY=4.
"""

OK, EINVAL, EBUSY = 0, 1, 4


class SlotTableModel:
    def __init__(self, num_slots, merge_interval):
        assert num_slots > 0 and merge_interval >= 1
        self.S = num_slots
        self.M = merge_interval
        self.n = [0] * num_slots            # log length of each slot
        self.base_of = list(range(num_slots))  # storage slot whose dense base a slot reads
        self.refs = [0] * num_slots         # number of other slots indexing this storage

    # -- validation helpers -------------------------------------------------
    def _check_list(self, slots):
        if len(slots) == 0:
            return OK
        if any(s < 0 or s >= self.S for s in slots):
            return EINVAL
        if len(set(slots)) != len(slots):
            return EINVAL
        return OK

    def _release(self, s):
        b = self.base_of[s]
        if b != s:
            self.refs[b] -= 1
            self.base_of[s] = s

    # -- operations ---------------------------------------------------------
    def step(self, slots):
        """One decode token for each listed slot.  Returns (code, plan) where plan
        lists (slot, base, n_before, is_merge) in argument order."""
        rc = self._check_list(slots)
        if rc != OK:
            return rc, []
        if any(self.refs[s] > 0 for s in slots):
            return EBUSY, []
        plan = []
        for s in slots:
            b, n = self.base_of[s], self.n[s]
            merge = (n + 1 == self.M)
            plan.append((s, b, n, merge))
            if merge:
                self._release(s)
                self.n[s] = 0
            else:
                self.n[s] = n + 1
        return OK, plan

    def step_eager(self, slots):
        """Eager step: allowed only on slots that own their base and have an empty log."""
        rc = self._check_list(slots)
        if rc != OK:
            return rc
        if any(self.refs[s] > 0 for s in slots):
            return EBUSY
        if any(self.n[s] != 0 or self.base_of[s] != s for s in slots):
            return EINVAL
        return OK

    def fork(self, src, dsts):
        if src < 0 or src >= self.S:
            return EINVAL
        rc = self._check_list(dsts)
        if rc != OK:
            return rc
        if src in dsts:
            return EINVAL
        if any(self.refs[d] > 0 for d in dsts):
            return EBUSY
        b, n = self.base_of[src], self.n[src]
        for d in dsts:
            self._release(d)
            self.base_of[d] = b
            self.n[d] = n
            self.refs[b] += 1
        return OK

    def set_state(self, slots):
        rc = self._check_list(slots)
        if rc != OK:
            return rc
        if any(self.refs[s] > 0 for s in slots):
            return EBUSY
        for s in slots:
            self._release(s)
            self.n[s] = 0
        return OK

    def merge(self, slots):
        rc = self._check_list(slots)
        if rc != OK:
            return rc
        if any(self.refs[s] > 0 for s in slots):
            return EBUSY
        for s in slots:
            self._release(s)
            self.n[s] = 0
        return OK

    def read_state(self, slots):
        return self._check_list(slots)

    def snapshot(self):
        return list(self.n), list(self.base_of), list(self.refs)
