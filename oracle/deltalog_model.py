"""fp64 model of DeltaLog execution: a dense base per slot plus a bounded log.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

It follows the DeltaLog page, section "Methodology — Base + Log" and the
two-phase decode cycle, in the page's order:
  * the active state of a slot is a dense base S̄ (history up to the last merge)
    plus a bounded log of compressed update factors (a_j, b_j) with log-decay
    metadata Λ_j;
  * append phase (the common case): S̄ is left unchanged, the token's factors
    and the current cumulative log-decay are appended to the log;
  * merge phase (every M-th step): base + replayed log entries are
    materialised back into S̄ and the log is cleared.
The "Kernel implementation — Staged execution" section says the replay
coefficients are computed once per slot-head; this model computes the same
coefficients (scalar products of logged keys with the current key/query,
weighted by decay differences) so that it states the algebra a staged
implementation uses.  The value-side factor a_j is u_j for the delta-rule
operators (GDN, KDA) and v_j for RWKV6; the key-side factor b_j is k_j.
Λ_j is cumulative since the last merge (a scalar per head for GDN, a d_k
vector for KDA and RWKV6); only differences Λ_t - Λ_j are exponentiated.

It is checked against the eager oracle at every step for every M (the method
changes the schedule of the state update, not the function it computes), and
its integer trace against ``SlotTableModel``.  Forking indexes the source's
base storage (Flide page, "Research method step by step", second step).

Shapes: S [H, dv, dk] per slot; per-token inputs [H, d] per slot, g [H] (GDN)
or [H, dk] (KDA, RWKV6), beta [H].
"""
import numpy as np

from .slot_table_model import SlotTableModel, OK

GDN, KDA, RWKV6 = 0, 1, 2


class DeltaLogModel:
    def __init__(self, op, num_slots, H, dk, dv, M, scale=1.0, bonus=None):
        self.op, self.H, self.dk, self.dv, self.M = op, H, dk, dv, M
        self.scale = float(scale)
        self.store = np.zeros((num_slots, H, dv, dk))
        self.table = SlotTableModel(num_slots, M)
        self.log = [[] for _ in range(num_slots)]   # entries (a [H,dv], k [H,dk], L [H] | [H,dk])
        self.bonus = None if bonus is None else np.asarray(bonus, np.float64)  # [H, dk]

    # -- helpers ---------------------------------------------------------------
    def _L_prev(self, s):
        if self.log[s]:
            return self.log[s][-1][2]
        return np.zeros(self.H) if self.op == GDN else np.zeros((self.H, self.dk))

    def _materialise(self, s, base, L_now, extra=None):
        """D ⊙ S̄[base] + Σ_j a_j (k_j ⊙ exp(L_now - L_j))^T over slot s's log (and one
        extra entry (a, k) with zero decay difference: the current token at a merge)."""
        Sb = self.store[base]
        if self.op == GDN:
            S = np.exp(L_now)[:, None, None] * Sb
        else:
            S = Sb * np.exp(L_now)[:, None, :]
        for a, kj, Lj in self.log[s]:
            if self.op == GDN:
                kt = kj * np.exp(L_now - Lj)[:, None]
            else:
                kt = kj * np.exp(L_now - Lj)
            S = S + a[:, :, None] * kt[:, None, :]
        if extra is not None:
            a, kj = extra
            S = S + a[:, :, None] * kj[:, None, :]
        return S

    # -- operations --------------------------------------------------------------
    def set_state(self, slots, S):
        rc = self.table.set_state(list(slots))
        assert rc == OK, rc
        for i, s in enumerate(slots):
            self.store[s] = np.asarray(S[i], np.float64)
            self.log[s] = []

    def fork(self, src, dsts):
        rc = self.table.fork(src, list(dsts))
        assert rc == OK, rc
        for d in dsts:
            self.log[d] = [(a.copy(), k.copy(), L.copy()) for a, k, L in self.log[src]]

    def read_state(self, slots):
        out = []
        for s in slots:
            out.append(self._materialise(s, self.table.base_of[s], self._L_prev(s)))
        return np.stack(out)

    def merge(self, slots):
        mats = [self._materialise(s, self.table.base_of[s], self._L_prev(s)) for s in slots]
        rc = self.table.merge(list(slots))
        assert rc == OK, rc
        for s, S in zip(slots, mats):
            self.store[s] = S
            self.log[s] = []

    def step(self, slots, q, k, v, g, beta=None):
        """One token for each listed slot; inputs are indexed like ``slots``.
        Returns o [len(slots), H, dv]."""
        slots = list(slots)
        rc, plan = self.table.step(slots)
        assert rc == OK, rc
        out = np.empty((len(slots), self.H, self.dv))
        for i, (s, base, n, merge) in enumerate(plan):
            qi, ki, vi = (np.asarray(x[i], np.float64) for x in (q, k, v))
            gi = np.asarray(g[i], np.float64)
            Sb = self.store[base]
            L_prev = self._L_prev(s)
            L_t = L_prev + gi
            if self.op in (GDN, KDA):
                bi = np.asarray(beta[i], np.float64)
                # replay coefficients, once per slot-head
                if self.op == GDN:
                    Sk = np.exp(L_t)[:, None] * np.einsum("hvd,hd->hv", Sb, ki)
                    Sq = np.exp(L_t)[:, None] * np.einsum("hvd,hd->hv", Sb, qi)
                    ckk = [np.exp(L_t - Lj) * np.einsum("hd,hd->h", kj, ki) for _, kj, Lj in self.log[s]]
                    ckq = [np.exp(L_t - Lj) * np.einsum("hd,hd->h", kj, qi) for _, kj, Lj in self.log[s]]
                else:
                    Sk = np.einsum("hvd,hd->hv", Sb, np.exp(L_t) * ki)
                    Sq = np.einsum("hvd,hd->hv", Sb, np.exp(L_t) * qi)
                    ckk = [np.einsum("hd,hd->h", kj * np.exp(L_t - Lj), ki) for _, kj, Lj in self.log[s]]
                    ckq = [np.einsum("hd,hd->h", kj * np.exp(L_t - Lj), qi) for _, kj, Lj in self.log[s]]
                # x = (decayed S_{t-1}) k_t from base + log
                x = Sk.copy()
                for c, (a, _, _) in zip(ckk, self.log[s]):
                    x += c[:, None] * a
                u = bi[:, None] * (vi - x)
                o = Sq.copy()
                for c, (a, _, _) in zip(ckq, self.log[s]):
                    o += c[:, None] * a
                o += np.einsum("hd,hd->h", ki, qi)[:, None] * u
                a_new = u
            else:  # RWKV6: output reads S_{t-1}; raw value update
                rhat = np.exp(L_prev) * qi
                o = np.einsum("hvd,hd->hv", Sb, rhat)
                for a, kj, Lj in self.log[s]:
                    o += np.einsum("hd,hd->h", kj * np.exp(L_prev - Lj), qi)[:, None] * a
                cb = np.einsum("hd,hd,hd->h", qi, self.bonus, ki)
                o += cb[:, None] * vi
                a_new = vi
            out[i] = self.scale * o
            if merge:
                self.store[s] = self._materialise(s, base, L_t, extra=(a_new, ki))
                self.log[s] = []
            else:
                self.log[s].append((a_new, ki.copy(), L_t))
        return out

    def meta(self):
        n, base_of, refs = self.table.snapshot()
        return list(n), list(base_of)
