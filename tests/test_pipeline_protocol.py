"""CPU model of the mbarrier protocol of the pipelined value-tile kernels.

The producer fills a ring of tile stages and a ring of aux slots with bulk
copies whose completions can arrive in any order; consumer warps wait with
parity tests, which cannot tell apart two phases of the same parity.  The
model replays the producer / consumer programs against that barrier semantic
under adversarial (newest-first) completion orders and flags any wait that
returns for a phase that has not completed, and any extra arrival.

The kernels' mapping (each consumer warp owns its stages; tile barrier waited
before the aux barrier) must pass; the earlier mapping (stage = tile mod ns,
shared by all warps; aux waited first) is kept as a negative control that the
model must catch.
"""
import random

import pytest

NCW = 8


class Bar:
    def __init__(self, count):
        self.count, self.done, self.pend, self.tx = count, 0, count, 0

    def arrive(self, tx=0):
        self.tx += tx
        self.pend -= 1
        if self.pend < 0:
            raise RuntimeError("extra arrival")
        self._check()

    def complete_tx(self, n):
        self.tx -= n
        if self.tx < 0:
            raise RuntimeError("tx underflow")
        self._check()

    def _check(self):
        if self.pend == 0 and self.tx == 0:
            self.done += 1
            self.pend = self.count

    def try_wait(self, parity):
        return (self.done % 2) != parity


def simulate(NS, NA, G, n_tiles, owned, tile_first, seed, p_complete=0.03, lifo=0.95,
             fused=False, ncw=NCW, npw=1, prep_by_unit=False, split=False):
    NCW_ = ncw
    rng = random.Random(seed)
    R = NS // NCW_
    if owned:
        stage = lambda i: (i % NCW_) * R + (i // NCW_) % R
        phase = lambda i: (i // NCW_) // R
    else:
        stage = lambda i: i % NS
        phase = lambda i: i // NS
    full = [Bar(1) for _ in range(NS)]
    empty = [Bar(1) for _ in range(NS)]
    afull = [Bar(1) for _ in range(NA)]
    aempty = [Bar(G) for _ in range(NA)]
    cready = [Bar(1) for _ in range(NA)]   # fused form: the prep warp's signal
    vready = [Bar(1) for _ in range(NA)]   # split: the unit's vectors, before cready
    inflight, violations = [], []
    prod = {"ti": 0, "ka": 0}
    # prep warp pw owns the aux slots x with x % npw == pw (npw divides NA) and
    # takes their units in order, so it sees every phase of those slots
    n_units = n_tiles // G
    prep = [{"ks": [k for k in range(n_units)
                    if (k % npw if prep_by_unit else (k % NA) % npw) == pw], "j": 0, "half": 0}
            for pw in range(npw)]
    cons = [{"i": w, "step": 0} for w in range(NCW_)]
    n_units = n_tiles // G

    def prep_warp(pw):
        if prep[pw]["j"] >= len(prep[pw]["ks"]):
            return
        k = prep[pw]["ks"][prep[pw]["j"]]
        x = k % NA
        if split and prep[pw]["half"] == 1:   # the coefficients, after the vectors
            cready[x].arrive()
            prep[pw]["half"] = 0
            prep[pw]["j"] += 1
            return
        if afull[x].try_wait((k // NA) & 1):
            if afull[x].done <= k // NA:
                violations.append(("prep", k))
            if split:
                vready[x].arrive()
                prep[pw]["half"] = 1
                return
            cready[x].arrive()
            prep[pw]["j"] += 1

    def producer():
        ti, ka = prod["ti"], prod["ka"]
        if ti >= n_tiles:
            return
        if ti // G == ka:
            x = ka % NA
            if aempty[x].try_wait(((ka // NA) & 1) ^ 1):
                afull[x].arrive(tx=3)
                inflight.extend([afull[x]] * 3)
                prod["ka"] += 1
            return
        s = stage(ti)
        if empty[s].try_wait((phase(ti) & 1) ^ 1):
            full[s].arrive(tx=1)
            inflight.append(full[s])
            prod["ti"] += 1

    def consumer(w):
        c = cons[w]
        i = c["i"]
        if i >= n_tiles:
            return
        kk = i // G
        x, s = kk % NA, stage(i)
        order = [(full[s], phase(i)), ((cready if fused else afull)[x], kk // NA)]
        if not tile_first:
            order.reverse()
        if split:   # tile, then vectors (the pass over the tile), then coefficients
            order = [(full[s], phase(i)), (vready[x], kk // NA), (cready[x], kk // NA)]
        if c["step"] < len(order):
            bar, ph = order[c["step"]]
            if bar.try_wait(ph & 1):
                if bar.done <= ph:
                    violations.append((w, i))
                c["step"] += 1
            return
        empty[s].arrive()
        aempty[x].arrive()
        c["i"] += NCW_
        c["step"] = 0

    try:
        for _ in range(2_000_000):
            r = rng.random()
            if r < p_complete and inflight:
                k = len(inflight) - 1 if rng.random() < lifo else rng.randrange(len(inflight))
                inflight.pop(k).complete_tx(1)
            elif r < p_complete + 0.2:
                producer()
            elif fused and r < p_complete + 0.3:
                prep_warp(rng.randrange(npw))
            else:
                consumer(rng.randrange(NCW_))
            if prod["ti"] >= n_tiles and all(c["i"] >= n_tiles for c in cons):
                return violations, True
    except RuntimeError:
        return violations + ["barrier accounting broken"], False
    return violations, False


@pytest.mark.parametrize("NS,NA,G", [(8, 3, 4), (8, 2, 4), (16, 9, 2), (16, 2, 1), (24, 16, 1),
                                     (24, 6, 2)])
def test_owned_stages_tile_first_is_safe(NS, NA, G):
    for seed in range(12):
        v, finished = simulate(NS, NA, G, NCW * 4 * 5, owned=True, tile_first=True, seed=seed)
        assert not v and finished, (seed, v[:3])


@pytest.mark.parametrize("ncw,NS,NA,G", [(4, 4, 2, 4), (4, 4, 2, 1), (3, 3, 2, 4), (8, 8, 3, 1),
                                          (4, 12, 2, 2)])
def test_fused_prep_stage_is_safe(ncw, NS, NA, G):
    """The fused form: a prep warp waits on each unit's inputs in order and
    signals a second barrier; consumers wait on their tile, then on that signal."""
    for seed in range(12):
        v, finished = simulate(NS, NA, G, 8 * 4 * 5, owned=True, tile_first=True, seed=seed,
                               fused=True, ncw=ncw)
        assert not v and finished, (seed, v[:3])


@pytest.mark.parametrize("npw,ncw,NS,NA,G", [(2, 4, 4, 2, 1), (2, 4, 4, 4, 1), (3, 3, 3, 6, 2),
                                              (2, 4, 8, 2, 4), (4, 4, 4, 8, 1), (1, 4, 4, 12, 4),
                                              (2, 4, 4, 16, 1), (1, 3, 3, 16, 4)])
def test_fused_several_prep_warps_is_safe(npw, ncw, NS, NA, G):
    """Several prep warps, each owning the aux slots x with x % npw == pw."""
    for seed in range(12):
        v, finished = simulate(NS, NA, G, 8 * 4 * 5, owned=True, tile_first=True, seed=seed,
                               fused=True, ncw=ncw, npw=npw)
        assert not v and finished, (seed, v[:3])


@pytest.mark.parametrize("npw,ncw,NS,NA,G", [(1, 4, 4, 2, 4), (1, 4, 4, 6, 4), (2, 4, 4, 4, 4),
                                            (2, 8, 8, 2, 4), (1, 2, 2, 3, 4)])
def test_fused_split_vectors_then_coefficients_is_safe(npw, ncw, NS, NA, G):
    """The fused form with prep warps as the kernel runs it: a prep warp
    arrives on a unit's vector barrier, then on its coefficient barrier; each
    consumer waits for its tile, then the vectors (its pass over the tile),
    then the coefficients (its epilogue)."""
    for seed in range(10):
        v, finished = simulate(NS, NA, G, ncw * G * 5, owned=True, tile_first=True, seed=seed,
                               fused=True, ncw=ncw, npw=npw, split=True)
        assert not v and finished, (seed, v[:3])


@pytest.mark.parametrize("ncw,NS,NA", [(4, 4, 4), (2, 4, 4), (2, 4, 6), (3, 3, 6), (4, 8, 8), (1, 1, 3)])
def test_consumer_prep_aux_first_on_owned_slots_is_safe(ncw, NS, NA):
    """One-tile units whose consumer warp computes the coefficients itself: it
    waits for the unit's inputs first, then for the tile.  With na a multiple of
    ncw each warp owns its aux slots as it owns its stages, so the aux wait is
    never a phase off even though it comes first."""
    for seed in range(12):
        v, finished = simulate(NS, NA, 1, 8 * 4 * 5, owned=True, tile_first=False, seed=seed,
                               ncw=ncw)
        assert not v and finished, (seed, v[:3])


def test_consumer_prep_aux_first_on_shared_slots_is_caught():
    """Negative control: with na not a multiple of ncw, slots pass between warps
    and an aux-first wait can pass a phase early."""
    caught = 0
    for seed in range(12):
        v, finished = simulate(4, 5, 1, 8 * 4 * 5, owned=True, tile_first=False, seed=seed, ncw=4)
        caught += bool(v) or not finished
    assert caught >= 3


def test_prep_warps_taking_every_npw_th_unit_is_caught():
    """Negative control: prep warps that take units pw, pw+npw, ... can wait on a
    slot whose earlier phase they never saw; the parity test then passes early."""
    caught = 0
    for seed in range(6):
        v, finished = simulate(4, 3, 1, 8 * 4 * 5, owned=True, tile_first=True, seed=seed,
                               fused=True, ncw=4, npw=2, prep_by_unit=True)
        caught += bool(v) or not finished
    assert caught >= 3


@pytest.mark.parametrize("ncw,NS,NA,G", [(4, 4, 2, 4), (3, 3, 2, 4), (4, 8, 3, 2)])
def test_owned_stages_two_ctas_shape_is_safe(ncw, NS, NA, G):
    for seed in range(12):
        v, finished = simulate(NS, NA, G, 8 * 4 * 5, owned=True, tile_first=True, seed=seed,
                               ncw=ncw)
        assert not v and finished, (seed, v[:3])


def test_shared_stages_aux_first_is_caught():
    caught = 0
    for seed in range(12):
        v, finished = simulate(12, 4, 4, NCW * 4 * 5, owned=False, tile_first=False, seed=seed)
        caught += bool(v) or not finished
    assert caught >= 6
