"""The chunked prefill's algebra, restated in plain fp64 numpy and checked
against the oracle's eager recurrence (CPU only).

The prefill kernel processes a context C tokens at a time: with S̄ the state
at the chunk start and Λ_j the log-decay accumulated inside the chunk, every
token's output and delta-rule factor follow from one product with S̄, pair
coefficients between the chunk's tokens and a forward substitution, and S̄ is
rewritten once at the chunk's end (the DeltaLog page's base + log algebra with
the chunk as the log).  This test writes those formulas out loop by loop, for
each op and a ragged last chunk, and requires them to reproduce the
token-by-token recurrence: a wrong decay index (RWKV6 reads Λ_{j-1}), a
missing bonus term or a wrong diagonal would fail it.  It shares nothing with
the CUDA path.
"""
import numpy as np
import pytest

import oracle

GDN, KDA, RWKV6 = 0, 1, 2


def chunked(op, S0, q, k, v, g, beta, bonus, C):
    """The chunk formulas for one slot-head: S0 [dv, dk], inputs [T, d]."""
    T, dk = k.shape
    S = S0.copy()
    o = np.zeros((T, S0.shape[0]))
    for t0 in range(0, T, C):
        idx = range(t0, min(T, t0 + C))
        n = len(idx)
        if op == GDN:
            L = np.cumsum([g[t] for t in idx])                       # Λ_j, one per token
            dec = lambda j, i: np.exp(L[j] - L[i]) * np.ones(dk)      # per channel, constant
            hat_k = [np.exp(L[j]) * k[t] for j, t in enumerate(idx)]
            hat_q = [np.exp(L[j]) * q[t] for j, t in enumerate(idx)]
        else:
            L = np.cumsum([g[t] for t in idx], axis=0)                # Λ_j[c]
            dec = lambda j, i: np.exp(L[j] - L[i])
            hat_k = [np.exp(L[j]) * k[t] for j, t in enumerate(idx)]
            if op == KDA:
                hat_q = [np.exp(L[j]) * q[t] for j, t in enumerate(idx)]
            else:                                                     # e^{Λ_{j-1}}, Λ_{-1} = 0
                hat_q = [(np.exp(L[j - 1]) if j > 0 else np.ones(dk)) * q[t]
                         for j, t in enumerate(idx)]
        a = []                                                        # appended factors
        for j, t in enumerate(idx):
            if op == RWKV6:
                y = S @ hat_q[j]
                for i in range(j):
                    y += np.sum(k[idx[i]] * q[t] * np.exp(L[j - 1] - L[i])) * v[idx[i]]
                y += np.sum(q[t] * bonus * k[t]) * v[t]
                a.append(v[t])
            else:
                x = S @ hat_k[j]
                for i in range(j):
                    x += np.sum(k[idx[i]] * k[t] * dec(j, i)) * a[i]
                u = beta[t] * (v[t] - x)
                a.append(u)
                y = S @ hat_q[j]
                for i in range(j + 1):
                    y += np.sum(k[idx[i]] * q[t] * dec(j, i)) * a[i]
            o[t] = y
        LC = L[n - 1]
        S = S * (np.exp(LC) if op == GDN else np.exp(LC)[None, :])
        for j in range(n):
            kt = k[idx[j]] * (np.exp(LC - L[j]) if op == GDN else np.exp(LC - L[j]))
            S = S + np.outer(a[j], kt)
    return o, S


@pytest.mark.parametrize("op", [GDN, KDA, RWKV6])
@pytest.mark.parametrize("T,C", [(11, 4), (9, 3), (5, 8)])
def test_chunk_formulas_reproduce_the_recurrence(op, T, C):
    rng = np.random.default_rng(40 + 7 * op + T)
    dk = dv = 6
    S0 = 0.3 * rng.standard_normal((dv, dk))
    q, k, v = (rng.standard_normal((T, dk)) for _ in range(3))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    if op == GDN:
        g = -0.1 * np.log1p(np.exp(rng.standard_normal(T)))
    elif op == KDA:
        g = -0.1 * np.log1p(np.exp(rng.standard_normal((T, dk))))
    else:
        g = -np.exp(-0.5 + 0.5 * rng.standard_normal((T, dk)))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(T)))
    bonus = 0.1 * rng.standard_normal(dk)
    o_c, S_c = chunked(op, S0, q, k, v, g, beta, bonus, C)
    one = lambda x: x[:, None]                        # [T, 1, ...]: one slot-head
    if op == GDN:
        o_e, S_e, _ = oracle.gdn_eager(S0[None], one(q), one(k), one(v), one(g), one(beta))
    elif op == KDA:
        o_e, S_e, _ = oracle.kda_eager(S0[None], one(q), one(k), one(v), one(g), one(beta))
    else:
        o_e, S_e, _ = oracle.rwkv6_eager(S0[None], one(q), one(k), one(v), one(g), bonus[None])
    assert np.max(np.abs(o_c - o_e[:, 0])) <= 1e-11 * max(1.0, np.max(np.abs(o_e)))
    assert np.max(np.abs(S_c - S_e[0])) <= 1e-11 * max(1.0, np.max(np.abs(S_e)))
