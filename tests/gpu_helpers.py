"""Shared helpers of the GPU parity tests: seeded inputs, a driver that runs the
CUDA path through the C ABI, and the oracle reference on the same inputs."""
import numpy as np
import torch

import oracle
from linear_attention_recurrent_gdn_gb300 import inputs as gen

OUT_TOL_BF16 = 5e-3     # max relative output error (DeltaLog page, "Results": < 0.005)
OUT_TOL_F32 = 1e-4
STATE_TOL = 1e-4        # fp32 state


def rel_err(x, ref):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-30))


def max_step_rel(o, o_ref):
    """Per-step max relative error (O13 reading), maximised over steps."""
    return max(rel_err(o[t], o_ref[t]) for t in range(o.shape[0]))


def make_case(op, B, H, d, T, seed, device="cpu"):
    x = gen.make_inputs(op, T, B, H, d, d, seed, device=device)
    S0 = gen.initial_state(B, H, d, d, seed, device=device)
    bonus = gen.rwkv6_bonus(H, d, seed, device=device) if op == gen.RWKV6 else None
    return x, S0, bonus


def oracle_run(op, x, S0, bonus, sel=None, snap=None):
    """Eager fp64 oracle on the (b, h) pairs `sel` (list of (b, h); all if None).
    Returns o [T, nsel, dv], S_final [nsel, dv, dk], S_snap."""
    T, B, H = x["q"].shape[:3]
    if sel is None:
        sel = [(b, h) for b in range(B) for h in range(H)]
    bi = torch.tensor([s[0] for s in sel])
    hi = torch.tensor([s[1] for s in sel])
    f64 = lambda t: t[:, bi, hi].to(torch.float64).numpy()
    S = S0[bi, hi].to(torch.float64).numpy()
    if op == gen.GDN:
        return oracle.gdn_eager(S, f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["g"]),
                                f64(x["beta"]), snap=snap)
    if op == gen.KDA:
        return oracle.kda_eager(S, f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["g"]),
                                f64(x["beta"]), snap=snap)
    bon = bonus[hi].to(torch.float64).numpy()
    return oracle.rwkv6_eager(S, f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["g"]), bon,
                              snap=snap)


def gpu_run(op, x, S0, bonus, M, out_bf16=True, eager=False, snap=(), slots=None,
            num_slots=None, staging=0):
    """Run T tokens on all B slots through the C ABI.  Returns o [T, B, H, dv] (fp32 host),
    a dict step -> state [B, H, dv, dk] (host) for steps in `snap`, and the context."""
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    T, B, H, d = x["q"].shape
    slots = list(range(B)) if slots is None else list(slots)
    ctx = dl.DeltaLog(op, num_slots or max(slots) + 1, H, d, d, M, out_bf16=out_bf16,
                      staging=staging)
    dev = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    ctx.set_state(slots, S0.cuda().contiguous())
    if bonus is not None:
        ctx.set_bonus(bonus.cuda().contiguous())
    outs, states = [], {}
    for t in range(T):
        args = [dev["q"][t], dev["k"][t], dev["v"][t], dev["g"][t],
                dev["beta"][t] if dev["beta"] is not None else None]
        o = (ctx.step_eager if eager else ctx.step)(slots, *args)
        outs.append(o.float())
        if t in snap:
            states[t] = ctx.read_state(slots).cpu()
    ctx.sync()
    o = torch.stack(outs).cpu()
    return o, states, ctx
