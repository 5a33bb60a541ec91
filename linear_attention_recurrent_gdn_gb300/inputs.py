"""Seeded synthetic decode inputs for GDN, KDA and RWKV6.

This module only draws random numbers with the distributions the decode
workloads state; it holds none of the recurrence arithmetic.  It is the one
piece shared by the CUDA path's tests and benchmark and by the oracle's tests.

Recipe (per token t of a run with seed s, generator seeded with s*100003 + t):
  GDN / KDA  q, k: N(0,1) rounded to bf16, L2-normalised in fp32 over the key
             dimension (eps 1e-6 inside the square root), rounded to bf16;
             v: N(0,1) rounded to bf16; beta = sigmoid(N(0,1)) fp32;
             g = log(alpha) = -0.1 * softplus(N(0,1)) fp32, one per head (GDN)
             or one per key channel (KDA).
  RWKV6      r, k, v: N(0,1) rounded to bf16 (not normalised);
             g = log(w) = -exp(N(-0.5, 0.5)) per key channel (second argument
             of N read as the standard deviation); bonus: 0.1 * N(0,1) [H, d_k].
  state      S_0 = 0.02 * N(0,1) fp32, [B, H, d_v, d_k] (value-major).
"""
import torch

GDN, KDA, RWKV6 = 0, 1, 2
OP_NAMES = {GDN: "gdn", KDA: "kda", RWKV6: "rwkv6"}


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normalised_bf16(x):
    xb = x.to(torch.bfloat16).to(torch.float32)
    n = torch.sqrt((xb * xb).sum(-1, keepdim=True) + 1e-6)
    return (xb / n).to(torch.bfloat16)


def step_inputs(op, B, H, dk, dv, seed, t, device="cpu"):
    """Inputs of one decode token for B slots: dict of q (r), k, v, g, beta."""
    gen = _gen(device, seed * 100003 + t)
    f32 = dict(dtype=torch.float32, device=device, generator=gen)
    if op in (GDN, KDA):
        q = _normalised_bf16(torch.randn(B, H, dk, **f32))
        k = _normalised_bf16(torch.randn(B, H, dk, **f32))
        v = torch.randn(B, H, dv, **f32).to(torch.bfloat16)
        gshape = (B, H) if op == GDN else (B, H, dk)
        g = -0.1 * torch.nn.functional.softplus(torch.randn(*gshape, **f32))
        beta = torch.sigmoid(torch.randn(B, H, **f32))
        return dict(q=q, k=k, v=v, g=g.contiguous(), beta=beta.contiguous())
    if op == RWKV6:
        r = torch.randn(B, H, dk, **f32).to(torch.bfloat16)
        k = torch.randn(B, H, dk, **f32).to(torch.bfloat16)
        v = torch.randn(B, H, dv, **f32).to(torch.bfloat16)
        g = -torch.exp(-0.5 + 0.5 * torch.randn(B, H, dk, **f32))
        return dict(q=r, k=k, v=v, g=g.contiguous(), beta=None)
    raise ValueError("unknown op %r" % (op,))


def make_inputs(op, T, B, H, dk, dv, seed, device="cpu", t0=0):
    """T consecutive tokens stacked on a leading axis: q,k [T,B,H,dk], v [T,B,H,dv],
    g [T,B,H] or [T,B,H,dk], beta [T,B,H] (None for RWKV6)."""
    steps = [step_inputs(op, B, H, dk, dv, seed, t0 + t, device) for t in range(T)]
    out = {}
    for key in ("q", "k", "v", "g", "beta"):
        vals = [s[key] for s in steps]
        out[key] = None if vals[0] is None else torch.stack(vals).contiguous()
    return out


def initial_state(B, H, dk, dv, seed, device="cpu"):
    gen = _gen(device, seed * 100003 + 99991)
    return 0.02 * torch.randn(B, H, dv, dk, dtype=torch.float32, device=device, generator=gen)


def rwkv6_bonus(H, dk, seed, device="cpu"):
    gen = _gen(device, seed * 100003 + 99989)
    return 0.1 * torch.randn(H, dk, dtype=torch.float32, device=device, generator=gen)
