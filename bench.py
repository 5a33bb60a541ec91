#!/usr/bin/env python3
"""Benchmark of DeltaLog recurrent-state decode on GB300.

One bench step = one full decode run of the workload: `tokens` decode tokens
for every slot, one AppendDecode launch per token (ReplayPrep fused in; two
launches with --staging kernels), all inputs pre-generated in HBM.  The decode
loop runs as CUDA graphs of M tokens (dl_window; --no-graph: one dl_step call
per token).  Default workload: GDN decode at serving batch, B=256 slots, H=32
heads, d_k=d_v=128, fp32 state (512 MiB, larger than L2), 512 tokens, merge
interval M=16; the M sweep {1,4,8,16,32} and the in-house eager kernel are
measured beside it.  The end-to-end figure runs the same decode from pinned
host buffers through dl_decode_host, copies included.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload gdn|kda|rwkv6] [--M 16] [--no-sweep] [--no-cpu]

Multi-GPU (torchrun): slots are independent, so every rank decodes its own
batch shard with no collective on the data path (weak scaling); the timing
is the max over ranks and the value sums all ranks' tokens·heads.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOADS = {
    # name: op, B, H, d, tokens, M (headline), seed
    "gdn_small": dict(op=0, B=1, H=4, d=64, tokens=64, M=8, seed=1000,
                      desc="GDN decode B=1 H=4 d_k=d_v=64 fp32 state, 64 tokens"),
    "gdn": dict(op=0, B=256, H=32, d=128, tokens=512, M=16, seed=1001,
                desc="GDN decode B=256 H=32 d_k=d_v=128 fp32 state, 512 tokens"),
    "kda": dict(op=1, B=128, H=32, d=128, tokens=512, M=16, seed=1002,
                desc="KDA decode B=128 H=32 d_k=d_v=128 fp32 state, 512 tokens"),
    "rwkv6": dict(op=2, B=128, H=40, d=64, tokens=512, M=16, seed=1003,
                  desc="RWKV6 decode B=128 H=40 head 64 fp32 state, 512 tokens"),
    "fork": dict(op=0, B=512, H=16, d=128, tokens=256, M=16, seed=1004, requests=64,
                 branches=8, ctx_tokens=2048,
                 desc="forked GDN decode: 64 requests x 2048 context tokens, 8 branches each "
                      "(512 branch slots) of U{16..256} tokens, H=16 d_k=d_v=128"),
}
METRIC = "state-update tokens·heads/s and achieved HBM GB/s vs ~8 TB/s; write bytes/step"
# Chunked prefill of the decode workloads' shapes: one call feeds every slot a
# 512-token context (the Flide page's first call, which builds a fork base).
PREFILL = {"prefill_gdn": "gdn", "prefill_kda": "kda", "prefill_rwkv6": "rwkv6"}
PREFILL_C = 32                      # tokens per chunk (csrc/prefill.cu)
# FP32 FMA peak from the unit counts and clock: 152 SMs x 128 FP32 lanes x
# 2 FLOP x 2.07 GHz (maximum SM clock).
FP32_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def log(*a):
    print(*a, file=sys.stderr, flush=True)


KERNEL_SOURCES = ["pipeline.cuh", "append_decode.cu", "append_launch.cuh", "append_fused_ne8.cu",
                  "append_fused_ne16.cu", "append_fused_ne32.cu", "dl_device.cuh", "layout.h"]


def strip_comments(src):
    """C/C++ source without comments and blank space, so that a change to a
    comment leaves the hash of the code unchanged."""
    import re
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def kernel_source_hash(read=None):
    """Hash of the AppendDecode sources (code only); ncu traffic figures are tied to it."""
    import hashlib
    read = read or (lambda f: open(os.path.join(ROOT, "linear_attention_recurrent_gdn_gb300",
                                                  "csrc", f)).read())
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(strip_comments(read(f)).encode())
    return h.hexdigest()[:16]


def measured_traffic(key):
    """DRAM bytes per launch (read + write) that an ncu capture recorded for this
    kernel and workload (profiles/traffic.txt), or None when the capture was
    taken on other kernel sources than the ones built now."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    src = kernel_source_hash()
    for line in open(path):
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == key and parts[2] == src:
            return float(parts[1])
    return None


# ------------------------------------------------------------ traffic model --
def algorithmic_bytes(op, d, M, n):
    """Algorithmic HBM bytes of one token for one slot-head with log length n
    before the step, split by kernel: returns (replay_prep, append_decode,
    append_decode_writes).  Counts each byte the step must move once:
    AppendDecode reads the dense base (d_v*d_k*4), the value-side log rows
    (n*d_v*4, bf16 for RWKV6), v_t (and k_t, q_t for GDN) and the coefficient
    block; it writes o_t (bf16) and appends u_t (delta-rule ops), or on a merge
    step writes the dense base back (and reads the key log rows for GDN).
    ReplayPrep reads k_t, q_t, g_t, beta_t and the key log (and log-decay) rows,
    writes the coefficient block and appends k_t, Λ_t (and v_t for RWKV6)."""
    dk = dv = d
    merge = (n + 1 == M)
    Mcap = max(M - 1, 1)
    Mcap4 = (Mcap + 3) // 4 * 4
    perkey = op != 0
    delta = op != 2
    P0 = 8 + 2 * Mcap4 + (2 * dk if perkey else 0)
    CB = P0 + (dk + M * dk if perkey else (M + 3) // 4 * 4)
    coef = (CB if merge else P0) * 4
    lw = dk * 4 if perkey else 4
    # ReplayPrep
    rp_r = 2 * dk * 2 + (dk * 4 if perkey else 4) + (4 if delta else 0) + n * (dk * 2 + lw)
    rp_w = coef + (0 if merge else dk * 2 + lw + (dv * 2 if op == 2 else 0))
    # AppendDecode
    esa = 4 if delta else 2
    ad_r = dv * dk * 4 + n * dv * esa + coef + (dv * 2) + (2 * dk * 2 if op == 0 else 0)
    if op == 0 and merge:
        ad_r += (n + 1) * dk * 2 - dk * 2     # key log rows (k_t already counted)
    ad_w = dv * 2 + (dv * dk * 4 if merge else (dv * 4 if delta else 0))
    return rp_r + rp_w, ad_r + ad_w, rp_w + ad_w


def fused_bytes(op, d, M, n):
    """Algorithmic HBM bytes of one token for one slot-head with log length n
    before the step, when the ReplayPrep stage runs inside AppendDecode (one
    kernel): returns (total, writes).  Reads: the dense base, k_t, q_t (r_t),
    v_t, g_t, beta_t, and n log rows (value side, key, log-decay).  The RWKV6
    bonus is [H, d_k] per step, shared by all slots, so it is not counted per
    slot-head.  Writes: o_t (bf16); on an append step the log row of this
    token (u_t fp32 or v_t bf16, k_t bf16, Λ_t); on the merge step the dense
    base.  No coefficient block leaves the chip."""
    dk = dv = d
    merge = (n + 1 == M)
    perkey = op != 0
    delta = op != 2
    esa = 4 if delta else 2
    lw = dk * 4 if perkey else 4
    r = dv * dk * 4 + 2 * dk * 2 + dv * 2 + lw + (4 if delta else 0) + n * (dv * esa + dk * 2 + lw)
    w = dv * 2 + (dv * dk * 4 if merge else dv * esa + dk * 2 + lw)
    return r + w, w


def eager_bytes(op, d):
    dk = dv = d
    r = dv * dk * 4 + 2 * dk * 2 + dv * 2 + (dk * 4 if op != 0 else 4) + (4 if op != 2 else 0)
    w = dv * dk * 4 + dv * 2
    return r + w, w


# --------------------------------------------------------------- clocks ------
class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t0 = time.time()
            while not self.rows and time.time() - t0 < 3.0:   # first sample before timing starts
                time.sleep(0.01)
            self.rows.clear()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4)
                          if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


# ------------------------------------------------------------ distributed ----
def dist_setup(want):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world <= 1:
        return 0, 1, None
    import torch.distributed as dist
    backend = "nccl" if want == "cuda" else "gloo"
    dist.init_process_group(backend=backend)
    return dist.get_rank(), dist.get_world_size(), dist


def reduce_max(dist, value, device):
    """Max of a float over ranks (identity when not distributed)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ------------------------------------------------------------- configs -------
def decode_loop(w, M, args, eager=False):
    """How the decode loop runs: CUDA graphs of M tokens unless --no-graph, the
    eager kernel, or a token count that is not a whole number of windows."""
    graphs = not (args.no_graph or eager or M == 1 or w["tokens"] % M)
    return "CUDA graphs, one per M tokens (dl_window)" if graphs else "dl_step per token"


def decode_config(w, M, args, world, eager=False):
    """The `config` object of a decode line; both arms print the same one."""
    B, H, d = w["B"], w["H"], w["d"]
    return {"workload": w["desc"] + (", eager dense step" if eager else ", merge interval M=%d" % M),
            "op": ("gdn", "kda", "rwkv6")[w["op"]], "B": B, "H": H, "d_k": d, "d_v": d,
            "tokens": w["tokens"], "M": M, "staging": args.staging,
            "loop": decode_loop(w, M, args, eager),
            "inputs": "bf16 q/k/v, fp32 g/beta, bf16 o",
            "l2": l2_note(w),
            "parallelism": "replicas/batch shards x%d" % world}


def l2_note(w):
    """How the timed region relates to L2 (129 MB on GB300): no flush between
    timed runs; the per-token inputs of one run are read once each."""
    B, H, d, T = w["B"], w["H"], w["d"], w["tokens"]
    state = B * H * d * d * 4
    per_tok = B * H * (3 * d * 2 + (d * 4 if w["op"] else 4) + (4 if w["op"] != 2 else 0))
    inputs = per_tok * T
    text = "no L2 flush; per-token inputs %.1f MB a run%s; fp32 state %.1f MB per rank" % (
        inputs / 1e6, " (larger than L2)" if inputs > 129e6 else "", state / 1e6)
    if state > 129e6:
        return "inputs larger than L2: " + text + " (larger than L2)"
    return text + " (fits in L2 and is re-read every token, as decoding does)"


def fork_plan(w, seed):
    """Branch lengths U{16..256} of the fork workload (uniform integers, seeded)."""
    import numpy as np
    return np.random.default_rng(seed).integers(16, 257, size=w["requests"] * w["branches"])


def fork_config(w, args, lens):
    return {"workload": w["desc"], "op": "gdn", "requests": w["requests"],
            "branches": w["branches"], "H": w["H"], "d_k": w["d"], "d_v": w["d"], "M": w["M"],
            "ctx_tokens": w["ctx_tokens"], "branch_tokens": int(lens.sum()),
            "staging": args.staging,
            "loop": ("dl_step per token" if args.no_graph else
                     "ragged CUDA graphs, one per M tokens (dl_window_*_ragged)"),
            "l2": "inputs larger than L2 (576 slots x 1 MiB state)"}


# ------------------------------------------------------------- reference -----
def run_reference(args):
    """Reference arm: the fp64 oracle (C, OpenMP) on the host cores, timed on a
    bounded sample of the same workload, reported in the same unit."""
    rank, world, dist = dist_setup("cpu")
    if rank != 0:
        return 0
    import torch
    import oracle
    from linear_attention_recurrent_gdn_gb300 import inputs as gen
    # a prefill computes the decode recurrence over its context, and a checkpoint
    # belongs to the GDN serving batch: same oracle
    w = WORKLOADS[PREFILL.get(args.workload, "gdn" if args.workload in ("checkpoint", "readstate")
                              else args.workload)]
    sample_sh = int(os.environ.get("DL_REF_SLOT_HEADS", "4096"))
    tokens = int(os.environ.get("DL_REF_TOKENS", "512"))
    oracle.build()
    res = cpu_baseline(w, sample_sh, tokens, args.steps, args.warmup)
    if args.workload == "fork":
        config = fork_config(w, args, fork_plan(w, w["seed"]))
    elif args.workload in WORKLOADS:
        config = decode_config(w, 1 if args.eager else (args.M or w["M"]), args, 1, args.eager)
    else:   # prefill, checkpoint and read-state lines: the decode workload they belong to
        config = {"workload": args.workload + " of " + w["desc"]}
    # n_gpus: the N the arm was launched with (rank 0 alone times the oracle on the
    # host cores; gpus_used says that no GPU takes part)
    out = {"metric": METRIC, "value": res["value"], "unit": "tokens·heads/s",
           "n_gpus": max(world, args.gpus), "gpus_used": 0,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "impl": "reference",
           "implementation": "fp64 eager oracle (C, OpenMP) on a bounded sample of the workload",
           "config": config,
           "cpu_baseline": {"value": res["value"], "unit": "tokens·heads/s",
                            "cores": res["cores"], "kind": "oracle", "sample": res["sample"]},
           "e2e": {"value": res["value"], "unit": "tokens·heads/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)
    return 0


def cpu_baseline(w, sample_sh, tokens, steps=1, warmup=0):
    """Time the fp64 eager oracle on `sample_sh` slot-heads x `tokens` tokens of
    the workload's input distributions (drawn on the CPU)."""
    import torch
    import oracle
    from linear_attention_recurrent_gdn_gb300 import inputs as gen
    op, d = w["op"], w["d"]
    H = min(w["H"], sample_sh)
    B = max(1, sample_sh // H)
    x = gen.make_inputs(op, tokens, B, H, d, d, w["seed"])
    S0 = gen.initial_state(B, H, d, d, w["seed"]).reshape(B * H, d, d).double().numpy()
    f = lambda t: t.reshape((tokens, B * H) + t.shape[3:]).double().numpy()
    if op == 2:
        bonus = gen.rwkv6_bonus(H, d, w["seed"]).double().numpy()
        extra = [bonus[h] for b in range(B) for h in range(H)]
        import numpy as np
        extra = np.stack(extra)
        fn = oracle.rwkv6_eager
    else:
        extra = f(x["beta"])
        fn = oracle.gdn_eager if op == 0 else oracle.kda_eager
    args = (S0, f(x["q"]), f(x["k"]), f(x["v"]), f(x["g"]), extra)
    for _ in range(warmup):
        fn(*args)
    times = []
    for _ in range(max(1, steps)):
        t0 = time.perf_counter()
        fn(*args)
        times.append(time.perf_counter() - t0)
    t = statistics.median(times)
    return {"value": B * H * tokens / t, "ms_per_step": t * 1e3, "cores": oracle.num_threads(),
            "sample": "%d slot-heads x %d tokens of the workload (fp64 eager, median of %d)"
                      % (B * H, tokens, len(times))}


# ------------------------------------------------------------------ ours -----
def roofline_window_bytes(op, d, M, T, slot_heads):
    """Algorithmic bytes per launch of the fused kernel, averaged over the T
    tokens of a decode run (token t has log length t mod M), and the writes."""
    tot = sum(fused_bytes(op, d, M, t % M)[0] for t in range(T)) * slot_heads / T
    wr = sum(fused_bytes(op, d, M, t % M)[1] for t in range(T)) * slot_heads / T
    return tot, wr


def measure_decode(w, args, dist, world, rank, local, dev, stream):
    """One decode workload at its merge interval, in its own timed region:
    W warm-up runs, then K runs of all its tokens (CUDA graphs of M tokens when
    the token count allows), inputs resident in HBM.  Returns the workload's
    entry: throughput, roofline of the fused kernel (one launch per token, so
    the launch time is the token time), algorithmic write cut against the eager
    kernel, clocks sampled during its own timed region."""
    import torch
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    from linear_attention_recurrent_gdn_gb300 import inputs as gen
    op, B, H, d, T, M = w["op"], w["B"], w["H"], w["d"], w["tokens"], w["M"]
    seed = w["seed"] + 7919 * rank
    x = gen.make_inputs(op, T, B, H, d, d, seed, device=dev)
    out = torch.empty((T, B, H, d), dtype=torch.bfloat16, device=dev)
    slots = list(range(B))
    c = dl.DeltaLog(op, B, H, d, d, M, out_bf16=True, stream=stream.cuda_stream,
                    staging=dl.STAGE_FUSED if args.staging == "fused" else dl.STAGE_KERNELS)
    c.set_state(slots, gen.initial_state(B, H, d, d, seed, device=dev))
    if op == 2:
        c.set_bonus(gen.rwkv6_bonus(H, d, seed, device=dev))
    graphs = decode_loop(w, M, args).startswith("CUDA graphs")
    sl = lambda key, j: x[key][j * M:(j + 1) * M] if x[key] is not None else None
    wins = ([c.window(slots, sl("q", j), sl("k", j), sl("v", j), sl("g", j), sl("beta", j),
                      out[j * M:(j + 1) * M]) for j in range(T // M)] if graphs else None)

    def one():
        if wins:
            for win in wins:
                win.launch()
            return
        for t in range(T):
            c.step(slots, x["q"][t], x["k"][t], x["v"][t], x["g"][t],
                   x["beta"][t] if x["beta"] is not None else None, out[t])

    ms, clocks = timed_steps(one, args, dist, local, dev, stream)
    for win in wins or []:
        win.close()
    c.close()
    fused = args.staging == "fused"
    sh = B * H
    bpl, wpl = roofline_window_bytes(op, d, M, T, sh)
    ew = eager_bytes(op, d)[1] * sh
    ms_tok = ms / T
    gbs = bpl / (ms_tok * 1e-3) / 1e9
    peak, src = hbm_peak()
    latency_bound = sh * d * d * 4 < (4 << 20)
    entry = {"value": sh * T * world / (ms / 1e3), "unit": "tokens·heads/s", "ms_per_step": ms,
             "us_per_token": ms_tok * 1e3, "config": decode_config(w, M, args, world),
             "roofline": {"bound": "latency" if latency_bound else "hbm", "achieved": gbs,
                          "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                          "traffic": measured_traffic("%s_%s_b%d_h%d_d%d_m%d" % (
                              "append_decode_fused" if fused else "append_decode",
                              ("gdn", "kda", "rwkv6")[op], B, H, d, M)),
                          "peak_source": src, "bytes_per_launch": bpl, "ms_per_launch": ms_tok,
                          "kernel": "AppendDecode (ReplayPrep fused)" if fused else "AppendDecode",
                          "timing": ("token time in the graph-captured decode loop" if graphs
                                     else "token time, one dl_step call per token")},
             "write_bytes_per_token": {"deltalog": wpl, "eager": ew},
             "write_cut_vs_eager": ew / wpl,
             "clocks": clocks,
             "gpu_launches": (1 if fused else 2) * T * args.steps * clocks.get("reps", 1)}
    if latency_bound:
        entry["note"] = ("%d KiB of state: launch latency, not HBM, bounds a token; the "
                         "fraction is reported for completeness" % (sh * d * d * 4 >> 10))
    del x, out
    torch.cuda.empty_cache()
    return entry


def run_ours(args):
    import torch
    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}))
        return 1
    rank, world, dist = dist_setup("cuda")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    from linear_attention_recurrent_gdn_gb300 import build
    if rank == 0:
        build.build()
    barrier(dist)
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    from linear_attention_recurrent_gdn_gb300 import inputs as gen

    w = dict(WORKLOADS[args.workload])
    if args.B:
        w["B"] = args.B
        w["desc"] += " [profiling override B=%d]" % args.B
    if args.tokens:
        w["tokens"] = args.tokens
        w["desc"] += " [profiling override tokens=%d]" % args.tokens
    op, B, H, d, T = w["op"], w["B"], w["H"], w["d"], w["tokens"]
    M = args.M or w["M"]
    seed = w["seed"] + 7919 * rank      # each rank decodes its own batch shard
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    t0 = time.time()
    x = gen.make_inputs(op, T, B, H, d, d, seed, device=dev)
    S0 = gen.initial_state(B, H, d, d, seed, device=dev)
    bonus = gen.rwkv6_bonus(H, d, seed, device=dev) if op == 2 else None
    out = torch.empty((T, B, H, d), dtype=torch.bfloat16, device=dev)
    slots = list(range(B))
    torch.cuda.synchronize()
    log("inputs generated in %.1fs" % (time.time() - t0))

    staging = dl.STAGE_FUSED if args.staging == "fused" else dl.STAGE_KERNELS

    def make_ctx(m):
        c = dl.DeltaLog(op, B, H, d, d, m, out_bf16=True, stream=stream.cuda_stream,
                        staging=staging)
        c.set_state(slots, S0)
        if bonus is not None:
            c.set_bonus(bonus)
        return c

    def decode_run(c, eager=False, wins=None):
        if wins:
            for win in wins:
                win.launch()
            return
        fn = c.step_eager if eager else c.step
        for t in range(T):
            fn(slots, x["q"][t], x["k"][t], x["v"][t], x["g"][t],
               x["beta"][t] if x["beta"] is not None else None, out[t])

    def make_windows(c, m):
        """The decode loop as CUDA graphs: one captured window per M tokens."""
        if args.no_graph or T % m or m == 1:   # a one-token window gains nothing from a graph
            return None
        sl = lambda key, j: x[key][j * m:(j + 1) * m] if x[key] is not None else None
        return [c.window(slots, sl("q", j), sl("k", j), sl("v", j), sl("g", j), sl("beta", j),
                         out[j * m:(j + 1) * m]) for j in range(T // m)]

    def timed(c, steps, warmup, eager=False, wins=None):
        for _ in range(warmup):
            decode_run(c, eager, wins)
        barrier(dist)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            decode_run(c, eager, wins)
        e1.record(stream)
        e1.synchronize()
        torch.cuda.synchronize()
        barrier(dist)
        return e0.elapsed_time(e1) / steps     # ms per bench step

    units_per_step = T * B * H                    # token·heads per rank per bench step

    # ---- headline: DeltaLog at M (or the eager kernel with --eager)
    if args.eager:
        M = 1
    ctx = make_ctx(M)
    wins = None if args.eager else make_windows(ctx, M)
    with ClockSampler(local) as clk:
        ms = timed(ctx, args.steps, args.warmup, eager=args.eager, wins=wins)
    ms_max = reduce_max(dist, ms, dev)
    value = units_per_step * world / (ms_max / 1e3)
    fused = args.staging == "fused" and not args.eager
    launches = (1 if (fused or args.eager) else 2) * T * args.steps * ((B + 1023) // 1024)
    for win in wins or []:
        win.close()

    # ---- per-kernel times (instrumented pass, token by token: events around every launch)
    ctx.set_timing(True)
    decode_run(ctx, eager=args.eager)
    kms, kcnt = ctx.get_timing()
    ctx.set_timing(False)
    n_seq = [t % M for t in range(T)]
    rp_b = ad_b = wr_all = 0
    for n in n_seq:
        if fused:
            b_, c_ = fused_bytes(op, d, M, n)
            a = 0
        else:
            a, b_, c_ = algorithmic_bytes(op, d, M, n)
        rp_b += a * B * H
        ad_b += b_ * B * H
        wr_all += c_ * B * H
    ad_ms = kms[1] / max(kcnt[1], 1)
    rp_ms = kms[0] / max(kcnt[0], 1)
    stepping_ms = ad_ms
    if fused and wins:
        # one launch per token in the graphs: the launch time is the token time
        # (inter-launch gaps included, so this never overstates the kernel)
        ad_ms = ms_max / T
    kernel_name = "AppendDecode (ReplayPrep fused)" if fused else "AppendDecode"
    if args.eager:
        eb_, ew_ = eager_bytes(op, d)
        ad_b, wr_all, rp_b = eb_ * B * H * T, ew_ * B * H * T, 0
        ad_ms = kms[2] / max(kcnt[2], 1)
        kernel_name = "EagerStep"
    ad_gbs = ad_b / T / (ad_ms * 1e-3) / 1e9
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        peak, peak_src = float(peaks["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        peak, peak_src = 6800.0, "fallback"
    step_bytes = (rp_b + ad_b) / T
    ctx.close()

    result = {
        "metric": METRIC, "value": value, "unit": "tokens·heads/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": decode_config(w, M, args, world, args.eager),
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "roofline": {"bound": "hbm", "achieved": ad_gbs, "peak": peak, "unit": "GB/s",
                     "frac": ad_gbs / peak,
                     "traffic": measured_traffic("%s_%s_b%d_h%d_d%d_m%d" % (
                         "eager_step" if args.eager else
                         "append_decode_fused" if fused else "append_decode",
                         gen.OP_NAMES[op], B, H, d, M)),
                     "kernel": kernel_name, "peak_source": peak_src + " hbm_gbs",
                     "bytes_per_launch": ad_b / T, "ms_per_launch": ad_ms,
                     "timing": ("token time in the graph-captured decode loop" if fused and wins
                                else "CUDA events around each launch"),
                     "ms_per_launch_stepping": stepping_ms},
        "kernels_ms_per_token": ({"EagerStep": ad_ms} if args.eager else
                                 {"AppendDecode (ReplayPrep fused)": ad_ms} if fused else
                                 {"ReplayPrep": rp_ms, "AppendDecode": ad_ms}),
        "step_gbs": step_bytes / (ms_max / T * 1e-3) / 1e9,
        "write_bytes_per_token": {"deltalog": wr_all / T,
                                  "deltalog_state_only": B * H * d * d * 4 / M},
    }

    # ---- end to end through the public API with host buffers (measured right
    #      after the headline, on the same inputs, before the other phases fill
    #      device and host memory)
    if not args.no_e2e:
        # pinned host buffers allocated as such and filled from the device (no
        # gigabytes of pageable temporaries freed just before the timed calls)
        pin = {}
        for k_, v_ in x.items():
            if v_ is not None:
                pin[k_] = torch.empty(v_.shape, dtype=v_.dtype, pin_memory=True)
                pin[k_].copy_(v_)
            else:
                pin[k_] = None
        hout = torch.empty((T, B, H, d), dtype=torch.bfloat16, pin_memory=True)
        torch.cuda.synchronize()
        c = make_ctx(M)

        def host_run():
            # one call per bench step: host inputs of all T tokens in, host outputs
            # out; the library overlaps each window's copies with its neighbours' compute
            c.decode_host(slots, pin["q"], pin["k"], pin["v"], pin["g"], pin["beta"], hout)
        for _ in range(max(args.warmup, 10)):
            host_run()
        barrier(dist)
        # up to 20 calls (about a second for the serving batch): a call now and
        # then runs ~20 ms long (no clock event, no host load behind it), and
        # more calls keep one such call from moving the mean by more than ~2 %
        e2e_steps = max(1, min(args.steps, 20))
        call_ms = []   # each call returns once its outputs are on the host
        with ClockSampler(local) as e2e_clk:
            t0 = time.perf_counter()
            for _ in range(e2e_steps):
                t1 = time.perf_counter()
                host_run()
                call_ms.append((time.perf_counter() - t1) * 1e3)
            torch.cuda.synchronize()
            e2e_ms = (time.perf_counter() - t0) * 1e3 / e2e_steps
        e2e_ms = reduce_max(dist, e2e_ms, dev)
        c.close()
        h2d = sum(v[0].numel() * v.element_size() for v in pin.values() if v is not None) * T
        d2h = hout[0].numel() * hout.element_size() * T
        group, path = decode_host_group(op, B, H, d, M, T)
        med_ms = reduce_max(dist, statistics.median(call_ms), dev)
        result["e2e"] = {"value": units_per_step * world / (e2e_ms / 1e3), "unit": "tokens·heads/s",
                         "value_median_call": units_per_step * world / (med_ms / 1e3),
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                         "ms_per_step": e2e_ms, "ms_per_call": [round(t, 2) for t in call_ms],
                         "clocks": e2e_clk.summary(), "api": "dl_decode_host", "path": path,
                         "copy_ceiling": copy_ceiling(pin, hout, dev, T, group,
                                                      units_per_step * world, args)}
        del pin, hout

    # ---- M sweep and the eager kernel (informational)
    if not args.no_sweep:
        sweep = {}
        for m in (1, 4, 8, 16, 32):
            c = make_ctx(m)
            ws = make_windows(c, m)
            sms = reduce_max(dist, timed(c, 2, 1, wins=ws), dev)
            sweep[str(m)] = units_per_step * world / (sms / 1e3)
            for win in ws or []:
                win.close()
            c.close()
        c = make_ctx(1)
        ems = reduce_max(dist, timed(c, 2, 1, eager=True), dev)
        c.close()
        eb, ew = eager_bytes(op, d)
        sweep["eager_kernel"] = units_per_step * world / (ems / 1e3)
        result["m_sweep"] = sweep
        result["eager_kernel_gbs"] = eb * B * H / (ems / T * 1e-3) / 1e9
        result["write_bytes_per_token"]["eager"] = ew * B * H
        result["write_cut_vs_eager"] = ew * B * H / result["write_bytes_per_token"]["deltalog"]
        result["note_writes"] = "algorithmic bytes; DRAM-measured writes are in profiles/"

    # ---- the other decode workloads, each in its own timed region
    if (not args.no_workloads and args.workload == "gdn" and not args.eager and not args.B
            and not args.tokens and not args.M):
        del x, out
        torch.cuda.empty_cache()
        result["workloads"] = {}
        for name in ("gdn_small", "kda", "rwkv6"):
            result["workloads"][name] = measure_decode(WORKLOADS[name], args, dist, world, rank,
                                                       local, dev, stream)
        result["workloads"]["fork"] = measure_fork(args, dist, world, rank, local, dev, stream)
        for name in PREFILL:   # chunked prefill of 512-token contexts at the decode shapes
            result["workloads"][name] = measure_prefill(name, args, dist, world, rank, local,
                                                        dev, stream)

    # ---- CPU baseline (rank 0, N = 1 only)
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        oracle.build()
        result["cpu_baseline"] = cpu_baseline(w, int(os.environ.get("DL_REF_SLOT_HEADS", "4096")),
                                              int(os.environ.get("DL_REF_TOKENS", "512")),
                                              steps=3, warmup=0)
        result["cpu_baseline"].update({"unit": "tokens·heads/s", "kind": "oracle"})
        result["cpu_baseline"].pop("ms_per_step", None)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def decode_host_group(op, S, H, d, M, T):
    """Tokens per copy group of dl_decode_host for S slots that start on their own
    bases with empty logs: a whole window of M tokens when T is a multiple of
    M >= 2 and four sets of such windows take at most 2 GiB (window graphs);
    otherwise small per-token tensors are grouped until a key tensor's copy
    reaches 2 MiB, at most 8 tokens and 64 MiB of staging a group.  Returns the
    group and the path's name."""
    key = S * H * d * 2
    per_tok = 2 * key + S * H * d * 2 + S * H * (d * 4 if op else 4) + S * H * 4 + S * H * d * 4
    if M >= 2 and T % M == 0 and 4 * M * per_tok <= (2 << 30):
        return M, "window graphs, one per M tokens"
    g = min(-(-(2 << 20) // key), (64 << 20) // per_tok)
    return max(1, min(8, g)), "token by token"


def copy_ceiling(pin, hout, dev, T, group, units, args):
    """The end-to-end run's copies alone: the same uploads (one copy per input
    tensor per group of tokens, pinned host to device) on one stream and the
    same downloads (one copy of the outputs per group) on another, with no
    compute.  Returns the throughput this bounds the end-to-end figure to and
    the bandwidth each direction reached, best of a few runs."""
    import torch
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    dbuf = {k: torch.empty((2 * group,) + tuple(v.shape[1:]), dtype=v.dtype, device=dev)
            for k, v in pin.items() if v is not None}
    dout = torch.empty((2 * group,) + tuple(hout.shape[1:]), dtype=hout.dtype, device=dev)
    h2d = sum(v[0].numel() * v.element_size() for v in pin.values() if v is not None) * T
    d2h = hout[0].numel() * hout.element_size() * T

    def run():
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        ev[0].record(up)
        ev[2].record(down)
        for g0 in range(0, T, group):
            n = min(group, T - g0)
            b = (g0 // group) % 2 * group
            with torch.cuda.stream(up):
                for k, v in pin.items():
                    if v is not None:
                        dbuf[k][b:b + n].copy_(v[g0:g0 + n], non_blocking=True)
            with torch.cuda.stream(down):
                hout[g0:g0 + n].copy_(dout[b:b + n], non_blocking=True)
        ev[1].record(up)
        ev[3].record(down)
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) * 1e3, ev[0].elapsed_time(ev[1]), ev[2].elapsed_time(ev[3])

    runs = [run() for _ in range(max(2, min(args.steps, 8)))]
    wall, t_up, t_dn = min(runs)
    return {"value": units / (wall / 1e3), "unit": "tokens·heads/s", "ms_per_step": wall,
            "ms_per_run": [round(r[0], 2) for r in runs],
            "h2d_gbs": h2d / (t_up * 1e-3) / 1e9, "d2h_gbs": d2h / (t_dn * 1e-3) / 1e9,
            "copies": "%d-token groups: one cudaMemcpyAsync per input tensor up, one down for "
                      "the outputs, on two streams, no compute" % group}


def prefill_mma_flops(op, d, C=PREFILL_C):
    """FLOPs (an FMA counts 2) the tensor-core prefill's MMAs execute per
    token·head, C = 32, every operand term and padded row included
    (csrc/prefill_tc.cu).  At d = 128: GDN D0 [K;Q;0]K^T (M=128, N=C, K=d), D1
    S̄[K;Q]^T in two terms (N=2C), D2 the rank-C rewrite in two terms (N=d, K=C),
    D3 the outputs' log terms in three (N=C, K=C); KDA the same with three terms
    each.  RWKV6 at d = 64 stacks two slot-heads in each M = 128 MMA and forms
    both heads' blocks of every product: [r̂;0][k̄;S̄]^T in three terms (N=2C+2d,
    K=d), [A;*]V^T in two (N=2d, K=C), D2 Vk̃ in two (N=2d, K=C), over 2C
    token·heads."""
    if op == 2:
        mac = 3 * 128 * (2 * C + 2 * d) * d + 2 * 128 * 2 * d * C + 2 * 128 * 2 * d * C
        return 2 * mac / (2 * C)
    terms = {0: (1, 2, 2, 3), 1: (3, 3, 3, 3)}[op]
    mac = (terms[0] * 128 * C * d + terms[1] * 128 * 2 * C * d + terms[2] * 128 * d * C
           + terms[3] * 128 * C * C)
    return 2 * mac / C


def prefill_flops(op, d, C=PREFILL_C):
    """FLOPs (an FMA counts 2) per token·head of the chunked prefill's
    contractions, d_k = d_v = d.  Per token: the products with S̄ (S̄K^T and S̄Q^T,
    2 d^2; RWKV6 only S̄R̂^T, d^2), S̄'s rewrite (the rank-C update d^2 and the
    chunk-end scaling d^2 / C), the decay-weighted pair products of the chunk's
    lower triangle (delta rule: k·k strictly below and k·q on and below the
    diagonal, C d; RWKV6: k·r strictly below, (C - 1) d / 2), and the forward
    substitution with the outputs (C d; RWKV6 the outputs, (C - 1) d / 2, and
    their bonus term, d).  Exponentials and elementwise scalings are not counted."""
    if op == 2:
        fma = 2 * d * d + d * d / C + C * d
    else:
        fma = 3 * d * d + d * d / C + 2 * C * d
    return 2 * fma


def gpu_setup():
    """Rank, world, process group, device and stream of this process, after the
    library is built (rank 0) and every rank has it."""
    import torch
    rank, world, dist = dist_setup("cuda")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    from linear_attention_recurrent_gdn_gb300 import build
    if rank == 0:
        build.build()
    barrier(dist)
    return rank, world, dist, local, torch.device("cuda", local), torch.cuda.current_stream()


MIN_REGION_S = 0.3   # shortest timed region: the clock sampler needs a few samples


def timed_steps(one, args, dist, local, dev, stream):
    """W untimed warm-up steps, then K steps between CUDA events on the launching
    stream (barrier + synchronize before), with the clocks sampled meanwhile.
    When K steps last less than MIN_REGION_S (latency-bound workloads), the
    timed region runs the K steps `reps` times over and the time per step is
    the region's time / (K * reps).  Returns (ms per step, max over ranks;
    clock summary, with `reps`)."""
    import torch
    for _ in range(args.warmup):
        one()
    barrier(dist)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    one()
    torch.cuda.synchronize()
    est = max(time.perf_counter() - t0, 1e-6) * max(args.steps, 1)
    reps = 1 if est >= MIN_REGION_S else int(MIN_REGION_S / est) + 1
    reps = int(reduce_max(dist, reps, dev))
    barrier(dist)
    with ClockSampler(local) as clk:
        e0.record(stream)
        for _ in range(args.steps * reps):
            one()
        e1.record(stream)
        e1.synchronize()
    summary = clk.summary()
    summary["reps"] = reps
    return reduce_max(dist, e0.elapsed_time(e1) / (args.steps * reps), dev), summary


def run_prefill(args):
    """Chunked prefill: one bench step is one dl_prefill call that feeds all B
    slots a T-token context (inputs resident in HBM)."""
    rank, world, dist, local, dev, stream = gpu_setup()
    result = measure_prefill(args.workload, args, dist, world, rank, local, dev, stream)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def measure_prefill(name, args, dist, world, rank, local, dev, stream):
    """One prefill workload (a PREFILL name) in its own timed region; returns its
    JSON object."""
    import torch
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    from linear_attention_recurrent_gdn_gb300 import inputs as gen
    w = WORKLOADS[PREFILL[name]]
    op, B, H, d, M = w["op"], args.B or w["B"], w["H"], w["d"], w["M"]
    T = args.tokens or w["tokens"]
    seed = w["seed"] + 7919 * rank
    x = gen.make_inputs(op, T, B, H, d, d, seed, device=dev)
    ctx = dl.DeltaLog(op, B, H, d, d, M, stream=stream.cuda_stream)
    slots = list(range(B))
    ctx.set_state(slots, gen.initial_state(B, H, d, d, seed, device=dev))
    if op == 2:
        ctx.set_bonus(gen.rwkv6_bonus(H, d, seed, device=dev))
    out = torch.empty((T, B, H, d), dtype=torch.bfloat16, device=dev)

    def one():
        ctx.prefill(slots, x["q"], x["k"], x["v"], x["g"], x["beta"], out=out)

    ms, clocks = timed_steps(one, args, dist, local, dev, stream)
    units = B * H * T
    tflops = units * prefill_flops(op, d) / (ms / 1e3) / 1e12
    # GDN and KDA at d = 128 and RWKV6 at d = 64 run on the tensor cores
    tensor = (op in (0, 1) and d == 128) or (op == 2 and d == 64)
    if tensor:
        try:
            bf16_peak = float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops"])
            bf16_src = "measured bf16_tflops (cuBLAS bf16 GEMM, burst)"
        except (OSError, KeyError, ValueError):
            bf16_peak, bf16_src = 1900.0, "fallback"
        mma = prefill_mma_flops(op, d)
        roofline = {"bound": "tensor", "achieved": tflops, "peak": bf16_peak, "unit": "TFLOP/s",
                    "frac": tflops / bf16_peak, "traffic": None, "peak_source": bf16_src,
                    "flops_per_token_head": prefill_flops(op, d),
                    "note": "algorithmic FLOPs of the chunk contractions (fp32 formulation) over "
                            "the dense bf16 tensor peak; the kernel's MMAs execute "
                            "mma_flops_per_token_head (hi/lo operand terms and padded rows)",
                    "mma_flops_per_token_head": mma,
                    "mma_tflops": units * mma / (ms / 1e3) / 1e12,
                    "fp32_equivalent_frac": tflops / FP32_PEAK_TFLOPS}
    else:
        roofline = {"bound": "alu", "achieved": tflops, "peak": FP32_PEAK_TFLOPS,
                    "unit": "TFLOP/s", "frac": tflops / FP32_PEAK_TFLOPS, "traffic": None,
                    "peak_source": "derived: 152 SMs x 128 FP32 lanes x 2 FLOP x 2.07 GHz",
                    "flops_per_token_head": prefill_flops(op, d)}
    result = {"metric": "prefill tokens·heads/s", "value": units * world / (ms / 1e3),
              "unit": "tokens·heads/s", "n_gpus": world, "steps": args.steps,
              "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
              "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
              "config": {"workload": "chunked prefill, " + w["desc"].split(",")[0] +
                         ", %d-token context per slot, outputs written" % T,
                         "op": gen.OP_NAMES[op], "B": B, "H": H, "d_k": d, "d_v": d,
                         "T": T, "chunk": PREFILL_C,
                         "l2": "inputs and state larger than L2"},
              "roofline": roofline,
              "clocks": clocks,
              "gpu_launches": args.steps * clocks.get("reps", 1) * ((B + 1023) // 1024)}
    ctx.close()
    del x, out
    torch.cuda.empty_cache()
    return result


def hbm_peak():
    """HBM copy bandwidth (GB/s): MEASURED_PEAKS.json, else the fallback figure."""
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return float(peaks["hbm_gbs"]), "measured hbm_gbs"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def run_checkpoint(args):
    """Prefix checkpoints: one bench step saves every slot of the GDN serving
    batch (its base, log rows and log length) into a device buffer and restores
    it.  Each slot holds an 8-entry log."""
    import torch
    rank, world, dist, local, dev, stream = gpu_setup()
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    from linear_attention_recurrent_gdn_gb300 import inputs as gen
    w = WORKLOADS["gdn"]
    op, B, H, d, M = w["op"], args.B or w["B"], w["H"], w["d"], w["M"]
    seed = w["seed"] + 7919 * rank
    ctx = dl.DeltaLog(op, B, H, d, d, M, stream=stream.cuda_stream)
    slots = list(range(B))
    ctx.set_state(slots, gen.initial_state(B, H, d, d, seed, device=dev))
    x = gen.make_inputs(op, 8, B, H, d, d, seed, device=dev)
    for t in range(8):
        ctx.step(slots, x["q"][t], x["k"][t], x["v"][t], x["g"][t], x["beta"][t])
    per = dl.dl_checkpoint_bytes(ctx._h)
    buf = torch.empty(B * per, dtype=torch.uint8, device=dev)

    def one():
        ctx.checkpoint_save(slots, buf)
        ctx.checkpoint_load(slots, buf)

    ms, clocks = timed_steps(one, args, dist, local, dev, stream)
    moved = 4 * B * per          # save reads and writes a record's bytes, restore too
    gbs = moved / (ms / 1e3) / 1e9
    peak, src = hbm_peak()
    result = {"metric": "checkpoint save + restore GB/s", "value": gbs * world, "unit": "GB/s",
              "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
              "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
              "data": "synthetic",
              "config": {"workload": "checkpoint save + restore of every slot, " +
                         w["desc"].split(",")[0] + ", M=%d, 8 log entries" % M,
                         "slots": B, "record_bytes": per,
                         "l2": "records larger than L2 (%.0f MB)" % (B * per / 1e6)},
              "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                           "frac": gbs / peak, "traffic": None, "peak_source": src},
              "clocks": clocks,
              "gpu_launches": args.steps * clocks.get("reps", 1) * 2 * ((B + 1023) // 1024)}
    if rank == 0:
        print(json.dumps(result), flush=True)
    ctx.close()
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_readstate(args):
    """Standalone Merge / ReadState kernel: one bench step materialises base +
    replayed log of every slot of the GDN serving batch (8-entry logs) into a
    caller buffer."""
    import torch
    rank, world, dist, local, dev, stream = gpu_setup()
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    from linear_attention_recurrent_gdn_gb300 import inputs as gen
    w = WORKLOADS["gdn"]
    op, B, H, d, M = w["op"], args.B or w["B"], w["H"], w["d"], w["M"]
    n_log = 8
    seed = w["seed"] + 7919 * rank
    ctx = dl.DeltaLog(op, B, H, d, d, M, stream=stream.cuda_stream)
    slots = list(range(B))
    ctx.set_state(slots, gen.initial_state(B, H, d, d, seed, device=dev))
    x = gen.make_inputs(op, n_log, B, H, d, d, seed, device=dev)
    for t in range(n_log):
        ctx.step(slots, x["q"][t], x["k"][t], x["v"][t], x["g"][t], x["beta"][t])
    out = torch.empty((B, H, d, d), dtype=torch.float32, device=dev)

    def one():
        ctx.read_state(slots, out)

    ms, clocks = timed_steps(one, args, dist, local, dev, stream)
    row = 4 * d + 2 * d + 4                       # one log entry: u fp32, k bf16, Λ
    moved = B * H * (2 * d * d * 4 + n_log * row)  # base read, state written, log rows read
    gbs = moved / (ms / 1e3) / 1e9
    peak, src = hbm_peak()
    result = {"metric": "read-state GB/s", "value": gbs * world, "unit": "GB/s",
              "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
              "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
              "data": "synthetic",
              "config": {"workload": "base + replayed log of every slot into a buffer, " +
                         w["desc"].split(",")[0] + ", M=%d, %d log entries" % (M, n_log),
                         "slots": B, "H": H, "d_k": d, "d_v": d,
                         "l2": "state larger than L2 (%.0f MB)" % (B * H * d * d * 4 / 1e6)},
              "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                           "frac": gbs / peak, "traffic": None, "peak_source": src},
              "clocks": clocks, "gpu_launches": args.steps * clocks.get("reps", 1)}
    if rank == 0:
        print(json.dumps(result), flush=True)
    ctx.close()
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_fork(args):
    """Forked decode as its own bench line (see measure_fork)."""
    rank, world, dist, local, dev, stream = gpu_setup()
    result = measure_fork(args, dist, world, rank, local, dev, stream)
    result.update({"metric": METRIC, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                   "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                   "dtype": "f32", "data": "synthetic"})
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def measure_fork(args, dist, world, rank, local, dev, stream):
    """Forked decode: bases are built once (setup, untimed); one bench step =
    fork every request into its branches (by index, no state copy) + the
    ragged branch decode until the longest branch ends."""
    import numpy as np
    import torch
    from linear_attention_recurrent_gdn_gb300 import deltalog as dl
    from linear_attention_recurrent_gdn_gb300 import inputs as gen
    w = WORKLOADS["fork"]
    R, NB, H, d, M, Tc = w["requests"], w["branches"], w["H"], w["d"], w["M"], w["ctx_tokens"]
    seed = w["seed"] + 7919 * rank
    lens = fork_plan(w, seed)
    order = np.argsort(-lens, kind="stable")
    Tq = int(lens.max())
    counts = [int((lens > t).sum()) for t in range(Tq)]
    S = R + R * NB
    fused = args.staging == "fused"
    ctx = dl.DeltaLog(0, S, H, d, d, M, stream=stream.cuda_stream,
                      staging=dl.STAGE_FUSED if fused else dl.STAGE_KERNELS)
    ctx.set_state(list(range(R)), gen.initial_state(R, H, d, d, seed, device=dev))
    t0 = time.time()
    xc = gen.make_inputs(0, Tc, R, H, d, d, seed, device=dev)     # the shared contexts
    ctx.prefill(list(range(R)), xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], want_out=False)
    torch.cuda.synchronize()
    del xc
    log("bases built (chunked prefill of %d tokens) in %.1fs" % (Tc, time.time() - t0))
    NBR = R * NB
    use_graph = not args.no_graph
    Tpad = (Tq + M - 1) // M * M if use_graph else Tq   # windows of M tokens; the tail is padding
    xq = gen.make_inputs(0, Tq, NBR, H, d, d, seed + 1, device=dev)
    if Tpad > Tq:
        xq = {k_: torch.cat([v_, torch.zeros((Tpad - Tq,) + tuple(v_.shape[1:]), dtype=v_.dtype,
                                             device=dev)]).contiguous()
              for k_, v_ in xq.items()}
    out = torch.empty((Tpad, NBR, H, d), dtype=torch.bfloat16, device=dev)
    act_slots = [[R + int(b) for b in order[:c]] for c in counts] + [[]] * (Tpad - Tq)
    branches = [[R + r * NB + i for i in range(NB)] for r in range(R)]
    wins = None
    if use_graph:
        wins = [ctx.window_ragged(NBR, xq["q"][w_ * M:(w_ + 1) * M], xq["k"][w_ * M:(w_ + 1) * M],
                                  xq["v"][w_ * M:(w_ + 1) * M], xq["g"][w_ * M:(w_ + 1) * M],
                                  xq["beta"][w_ * M:(w_ + 1) * M], out[w_ * M:(w_ + 1) * M])
                for w_ in range(Tpad // M)]

    def one():
        for r in range(R):
            ctx.fork(r, branches[r])
        if wins:
            for w_, win in enumerate(wins):
                win.launch(act_slots[w_ * M:(w_ + 1) * M])
            return
        for t in range(Tq):
            c = counts[t]
            ctx.step(act_slots[t], xq["q"][t][:c], xq["k"][t][:c], xq["v"][t][:c],
                     xq["g"][t][:c], xq["beta"][t][:c], out[t][:c])

    ms, clocks = timed_steps(one, args, dist, local, dev, stream)
    units = int(lens.sum()) * H
    # every branch starts at the source's log length 0, so the branches active at
    # token t all step with log length t mod M
    step_bytes = sum(counts[t] * H * fused_bytes(0, d, M, t % M)[0] for t in range(Tq))
    step_writes = sum(counts[t] * H * fused_bytes(0, d, M, t % M)[1] for t in range(Tq))
    eager_writes = units * eager_bytes(0, d)[1]
    gbs = step_bytes / (ms / 1e3) / 1e9
    peak, peak_src = hbm_peak()
    result = {"value": units * world / (ms / 1e3), "unit": "tokens·heads/s", "ms_per_step": ms,
              "config": fork_config(w, args, lens),
              "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                           "frac": gbs / peak, "traffic": None, "peak_source": peak_src,
                           "kernel": "AppendDecode over the ragged branch batch, fork "
                                     "launches included",
                           "bytes_per_step": step_bytes,
                           "timing": "whole bench step (forks + every branch token)"},
              "write_bytes_per_step": {"deltalog": step_writes, "eager": eager_writes},
              "write_cut_vs_eager": eager_writes / step_writes,
              "clocks": clocks,
              "gpu_launches": (R + (1 if fused else 2) * Tpad) * args.steps * clocks.get("reps", 1)}
    for win in wins or []:
        win.close()
    ctx.close()
    del xq, out
    torch.cuda.empty_cache()
    return result


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gdn",
                    choices=sorted(WORKLOADS) + sorted(PREFILL) + ["checkpoint", "readstate"])
    ap.add_argument("--M", type=int, default=0)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--B", type=int, default=0, help="override the batch (profiling runs only)")
    ap.add_argument("--tokens", type=int, default=0, help="override the token count (profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the decode loop as one dl_step call per token instead of CUDA graphs")
    ap.add_argument("--staging", default="fused", choices=["fused", "kernels"],
                    help="ReplayPrep as a warp role of AppendDecode (fused) or its own kernel")
    ap.add_argument("--eager", action="store_true",
                    help="time the in-house eager kernel (dense read-modify-write) instead")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other decode workloads the default run measures beside "
                         "the headline")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "fork":
        return run_fork(args)
    if args.workload in PREFILL:
        return run_prefill(args)
    if args.workload == "checkpoint":
        return run_checkpoint(args)
    if args.workload == "readstate":
        return run_readstate(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
