"""Benchmark: sparse-FFN decode tokens/s at batch 1 on one GB300, with the
achieved HBM bandwidth on the bytes the method must move.

Default workload: the OPT-175B-shaped INT4 FFN stack at full depth (96 layers,
d=12288, F=49152, predictor rank 1024, group-32 INT4 weights with fp16 scales,
Zipf(1.1) firing at 6%), one token per step through all 96 layers (predictor
-> compaction -> FC1 -> FC2, RMS normalisation between layers), inputs cycling
over the run's 64 seeded tokens.  The 77 GB of layer weights read per step are
far larger than L2, so no flush is needed.  After the headline, the other
workloads are timed the same way at batch 1 and full depth (OPT-125M-shaped
layer in rotation over copies larger than L2, OPT-6.7B-, OPT-30B- and
LLaMA-70B-shaped stacks) and listed under "other_workloads", with the launch
floor of the persistent kernel and one batch-1 call of the head-sparse
attention block of the same model shape ("attention_heads").

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config c5] [--impl ours|reference]

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle
instead (bounded sample of the same workload, scaled to tokens/s).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-FFN decode tokens/s at batch 1 and achieved HBM GB/s vs ~8 TB/s"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ ranks

def max_over_ranks(value: float, device: str = "cuda") -> float:
    """The largest `value` over all ranks (the slowest rank bounds the job);
    the value itself with one process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(ms_max: float, steps: int, batch: int, world: int) -> float:
    """Whole-job tokens/s: every rank runs `steps` steps of `batch` tokens on
    its own GPU (independent replicas, weak scaling); the job takes as long as
    its slowest rank."""
    return world * steps * batch / (ms_max / 1e3)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        except Exception:
            pass
        finally:
            if self.path and os.path.exists(self.path):
                os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------- algorithmic bytes

def layer_bytes(cfg, r, n_pred, n_relu, batch=1):
    """Bytes the method must move for one layer and one decode step:
    the predictor (P1, P2, bias) in full, the FC1 rows of the predicted-active
    neurons (gate + up rows when gated), the FC2 rows of the neurons whose FC1
    output is non-zero, and the small vectors (x, y, b2, mask, index list, h)."""
    d, F = cfg.d, cfg.F
    row = d // 2 + 2 * (d // 32) if cfg.int4 else 2 * d
    pred = 2 * (r * d + F * r) + 2 * F
    fc1 = n_pred * row * (2 if cfg.gated else 1)
    fc2 = n_relu * row + 2 * d
    small = batch * (2 * d + 4 * d) + batch * ((F + 31) // 32) * 4 + 4 * n_pred * (1 + batch)
    return dict(predict=pred, fc1=fc1, fc2=fc2, small=small, total=pred + fc1 + fc2 + small)


def measure_counts(st, tokens, B=1):
    """Untimed pass: per step (B tokens) and layer, the predicted-active count
    (the union of the B tokens' masks) and the number of listed neurons with a
    non-zero FC1 output for some token (one stack launch per step, through
    pi_ffn_stack's layer_counts output)."""
    out = []
    for t in range(0, tokens.shape[0], B):
        cnt = st.step_counts(tokens[t:t + B])
        out.append([tuple(int(v) for v in row) for row in cnt.cpu().tolist()])
    return out


def kernel_source_hash():
    """Hash of the fused kernel's sources: an ncu traffic figure is only
    reported while it was taken on the current kernel."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "activation_sparse_ffn_layer_gb300", "csrc")
    for name in ("pi_fused.cu", "pi_common.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(config_key):
    """DRAM bytes per launch of the fused kernel from the committed ncu summary
    of this workload, or None if absent or taken on a different kernel."""
    path = os.path.join(ROOT, "profiles", f"fused_stack_{config_key}_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ our arm

def step_bytes_of(cfg, layers, counts, B):
    """Algorithmic bytes of each step of the run (list over steps)."""
    L = len(layers)
    per_step = []
    for per in counts:
        tot = 0
        for l, (n, nz) in enumerate(per):
            tot += layer_bytes(cfg, layers[l].r, n, nz, B)["total"]
        tot += (L - 1) * B * (4 * cfg.d + 2 * cfg.d)   # inter-layer norm: read y, write x
        per_step.append(tot)
    return per_step


def measure_stack(cfg, B, L, K, W, sample_clocks=True):
    """Build a workload's stack on the GPU, count its algorithmic bytes
    (untimed pass), capture one step as a CUDA graph and time K replays after
    W warm-up replays.  Returns (result dict, objects for the e2e and CPU legs)."""
    import torch
    from activation_sparse_ffn_layer_gb300.runtime import DecodeStack
    from synth import make_layer, make_tokens

    t_gen = time.perf_counter()
    layers = [make_layer(cfg, l, device="cuda") for l in range(L)]
    torch.cuda.synchronize()
    t_gen = time.perf_counter() - t_gen
    NS = max(cfg.tokens // B, 4)          # distinct steps of B tokens, cycled
    T = NS * B
    tokens = make_tokens(cfg, 0, T, device="cuda")
    st = DecodeStack(layers, batch=B, tau=cfg.tau, eps=cfg.rms_eps)
    weight_bytes = sum(w.nbytes() for w in layers)
    # a stack whose weights fit in L2 (c1) is timed over R copies of itself in
    # rotation (one copy per step, more than twice L2 in all), so every step
    # reads its weights from HBM
    R = 1
    if weight_bytes < 2 * L2_BYTES:
        R = min(32, -(-2 * L2_BYTES // weight_bytes))
    stacks = [st] + [DecodeStack([clone_layer(w) for w in layers], batch=B, tau=cfg.tau, eps=cfg.rms_eps)
                     for _ in range(R - 1)]

    counts = measure_counts(st, tokens, B)
    per_step = step_bytes_of(cfg, layers, counts, B)
    n_pred_mean = sum(n for per in counts for n, _ in per) / (NS * L)
    n_relu_mean = sum(z for per in counts for _, z in per) / (NS * L)

    for s_ in stacks:
        s_.capture()
    stream = torch.cuda.current_stream()
    for i in range(max(W, R)):
        s_ = stacks[i % R]
        s_.x_in.copy_(tokens[(i % NS) * B:(i % NS + 1) * B])
        s_.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ka = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    kb = [torch.cuda.Event(enable_timing=True) for _ in range(K)]

    def timed():
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(K):
            t = (W + i) % NS
            s_ = stacks[(W + i) % R]
            s_.x_in.copy_(tokens[t * B:(t + 1) * B])
            ka[i].record(stream)
            s_.replay()
            kb[i].record(stream)
        e1.record(stream)
        torch.cuda.synchronize()

    clocks = None
    if sample_clocks:
        with ClockSampler(torch.cuda.current_device()) as clk:
            timed()
        clocks = clk.summary()
    else:
        timed()
    ms = e0.elapsed_time(e1)
    kernel_ms = sum(a.elapsed_time(b) for a, b in zip(ka, kb))
    step_bytes = sum(per_step[(W + i) % NS] for i in range(K)) / K
    res = dict(cfg=cfg, B=B, L=L, K=K, ms=ms, kernel_ms=kernel_ms, step_bytes=step_bytes,
               n_pred=n_pred_mean, n_relu=n_relu_mean, weight_bytes=weight_bytes, R=R, T=T,
               launches=st.launches_per_step(), clocks=clocks, gen_s=t_gen)
    return res, (layers, st, tokens, stacks)


def summary_line(res, peak):
    """Compact per-workload figures for the extra-workload list."""
    cfg, K, B = res["cfg"], res["K"], res["B"]
    per_launch = res["kernel_ms"] / K
    achieved = res["step_bytes"] / (per_launch / 1e3) / 1e9
    return {"workload": f"{cfg.key}: {cfg.name}, batch {B}, {res['L']} layers per step",
            "tokens_per_s": round(K * B / (res["ms"] / 1e3), 2), "us_per_step": round(res["ms"] / K * 1e3, 2),
            "bytes_per_step": int(res["step_bytes"]), "achieved_gbs": round(achieved, 1),
            "frac": round(achieved / peak, 4), "predicted_per_layer": round(res["n_pred"], 1),
            "l2": ("inputs larger than L2" if res["R"] == 1 else
                   f"{res['R']} copies of the stack in rotation, one per step"),
            "traffic": recorded_traffic(cfg.key) if res["launches"] == 1 and B == 1 and res["L"] == cfg.layers else None,
            "steps": K}


def launch_floor(K=200, W=20):
    """Time of one graph-replayed step of the smallest stack the persistent
    kernel takes (one layer, d = 256, F = 256, rank 8): the fixed cost of a
    launch and its two grid barriers (a one-layer step), with almost no bytes
    to move."""
    import torch
    from activation_sparse_ffn_layer_gb300.runtime import DecodeStack
    from synth import CONFIGS, make_layer, make_tokens, small
    cfg = small(CONFIGS["c1"], d=256, F=256, rank=8)
    w = make_layer(cfg, 0, device="cuda")
    st = DecodeStack([w], batch=1, tau=cfg.tau, eps=cfg.rms_eps)
    st.x_in.copy_(make_tokens(cfg, 0, 1, device="cuda"))
    st.capture()
    for _ in range(W):
        st.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        st.replay()
    e1.record()
    torch.cuda.synchronize()
    return round(e0.elapsed_time(e1) / K * 1e3, 2)


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)

    import __graft_entry__
    __graft_entry__.build()
    from synth import CONFIGS

    cfg = CONFIGS[args.config]
    B = args.batch
    L = args.layers if args.layers else cfg.layers
    K, W = args.steps, args.warmup
    if world > 1:
        dist.barrier()
    res, (layers, st, tokens, _stacks) = measure_stack(cfg, B, L, K, W)
    ms = res["ms"]
    if world > 1:
        ms = max_over_ranks(ms, "cuda")
        dist.barrier()
    kernel_ms = res["kernel_ms"]
    step_bytes = res["step_bytes"]
    tok_s = job_throughput(ms, K, B, world)
    peak, peak_kind = _peaks()

    # batch 1: a step is one launch of the fused stack kernel (the dominant and
    # only kernel); batch > 1: the per-step kernels of the graph, timed together
    per_launch = kernel_ms / K
    achieved = step_bytes / (per_launch / 1e3) / 1e9
    fused = res["launches"] == 1
    traffic = recorded_traffic(cfg.key) if fused and B == 1 and L == cfg.layers else None
    roofline = {"kernel": "k_fused_stack (pi_ffn_stack)" if fused else "batched step (pi_ffn_stack graph)",
                "bound": "hbm", "achieved": round(achieved, 1),
                "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": traffic, "peak_kind": peak_kind, "bytes_per_launch": int(step_bytes),
                "us_per_launch": round(per_launch * 1e3, 2), "share_of_step": round(kernel_ms / ms, 3)}

    e2e = time_e2e(st, tokens, K=min(K, 512), W=W, B=B)
    weight_bytes, R, T = res["weight_bytes"], res["R"], res["T"]
    out = {
        "metric": METRIC, "value": round(tok_s, 2), "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(ms / K, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{cfg.key}: {cfg.name}, batch {B}, {L} layers per step",
                   "batch": B, "layers": L, "d": cfg.d, "ffn": cfg.F, "tokens_cycled": T,
                   "weights": "int4-g32" if cfg.int4 else "fp16",
                   "l2": (f"inputs larger than L2 ({weight_bytes / 1e9:.1f} GB of layer weights per step)" if R == 1 else
                          f"inputs larger than L2: {R} copies of the {weight_bytes / 1e6:.1f} MB stack in rotation, "
                          f"one per step ({R * weight_bytes / 1e6:.0f} MB)"),
                   "parallelism": "replicas" if world > 1 else "single"},
        "achieved_gbs_step": round(step_bytes / (ms / K / 1e3) / 1e9, 1),
        "frac_step": round(step_bytes / (ms / K / 1e3) / 1e9 / peak, 4),
        "bytes_per_step": int(step_bytes),
        "active": {"predicted_per_layer": round(res["n_pred"], 1), "relu_nonzero_per_layer": round(res["n_relu"], 1),
                   "F": cfg.F},
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": K * res["launches"],
        "clocks": res["clocks"],
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(cfg, layers, st, tokens, budget_s=args.cpu_seconds)
    if rank == 0 and world == 1 and B == 1 and not args.no_extras:
        # the other workloads at batch 1 and full depth, each timed the same way
        del layers, st, tokens, _stacks
        torch.cuda.empty_cache()
        extras = []
        for key in args.extras.split(","):
            if not key or key == cfg.key:
                continue
            ec = CONFIGS[key]
            r_, objs = measure_stack(ec, 1, ec.layers, min(K, args.extra_steps) if ec.layers > 1 else
                                     max(K, 200), W, sample_clocks=False)
            extras.append(summary_line(r_, peak))
            del objs
            torch.cuda.empty_cache()
        out["other_workloads"] = extras
        out["launch_floor_us"] = launch_floor()
        # the head-sparse attention block of the same model shape, batch 1
        from activation_sparse_ffn_layer_gb300.entry_bench import run_attn
        if cfg.key in ("c2", "c3", "c4", "c5"):
            a = run_attn(cfg.key, 1, quiet=True)
            out["attention_heads"] = {k: a[k] for k in ("workload", "batch", "us", "bytes", "gbs", "frac_of_peak",
                                                        "heads", "union_heads", "cache_lengths")}
            torch.cuda.empty_cache()
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


L2_BYTES = 129 * 1000 * 1000   # GB300 L2 (nominal)


def clone_layer(w):
    """A copy of a layer's weights in fresh device memory (same values)."""
    import dataclasses
    import torch
    kw = {}
    for f in dataclasses.fields(w):
        v = getattr(w, f.name)
        kw[f.name] = v.clone() if isinstance(v, torch.Tensor) and v.is_cuda else v
    return type(w)(**kw)


def time_e2e(st, tokens, K, W, B=1):
    """Through the public API with host buffers: per step, copy the step's B
    tokens from pinned host memory, run the step, copy y back and read it on
    the host."""
    import torch
    NS = tokens.shape[0] // B
    host_x = tokens.cpu().pin_memory()
    host_y = torch.empty(st.y.shape, dtype=st.y.dtype).pin_memory()
    stream = torch.cuda.current_stream()
    for i in range(W):
        t = i % NS
        st.x_in.copy_(host_x[t * B:(t + 1) * B], non_blocking=True)
        st.replay()
        host_y.copy_(st.y, non_blocking=True)
        stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    acc = 0.0
    e0.record(stream)
    for i in range(K):
        t = i % NS
        st.x_in.copy_(host_x[t * B:(t + 1) * B], non_blocking=True)
        st.replay()
        host_y.copy_(st.y, non_blocking=True)
        stream.synchronize()
        acc += float(host_y[0, 0])                 # the host reads the step's result
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    return {"value": round(K * B / (ms / 1e3), 2), "unit": "tokens/s",
            "h2d_bytes_per_step": int(host_x[0:B].numel() * 2), "d2h_bytes_per_step": int(host_y.numel() * 4)}


def cpu_baseline(cfg, layers, st, tokens, budget_s=15.0):
    """The CPU oracle, as it stands, on a bounded sample: sampled layers of the
    first tokens, each fed with the GPU's input to that layer; scaled to
    tokens/s over the full depth."""
    import oracle
    cores = _cores()
    oracle.set_threads(cores)
    L = len(layers)
    B = st.batch
    NS = tokens.shape[0] // B
    sample_layers = sorted({0, 1, L // 2, L - 1}) if L > 1 else [0]
    hosts = {l: oracle.host_layer(layers[l].to("cpu")) for l in sample_layers}
    times = []
    t_start = time.perf_counter()
    t = 0
    while True:
        k = t % NS  # the first token of each step is evaluated
        xs, _ = st.step_trace(tokens[k * B:(k + 1) * B])
        for l in sample_layers:
            x = xs[l][0].cpu()
            t0 = time.perf_counter()
            oracle.layer_step(x, hosts[l], cfg.tau)
            times.append(time.perf_counter() - t0)
        t += 1
        if time.perf_counter() - t_start > budget_s and len(times) >= len(sample_layers):
            break
    per_layer = sum(times) / len(times)
    return {"value": round(1.0 / (per_layer * L), 4), "unit": "tokens/s", "cores": oracle.threads(),
            "kind": "oracle",
            "sample": f"{len(times)} layer-token evaluations (layers {sample_layers}, {t} tokens), "
                      f"mean {per_layer * 1e3:.1f} ms per layer, scaled to {L} layers"}


# ------------------------------------------------------------ reference arm

def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch
    import oracle
    from synth import CONFIGS, make_layer, make_tokens

    cfg = CONFIGS[args.config]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    L = cfg.layers
    sample_layers = sorted({0, 1, L // 2, L - 1}) if L > 1 else [0]
    hosts = {l: oracle.host_layer(make_layer(cfg, l, device=dev).to("cpu")) for l in sample_layers}
    toks = make_tokens(cfg, 0, cfg.tokens, device="cpu")
    cores = _cores()
    oracle.set_threads(cores)

    def one_step(i):
        # a bounded sample of one decode step: one sampled layer of one token
        l = sample_layers[i % len(sample_layers)]
        x = toks[i % cfg.tokens]
        oracle.layer_step(x, hosts[l], cfg.tau)

    for i in range(args.warmup):
        one_step(i)
    t0 = time.perf_counter()
    done = 0
    for i in range(args.steps):
        one_step(args.warmup + i)
        done += 1
        if time.perf_counter() - t0 > args.ref_seconds:
            break
    el = time.perf_counter() - t0
    per_layer = el / done
    value = 1.0 / (per_layer * L)
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": world,
           "steps": done, "warmup": args.warmup, "ms_per_step": round(per_layer * L * 1e3, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": f"{cfg.key}: {cfg.name}, batch 1, {L} layers per step", "batch": 1,
                      "layers": L},
           "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": oracle.threads(),
                            "kind": "oracle",
                            "sample": f"{done} layer evaluations over layers {sample_layers} "
                                      f"(token inputs of layer 0 used for every sampled layer), "
                                      f"scaled to {L} layers per token"},
           "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--config", default="c5")
    ap.add_argument("--batch", type=int, default=1, help="tokens per step (the headline workload is 1)")
    ap.add_argument("--layers", type=int, default=0, help="layers of the stack (0: the workload's own)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="time the headline workload only")
    ap.add_argument("--extras", default="c1,c2,c3,c4", help="other batch-1 workloads timed after the headline")
    ap.add_argument("--extra-steps", type=int, default=64)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
