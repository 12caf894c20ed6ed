"""Timing of the C-ABI entry points one by one on a workload's layer.

For a configuration and batch size this times, through the library's own
calls, ``pi_predict``, ``pi_compact``, ``pi_sparse_fc1``, ``pi_sparse_fc2``,
``pi_rmsnorm_half`` and ``pi_ffn_layer`` (CUDA graphs of 10 calls, CUDA events,
two layers in alternation so that neither is left in L2 by the previous call)
and prints one JSON line per call with its time and the algorithmic bytes it
moves: the predictor weights for ``pi_predict``, the listed rows for the FC
calls (FC2 counts the rows whose FC1 output is non-zero for some token).

    python -m activation_sparse_ffn_layer_gb300.entry_bench --config c2 --batch 1
    python -m activation_sparse_ffn_layer_gb300.entry_bench --config c5 --batch 4 --once
    python -m activation_sparse_ffn_layer_gb300.entry_bench --config c4 --cold host

``--attn`` times ``pi_attn_heads`` (the head-sparse attention block) instead,
on the workload's attention shape with a decode-length cache; its bytes are
the head predictor, the query rows of the heads some token uses, every key
and value row, the output-projection rows of those heads and the cache rows
the active (head, token) pairs read.

``--once`` runs every call a few times eagerly and then once more, without
graphs or timing, which is the shape a profiler capture wants.  ``--cold host``
times the tiered FC calls instead, with the FC rows from ``--n-hot`` on (default
0: all of them) in pinned host memory, read by the GPU directly.
"""
from __future__ import annotations

import argparse
import json
import os

import torch

from . import binding as B

HERE = os.path.dirname(os.path.abspath(__file__))


def _peak_gbs() -> float:
    try:
        with open(os.path.join(os.path.dirname(HERE), "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"])
    except Exception:
        return 6800.0


def _time(fn, reps: int = 200) -> float:
    """Microseconds per call: graph-replayed batches of 10 calls."""
    for _ in range(5):
        fn()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(10):
            fn()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps // 10):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps * 1e3


def _cold_rows(w, n_hot: int, where: str):
    """The FC rows of w from n_hot on, in pinned host memory or a device buffer."""
    def cold(t):
        if t is None:
            return None
        c = t[n_hot:].contiguous()
        return c.cpu().pin_memory() if where == "host" else c.clone()
    if w.int4:
        return dict(w1=cold(w.w1_q), w1_scales=cold(w.w1_s), w2t=cold(w.w2t_q), w2t_scales=cold(w.w2t_s))
    return dict(w1=cold(w.w1), wu=cold(w.wu), w2t=cold(w.w2t))


def run(config: str, batch: int, once: bool = False, cold: str = "", n_hot: int = 0):
    from synth import CONFIGS, make_layer, make_tokens

    B.lib()
    cfg = CONFIGS[config]
    dev = "cuda"
    layers = [make_layer(cfg, l, device=dev) for l in range(2)]
    d, F = cfg.d, cfg.F
    x = make_tokens(cfg, 0, batch, device=dev)
    desc = B.layer_desc(layers[0], batch)
    ws = torch.zeros(B.pi_workspace_bytes(desc), dtype=torch.uint8, device=dev)
    W = (F + 31) // 32
    mask = torch.zeros(batch, W, dtype=torch.int32, device=dev)
    idx = torch.zeros(F, dtype=torch.int32, device=dev)
    cnt = torch.zeros(1, dtype=torch.int32, device=dev)
    h = torch.zeros(F * batch, dtype=torch.float32, device=dev)
    y = torch.zeros(batch, d, dtype=torch.float32, device=dev)
    xn = torch.zeros(batch, d, dtype=torch.float16, device=dev)
    wst = [B.weights_struct(w) for w in layers]
    turn = [0]

    def nxt() -> int:
        turn[0] += 1
        return turn[0] % 2

    def predict():
        w = layers[nxt()]
        B.pi_predict(desc, x, w.p1, w.p2, w.b1, cfg.tau, mask, ws)

    def compact():
        B.pi_compact(desc, mask, None, idx, None, cnt)

    def fc1():
        B.pi_sparse_fc1(desc, x, wst[nxt()], idx, cnt, mask if batch > 1 else None, h, ws)

    def fc2():
        B.pi_sparse_fc2(desc, h, idx, cnt, wst[nxt()], y, ws)

    def norm():
        B.pi_rmsnorm_half(d, batch, y, cfg.rms_eps, xn)

    def layer():
        B.pi_ffn_layer(desc, x, wst[nxt()], cfg.tau, ws, y)

    # one real pass so that the list, h and y hold this layer's values
    predict()
    compact()
    fc1()
    fc2()
    torch.cuda.synchronize()
    n = int(cnt.item())
    live = int((h[: n * batch].view(n, batch) != 0).any(dim=1).sum().item()) if n else 0
    calls = [("pi_predict", predict), ("pi_compact", compact), ("pi_sparse_fc1", fc1),
             ("pi_sparse_fc2", fc2), ("pi_rmsnorm_half", norm), ("pi_ffn_layer", layer)]
    if cold:
        # the rows from n_hot on in a second tier (0: every FC row)
        keep = [_cold_rows(w, n_hot, cold) for w in layers]
        tiers = [B.cold_tier(n_hot, **k) for k in keep]

        def fc1_t():
            k = nxt()
            B.pi_sparse_fc1_tiered(desc, x, wst[k], tiers[k], idx, cnt, mask if batch > 1 else None, h)

        def fc2_t():
            k = nxt()
            B.pi_sparse_fc2_tiered(desc, h, idx, cnt, wst[k], tiers[k], y, ws)

        def layer_t():
            k = nxt()
            B.pi_ffn_layer_tiered(desc, x, wst[k], tiers[k], cfg.tau, ws, y)
        calls = [("pi_sparse_fc1_tiered", fc1_t), ("pi_sparse_fc2_tiered", fc2_t),
                 ("pi_ffn_layer_tiered", layer_t)]
    if once:
        for name, fn in calls:
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            fn()
            torch.cuda.synchronize()
        print(json.dumps({"config": config, "batch": batch, "listed": n, "live": live, "mode": "once"}))
        return
    w0 = layers[0]
    row = d // 2 + d // 16 if cfg.int4 else 2 * d
    pred_b = 2 * (w0.r * d + F * w0.r) + 2 * F
    fc1_b = n * row * (2 if cfg.gated else 1)
    fc2_b = live * row
    moved = {"pi_predict": pred_b, "pi_compact": 4 * batch * W + 4 * n, "pi_sparse_fc1": fc1_b,
             "pi_sparse_fc2": fc2_b, "pi_rmsnorm_half": batch * d * 6,
             "pi_ffn_layer": pred_b + fc1_b + fc2_b, "pi_sparse_fc1_tiered": fc1_b,
             "pi_sparse_fc2_tiered": fc2_b, "pi_ffn_layer_tiered": pred_b + fc1_b + fc2_b}
    extra = {}
    if cold:
        listed = idx[:n].cpu()
        extra = {"cold": cold, "n_hot": n_hot, "listed_cold": int((listed >= n_hot).sum().item())}
    peak = _peak_gbs()
    for name, fn in calls:
        us = _time(fn)
        gbs = moved[name] / us / 1e3
        print(json.dumps({"call": name, "config": config, "batch": batch, "us": round(us, 2),
                          "bytes": moved[name], "gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
                          "listed": n, "live": live, **extra}), flush=True)


def run_attn(config: str, batch: int, once: bool = False, max_seq: int = 1024, quiet: bool = False,
             context: int = 0):
    """Times pi_attn_heads; returns the result line as a dict (also printed
    unless quiet).  context > 0: every sequence's cache holds that many
    positions (the capacity grows to fit) instead of the decode-length mix."""
    from synth import ATTN_CONFIGS, decode_lengths, make_attn, make_kv_cache

    B.lib()
    cfg = ATTN_CONFIGS[config]
    dev = "cuda"
    blocks = [make_attn(cfg, l, device=dev) for l in range(2)]
    H, KVH, dh, d = cfg.heads, cfg.kv_heads, cfg.head_dim, cfg.d
    lengths = decode_lengths(cfg, batch)
    if context > 0:
        lengths = [context] * batch
        max_seq = max(max_seq, context + 1)
    caches = [make_kv_cache(cfg, lengths, seed=l, device=dev, max_seq=max_seq) for l in range(2)]
    g = torch.Generator(device=dev).manual_seed(7)
    x = torch.randn(batch, d, generator=g, device=dev).to(torch.float16)
    desc = B.attn_desc(blocks[0], batch, max_seq)
    ws = torch.empty(B.pi_attn_workspace_bytes(desc), dtype=torch.uint8, device=dev)
    pos = torch.tensor(lengths, dtype=torch.int32, device=dev)
    mask = torch.zeros(batch, (H + 31) // 32, dtype=torch.int32, device=dev)
    y = torch.zeros(batch, d, dtype=torch.float32, device=dev)
    st = [B.attn_weights_struct(w) for w in blocks]
    turn = [0]

    def call():
        turn[0] += 1
        k = turn[0] % 2
        B.pi_attn_heads(desc, x, st[k], caches[k][0], caches[k][1], pos, cfg.tau, mask, y, ws)

    call()
    torch.cuda.synchronize()
    if once:
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        call()
        torch.cuda.synchronize()
        print(json.dumps({"call": "pi_attn_heads", "config": config, "batch": batch, "mode": "once"}))
        return
    # bytes of the block for the masks the call computes (both blocks alike)
    call()
    torch.cuda.synchronize()
    m = mask.cpu().numpy().astype("int64") & 0xFFFFFFFF
    on = [[(int(m[b, h // 32]) >> (h % 32)) & 1 for h in range(H)] for b in range(batch)]
    union = sum(1 for h in range(H) if any(on[b][h] for b in range(batch)))
    pairs_kv = sum(lengths[b] * on[b][h] for b in range(batch) for h in range(H))
    w0 = blocks[0]
    row = 2 * d
    moved = (2 * (w0.r * d + H * w0.r + H) + (union + 2 * KVH) * dh * row + 2 * (union + 2 * KVH) * dh
             + union * dh * row + pairs_kv * 2 * dh * 2 + batch * d * 2 + batch * d * 4)
    us = _time(call)
    gbs = moved / us / 1e3
    peak = _peak_gbs()
    res = {"call": "pi_attn_heads", "config": config, "workload": cfg.name, "batch": batch, "us": round(us, 2),
           "bytes": moved, "gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
           "heads": H, "union_heads": union, "active_pairs": int(sum(map(sum, on))),
           "cache_lengths": lengths[:4], "max_seq": max_seq}
    if not quiet:
        print(json.dumps(res), flush=True)
    return res


def main(argv=None):
    ap = argparse.ArgumentParser(description="time the C-ABI entry points on one layer of a workload")
    ap.add_argument("--config", default="c2")
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--once", action="store_true", help="run each call once after a warm-up (profiler captures)")
    ap.add_argument("--cold", default="", choices=["", "host", "device"],
                    help="time the tiered FC calls with the rows past the hot prefix in pinned host memory "
                         "or in a second device buffer")
    ap.add_argument("--n-hot", type=int, default=0, help="rows kept in the first tier with --cold (0: none)")
    ap.add_argument("--attn", action="store_true", help="time the head-sparse attention block instead")
    ap.add_argument("--context", type=int, default=0, help="with --attn: cache positions per sequence "
                    "(default: a 128-token prompt plus ragged decode steps)")
    args = ap.parse_args(argv)
    assert torch.cuda.is_available(), "needs a CUDA GPU"
    if args.attn:
        run_attn(args.config, args.batch, args.once, context=args.context)
    else:
        run(args.config, args.batch, args.once, args.cold, args.n_hot)


if __name__ == "__main__":
    main()
