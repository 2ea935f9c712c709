"""Measure the kernel and tile choices the planner makes, over a sweep of
YOLO-shaped layers, against every alternative the kernels can run.

"Fusing an Epilogue" (section "Three kernels for one operation") keeps its
kernel choice as hand-picked thresholds that somebody measures and writes
down, with a bench whose job is to check they still hold.  This is that
bench for this library: for each layer shape it times the planner's own
choice ("auto"), the CUDA-core direct kernel, and each tcgen05 tiling the
shape admits (pixel-major or channel-major tiles, whole tiles or stream-K,
single CTAs or 2-CTA pairs, 128- or 256-wide tiles; channel-major tiles dealt
whole or as equal runs of 32-pixel chunks), each call alone with
the L2 flushed before it, and reports how far the planner's choice is from
the fastest.

    python -m conv2d_batchnorm_silu_gb300.tune [--iters 24] [--json out.json]

Needs a GPU.  Every variant's output is checked against the planner's own
(bf16 results, same tolerance as the layer's) so that a fast wrong variant
cannot win.
"""
from __future__ import annotations

import argparse
import itertools
import json
import statistics
import sys

import torch

from . import capi
from .synthetic import LAYERS, LayerShape, bits_to_torch_bf16, make_layer_inputs

# YOLO-style backbone layers at 640x640 input, batch 8 (stem, downsampling 3x3
# stride-2 convolutions, C2f 1x1 and 3x3 bottleneck convolutions, SPPF 1x1),
# plus the five layers of the benchmark step.
SWEEP = [
    LayerShape("stem640", 8, 640, 640, 3, 32, 3, 3, 2, 1),
    LayerShape("down320", 8, 320, 320, 32, 64, 3, 3, 2, 1),
    LayerShape("c2f160_1x1", 8, 160, 160, 64, 64, 1, 1, 1, 0),
    LayerShape("bneck160", 8, 160, 160, 32, 32, 3, 3, 1, 1),
    LayerShape("down160", 8, 160, 160, 64, 128, 3, 3, 2, 1),
    LayerShape("c2f80_1x1", 8, 80, 80, 128, 128, 1, 1, 1, 0),
    LayerShape("bneck80", 8, 80, 80, 64, 64, 3, 3, 1, 1),
    LayerShape("down80", 8, 80, 80, 128, 256, 3, 3, 2, 1),
    LayerShape("c2f40_1x1", 8, 40, 40, 256, 256, 1, 1, 1, 0),
    LayerShape("bneck40", 8, 40, 40, 128, 128, 3, 3, 1, 1),
    LayerShape("down40", 8, 40, 40, 256, 512, 3, 3, 2, 1),
    LayerShape("c2f20_1x1", 8, 20, 20, 512, 512, 1, 1, 1, 0),
    LayerShape("bneck20", 8, 20, 20, 256, 256, 3, 3, 1, 1),
    LayerShape("sppf20_1x1", 8, 20, 20, 512, 256, 1, 1, 1, 0),
    LayerShape("head80_3x3", 8, 80, 80, 128, 64, 3, 3, 1, 1),
] + [LAYERS[n] for n in ("tiny", "stem", "down", "pointwise", "deep")]


def variants():
    """(label, overrides) for every alternative; unsupported ones are skipped per shape."""
    yield "auto", {}
    yield "direct", {"algo": "direct"}
    # channel-major tiles on the kernel of tc_cmajor.cu: x in boxes of whole output rows (or of
    # the [M][C] matrix of a 1x1 layer) or in im2col boxes, the weights streamed or resident
    yield "rows", {"algo": "tcgen05", "row_boxes": 1, "weights_resident": 0}
    yield "rows-wres", {"algo": "tcgen05", "row_boxes": 1, "weights_resident": 1}
    yield "wres", {"algo": "tcgen05", "row_boxes": 0, "weights_resident": 1}
    for swap, sk, pair, bn in itertools.product((0, 1), (0, 1), (0, 1), (128, 256)):
        if swap and (sk or pair or bn != 256):
            continue
        if pair and (not sk or bn != 256):
            continue
        if swap:
            # channel-major: equal runs of 32-pixel chunks, or whole 256-pixel tiles
            yield "swap", {"algo": "tcgen05", "swap_ab": 1, "stream_k": 0, "pair": 0, "block_n": 0, "balanced": 1,
                           "weights_resident": 0, "row_boxes": 0}
            yield "swap-tiles", {"algo": "tcgen05", "swap_ab": 1, "stream_k": 0, "pair": 0, "block_n": 0,
                                 "balanced": 0, "weights_resident": 0, "row_boxes": 0}
            continue
        label = f"n{bn}{'-sk' if sk else ''}{'-pair' if pair else ''}"
        yield label, {"algo": "tcgen05", "swap_ab": swap, "stream_k": sk, "pair": pair, "block_n": bn}


def _time(call, iters, flush, stream):
    evs = []
    with torch.cuda.stream(stream):
        for _ in range(iters):
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            evs.append((a, b))
    torch.cuda.synchronize()
    # Event times come in steps of about 2 us on this GPU; the mean of the middle half of
    # the samples resolves differences below that step (the flush and launch jitter spread
    # the samples across it), where a median would land on one step.
    ts = sorted(a.elapsed_time(b) for a, b in evs)
    mid = ts[len(ts) // 4: len(ts) - len(ts) // 4] or ts
    return 1e3 * statistics.fmean(mid)


def _close(a: torch.Tensor, b: torch.Tensor) -> bool:
    fa, fb = a.float(), b.float()
    return bool(torch.all((fa - fb).abs() <= 2e-2 + 2e-2 * fb.abs()).item())


def sweep(iters: int = 24, shapes=SWEEP, log=sys.stderr) -> list[dict]:
    dev = torch.device("cuda:0")
    stream = torch.cuda.Stream(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    rows = []
    for sh in shapes:
        inp = make_layer_inputs(sh)
        x = bits_to_torch_bf16(inp.x_bits).to(dev)
        w = bits_to_torch_bf16(inp.w_bits).to(dev)
        g, b, m, v = (torch.from_numpy(t).to(dev) for t in (inp.gamma, inp.beta, inp.mean, inp.var))
        scale, bias = capi.fold(g, b, m, v, inp.eps)
        ref = capi.forward(x, w, scale, bias, sh.stride, sh.pad)
        auto_plan = capi.plan(sh.n, sh.h, sh.w, sh.c, sh.k, sh.r, sh.s, sh.stride, sh.pad, "auto", sms)
        times = {}
        for label, ov in variants():
            try:
                capi.plan_request(sh.n, sh.h, sh.w, sh.c, sh.k, sh.r, sh.s, sh.stride, sh.pad, sms, **ov)
            except capi.CbsError:
                continue
            y = torch.empty_like(ref)

            def call(ov=ov, y=y):
                capi.forward_request(x, w, scale, bias, sh.stride, sh.pad, y=y, stream=stream, **ov)

            with torch.cuda.stream(stream):
                for _ in range(2):
                    call()
            torch.cuda.synchronize()
            capi.check(stream)
            if not _close(y, ref):
                times[label] = None  # a variant that disagrees never counts
                continue
            times[label] = round(_time(call, iters, flush, stream), 3)
        valid = {k: t for k, t in times.items() if t is not None}
        best = min(valid, key=valid.get)
        row = {"layer": sh.name, "shape": [sh.n, sh.h, sh.w, sh.c, sh.k, sh.r, sh.s, sh.stride, sh.pad],
               "gflop": round(sh.flops / 1e9, 3), "planner": _plan_label(auto_plan), "times_us": times,
               "best": best, "auto_over_best": round(valid["auto"] / valid[best], 3)}
        rows.append(row)
        print(json.dumps(row), file=log, flush=True)
    return rows


def _plan_label(pl: dict) -> str:
    if pl["algo"] == "direct":
        return "direct"
    if pl["threads"] == 288:  # the thin-input kernel's CTA
        return "thin-input"
    if pl.get("row_boxes"):
        return "rows-wres" if pl.get("weights_resident") else "rows"
    if pl.get("weights_resident"):
        return "wres"
    if pl["swap_ab"]:
        return "swap" if pl.get("balanced") else "swap-tiles"
    return f"n{pl['block_n']}{'-sk' if pl['stream_k'] else ''}{'-pair' if pl['cluster'] == 2 else ''}"


def markdown(rows: list[dict]) -> str:
    out = ["| layer | N,H,W,C -> K, RxS/s/p | GFLOP | planner | auto us | best | best us | auto/best |",
           "|---|---|---|---|---|---|---|---|"]
    for r in rows:
        n, h, w, c, k, rr, s, st, p = r["shape"]
        t = r["times_us"]
        out.append(f"| {r['layer']} | {n},{h},{w},{c} -> {k}, {rr}x{s}/{st}/{p} | {r['gflop']} | {r['planner']} | "
                   f"{t['auto']} | {r['best']} | {t[r['best']]} | {r['auto_over_best']} |")
    return "\n".join(out)


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--iters", type=int, default=24)
    ap.add_argument("--json", default=None, help="write the rows to this file")
    args = ap.parse_args(argv)
    if not torch.cuda.is_available():
        print("tune: needs a CUDA device", file=sys.stderr)
        return 2
    rows = sweep(args.iters)
    if args.json:
        with open(args.json, "w") as f:
            json.dump(rows, f, indent=1)
    print(markdown(rows))
    worst = max(r["auto_over_best"] for r in rows)
    print(f"\nplanner within {100 * (worst - 1):.1f}% of the fastest measured variant on every layer"
          if worst <= 1.05 else f"\nplanner up to {100 * (worst - 1):.1f}% slower than the fastest variant")
    return 0


if __name__ == "__main__":
    sys.exit(main())
