"""Offline sweep of the dispatcher's choices on the current GPU, and the least-squares
fit of its split cost model: the tile-config sweep that feeds the dispatch rules in
csrc/api.cu (decode_block_cols, make_plan's tile heights and its split cost model).

    python -m weight_only_int4_02_gb300.tune [--shapes M,K,N ...] [--group 128] [--out sweep.json]

Every setting runs in a fresh process, because the library reads its ablation knobs
once, from the environment: W4A16_DECODE_CB (columns per block of the decode kernel),
W4A16_TILE_M (rows of X per tile of the tensor-core kernel) and W4A16_SPLIT (parts a
tile is cut into when there are fewer tiles than SMs). A shape is timed the way the
benchmark times a layer: a CUDA Graph of launches back to back over rotating copies of
its packed weights (more bytes than L2), so that each launch streams its weights from
HBM and overlaps its predecessor as it would in a model; microseconds per launch, the
best of three replays. The report gives, per shape, the dispatcher's own time, the
fastest setting and the ratio; the fit gives, per tile height, the split cost model's
four constants from the split sweep.

This is a tuning tool (it needs a GPU and runs for minutes); nothing in the library or
the benchmark runs it.
"""
import argparse
import json
import os
import subprocess
import sys

import numpy as np

from weight_only_int4_02_gb300 import inputs

KNOBS = ("W4A16_DECODE_CB", "W4A16_TILE_M", "W4A16_SPLIT", "W4A16_SPLIT_ALL", "W4A16_MIN_ITERS")
DEFAULT_SHAPES = [(M, K, N) for M in (1, 8, 16, 32, 64, 128)
                  for (K, N) in ((4096, 12288), (4096, 4096), (4096, 22016), (11008, 4096))]


def sweep_plan(shapes, sms=152):
    """The settings to time: the dispatcher's own choice for every shape, the decode
    kernel's block widths for up to sixteen rows of X (K a multiple of 32), the tensor-core
    kernel's tile heights, and its split parts where a shape has fewer tiles than SMs.
    Returns [(env, force_path, shapes)]."""
    plan = [({}, 0, list(shapes))]
    dec = [s for s in shapes if s[0] <= 16 and s[1] % 32 == 0]
    for cb in (16, 32, 48, 64, 80, 128):
        cbs = [s for s in dec if s[0] <= 8 or cb not in (48, 80)]
        if cbs:
            plan.append(({"W4A16_DECODE_CB": str(cb)}, 3, cbs))
    for tm in (16, 32, 64, 128, 256):
        # tile heights from an eighth of the dispatcher's to twice it
        tms = [s for s in shapes if default_tm(s[0]) // 8 <= tm <= 2 * default_tm(s[0])]
        if tms:
            plan.append(({"W4A16_TILE_M": str(tm)}, 2, tms))
    few = [s for s in shapes if -(-s[2] // 128) * -(-s[0] // default_tm(s[0])) < sms]
    for sp in (1, 2, 3, 4, 6, 8):
        if few:
            plan.append(({"W4A16_SPLIT": str(sp)}, 2, few))
    return plan


def default_tm(M):
    """Rows of X per tile the dispatcher takes for M rows (make_plan)."""
    return 16 if M <= 16 else 32 if M <= 32 else 64 if M <= 64 else 128 if M <= 128 else 256


def split_features(iters, s, ring, rows):
    """The split cost model's terms for a tile of `iters` stages cut into s parts (make_plan):
    stages of the longest part prefetched (up to `ring`), stages streamed after them, and
    the fix-up's fixed and per-row terms."""
    n = -(-iters // s)
    pre = min(n, ring)
    return [pre, n - pre, 1.0 if s > 1 else 0.0, rows * (s - 1) if s > 1 else 0.0]


def fit_split_model(samples, ring):
    """Least-squares constants (prefetched_us, streamed_us, fixup_us, fixup_row_us) of
    the split cost model from samples [(iters, s, rows, us)], for a given ring depth."""
    A = np.array([split_features(it, s, ring, rows) for (it, s, rows, _) in samples], dtype=np.float64)
    b = np.array([us for (*_, us) in samples], dtype=np.float64)
    coef, *_ = np.linalg.lstsq(A, b, rcond=None)
    resid = float(np.sqrt(np.mean((A @ coef - b) ** 2))) if len(b) else 0.0
    return [float(c) for c in coef], resid


def best_settings(results):
    """Per shape: the dispatcher's own time, the fastest setting and its time.
    results: {setting label: {shape key: us}}, the label "default" for no knob."""
    out = {}
    for label, times in results.items():
        for key, us in times.items():
            e = out.setdefault(key, {"default_us": None, "best": None, "best_us": None})
            if label == "default":
                e["default_us"] = us
            if e["best_us"] is None or us < e["best_us"]:
                e["best"], e["best_us"] = label, us
    for e in out.values():
        if e["default_us"]:
            e["best_over_default"] = e["best_us"] / e["default_us"]
    return out


def _worker(force, shapes, G, reps):
    import torch
    from weight_only_int4_02_gb300 import w4a16
    w4a16.force_path(force)
    out = {}
    for (M, K, N) in shapes:
        q = torch.from_numpy(inputs.codes(K, N, 0)).cuda()
        s = torch.from_numpy(inputs.scales(K, N, G, 0)).cuda()
        packed, sp = w4a16.pack(q, s, G)
        del q, s
        nbytes = packed.numel() * 4 + sp.numel() * 2
        copies = [(packed, sp)] + [(packed.clone(), sp.clone()) for _ in range(max(1, int(400e6 // nbytes)))]
        x = torch.from_numpy(inputs.activations(M, K, 0)).cuda()
        y = torch.empty((M, N), dtype=torch.float16, device="cuda")
        for c in copies:
            w4a16.gemm(x, c[0], c[1], N, G, y=y)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=torch.cuda.Stream()):
            for r in range(reps):
                w4a16.gemm(x, copies[r % len(copies)][0], copies[r % len(copies)][1], N, G, y=y)
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        best = float("inf")
        for _ in range(3):
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b) * 1e3 / reps)
        if w4a16.check_device_status() != w4a16.OK:
            raise RuntimeError("a kernel wait timed out")
        out["%d,%d,%d" % (M, K, N)] = {"us": best, "plan": list(w4a16.plan(M, N, K, G))}
        del copies, packed, sp, g
        torch.cuda.empty_cache()
    print(json.dumps(out), flush=True)


def run_sweep(shapes, G, reps):
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    results, plans = {}, {}
    for env, force, sub in sweep_plan(shapes, sms):
        label = ",".join("%s=%s" % kv for kv in env.items()) or "default"
        e = dict(os.environ)
        for k in KNOBS:
            e.pop(k, None)
        e.update(env)
        cmd = [sys.executable, "-m", "weight_only_int4_02_gb300.tune", "--worker", str(force), "--group", str(G),
               "--reps", str(reps), "--shapes"] + ["%d,%d,%d" % s for s in sub]
        r = subprocess.run(cmd, env=e, capture_output=True, text=True, check=True)
        got = json.loads(r.stdout.strip().splitlines()[-1])
        results[label] = {k: v["us"] for k, v in got.items()}
        plans[label] = {k: v["plan"] for k, v in got.items()}
    return results, plans, sms


def fit_from_sweep(results, plans, shapes, sms, G):
    """Split cost model constants per tile height from the W4A16_SPLIT runs."""
    per_tm = {}
    for label, times in results.items():
        if not label.startswith("W4A16_SPLIT="):
            continue
        for key, us in times.items():
            M, K, N = (int(v) for v in key.split(","))
            path, tm, grid = plans[label][key]
            tiles = -(-N // 128) * -(-M // tm)
            if path != 2 or tiles >= sms:
                continue
            s = grid // tiles
            chunks = -(-K // 64)                     # 64-value chunks of k
            kc = -(-chunks // 4) * 4                 # padded to a multiple of four (make_plan's KC)
            iters = kc // (4 if tm <= 64 else 2)     # stages of 256 (or 128) values
            per_tm.setdefault(tm, []).append((iters, s, M if M <= tm else tm, us))
    out = {}
    for tm, samples in sorted(per_tm.items()):
        ring = 8.0 if tm <= 32 else 0.0
        coef, resid = fit_split_model(samples, ring)
        out[str(tm)] = {"ring": ring, "prefetched_us": coef[0], "streamed_us": coef[1], "fixup_us": coef[2],
                        "fixup_row_us": coef[3], "rms_us": resid, "samples": len(samples)}
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--shapes", nargs="*", default=None, help="M,K,N (default: the Llama-2-7B-like layers, M 1..128)")
    ap.add_argument("--group", type=int, default=128)
    ap.add_argument("--reps", type=int, default=40)
    ap.add_argument("--out", default=None, help="write the sweep, the best settings and the fit as JSON")
    ap.add_argument("--worker", type=int, default=None, help=argparse.SUPPRESS)
    a = ap.parse_args(argv)
    shapes = [tuple(int(v) for v in s.split(",")) for s in a.shapes] if a.shapes else DEFAULT_SHAPES
    if a.worker is not None:
        _worker(a.worker, shapes, a.group, a.reps)
        return
    results, plans, sms = run_sweep(shapes, a.group, a.reps)
    report = {"sms": sms, "results_us": results, "plans": plans, "best": best_settings(results),
              "split_model": fit_from_sweep(results, plans, shapes, sms, a.group)}
    for key, e in sorted(report["best"].items(), key=lambda kv: [int(v) for v in kv[0].split(",")]):
        print("%-16s dispatcher %7.2f us  best %-22s %7.2f us  (%.3f)" % (
            key, e["default_us"] or float("nan"), e["best"], e["best_us"], e.get("best_over_default", float("nan"))))
    for tm, f in report["split_model"].items():
        print("split model, %s-row tiles: %s" % (tm, json.dumps(f)))
    if a.out:
        with open(a.out, "w") as fh:
            json.dump(report, fh, indent=1)


if __name__ == "__main__":
    main()
