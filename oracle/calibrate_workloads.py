"""Write ``workloads/calibration.json``: the routing structure of the named
workloads, computed with the oracle's router.  TEST INFRASTRUCTURE; run once
(``python -m oracle.calibrate_workloads``) and commit its output.

For every workload, tokens whose k-th and (k+1)-th ranking scores (s + b) lie
closer than GAP_MIN are re-drawn from the next stream of the generator until
the gap holds, so that the selected expert set is decided by a margin far above
float32 rounding.  For the "zipf" workload the correction bias is fitted by a
fixed-point iteration so that the expert loads follow min(T, C * rank^-s) with
sum T*k over the live experts, the last ``zipf_dead`` experts of the seeded
permutation getting bias -2 (they are never selected).
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import numpy as np
import torch

import workloads as wl
from oracle.moe_oracle import router_scores, topk_gap

GAP_MIN = 1e-3


def zipf_targets(T: int, k: int, n_live: int, s: float) -> np.ndarray:
    """Water-filled Zipf loads: c_i = min(T, C * i**-s), i = 1..n_live, sum = T*k."""
    ranks = np.arange(1, n_live + 1, dtype=np.float64)
    lo, hi = 0.0, float(T * k) * 10
    for _ in range(200):
        C = 0.5 * (lo + hi)
        if np.minimum(T, C * ranks ** -s).sum() < T * k:
            lo = C
        else:
            hi = C
    return np.minimum(T, hi * ranks ** -s)


def _topk_counts(r: np.ndarray, k: int) -> np.ndarray:
    idx = np.argpartition(-r, k - 1, axis=1)[:, :k]
    return np.bincount(idx.ravel(), minlength=r.shape[1])


def fit_bias(s: np.ndarray, target: np.ndarray, dead: np.ndarray, k: int, b0: np.ndarray,
             iters: int = 600) -> np.ndarray:
    b = b0.copy()
    b[dead] = -2.0
    live = ~dead
    for it in range(iters):
        cnt = _topk_counts(s + b[None, :], k)
        err = np.log(target + 0.5) - np.log(cnt + 0.5)
        step = 0.02 if it < iters // 2 else 0.005
        b[live] += step * err[live]
    return b


def redraw(w: wl.Workload, x: torch.Tensor, W: np.ndarray, b: np.ndarray,
           attempts: dict, max_rounds: int = 200) -> np.ndarray:
    """Re-draw tokens until every gap >= GAP_MIN.  Updates ``x`` and ``attempts``.
    Returns the final s [T, E]."""
    xf = x.to(torch.float64).numpy()
    _, s, r = router_scores(xf, W, b)
    for _ in range(max_rounds):
        bad = np.nonzero(topk_gap(r, w.k) < GAP_MIN)[0]
        if len(bad) == 0:
            return s
        for t in bad:
            attempts[int(t)] = attempts.get(int(t), 0) + 1
        xb = wl.gen_x(w, tokens=bad, attempts=attempts)
        x[bad] = xb
        _, sb, rb = router_scores(xb.to(torch.float64).numpy(), W, b)
        s[bad] = sb
        r[bad] = rb
    raise RuntimeError(f"{w.name}: gap not reached after {max_rounds} rounds")


def calibrate(w: wl.Workload) -> dict:
    attempts: dict = {}
    x = wl.gen_x(w, attempts={})
    Wt, bt = wl.gen_router(w)  # zipf: default bias before fitting
    W = Wt.numpy().astype(np.float64)
    out: dict = {}
    if w.routing == "zipf":
        perm = wl.expert_permutation(w).numpy()
        n_live = w.E - w.zipf_dead
        dead = np.zeros(w.E, dtype=bool)
        dead[perm[n_live:]] = True
        tgt = np.zeros(w.E)
        tgt[perm[:n_live]] = zipf_targets(w.T, w.k, n_live, w.zipf_s)
        b = np.zeros(w.E)
        for _ in range(3):
            _, s, _ = router_scores(x.to(torch.float64).numpy(), W, np.zeros(w.E))
            b = fit_bias(s, tgt, dead, w.k, b)
            b32 = b.astype(np.float32)
            redraw(w, x, W, b32.astype(np.float64), attempts)
        b32 = b.astype(np.float32)
        out["bias_bits"] = [int(v) for v in b32.view(np.uint32)]
        out["zipf_target"] = [round(float(v), 2) for v in tgt]
        bias = b32.astype(np.float64)
    else:
        bias = bt.numpy().astype(np.float64)
    s = redraw(w, x, W, bias, attempts)
    r = s + bias[None, :]
    gap = topk_gap(r, w.k)
    idx = np.argsort(-r, axis=1, kind="stable")[:, : w.k]
    counts = np.bincount(idx.ravel(), minlength=w.E)
    out["resample"] = {str(t): a for t, a in sorted(attempts.items())}
    out["min_gap"] = float(gap.min())
    out["counts"] = [int(c) for c in counts]
    out["active_experts"] = int((counts > 0).sum())
    return out


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("names", nargs="*", default=list(wl.WORKLOADS))
    args = ap.parse_args(argv)
    path = os.path.join(os.path.dirname(wl.__file__), "calibration.json")
    data = {}
    if os.path.exists(path):
        with open(path) as f:
            data = json.load(f)
    data["gap_min"] = GAP_MIN
    for name in args.names:
        w = wl.WORKLOADS[name]
        res = calibrate(w)
        data[name] = res
        print(f"{name}: redrawn {len(res['resample'])} tokens, min gap {res['min_gap']:.3e}, "
              f"active experts {res['active_experts']}, max count {max(res['counts'])}",
              file=sys.stderr)
    with open(path, "w") as f:
        json.dump(data, f, indent=0, sort_keys=True)
        f.write("\n")


if __name__ == "__main__":
    main()
