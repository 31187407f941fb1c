"""Shared test utilities: conditioned inputs, device weights, tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
import workloads as wl
from oracle import inputs as oi

# Float tolerance of the layer output against the fp64 oracle (relative L2 and
# max-abs as a fraction of the oracle's RMS).
REL_L2 = 5e-3
MAX_ABS_FRAC = 3e-2
GAP_MIN = 1e-3


def conditioned_attempts(w: wl.Workload, max_rounds: int = 100) -> dict:
    """Re-draw counters that give every token a top-k gap >= GAP_MIN (oracle router).

    Named workloads use the stored calibration; other shapes are conditioned here."""
    if w.name in wl.calibration() and w.T == wl.WORKLOADS[w.name].T and w.H == wl.WORKLOADS[w.name].H \
            and w.E == wl.WORKLOADS[w.name].E and w.k == wl.WORKLOADS[w.name].k:
        return wl.resample_counts(w)
    W, b = wl.gen_router(w)
    attempts: dict = {}
    x = wl.gen_x(w, attempts=attempts)
    for _ in range(max_rounds):
        rt = O.route(oi.x_f64(x), W.numpy(), b.numpy(), w.k, w.renorm)
        bad = np.nonzero(O.topk_gap(rt.r, w.k) < GAP_MIN)[0]
        if len(bad) == 0:
            return attempts
        for t in bad:
            attempts[int(t)] = attempts.get(int(t), 0) + 1
        x[bad] = wl.gen_x(w, tokens=bad, attempts=attempts)
    raise RuntimeError("could not condition the router gap")


def device_weights(w: wl.Workload, device, router=None, latent=None):
    if router is None:
        router = wl.gen_router(w)
    if latent is None and w.L:
        latent = wl.gen_latent(w)
    W, b = router
    out = {"router_w": W.to(device), "router_bias": b.to(device), **wl.gen_experts(w, device)}
    if latent is not None:
        out.update({k: v.to(device) for k, v in latent.items()})
    return out


def rel_l2(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def assert_close(got, ref, rel=REL_L2, max_abs_frac=MAX_ABS_FRAC, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    e = rel_l2(got, ref)
    rms = np.sqrt(np.mean(ref * ref))
    mx = float(np.abs(got - ref).max()) if got.size else 0.0
    assert e <= rel, f"{what}: relative L2 {e:.3e} > {rel:.1e}"
    assert mx <= max_abs_frac * rms, f"{what}: max abs {mx:.3e} > {max_abs_frac:.0e} * rms {rms:.3e}"
    return e


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return oi.bf16_bits(t)


def random_topk(T: int, E: int, k: int, rng: np.random.Generator, hot=None) -> np.ndarray:
    """Random valid top-k lists (distinct experts per token); ``hot`` experts
    are preferred with the given probability weights when set."""
    out = np.empty((T, k), dtype=np.int32)
    p = None
    if hot is not None:
        p = np.asarray(hot, dtype=np.float64)
        p = p / p.sum()
    for t in range(T):
        out[t] = rng.choice(E, size=k, replace=False, p=p)
    return out


def fp32_group_chain(P, scale_bits, x_scale) -> np.ndarray:
    """The fp32 evaluation the library states for act_bits 8 (include/moe.h,
    moe_int4_linear): acc = fma(scale[n, g], P[r, n, g], acc) over the groups
    g in K order from acc = 0, then y = x_scale[r] * acc, all IEEE fp32.

    P [R, N, G] exact integers (int64), scale_bits bf16 [N, G], x_scale fp32
    [R].  Every product scale * P is exact in fp32 (8 significant bits times
    at most 15), so each fma is one fp32 addition of the exact product."""
    P = np.asarray(P)
    s = O.bf16_bits_to_f64(scale_bits).astype(np.float32)  # exact
    acc = np.zeros(P.shape[:2], dtype=np.float32)
    for g in range(P.shape[2]):
        prod = s[None, :, g] * P[:, :, g].astype(np.float32)  # exact in fp32
        acc = (acc + prod).astype(np.float32)
    return (acc * np.asarray(x_scale, dtype=np.float32)[:, None]).astype(np.float32)


def _round_f32(x) -> float:
    """The float32 nearest to the exact rational x (ties to even), as a float."""
    from fractions import Fraction
    x = Fraction(x)
    if x == 0:
        return 0.0
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)                       # subnormal spacing below 2^-126
    step = Fraction(2) ** (e - 23)
    m = a / step
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return float(sign * n * step)


def fp32_fma_chain(P, scale_bits, x_scale) -> np.ndarray:
    """acc = fma(scale[n, g], P[r, n, g], acc) over g in K order from 0, then
    y = x_scale[r] * acc, each fma and the product rounded once to fp32 (IEEE,
    ties to even), evaluated with exact rationals: for partials whose
    products with the scale are not exact in fp32 (the int16 reading)."""
    from fractions import Fraction
    P = np.asarray(P)
    s = O.bf16_bits_to_f64(scale_bits)
    R, N, G = P.shape
    out = np.empty((R, N), dtype=np.float32)
    for r in range(R):
        for n in range(N):
            acc = 0.0
            for g in range(G):
                acc = _round_f32(Fraction(float(s[n, g])) * int(P[r, n, g]) + Fraction(acc))
            out[r, n] = _round_f32(Fraction(float(np.float32(x_scale[r]))) * Fraction(acc))
    return out


def _expert_rows(job):
    """Worker: one expert's gated MLP on its rows (oracle, fp64)."""
    w, e, u, act_bits = job
    return O.expert_ffn(u, oi.expert_arrays(w, e), act_bits)


def oracle_tokens(w: wl.Workload, x, router, latent, tokens, workers: int = 8) -> np.ndarray:
    """The oracle's layer output for the listed tokens of workload ``w``.

    Same arithmetic as ``oracle.moe_forward(x, params, tokens)`` (routing,
    expert input, per-slot expert outputs summed in slot order, latent
    wrap), with the rows of each selected expert evaluated together and the
    experts spread over a pool of processes (started with spawn, so it is
    safe after CUDA has been initialised).  Every row is independent in the
    definition, so grouping changes no value."""
    import multiprocessing as mp
    p = oi.layer_params(w, router=router, latent=latent)
    xs = oi.x_f64(x)[np.asarray(tokens)]
    rt = O.route(xs, p.w_router, p.bias, w.k, w.renorm)
    u = O.expert_input(xs, p)
    experts = sorted({int(e) for e in rt.idx.ravel()})
    rows = {e: np.nonzero((rt.idx == e).any(axis=1))[0] for e in experts}
    jobs = [(w, e, u[rows[e]], w.act_bits) for e in experts]
    if workers > 1 and len(jobs) > 1:
        with mp.get_context("spawn").Pool(min(workers, len(jobs))) as pool:
            outs = pool.map(_expert_rows, jobs, chunksize=1)
    else:
        outs = [_expert_rows(j) for j in jobs]
    y = {e: dict(zip(rows[e].tolist(), o)) for e, o in zip(experts, outs)}
    out = np.zeros_like(u)
    for i in range(len(xs)):
        for j in range(w.k):
            e = int(rt.idx[i, j])
            out[i] += rt.weight[i, j] * y[e][i]
    return O.latent_out(out, p)


def targeted_tokens(w: wl.Workload, x, router, n: int = 32, seed: int = 2024) -> list:
    """n tokens of workload ``w`` chosen to reach the expert kernels' edge
    cases: the last token, the rows of the hottest experts' last (ragged)
    128-row chunk, every 128-row chunk boundary of the hottest experts,
    experts of exactly 16 and 17 rows (one and two 16-row stream chunks; on
    the tensor cores in prefill-shaped batches), then random tokens.  Routing
    is the oracle's."""
    if w.T <= n:
        return list(range(w.T))
    W, b = router
    rt = O.route(oi.x_f64(x), W.numpy(), b.numpy(), w.k, w.renorm)
    toks = {w.T - 1}
    counts = np.bincount(rt.idx.ravel(), minlength=w.E)
    rows_of = lambda e: np.nonzero((rt.idx == e).any(axis=1))[0]   # ascending token ids
    for e in np.argsort(-counts, kind="stable")[:3]:
        r = rows_of(e)
        last0 = (len(r) - 1) // 128 * 128                 # first row of the last chunk
        toks.update(int(t) for t in (r[last0], r[-1]))
        toks.update(int(r[c]) for c in range(127, len(r), 128)[:3])   # chunk edges
        toks.update(int(r[c]) for c in range(128, len(r), 128)[:3])
    for size in (16, 17):
        for e in np.nonzero(counts == size)[0][:2]:
            r = rows_of(e)
            toks.update(int(t) for t in (r[0], r[-1]))
    rng = np.random.default_rng(seed)
    while len(toks) < n:
        toks.add(int(rng.integers(w.T)))
    return sorted(toks)[: max(n, len(toks))]
