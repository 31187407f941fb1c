"""The seeded generator and the stored routing calibration.

The calibration file is data written by ``oracle/calibrate_workloads.py``; these
tests re-derive its claims with the oracle's router: every token of a named
workload has a top-k gap of at least 1e-3, the recorded expert loads are the
realised ones, the exact-mode routing is adversarial and the prefill load is
Zipf-shaped with idle experts.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as wl

GAP_MIN = 1e-3


def test_hash_tensor_and_int_agree():
    xs = [0, 1, 12345, 2 ** 31, 2 ** 32 - 1]
    t = wl.mix32(torch.tensor(xs, dtype=torch.int64))
    assert t.tolist() == [wl.mix32(v) for v in xs]
    assert all(0 <= v < 2 ** 32 for v in t.tolist())
    # a bijection: no collisions on a dense range
    r = wl.mix32(torch.arange(1 << 20, dtype=torch.int64))
    assert torch.unique(r).numel() == 1 << 20


def test_generator_is_deterministic_and_sliceable():
    w = wl.WORKLOADS["tiny"]
    x1, x2 = wl.gen_x(w), wl.gen_x(w)
    assert torch.equal(x1, x2)
    assert torch.equal(wl.gen_x(w, tokens=[5, 2]), x1[[5, 2]])
    e1 = wl.gen_expert(w, 3)
    stacked = wl.gen_experts(w)
    for name, t in e1.items():
        assert torch.equal(stacked[name][3], t)


def test_value_distributions():
    w = wl.WORKLOADS["tiny"]
    x = wl.gen_x(w).float()
    assert abs(x.mean().item()) < 0.05 and abs(x.std().item() - 1.0) < 0.05
    W, b = wl.gen_router(w)
    assert W.dtype == torch.float32 and abs(W.std().item() - 0.02) < 0.002
    ex = wl.gen_expert(wl.WORKLOADS["decode"], 0)
    s = ex["gate_scale"].float()
    # bounds of U(0.002, 0.01) after rounding to bf16 (8 significant bits)
    assert s.min().item() >= 0.002 * (1 - 2 ** -8) and s.max().item() <= 0.01 * (1 + 2 ** -8)
    codes = O.unpack_int4(ex["gate_packed"][:64].numpy())
    hist = np.bincount(codes.ravel() + 8, minlength=16)
    assert hist.min() > 0.9 * hist.mean()   # uniform over [-8, 7]


def _route(w, tokens=None):
    W, b = wl.gen_router(w)
    x = wl.gen_x(w, tokens=tokens)
    return O.route(x.to(torch.float64).numpy(), W.numpy(), b.numpy(), w.k, w.renorm)


@pytest.mark.parametrize("name", ["tiny", "decode", "exact"])
def test_calibrated_gap_and_counts_full(name):
    w = wl.WORKLOADS[name]
    rt = _route(w)
    assert O.topk_gap(rt.r, w.k).min() >= GAP_MIN
    counts = np.bincount(rt.idx.ravel(), minlength=w.E)
    assert counts.tolist() == wl.calibration()[name]["counts"]


@pytest.mark.parametrize("name", ["prefill", "latent"])
def test_calibrated_gap_sampled(name):
    w = wl.WORKLOADS[name]
    redrawn = sorted(int(t) for t in wl.resample_counts(w))
    rng = np.random.default_rng(7)
    toks = sorted(set(redrawn[:256]) | set(rng.choice(w.T, 256, replace=False).tolist()))
    rt = _route(w, tokens=toks)
    assert O.topk_gap(rt.r, w.k).min() >= GAP_MIN


def test_exact_routing_is_adversarial():
    w = wl.WORKLOADS["exact"]
    chosen = set(wl.expert_permutation(w)[: w.k].tolist())
    counts = np.array(wl.calibration()["exact"]["counts"])
    assert set(np.nonzero(counts)[0].tolist()) == chosen
    assert all(counts[e] == w.T for e in chosen)


def test_prefill_load_is_zipf_with_idle_experts():
    w = wl.WORKLOADS["prefill"]
    c = wl.calibration()["prefill"]
    counts = np.array(c["counts"])
    target = np.array(c["zipf_target"])
    assert counts.sum() == w.T * w.k and counts.max() <= w.T
    assert (counts == 0).sum() == w.zipf_dead
    big = target >= 200
    assert np.all(np.abs(counts[big] - target[big]) <= 0.1 * target[big])
    # heavier rank -> larger load, on the head of the distribution
    order = np.argsort(-target)[:10]
    assert np.all(np.diff(counts[order]) < 0)


def test_oracle_input_adapters():
    """oracle.inputs hands the oracle exactly the generator's values."""
    from oracle import inputs as oi
    w = wl.workload("tiny", name="adapt", L=128, I=128, norm_gain_std=0.1)
    x = wl.gen_x(w)
    assert np.array_equal(O.bf16_bits_to_f64(oi.bf16_bits(x)), oi.x_f64(x))
    ex = wl.gen_expert(w, 3, "cpu")
    arr = oi.expert_arrays(w, 3)
    assert set(arr) == set(ex)
    for name, t in ex.items():
        want = oi.bf16_bits(t) if t.dtype == torch.bfloat16 else t.numpy()
        assert arr[name].dtype == want.dtype and np.array_equal(arr[name], want), name
    assert np.array_equal(O.unpack_int4(arr["gate_packed"]).shape, (w.I, w.D))
    # the lazy cache evicts and regenerates the same arrays
    lazy = oi.LazyExperts(w, keep=2)
    first = {e: lazy(e)["down_scale"].copy() for e in range(4)}
    assert len(lazy._cache) == 2
    for e in range(4):
        assert np.array_equal(lazy(e)["down_scale"], first[e])
    router = wl.gen_router(w)
    lat = wl.gen_latent(w)
    p = oi.layer_params(w, router=router, latent=lat)
    assert (p.k, p.renorm, p.act_bits, p.E, p.eps) == (w.k, w.renorm, w.act_bits, w.E, w.eps)
    assert np.array_equal(p.w_router, router[0].numpy().astype(np.float64))
    assert np.array_equal(p.lat_up, oi.bf16_bits(lat["lat_up"])) and p.lat_up.shape == (w.H, w.L)
    assert p.lat_down.shape == (w.L, w.H) and p.lat_norm.shape == (w.L,)
