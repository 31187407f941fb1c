"""GPU parity of each C-ABI stage against the fp64 oracle.

Integer and index results are compared bit for bit (routing sets, counts,
offsets, permutation, int8 codes and scales, integer accumulators); float
results within tolerances derived from their arithmetic (stated per test).
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as wl
from oracle import inputs as oi
from tests._helpers import (assert_close, bf16_bits, conditioned_attempts, fp32_fma_chain,
                            fp32_group_chain, random_topk, rel_l2)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def moe():
    from int4_routed_expert_fp32_gb300.build import build
    build()
    import int4_routed_expert_fp32_gb300 as m
    torch.cuda.set_device(DEV)
    assert m.check_error() == 0
    yield m
    assert m.check_error() == 0


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def test_generator_cpu_and_cuda_agree(moe):
    w = wl.WORKLOADS["decode"]
    cpu = wl.gen_expert(w, 17, "cpu")
    gpu = wl.gen_expert(w, 17, DEV)
    for name in cpu:
        assert torch.equal(cpu[name], gpu[name].cpu()), name


# --------------------------------------------------------------------- router

ROUTE_CASES = {
    "tiny": wl.WORKLOADS["tiny"],
    "decode": wl.WORKLOADS["decode"],
    "exact": wl.WORKLOADS["exact"],
    "ragged": wl.workload("tiny", name="ragged", T=77, H=512, E=40, k=6, seed=3),
    "k1": wl.workload("tiny", name="k1", T=33, H=128, E=5, k=1, seed=4),
    "k_eq_E": wl.workload("tiny", name="kE", T=9, H=64, E=4, k=4, seed=5),
    "no_renorm": wl.workload("tiny", name="nr", T=40, H=256, E=24, k=3, renorm=False, seed=6),
    # from 512 tokens the logits come from the tensor cores: ragged in both
    # the 128-token and the 256-logit tiles
    "tc_ragged": wl.workload("tiny", name="tc_ragged", T=601, H=512, E=100, k=6, seed=7),
    # the one-warp top-k (from 64 tokens) at 8 and 16 scores per lane (E in
    # (128, 256] and (384, 512]); above 512 experts the one-CTA top-k
    "E200": wl.workload("tiny", name="E200", T=70, H=256, E=200, k=8, seed=22),
    "E500_k32": wl.workload("tiny", name="E500", T=64, H=256, E=500, k=32, seed=23),
    # the library's limits: 2048 experts, top-32
    "max_E_k": wl.workload("tiny", name="max_E_k", T=24, H=256, E=2048, k=32, seed=21),
}


@pytest.mark.parametrize("case", list(ROUTE_CASES))
def test_route_parity(moe, case):
    w = ROUTE_CASES[case]
    x = wl.gen_x(w, attempts=conditioned_attempts(w))
    W, b = wl.gen_router(w)
    idx, wt = moe.route(x.to(DEV), W.to(DEV), b.to(DEV), w.k, w.renorm)
    assert moe.check_error() == 0
    gi, gw = idx.cpu().numpy(), wt.cpu().numpy()
    rt = O.route(oi.x_f64(x), W.numpy(), b.numpy(), w.k, w.renorm)
    # the selected expert sets are bit-exact
    assert np.array_equal(np.sort(gi, 1), np.sort(rt.idx, 1))
    # each slot's weight is the oracle weight of the same expert (fp32 vs fp64)
    for t in range(w.T):
        ref = dict(zip(rt.idx[t].tolist(), rt.weight[t].tolist()))
        for j in range(w.k):
            assert abs(gw[t, j] - ref[int(gi[t, j])]) <= 2e-6 * max(1.0, abs(ref[int(gi[t, j])]))
        # slots in descending ranking score (up to fp32 rounding of the scores)
        r = rt.r[t, gi[t]]
        assert np.all(np.diff(r) <= 1e-6)


def test_router_prepare_terms_sum_exactly(moe):
    """moe_router_prepare's three bf16 terms add up to the fp32 router weight
    exactly (the sum is formed in fp64 here), for weights from 2^-100 to 2^100
    (the split is exact from 2^-110 on) and the fp32 values that need all
    three terms."""
    rng = np.random.default_rng(61)
    E, H = 40, 192
    mant = rng.uniform(1.0, 2.0, size=(E, H))
    expo = rng.integers(-100, 100, size=(E, H))
    sign = rng.choice([-1.0, 1.0], size=(E, H))
    W = (sign * mant * np.exp2(expo)).astype(np.float32)
    W[0, :8] = [0.0, -0.0, 1.0, np.float32(1 + 2 ** -23), np.float32(3.0000002),
                np.float32(-1e-30), np.float32(1e30), np.float32(2 ** -126)]
    terms = moe.router_prepare(torch.from_numpy(W).to(DEV))
    assert moe.check_error() == 0
    t = terms.view(torch.int16).cpu().numpy().astype(np.uint16).astype(np.uint32) << 16
    t = t.view(np.float32).astype(np.float64)
    assert np.array_equal(t[0] + t[1] + t[2], W.astype(np.float64))


@pytest.mark.parametrize("T,kernels", [(40, 2), (512, 3)])
def test_route_launch_count(moe, T, kernels):
    # the library counts its launches: SIMT logits + top-k below 512 tokens,
    # weight split + tensor-core logits + top-k from 512
    w = wl.workload("tiny", name="lc", T=T, H=256, E=24, k=3, seed=8)
    x = wl.gen_x(w)
    W, b = wl.gen_router(w)
    xd, Wd, bd = x.to(DEV), W.to(DEV), b.to(DEV)
    n0 = moe.launch_count()
    moe.route(xd, Wd, bd, w.k, w.renorm)
    assert moe.launch_count() - n0 == kernels
    assert moe.check_error() == 0


@pytest.mark.parametrize("name", ["prefill", "latent"])
def test_route_tensor_core_full(moe, name):
    """The tensor-core router at full width (H = 7168, 8192 and 2048 tokens):
    sets bit-exact, the prefill counts as calibrated, every weight within
    2e-6 of the oracle's (fp32 partial logits over 1024-column slices of the
    three exact bf16 terms of the weight)."""
    w = wl.WORKLOADS[name]
    x = wl.gen_x(w)
    W, b = wl.gen_router(w)
    idx, wt = moe.route(x.to(DEV), W.to(DEV), b.to(DEV), w.k, w.renorm)
    gi, gw = idx.cpu().numpy(), wt.cpu().numpy().astype(np.float64)
    rt = O.route(oi.x_f64(x), W.numpy(), b.numpy(), w.k, w.renorm)
    assert np.array_equal(np.sort(gi, 1), np.sort(rt.idx, 1))
    if name == "prefill":
        counts = np.bincount(gi.ravel(), minlength=w.E)
        assert counts.tolist() == wl.calibration()["prefill"]["counts"]
    order_g, order_r = np.argsort(gi, 1), np.argsort(rt.idx, 1)
    got = np.take_along_axis(gw, order_g, 1)
    ref = np.take_along_axis(rt.weight, order_r, 1)
    assert np.max(np.abs(got - ref) / np.maximum(1.0, np.abs(ref))) <= 2e-6


# ------------------------------------------------------------------- dispatch

def _dispatch_case(name):
    rng = np.random.default_rng(11)
    if name == "random":
        T, E, k, D = 77, 40, 6, 192
        idx = random_topk(T, E, k, rng)
    elif name == "adversarial":
        T, E, k, D = 100, 32, 4, 128
        idx = np.tile(np.array([[7, 30, 2, 11]], np.int32), (T, 1))
    elif name == "one_token":
        T, E, k, D = 1, 16, 3, 64
        idx = np.array([[15, 0, 4]], np.int32)
    elif name == "zipf_prefill":
        T, E, k, D = 8192, 384, 8, 256
        p = np.arange(1, E + 1, dtype=np.float64) ** -1.1
        p[-16:] = 0
        idx = random_topk(T, E, k, rng, hot=p)
    else:
        raise KeyError(name)
    x = _bf16(rng.normal(size=(T, D)))
    return idx, x, E


@pytest.mark.parametrize("name", ["random", "adversarial", "one_token", "zipf_prefill"])
@pytest.mark.parametrize("act_bits", [16, 8])
def test_dispatch_parity(moe, name, act_bits):
    idx, x, E = _dispatch_case(name)
    T, k = idx.shape
    out = moe.dispatch(torch.from_numpy(idx).to(DEV), x.to(DEV), E, act_bits)
    assert moe.check_error() == 0
    d = O.dispatch(idx, E)
    got = {n: t.cpu().numpy() for n, t in out.items() if t is not None and t.dtype != torch.bfloat16}
    assert got["counts"].tolist() == d.counts.tolist()
    assert got["offsets"].tolist() == d.offsets.tolist()
    assert got["row_token"].tolist() == d.row_token.tolist()
    assert got["row_slot"].tolist() == d.row_slot.tolist()
    assert got["inv_row"].tolist() == d.inv_row.tolist()
    if act_bits == 16:
        assert np.array_equal(bf16_bits(out["x_sorted"]), bf16_bits(x)[d.row_token])
    else:
        q, sc = O.quantize_rows_int8(x.float().numpy())
        assert np.array_equal(got["x_sorted"], q[d.row_token])
        assert np.array_equal(got["x_scale"].view(np.uint32), sc[d.row_token].view(np.uint32))


def _pair_columns(C):
    """Natural column stored at each position of the pair order (blocks of 8:
    0 4 1 5 2 6 3 7)."""
    blk = np.array([0, 4, 1, 5, 2, 6, 3, 7])
    return (np.arange(C // 8)[:, None] * 8 + blk[None, :]).ravel()


@pytest.mark.parametrize("name", ["random", "one_token", "zipf_prefill"])
@pytest.mark.parametrize("act_bits", [16, 8])
def test_dispatch_pairs_layout(moe, name, act_bits):
    """moe_dispatch_pairs: the same permutation as moe_dispatch, rows in pair
    order as fp16 (exact for these values) or int8, bit for bit."""
    idx, x, E = _dispatch_case(name)
    ti = torch.from_numpy(idx).to(DEV)
    nat = moe.dispatch(ti, x.to(DEV), E, act_bits)
    prs = moe.dispatch(ti, x.to(DEV), E, act_bits, pairs=True)
    assert moe.check_error() == 0
    for n in ("counts", "offsets", "row_token", "row_slot", "inv_row"):
        assert torch.equal(nat[n], prs[n]), n
    cols = _pair_columns(x.shape[1])
    if act_bits == 16:
        want = nat["x_sorted"].float().cpu().numpy().astype(np.float16)[:, cols]
        assert np.array_equal(prs["x_sorted"].cpu().numpy().view(np.uint16), want.view(np.uint16))
    else:
        assert np.array_equal(prs["x_sorted"].cpu().numpy(), nat["x_sorted"].cpu().numpy()[:, cols])
        assert torch.equal(prs["x_scale"], nat["x_scale"])


def test_dispatch_pairs_reports_fp16_overflow(moe):
    idx, x, E = _dispatch_case("random")
    x = x.clone()
    x[5, 17] = 1.0e5  # beyond the fp16 range
    moe.dispatch(torch.from_numpy(idx).to(DEV), x.to(DEV), E, 16, pairs=True)
    assert moe.check_error() == moe.capi.MOE_ERR_UNSUPPORTED
    assert moe.check_error() == 0


def test_quantize_rows_bit_exact(moe, golden_dir):
    import json
    import os
    rng = np.random.default_rng(5)
    v = rng.normal(size=(37, 448)) * rng.uniform(1e-3, 50, size=(37, 1))
    v[3] = 0.0                                     # zero row
    v[4, :] = np.round(v[4, :] * 0) + 1.0          # constant row
    vb = _bf16(v)
    q, s = moe.quantize_rows(vb.to(DEV))
    qo, so = O.quantize_rows_int8(vb.float().numpy())
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))
    # the golden cases, padded to 64 columns with zeros
    with open(os.path.join(golden_dir, "quantizer_cases.json")) as f:
        cases = json.load(f)["cases"]
    rows = np.zeros((len(cases), 64), np.float32)
    for i, c in enumerate(cases):
        rows[i, :len(c["v"])] = c["v"]
    q, s = moe.quantize_rows(_bf16(rows).to(DEV))
    for i, c in enumerate(cases):
        assert q[i, :len(c["q"])].cpu().tolist() == c["q"]
        assert float(s[i]) == c["scale"]


# ------------------------------------------------------------ int4 linear

def _segments(counts):
    off = np.zeros(len(counts) + 1, np.int32)
    off[1:] = np.cumsum(counts)
    return off


def _random_int4(rng, E, N, K, lo=0.002, hi=0.01):
    packed = rng.integers(0, 2 ** 32, size=(E, N, K // 8), dtype=np.uint64).astype(np.uint32).view(np.int32)
    scale = O.f32_to_bf16_bits(rng.uniform(lo, hi, size=(E, N, K // 32)).astype(np.float32))
    return packed, scale


def _t(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(DEV)


class _tc_kernels:
    """Within the block, run the act_bits 16 tensor-core GEMMs on the
    CTA-pair kernels (pair=True, the default) or the one-CTA kernels."""

    def __init__(self, moe, pair: bool):
        self.moe, self.pair = moe, pair

    def __enter__(self):
        self.prev = self.moe.set_tc_pair(self.pair)

    def __exit__(self, *exc):
        self.moe.set_tc_pair(self.prev)



# ------------------------------------------------------------ int4 weight quantiser

@pytest.mark.parametrize("shape", [(3, 40, 96), (1, 7, 32), (2, 513, 7168)])
def test_quantize_int4_bit_exact(moe, shape):
    """Codes and bf16 scales equal the oracle's bit for bit (float32 steps on
    both sides), over magnitudes from 1e-4 to 1e3, zero groups and ties."""
    rng = np.random.default_rng(sum(shape))
    E, N, K = shape
    w = rng.normal(size=shape) * rng.uniform(1e-4, 1e3, size=(E, N, 1))
    w[:, :, :32] *= rng.random((E, N, 1)) < 0.8        # some all-zero groups
    if K >= 64:
        w[0, 0, 32:64] = np.concatenate([np.arange(29) * 0.5 - 7, [0, 0, 0]])  # s = 1: ties
    wb = _bf16(w)
    packed, scale = moe.quantize_int4(wb.to(DEV))
    assert moe.check_error() == 0
    ref_p, ref_s = O.quantize_weight_int4(wb.float().numpy().reshape(E * N, K))
    assert np.array_equal(packed.cpu().numpy().reshape(E * N, K // 8), ref_p)
    assert np.array_equal(bf16_bits(scale.cpu()).reshape(E * N, K // 32), ref_s)


def test_quantize_int4_feeds_int4_linear(moe):
    """Quantised bf16 weights run through the expert GEMM: the result equals
    the oracle's product with the dequantised weights."""
    rng = np.random.default_rng(11)
    E, N, K, counts = 3, 256, 1024, [5, 0, 60]
    off = _segments(counts)
    R = int(off[-1])
    w = _bf16(rng.normal(size=(E, N, K)) * 0.02)
    packed, scale = moe.quantize_int4(w.to(DEV))
    x = _bf16(rng.normal(size=(R, K)))
    got = moe.int4_linear(x.to(DEV), None, _t(off), packed, scale, 16)
    assert moe.check_error() == 0
    got = got.cpu().numpy()
    pk = packed.cpu().numpy()
    sb = bf16_bits(scale.cpu())
    xf = oi.x_f64(x)
    for e in range(E):
        a, b = off[e], off[e + 1]
        if a < b:
            ref = O.int4_linear(xf[a:b], pk[e], sb[e], 16)
            assert rel_l2(got[a:b], ref) <= 1e-5
    # and the dequantised weights are within half a step of the bf16 weights
    wq = O.dequantize(pk.reshape(E * N, K // 8), sb.reshape(E * N, K // 32))
    step = np.repeat(O.bf16_bits_to_f64(sb.reshape(E * N, K // 32)), 32, axis=1)
    assert np.all(np.abs(wq - w.float().numpy().reshape(E * N, K)) <= 0.5 * step * (1 + 2.0 ** -20))


def test_quantize_int4_reports_nonfinite_weights(moe):
    w = torch.zeros(4, 64, dtype=torch.bfloat16)
    w[2, 40] = float("inf")
    w[3, 3] = float("nan")
    packed, scale = moe.quantize_int4(w.to(DEV))
    assert moe.check_error() == moe.capi.MOE_ERR_UNSUPPORTED
    s = bf16_bits(scale.cpu())
    assert s[2, 1] == 0 and s[3, 0] == 0
    # the next call is clean
    moe.quantize_int4(torch.ones(2, 32, dtype=torch.bfloat16, device=DEV))
    assert moe.check_error() == 0


# ------------------------------------------------ int16 reading of act_bits 16

def test_quantize_rows_int16_bit_exact(moe):
    """Codes and scales equal the oracle's bit for bit (float32 steps on both
    sides): random magnitudes, a zero row, half steps at scale 1 and the row
    that separates float32 from float64 quantisation."""
    rng = np.random.default_rng(16)
    v = (rng.normal(size=(40, 320)) * rng.uniform(1e-3, 1e3, size=(40, 1))).astype(np.float32)
    v[3] = 0.0
    v[5, :6] = [32767.0, 0.5, 1.5, 2.5, -2.5, -100.5]
    v[5, 6:] = 0.0
    a = np.float32(1.925695538520813)
    v[7] = 0.0
    v[7, :3] = [a, a / np.float32(2), -a / np.float32(2)]
    vb = _bf16(v)
    q, s = moe.quantize_rows_int16(vb.to(DEV))
    assert moe.check_error() == 0
    rq, rs = O.quantize_rows_int16(vb.float().numpy())
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))


@pytest.mark.parametrize("K,N,counts", [
    (320, 300, [0, 1, 33, 70, 8]),
    (7168, 136, [5, 17, 40, 130, 0]),
    (8160, 64, [3, 16]),                # the largest K with an exact int32 whole-K sum
])
def test_int4_linear_int16_partials_and_output(moe, K, N, counts):
    """The int16 reading: every group partial equals the oracle's exact integer
    (codes from the oracle's own int16 quantiser), the output matches the
    oracle's fp64 result, and sampled outputs equal the fp32 fma chain the
    header states, evaluated with exact rationals."""
    rng = np.random.default_rng(K + N)
    E = len(counts)
    off = _segments(counts)
    R = int(off[-1])
    packed, scale = _random_int4(rng, E, N, K, 0.005, 0.02)
    x = _bf16(rng.normal(size=(R, K)) * rng.uniform(0.1, 10, size=(R, 1)))
    out, part = moe.int4_linear_int16(x.to(DEV), _t(off), _t(packed), _t(scale, torch.bfloat16),
                                      partials=True)
    assert moe.check_error() == 0
    out, part = out.cpu().numpy(), part.cpu().numpy()
    q16, sx = O.quantize_rows_int16(x.float().numpy())
    for e in range(E):
        a, b = off[e], off[e + 1]
        if a == b:
            continue
        P = O.int16_group_partials(q16[a:b], packed[e])
        assert np.array_equal(part[a:b], P), e
        ref = O.int4_linear_int16(oi.x_f64(x)[a:b], packed[e], scale[e])
        assert rel_l2(out[a:b], ref) <= 2e-6, e
        rows = [a, b - 1]
        cols = [0, N // 2, N - 1]
        chain = fp32_fma_chain(P[[r - a for r in rows]][:, cols], scale[e][cols], sx[rows])
        assert np.array_equal(out[np.ix_(rows, cols)], chain), e


def test_int4_linear_int16_rejections(moe):
    x = torch.zeros(4, 96, dtype=torch.bfloat16, device=DEV)
    off = _t(np.array([0, 4], np.int32))
    w = torch.zeros(1, 8, 96 // 8, dtype=torch.int32, device=DEV)
    sc = torch.zeros(1, 8, 3, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(moe.MoeError):
        moe.int4_linear_int16(torch.zeros(4, 8192, dtype=torch.bfloat16, device=DEV), off,
                              torch.zeros(1, 8, 1024, dtype=torch.int32, device=DEV),
                              torch.zeros(1, 8, 256, dtype=torch.bfloat16, device=DEV))
    bad = _t(np.array([0, 9], np.int32))      # offsets beyond the rows
    moe.int4_linear_int16(x, bad, w, sc)
    assert moe.check_error() == moe.capi.MOE_ERR_INVALID
    moe.int4_linear_int16(x, off, w, sc)
    assert moe.check_error() == 0


# ------------------------------------------------------------ int8 weight quantiser

@pytest.mark.parametrize("shape", [(3, 40, 96), (1, 7, 32), (2, 513, 7168)])
def test_quantize_int8_bit_exact(moe, shape):
    """Codes and bf16 scales equal the oracle's bit for bit (float32 steps on
    both sides), over magnitudes from 1e-4 to 1e3, zero groups and ties."""
    rng = np.random.default_rng(sum(shape) + 8)
    E, N, K = shape
    w = rng.normal(size=shape) * rng.uniform(1e-4, 1e3, size=(E, N, 1))
    w[:, :, :32] *= rng.random((E, N, 1)) < 0.8        # some all-zero groups
    if K >= 64:  # s = 1: max 127 and half steps
        w[0, 0, 32:64] = np.concatenate([[127.0], np.arange(31) * 0.5 - 7.5])
    wb = _bf16(w)
    q, scale = moe.quantize_int8(wb.to(DEV))
    assert moe.check_error() == 0
    ref_q, ref_s = O.quantize_weight_int8(wb.float().numpy().reshape(E * N, K))
    assert np.array_equal(q.cpu().numpy().reshape(E * N, K), ref_q)
    assert np.array_equal(bf16_bits(scale.cpu()).reshape(E * N, K // 32), ref_s)


def test_quantize_int8_reports_nonfinite_weights(moe):
    w = torch.zeros(4, 64, dtype=torch.bfloat16)
    w[2, 40] = float("inf")
    w[3, 3] = float("nan")
    w[1, 5] = 2.0
    q, scale = moe.quantize_int8(w.to(DEV))
    assert moe.check_error() == moe.capi.MOE_ERR_UNSUPPORTED
    s = bf16_bits(scale.cpu())
    assert s[2, 1] == 0 and s[3, 0] == 0
    qc = q.cpu().numpy()
    assert not qc[2, 32:].any() and not qc[3, :32].any() and qc[1, 5] == 127
    # the next call is clean
    moe.quantize_int8(torch.ones(2, 32, dtype=torch.bfloat16, device=DEV))
    assert moe.check_error() == 0


@pytest.mark.parametrize("pair", [True, False])
@pytest.mark.parametrize("K,N,counts", [
    (320, 300, [0, 1, 33, 70, 8]),        # ragged K tail, ragged N tile, multi-chunk experts
    (2048, 512, [5, 0, 0, 64, 2]),
    (128, 64, [3, 3]),                    # K below one stage, N below one tile
    (256, 320, [256, 257, 31, 32, 33, 0, 300]),  # 256-row chunks and their ragged tails
])
def test_int4_linear_w4a16(moe, K, N, counts, pair):
    """Both tensor-core kernels (CTA pairs and one CTA) on prefill-shaped
    batches (the stream kernel on the others)."""
    rng = np.random.default_rng(K + N)
    E = len(counts)
    off = _segments(counts)
    R = int(off[-1])
    packed, scale = _random_int4(rng, E, N, K)
    x = _bf16(rng.normal(size=(R, K)))
    with _tc_kernels(moe, pair):
        got = moe.int4_linear(x.to(DEV), None, _t(off), _t(packed), _t(scale, torch.bfloat16), 16)
    assert moe.check_error() == 0
    got = got.cpu().numpy()
    xf = oi.x_f64(x)
    for e in range(E):
        a, b = off[e], off[e + 1]
        if a == b:
            continue
        ref = O.int4_linear(xf[a:b], packed[e], scale[e], 16)
        # fp32 accumulation of exact products over K terms
        assert rel_l2(got[a:b], ref) <= 1e-5


def _extreme_scales(rng, E, N, K, lo=1e-30, tiny=1e-7, big=1e2, huge=2e4, small=3e-6):
    """bf16 group scales spanning ``lo`` .. ``huge`` in chosen weight rows:
    all tiny, tiny and large mixed, all large, huge (q * s beyond 65504 when
    huge > 8160), just below 2^-17 (``small``), zero, extremely small, six
    decades in one row; the other rows U(0.002, 0.01)."""
    G = K // 32
    s = rng.uniform(0.002, 0.01, size=(E, N, G)).astype(np.float32)
    s[:, 0] = tiny
    s[:, 1, 0::2], s[:, 1, 1::2] = tiny, big
    s[:, 2] = big
    s[:, 3] = huge
    s[:, 4] = small
    s[:, 5] = 0.0
    s[:, 6] = lo
    s[:, 7] = rng.choice([tiny * 10, 1e-3, 1.0, big / 4], size=(E, G))
    return O.f32_to_bf16_bits(s)


def _check_columns(got, ref, what):
    """Every weight row (output column) against the oracle on its own, so a
    row of tiny scales cannot hide behind rows of large ones."""
    for n in range(ref.shape[1]):
        g, r = got[:, n], ref[:, n]
        if not np.any(r):
            assert not np.any(g), (what, n)
            continue
        assert rel_l2(g, r) <= 3e-5, (what, n, rel_l2(g, r))


@pytest.mark.parametrize("act_bits", [16, 8])
def test_int4_linear_extreme_scales_both_kernels(moe, act_bits):
    """Weight scales from 1e-30 to 2e4 on both expert kernels (9 + 30 rows: a
    decode-shaped batch, the stream kernel; 9 + 60 rows: a prefill-shaped
    batch, every expert on the tensor cores), each weight row checked on its
    own: relative L2 <= 3e-5 per column, and the exact mode's fp32 chain bit
    for bit.  The bound: fp32 accumulation of exact products, plus, on the
    stream kernel, the start value -(1032 S_lo + 72 S_hi) of each group's
    fp16 chain, which leaves an absolute error of about 2^-24 * 1040 * sum|x|
    per group (~1e-5 relative on one column; 1e-5 over a whole matrix, as
    test_int4_linear_w4a16 checks).

    The stream kernel and the exact mode apply scales in fp32 and take any
    scale.  The act_bits 16 tensor-core kernel multiplies q * scale in fp16,
    exact for scales in [2^-17, 8160]: outside that range it records
    MOE_ERR_UNSUPPORTED (checked here), and inside it (scales 1e-5 .. 8000)
    it matches like the stream kernel."""
    rng = np.random.default_rng(17 + act_bits)
    K, N = 2048, 136
    E = 2
    packed = rng.integers(0, 2 ** 32, size=(E, N, K // 8), dtype=np.uint64).astype(np.uint32).view(np.int32)

    def run(counts, scale):
        off = _segments(counts)
        R = int(off[-1])
        x = _bf16(rng.normal(size=(R, K)))
        q, sx = O.quantize_rows_int8(x.float().numpy())
        if act_bits == 16:
            got = moe.int4_linear(x.to(DEV), None, _t(off), _t(packed),
                                  _t(scale, torch.bfloat16), 16).cpu().numpy()
        else:
            got = moe.int4_linear(_t(q), _t(sx), _t(off), _t(packed), _t(scale, torch.bfloat16),
                                  8).cpu().numpy()
        return off, oi.x_f64(x), q, sx, got, moe.check_error()

    def check(off, xf, q, sx, got, scale):
        for e in range(E):
            a, b = off[e], off[e + 1]
            ref = O.int4_linear(xf[a:b], packed[e], scale[e], act_bits)
            if act_bits == 8:
                P = O.int4_group_partials(q[a:b], packed[e])
                assert np.array_equal(got[a:b], fp32_group_chain(P, scale[e], sx[a:b])), e
            _check_columns(got[a:b], ref, f"expert {e}")

    scale = _extreme_scales(rng, E, N, K)
    # stream kernel (no expert holds 48 rows): any scale
    off, xf, q, sx, got, status = run([9, 30], scale)
    assert status == 0
    check(off, xf, q, sx, got, scale)
    # tensor cores (an expert of 60 rows)
    off, xf, q, sx, got, status = run([9, 60], scale)
    if act_bits == 8:
        assert status == 0
        check(off, xf, q, sx, got, scale)
        return
    assert status == moe.capi.MOE_ERR_UNSUPPORTED
    # the tensor-core kernel's exact range: 2^-17 (7.6e-6) .. 8160
    scale = _extreme_scales(rng, E, N, K, lo=8e-6, tiny=1e-5, big=64.0, huge=8000.0, small=7.7e-6)
    off, xf, q, sx, got, status = run([9, 60], scale)
    assert status == 0
    check(off, xf, q, sx, got, scale)


@pytest.mark.parametrize("K,N,counts", [
    (320, 300, [0, 1, 33, 70, 8]),   # every expert on the tensor cores (112 rows)
    (7168, 256, [2, 40]),            # all on the stream kernel (fewer than 48 rows)
    (7168, 256, [2, 48, 17]),        # all on the tensor cores, full hidden width
])
def test_int4_linear_exact_integer_accumulators(moe, K, N, counts):
    """Unit scales and an int8 input of scale 1: the output is the integer sum
    itself and must match the int64 oracle bit for bit (|sum| <= K*8*127 < 2^24)."""
    rng = np.random.default_rng(7)
    E = len(counts)
    off = _segments(counts)
    R = int(off[-1])
    packed = rng.integers(0, 2 ** 32, size=(E, N, K // 8), dtype=np.uint64).astype(np.uint32).view(np.int32)
    packed[:, :, :4] = np.int32(-2004318072)   # 0x88888888: every nibble -8 (extreme)
    scale = np.full((E, N, K // 32), 0x3F80, np.uint16)
    q = rng.integers(-127, 128, size=(R, K)).astype(np.int8)
    q[:, 0] = 127
    q[:, 1:32] = -127                           # extreme products in the first group
    xs = np.ones(R, np.float32)
    got = moe.int4_linear(_t(q), _t(xs), _t(off), _t(packed), _t(scale, torch.bfloat16), 8)
    assert moe.check_error() == 0
    got = got.cpu().numpy()
    for e in range(E):
        a, b = off[e], off[e + 1]
        if a == b:
            continue
        P = O.int4_group_partials(q[a:b], packed[e]).sum(axis=2)
        assert np.array_equal(got[a:b].astype(np.int64), P)
        assert np.all(got[a:b] == P)   # exactly integral in fp32


@pytest.mark.parametrize("K,N,counts", [
    (512, 384, [9, 0, 41, 70]),      # every expert on the tensor cores
    (7168, 300, [5, 17, 0, 40, 130]),  # full width, ragged N tile, one expert of two chunks
])
def test_int4_linear_exact_mode_scaled(moe, K, N, counts):
    """Real (non-unit) scales: the output is the fp32 chain of the exact group
    partials that the header states, bit for bit, on the library's own
    choice of kernel per expert; and within fp32 rounding of the fp64
    oracle's sum."""
    rng = np.random.default_rng(8 + K)
    E = len(counts)
    off = _segments(counts)
    R = int(off[-1])
    packed, scale = _random_int4(rng, E, N, K, 0.002, 0.02)
    x = _bf16(rng.normal(size=(R, K)) * 3)
    q, sx = O.quantize_rows_int8(x.float().numpy())
    got = moe.int4_linear(_t(q), _t(sx), _t(off), _t(packed), _t(scale, torch.bfloat16), 8)
    assert moe.check_error() == 0
    got = got.cpu().numpy()
    for e in range(E):
        a, b = off[e], off[e + 1]
        if a == b:
            continue
        P = O.int4_group_partials(q[a:b], packed[e])
        assert np.array_equal(got[a:b], fp32_group_chain(P, scale[e], sx[a:b])), e
        ref = O.int4_linear(oi.x_f64(x)[a:b], packed[e], scale[e], 8)
        assert rel_l2(got[a:b], ref) <= 1e-6


@pytest.mark.parametrize("kernel", [0, 1])
def test_int4_linear_exact_group_partials(moe, kernel):
    """The int32 group partials of the exact mode, read out of either kernel
    (0: stream, 1: tensor cores), equal the oracle's int64 partials bit for
    bit at K = 7168 with non-unit scales, for experts of 5, 17, 40 and 130
    rows (one 128-row tile plus a ragged one) and a ragged output tile; the
    output is their fp32 chain, the same bits on both kernels."""
    rng = np.random.default_rng(11)
    K, N, counts = 7168, 300, [5, 17, 0, 40, 130]
    E = len(counts)
    off = _segments(counts)
    R = int(off[-1])
    packed, scale = _random_int4(rng, E, N, K, 0.002, 0.02)
    packed[:, :, :4] = np.int32(-2004318072)   # 0x88888888: every nibble -8
    packed[:, 7, 8:12] = np.int32(0x77777777)  # every nibble +7
    q = rng.integers(-127, 128, size=(R, K)).astype(np.int8)
    q[:, :32] = -127                            # extreme products in the first group
    q[:, 64:96] = 127
    xs = rng.uniform(1e-3, 1e-1, size=R).astype(np.float32)
    out, P = moe.int4_linear_partials(_t(q), _t(xs), _t(off), _t(packed),
                                      _t(scale, torch.bfloat16), kernel)
    assert moe.check_error() == 0
    out, P = out.cpu().numpy(), P.cpu().numpy()
    for e in range(E):
        a, b = off[e], off[e + 1]
        if a == b:
            continue
        ref = O.int4_group_partials(q[a:b], packed[e])
        assert np.array_equal(P[a:b].astype(np.int64), ref), e
        assert np.array_equal(out[a:b], fp32_group_chain(ref, scale[e], xs[a:b])), e
    # the library's own routing of the same call gives the same bits
    lib = moe.int4_linear(_t(q), _t(xs), _t(off), _t(packed), _t(scale, torch.bfloat16), 8)
    assert np.array_equal(lib.cpu().numpy(), out)


# ------------------------------------------------------------- expert FFN

@pytest.mark.parametrize("act_bits,pair", [(16, True), (16, False), (8, True)])
@pytest.mark.parametrize("D,I,counts", [
    # decode-shaped batches (no expert holds 48 rows): the stream kernel
    (320, 192, [0, 3, 20, 1, 0, 9]),
    (256, 128, [16, 16]),
    (256, 128, [16, 17, 14]),            # one and two 16-row stream chunks
    (320, 192, [0, 3, 40, 1, 0, 9]),     # 53 rows: tensor-core kernels launched, no tile
    (256, 128, [16, 16, 16, 0, 3]),      # the same with experts of <= 16 rows
    # prefill-shaped batches: every expert on the tensor cores
    (256, 128, [48, 1, 2, 16, 17]),      # the threshold, and 1- to 17-row experts
    (1024, 512, [1, 2, 65, 0]),
    (320, 192, [130, 5, 64, 0, 16, 17]), # ragged token tiles, ragged N tiles
    (256, 192, [400, 3, 0, 193]),        # several 128-row chunks per expert, ragged last chunks
    (320, 192, [48, 3, 64, 17, 33, 0]),  # partial 128-row tiles
    (256, 128, [70, 40, 40, 40, 40, 40, 40, 40]),
    (256, 192, [256, 257, 31, 32, 33, 100, 511, 0]),  # 256-row chunks (CTA pairs), ragged tails
    (320, 192, [300, 48, 200]),          # a down tile of 256 outputs and a ragged one of 64
])
def test_expert_ffn_parity(moe, act_bits, pair, D, I, counts):
    """act_bits 16 on both tensor-core kernels (CTA pairs, one CTA), act_bits 8
    on its own; the decode-shaped cases run the stream kernel either way."""
    rng = np.random.default_rng(D + I + act_bits)
    E = len(counts)
    off = _segments(counts)
    R = int(off[-1])
    gp, gs = _random_int4(rng, E, I, D, 0.005, 0.02)
    up, us = _random_int4(rng, E, I, D, 0.005, 0.02)
    dp, ds = _random_int4(rng, E, D, I, 0.005, 0.02)
    x = _bf16(rng.normal(size=(R, D)))
    ex = {"gate_packed": _t(gp), "gate_scale": _t(gs, torch.bfloat16),
          "up_packed": _t(up), "up_scale": _t(us, torch.bfloat16),
          "down_packed": _t(dp), "down_scale": _t(ds, torch.bfloat16)}
    if act_bits == 16:
        xin, xs = x.to(DEV), None
    else:
        q, s = O.quantize_rows_int8(x.float().numpy())
        xin, xs = _t(q), _t(s)
    with _tc_kernels(moe, pair):
        y = moe.expert_ffn(xin, xs, _t(off), ex, act_bits)
    assert moe.check_error() == 0
    y = y.float().cpu().numpy()
    xf = oi.x_f64(x)
    refs, gots = [], []
    for e in range(E):
        a, b = off[e], off[e + 1]
        if a == b:
            continue
        exn = {"gate_packed": gp[e], "gate_scale": gs[e], "up_packed": up[e], "up_scale": us[e],
               "down_packed": dp[e], "down_scale": ds[e]}
        refs.append(O.expert_ffn(xf[a:b], exn, act_bits))
        gots.append(y[a:b])
    assert_close(np.concatenate(gots), np.concatenate(refs), what=f"ffn act{act_bits}")


@pytest.mark.parametrize("act_bits", [16, 8])
def test_expert_ffn_pairs_equals_expert_ffn(moe, act_bits):
    """moe_dispatch_pairs + moe_expert_ffn_pairs (the layer's path) give the
    bits of moe_dispatch + moe_expert_ffn (same kernels after the copy)."""
    rng = np.random.default_rng(31)
    T, k, E, D, I = 40, 4, 6, 320, 192
    idx = random_topk(T, E, k, rng)       # ~27 rows per expert: the stream kernel
    x = _bf16(rng.normal(size=(T, D)))
    gp, gs = _random_int4(rng, E, I, D, 0.005, 0.02)
    up, us = _random_int4(rng, E, I, D, 0.005, 0.02)
    dp, ds = _random_int4(rng, E, D, I, 0.005, 0.02)
    ex = {"gate_packed": _t(gp), "gate_scale": _t(gs, torch.bfloat16),
          "up_packed": _t(up), "up_scale": _t(us, torch.bfloat16),
          "down_packed": _t(dp), "down_scale": _t(ds, torch.bfloat16)}
    ti = torch.from_numpy(idx).to(DEV)
    nat = moe.dispatch(ti, x.to(DEV), E, act_bits)
    prs = moe.dispatch(ti, x.to(DEV), E, act_bits, pairs=True)
    y0 = moe.expert_ffn(nat["x_sorted"], nat["x_scale"], nat["offsets"], ex, act_bits)
    y1 = moe.expert_ffn(prs["x_sorted"], prs["x_scale"], prs["offsets"], ex, act_bits, pairs=True)
    assert moe.check_error() == 0
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))


def test_tc_pair_and_one_cta_kernels_agree(moe):
    """The CTA-pair and one-CTA tensor-core kernels take the same K steps of
    16 columns for every output, so y and h agree bit for bit, whichever
    tokens share an MMA (a prefill-shaped batch with chunks of 1 to 300 rows)."""
    rng = np.random.default_rng(53)
    D, I = 512, 384
    counts = [300, 1, 17, 64, 129, 0, 256, 48]
    E = len(counts)
    off = _segments(counts)
    R = int(off[-1])
    gp, gs = _random_int4(rng, E, I, D, 0.005, 0.02)
    up, us = _random_int4(rng, E, I, D, 0.005, 0.02)
    dp, ds = _random_int4(rng, E, D, I, 0.005, 0.02)
    ex = {"gate_packed": _t(gp), "gate_scale": _t(gs, torch.bfloat16),
          "up_packed": _t(up), "up_scale": _t(us, torch.bfloat16),
          "down_packed": _t(dp), "down_scale": _t(ds, torch.bfloat16)}
    x = _bf16(rng.normal(size=(R, D))).to(DEV)
    ys = []
    for pair in (True, False):
        with _tc_kernels(moe, pair):
            ys.append(moe.expert_ffn(x, None, _t(off), ex, 16))
    assert moe.check_error() == 0
    assert torch.equal(ys[0].view(torch.int16), ys[1].view(torch.int16))


@pytest.mark.parametrize("act_bits", [16, 8])
@pytest.mark.parametrize("counts,bound", [([5, 30, 0, 12], 30), ([5, 60, 200, 17], 200),
                                          ([5, 60, 200, 17], 10)])
def test_expert_ffn_pairs_bounded_gives_the_same_bits(moe, act_bits, counts, bound):
    """moe_expert_ffn_pairs_bounded with a true bound on the rows per expert
    gives the bits of moe_expert_ffn_pairs; a bound below the true count (10
    rows for a batch with 200) moves every expert to the stream kernel: the
    same values within the kernels' rounding."""
    rng = np.random.default_rng(71 + act_bits + bound)
    D, I = 256, 192
    E = len(counts)
    off = _segments(counts)
    R = int(off[-1])
    gp, gs = _random_int4(rng, E, I, D, 0.005, 0.02)
    up, us = _random_int4(rng, E, I, D, 0.005, 0.02)
    dp, ds = _random_int4(rng, E, D, I, 0.005, 0.02)
    ex = {"gate_packed": _t(gp), "gate_scale": _t(gs, torch.bfloat16),
          "up_packed": _t(up), "up_scale": _t(us, torch.bfloat16),
          "down_packed": _t(dp), "down_scale": _t(ds, torch.bfloat16)}
    T = R  # one token per row
    idx = np.zeros((T, 1), dtype=np.int32)
    for e in range(E):
        idx[off[e]:off[e + 1], 0] = e
    x = _bf16(rng.normal(size=(T, D)))
    d = moe.dispatch(torch.from_numpy(idx).to(DEV), x.to(DEV), E, act_bits, pairs=True)
    y0 = moe.expert_ffn(d["x_sorted"], d["x_scale"], d["offsets"], ex, act_bits, pairs=True)
    y1 = moe.expert_ffn(d["x_sorted"], d["x_scale"], d["offsets"], ex, act_bits, pairs=True,
                        max_rows_per_expert=bound)
    assert moe.check_error() == 0
    if bound >= max(counts):
        assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    else:
        assert rel_l2(y1.float().cpu().numpy(), y0.float().cpu().numpy()) <= 5e-3


@pytest.mark.parametrize("counts", [[5, 30], [5, 60]])
def test_expert_ffn_reports_fp16_overflow_and_recovers(moe, counts):
    """An intermediate h beyond the fp16 range, on both expert kernels (5 + 30
    rows: the stream kernel; 5 + 60 rows: the tensor cores), records
    MOE_ERR_UNSUPPORTED; the call finishes and the next call is clean."""
    rng = np.random.default_rng(41)
    D, I = 256, 128
    E = len(counts)
    off = _segments(counts)
    R = int(off[-1])
    gp, gs = _random_int4(rng, E, I, D, 0.005, 0.02)
    up, us = _random_int4(rng, E, I, D, 0.005, 0.02)
    dp, ds = _random_int4(rng, E, D, I, 0.005, 0.02)
    ex = {"gate_packed": _t(gp), "gate_scale": _t(gs, torch.bfloat16),
          "up_packed": _t(up), "up_scale": _t(us, torch.bfloat16),
          "down_packed": _t(dp), "down_scale": _t(ds, torch.bfloat16)}
    big = _bf16(rng.normal(size=(R, D)) * 3000.0)
    moe.expert_ffn(big.to(DEV), None, _t(off), ex, 16)
    assert moe.check_error() == moe.capi.MOE_ERR_UNSUPPORTED
    assert moe.check_error() == 0
    small = _bf16(rng.normal(size=(R, D)))
    moe.expert_ffn(small.to(DEV), None, _t(off), ex, 16)
    assert moe.check_error() == 0


def test_status_word_is_a_report_only(moe):
    """An error that one call records (an fp16 overflow in a prefill-shaped
    batch, on the tensor cores; a bounded wait that ran out) leaves later
    calls unchanged, with
    no moe_check_error in between: they give the bits of a clean call, and
    the status word keeps the first error until it is read."""
    rng = np.random.default_rng(43)
    D, I, counts = 256, 128, [5, 60]
    E = len(counts)
    off = _t(_segments(counts))
    R = sum(counts)
    gp, gs = _random_int4(rng, E, I, D, 0.005, 0.02)
    up, us = _random_int4(rng, E, I, D, 0.005, 0.02)
    dp, ds = _random_int4(rng, E, D, I, 0.005, 0.02)
    ex = {"gate_packed": _t(gp), "gate_scale": _t(gs, torch.bfloat16),
          "up_packed": _t(up), "up_scale": _t(us, torch.bfloat16),
          "down_packed": _t(dp), "down_scale": _t(ds, torch.bfloat16)}
    small = _bf16(rng.normal(size=(R, D))).to(DEV)
    big = _bf16(rng.normal(size=(R, D)) * 3000.0).to(DEV)
    clean = moe.expert_ffn(small, None, off, ex, 16)
    assert moe.check_error() == 0
    moe.expert_ffn(big, None, off, ex, 16)          # records UNSUPPORTED
    after_unsupported = moe.expert_ffn(small, None, off, ex, 16)
    moe.wait_selftest(20_000_000)                   # a wait runs out (TIMEOUT, not kept)
    after_timeout = moe.expert_ffn(small, None, off, ex, 16)
    assert moe.check_error() == moe.capi.MOE_ERR_UNSUPPORTED   # the first error
    assert torch.equal(after_unsupported.view(torch.int16), clean.view(torch.int16))
    assert torch.equal(after_timeout.view(torch.int16), clean.view(torch.int16))
    moe.wait_selftest(20_000_000)
    again = moe.expert_ffn(small, None, off, ex, 16)
    assert moe.check_error() == moe.capi.MOE_ERR_TIMEOUT
    assert torch.equal(again.view(torch.int16), clean.view(torch.int16))
    assert moe.check_error() == 0


def test_ffn_rejects_offsets_beyond_capacity(moe):
    rng = np.random.default_rng(1)
    E, D, I = 2, 128, 128
    gp, gs = _random_int4(rng, E, I, D)
    dp, ds = _random_int4(rng, E, D, I)
    ex = {"gate_packed": _t(gp), "gate_scale": _t(gs, torch.bfloat16), "up_packed": _t(gp),
          "up_scale": _t(gs, torch.bfloat16), "down_packed": _t(dp), "down_scale": _t(ds, torch.bfloat16)}
    x = torch.zeros(8, D, dtype=torch.bfloat16, device=DEV)
    bad = _t(np.array([0, 5, 3], np.int32))      # decreasing
    moe.expert_ffn(x, None, bad, ex, 16)
    assert moe.check_error() == moe.capi.MOE_ERR_INVALID
    assert moe.check_error() == 0


# ---------------------------------------------------------------- combine

def test_combine_rejects_rows_outside_y(moe):
    """A row index outside [0, T*k) is skipped and recorded (MOE_ERR_INVALID);
    the other slots of the token still add up."""
    rng = np.random.default_rng(5)
    T, k, D = 4, 2, 128
    y = _bf16(rng.normal(size=(T * k, D)))
    inv = np.arange(T * k, dtype=np.int32)
    inv[3] = T * k          # one past the last row
    inv[6] = -1
    w = np.full((T, k), 0.5, np.float32)
    out = moe.combine(y.to(DEV), _t(inv), _t(w))
    assert moe.check_error() == moe.capi.MOE_ERR_INVALID
    assert moe.check_error() == 0
    got = out.float().cpu().numpy()
    yf = oi.x_f64(y)
    assert np.array_equal(got[1], (0.5 * yf[2]).astype(np.float32))   # slot 1 skipped
    assert np.array_equal(got[3], (0.5 * yf[7]).astype(np.float32))   # slot 0 skipped
    ref0 = 0.5 * yf[0] + 0.5 * yf[1]
    assert np.all(np.abs(got[0] - ref0) <= 2 ** -8 * np.abs(ref0) + 1e-6)


def test_combine_parity(moe):
    rng = np.random.default_rng(3)
    T, k, D = 70, 6, 448
    R = T * k
    y = _bf16(rng.normal(size=(R, D)))
    inv = rng.permutation(R).astype(np.int32)
    w = rng.uniform(0, 1, size=(T, k)).astype(np.float32)
    out = moe.combine(y.to(DEV), _t(inv), _t(w))
    got = out.float().cpu().numpy()
    yf = oi.x_f64(y)
    ref = (yf[inv].reshape(T, k, D) * w.astype(np.float64)[:, :, None]).sum(1)
    # fp32 accumulation, one bf16 rounding of the result (2^-9 relative)
    assert np.all(np.abs(got - ref) <= 2 ** -8 * np.abs(ref) + 1e-5)


def test_linear_bf16_and_rmsnorm(moe):
    rng = np.random.default_rng(4)
    M, N, K = 100, 136, 96
    x = _bf16(rng.normal(size=(M, K)))
    W = _bf16(rng.normal(size=(N, K)) * 0.1)
    y = moe.linear_bf16(x.to(DEV), W.to(DEV)).float().cpu().numpy()
    ref = oi.x_f64(x) @ oi.x_f64(W).T
    assert np.all(np.abs(y - ref) <= 2 ** -8 * np.abs(ref) + 1e-5 * np.abs(ref).max())
    g = _bf16(rng.uniform(0.5, 1.5, size=192))
    v = _bf16(rng.normal(size=(33, 192)) * 4)
    out = moe.rmsnorm(v.to(DEV), g.to(DEV), 1e-6).float().cpu().numpy()
    ref = O.rmsnorm(oi.x_f64(v), bf16_bits(g), 1e-6)
    assert np.all(np.abs(out - ref) <= 2 ** -8 * np.abs(ref) + 1e-6)


# ---------------------------------------------------------- bounded waits

def test_bounded_wait_reports_timeout_and_context_survives(moe):
    moe.wait_selftest(20_000_000)   # 20 ms on a barrier that nothing completes
    assert moe.check_error() == moe.capi.MOE_ERR_TIMEOUT
    assert moe.check_error() == 0   # cleared
    q, s = moe.quantize_rows(torch.ones(2, 64, dtype=torch.bfloat16, device=DEV))
    assert float(s[0]) == float(np.float32(1.0) / np.float32(127.0))
    assert moe.check_error() == 0


@pytest.mark.parametrize("act_bits,kernel", [(16, 0), (8, 0), (16, 1), (8, 1), (16, 2), (16, 3)])
def test_pipelined_kernel_exit_paths(moe, kernel, act_bits):
    """A producer that stops before its fourth copy stage (a test build of the
    stream, tensor-core (both tile layouts) and CTA-pair kernels): the other roles' bounded waits
    (20 ms) run out, the kernel records MOE_ERR_TIMEOUT, drains its copies and
    MMAs, frees its tensor memory and returns (a CTA pair after both CTAs'
    roles have stopped); the next call is correct and clean."""
    rng = np.random.default_rng(77 + kernel + act_bits)
    K, N, counts = 2048, 512, [20, 40]
    E = len(counts)
    off = _segments(counts)
    R = int(off[-1])
    packed, scale = _random_int4(rng, E, N, K, 0.002, 0.02)
    x = _bf16(rng.normal(size=(R, K)))
    if act_bits == 16:
        xin, xs = x.to(DEV), None
    else:
        q, sx = O.quantize_rows_int8(x.float().numpy())
        xin, xs = _t(q), _t(sx)
    args = (xin, xs, _t(off), _t(packed), _t(scale, torch.bfloat16))
    moe.int4_linear_stall_selftest(*args, act_bits, kernel, 3, 20_000_000)
    assert moe.check_error() == moe.capi.MOE_ERR_TIMEOUT
    assert moe.check_error() == 0
    got = moe.int4_linear(*args, act_bits).cpu().numpy()
    assert moe.check_error() == 0
    xf = oi.x_f64(x)
    for e in range(E):
        a, b = off[e], off[e + 1]
        assert rel_l2(got[a:b], O.int4_linear(xf[a:b], packed[e], scale[e], act_bits)) <= 1e-5


def test_limits_are_enforced(moe):
    """One past each limit (2048 experts, top-32) is rejected before any launch."""
    x = torch.zeros(4, 256, dtype=torch.bfloat16, device=DEV)
    for E, k in [(2049, 8), (64, 33)]:
        W = torch.zeros(E, 256, device=DEV)
        b = torch.zeros(E, device=DEV)
        with pytest.raises(moe.MoeError) as ei:
            moe.route(x, W, b, k, True)
        assert "UNSUPPORTED" in str(ei.value)
    assert moe.check_error() == 0
