"""Whole-layer GPU parity against the fp64 oracle, at small sizes (every token)
and at every full workload size in the launch configuration the benchmark
times (sampled tokens, evaluated one by one by the oracle).

Tolerance (layer output, bf16): relative L2 <= 5e-3 and max abs <= 3e-2 x RMS
of the oracle output.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as wl
from oracle import inputs as oi
from tests._helpers import (assert_close, conditioned_attempts, device_weights, oracle_tokens,
                            targeted_tokens)

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


def _layer(moe, w, weights):
    return moe.MoeLayer(w.T, w.H, w.E, w.k, w.I, weights, L=w.L, act_bits=w.act_bits,
                        renorm=w.renorm, eps=w.eps)


SMALL = {
    "tiny": wl.WORKLOADS["tiny"],
    "tiny_exact": wl.workload("tiny", act_bits=8),
    "ragged": wl.workload("tiny", name="ragged", T=77, H=512, E=40, k=6, I=192, seed=3),
    "ragged_exact": wl.workload("tiny", name="ragged", T=77, H=512, E=40, k=6, I=192, seed=3,
                                act_bits=8),
    "small_latent": wl.workload("tiny", name="small_latent", T=50, H=512, L=256, E=16, k=4,
                                I=128, seed=9, norm_gain_std=0.1),
    # exact mode on the latent width: the int8 rows are the bf16 latent
    # projection's, and the expert outputs stay fp32 into the RMSNorm
    "small_latent_exact": wl.workload("tiny", name="small_latent_exact", T=50, H=512, L=256,
                                      E=16, k=4, I=128, seed=9, norm_gain_std=0.1, act_bits=8),
    "small_adversarial": wl.workload("tiny", name="small_adv", T=60, H=512, E=16, k=4, I=192,
                                     seed=10, act_bits=8, routing="adversarial"),
    "one_token": wl.workload("tiny", name="one", T=1, H=256, E=8, k=2, I=128, seed=12),
    "multi_chunk": wl.workload("tiny", name="multi", T=200, H=256, E=4, k=2, I=128, seed=13),
    "no_renorm": wl.workload("tiny", name="nr", T=40, H=256, E=24, k=3, I=64, renorm=False, seed=6),
    # the library's limits: 2048 experts, top-32
    "max_E_k": wl.workload("tiny", name="max_E_k", T=20, H=256, E=2048, k=32, I=64, seed=21),
    "max_E_k_exact": wl.workload("tiny", name="max_E_k_exact", T=20, H=256, E=2048, k=32, I=64,
                                 seed=21, act_bits=8),
}


@pytest.mark.parametrize("case", list(SMALL))
def test_layer_small_all_tokens(moe, case):
    w = SMALL[case]
    x = wl.gen_x(w, attempts=conditioned_attempts(w))
    router = wl.gen_router(w)
    lat = wl.gen_latent(w)
    layer = _layer(moe, w, device_weights(w, DEV, router, lat))
    out = layer.forward(x.to(DEV))
    assert moe.check_error() == 0
    ref = O.moe_forward(oi.x_f64(x), oi.layer_params(w, router=router, latent=lat))
    assert_close(out.float().cpu().numpy(), ref, what=case)


# ----------------------------------------------------------- full sizes

@pytest.mark.parametrize("name", ["decode", "prefill", "latent", "exact"])
def test_layer_full_size_sampled(moe, name):
    """The full workloads against the oracle on at least 32 tokens each (all
    32 at decode), chosen to reach the hottest experts' last ragged chunks,
    128-row chunk boundaries and experts of exactly 16 and 17 rows (the
    smallest experts, which in these prefill-shaped batches also run on the
    tensor cores)."""
    w = wl.WORKLOADS[name]
    x = wl.gen_x(w)
    router = wl.gen_router(w)
    lat = wl.gen_latent(w)
    layer = _layer(moe, w, device_weights(w, DEV, router, lat))
    out = layer.forward(x.to(DEV))
    assert moe.check_error() == 0
    out = out.float().cpu().numpy()
    assert np.all(np.isfinite(out))
    toks = targeted_tokens(w, x, router)
    assert len(toks) >= min(32, w.T)
    ref = oracle_tokens(w, x, router, lat, toks)
    assert_close(out[toks], ref, what=name)


def test_layer_deterministic_and_host_variant(moe):
    w = wl.WORKLOADS["decode"]
    x = wl.gen_x(w)
    layer = _layer(moe, w, device_weights(w, DEV))
    a = layer.forward(x.to(DEV))
    b = layer.forward(x.to(DEV))
    assert torch.equal(a, b)
    xh = x.pin_memory()
    oh = torch.empty_like(x).pin_memory()
    layer.forward_host(xh, oh)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(oh, a.cpu())
    assert moe.check_error() == 0


def test_layer_router_prepared_terms_give_the_same_bits(moe):
    """From 512 tokens the router's logits run on the tensor cores with the
    fp32 weight split into three bf16 terms; a layer given the terms once
    (moe_router_prepare, MoeLayer's default) and one that splits the weight on
    every call give the same bits."""
    w = wl.workload("tiny", name="prep", T=600, H=512, E=48, k=4, I=128, seed=31)
    x = wl.gen_x(w).to(DEV)
    weights = device_weights(w, DEV)
    a = moe.MoeLayer(w.T, w.H, w.E, w.k, w.I, weights).forward(x)
    b = moe.MoeLayer(w.T, w.H, w.E, w.k, w.I, weights, prepare_router=False).forward(x)
    assert moe.check_error() == 0
    assert torch.equal(a, b)


def test_layer_zero_tokens(moe):
    w = wl.workload("tiny", T=0)
    weights = device_weights(wl.WORKLOADS["tiny"], DEV)
    layer = _layer(moe, w, weights)
    out = layer.forward(torch.empty(0, w.H, dtype=torch.bfloat16, device=DEV))
    assert out.shape == (0, w.H)
    assert moe.check_error() == 0


# ----------------------------------------------------------- shared expert

def _shared_weights(rng, H, Is, std=0.02):
    mk = lambda *s: O.f32_to_bf16_bits((rng.normal(size=s) * std).astype(np.float32))
    return mk(Is, H), mk(Is, H), mk(H, Is)


def _bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits)).view(torch.bfloat16).to(DEV)


@pytest.mark.parametrize("T,H,Is,acc", [(5, 512, 256, False), (32, 1024, 320, True),
                                        (300, 768, 192, True), (1, 7168, 2048, False)])
def test_shared_expert_parity(moe, T, H, Is, acc):
    """out (+)= down(bf16(SiLU(gate x) * up x)) against the fp64 oracle; the
    split-K slices (many when T is small) are summed in fp32."""
    rng = np.random.default_rng(T + H + Is)
    g, u, d = _shared_weights(rng, H, Is)
    x = torch.from_numpy(rng.normal(size=(T, H)).astype(np.float32)).to(torch.bfloat16)
    base = torch.from_numpy(rng.normal(size=(T, H)).astype(np.float32) * 0.1).to(torch.bfloat16)
    out = base.to(DEV) if acc else None
    got = moe.shared_expert(x.to(DEV), _bf16_dev(g), _bf16_dev(u), _bf16_dev(d), out)
    assert moe.check_error() == 0
    ref = O.shared_expert(oi.x_f64(x), g, u, d)
    if acc:
        ref = ref + base.double().numpy()
    assert_close(got.float().cpu().numpy(), ref, what=f"shared {T}x{H}x{Is}")


@pytest.mark.parametrize("case", ["tiny", "small_latent", "tiny_exact", "small_latent_exact"])
def test_layer_with_shared_expert(moe, case):
    w = SMALL[case]
    Is = 192
    rng = np.random.default_rng(31)
    g, u, d = _shared_weights(rng, w.H, Is)
    x = wl.gen_x(w, attempts=conditioned_attempts(w))
    router = wl.gen_router(w)
    lat = wl.gen_latent(w)
    weights = device_weights(w, DEV, router, lat)
    weights.update({"shared_gate": _bf16_dev(g), "shared_up": _bf16_dev(u),
                    "shared_down": _bf16_dev(d)})
    layer = moe.MoeLayer(w.T, w.H, w.E, w.k, w.I, weights, L=w.L, act_bits=w.act_bits,
                         renorm=w.renorm, eps=w.eps, I_shared=Is)
    out = layer.forward(x.to(DEV))
    assert moe.check_error() == 0
    p = oi.layer_params(w, router=router, latent=lat)
    p.shared_gate, p.shared_up, p.shared_down = g, u, d
    ref = O.moe_forward(oi.x_f64(x), p)
    assert_close(out.float().cpu().numpy(), ref, what=case + "+shared")


@pytest.mark.parametrize("case", ["tiny", "small_latent", "small_adversarial"])
def test_layer_forward_replays_from_a_cuda_graph(moe, case):
    """The layer call allocates nothing and never synchronises the host, so a
    captured CUDA graph of it replays to the same bits as stream launches."""
    w = SMALL[case]
    x = wl.gen_x(w, attempts=conditioned_attempts(w)).to(DEV)
    router = wl.gen_router(w)
    lat = wl.gen_latent(w)
    layer = _layer(moe, w, device_weights(w, DEV, router, lat))
    ref = layer.forward(x)
    out = torch.zeros_like(ref)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.forward(x, out)  # warm-up on the capture stream
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            layer.forward(x, out)
        out.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert moe.check_error() == 0
    assert torch.equal(out, ref)


@pytest.mark.parametrize("case", ["tiny", "small_latent", "small_adversarial", "tiny_exact"])
def test_layer_graph_launches_replay_the_call(moe, case):
    """moe_layer_graph_create / _launch: every launch of the captured call
    gives the bits of moe_layer_forward (and of forward_host through pinned
    buffers), and moe_launch_count advances by the captured kernel count."""
    w = SMALL[case]
    x = wl.gen_x(w, attempts=conditioned_attempts(w))
    router = wl.gen_router(w)
    lat = wl.gen_latent(w)
    layer = _layer(moe, w, device_weights(w, DEV, router, lat))
    xd = x.to(DEV)
    ref = layer.forward(xd)
    torch.cuda.synchronize()
    n0 = moe.launch_count()
    layer.forward(xd, torch.empty_like(ref))
    per_call = moe.launch_count() - n0
    out = torch.zeros_like(ref)
    g = layer.graph(xd, out)
    assert not out.any()                      # capturing runs nothing
    n1 = moe.launch_count()
    for _ in range(2):
        out.zero_()
        g.launch()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    assert moe.launch_count() - n1 == 2 * per_call
    g.close()
    xh = x.pin_memory()
    oh = torch.zeros_like(x).pin_memory()
    gh = layer.graph(xh, oh, host=True)
    gh.launch()
    torch.cuda.synchronize()
    assert torch.equal(oh, ref.cpu())
    gh.close()
    assert moe.check_error() == 0


@pytest.mark.parametrize("case", ["tiny", "small_latent", "tiny_exact"])
def test_layer_pipe_gives_each_call_its_bits(moe, case):
    """Five calls with different inputs through a pipe (input and output
    copies on the pipe's own streams, overlapping the neighbouring calls'
    compute, two device slots used in turn) give, in each call's own host
    buffer, the bits of forward on that input."""
    w = SMALL[case]
    layer = _layer(moe, w, device_weights(w, DEV))
    x0 = wl.gen_x(w)
    xs = [torch.roll(x0, i, dims=0).contiguous() for i in range(5)]
    want = [layer.forward(x.to(DEV)).cpu() for x in xs]
    pipe = layer.pipe()
    xh = [x.pin_memory() for x in xs]
    oh = [torch.empty_like(x).pin_memory() for x in xs]
    for a, b in zip(xh, oh):
        pipe.submit(a, b)
    pipe.join()
    torch.cuda.current_stream().synchronize()
    assert moe.check_error() == 0
    for i in range(5):
        assert torch.equal(oh[i], want[i]), i
    # a second round through the same pipe
    for a, b in zip(xh[::-1], oh):
        pipe.submit(a, b)
    pipe.join()
    torch.cuda.current_stream().synchronize()
    for i in range(5):
        assert torch.equal(oh[i], want[4 - i]), i
    # host buffers that are not pinned, or on the device, are refused
    with pytest.raises(ValueError):
        pipe.submit(xs[0], oh[0])
    with pytest.raises(ValueError):
        pipe.submit(xh[0], want[0].to(DEV))
    pipe.close()
    with pytest.raises(ValueError):
        pipe.submit(xh[0], oh[0])
    assert moe.check_error() == 0


def test_layer_graph_rejects_bad_arguments_before_capture(moe):
    w = SMALL["tiny"]
    layer = _layer(moe, w, device_weights(w, DEV))
    x = torch.zeros(w.T, w.H, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ValueError):
        layer.graph(x[:-1], torch.empty_like(x))
    with pytest.raises(ValueError):
        layer.graph(x.cpu(), torch.empty_like(x).cpu(), host=True)   # not pinned
    bad = moe.capi.MoeConfig(w.T, w.H, w.E, w.k + w.E, w.I, 0, 16, 1, 1e-6, 0)  # k > E
    h = moe.capi.c_void_p(123)
    rc = moe.lib.moe_layer_graph_create(moe.capi.ctypes.byref(bad), moe.capi.ctypes.byref(layer.wstruct),
                                        x.data_ptr(), x.data_ptr(), 0, layer.ws.data_ptr(),
                                        layer.ws.numel(), None, moe.capi.ctypes.byref(h))
    assert rc == moe.capi.MOE_ERR_UNSUPPORTED and not h.value
    moe.lib.moe_layer_graph_destroy(None)
    assert moe.check_error() == 0


def test_layer_rejects_mis_sized_buffers_before_any_launch(moe):
    w = SMALL["tiny"]
    layer = _layer(moe, w, device_weights(w, DEV))
    n0 = moe.launch_count()
    for x, out in [(torch.zeros(w.T - 1, w.H, dtype=torch.bfloat16, device=DEV), None),
                   (torch.zeros(w.T, w.H, dtype=torch.bfloat16, device=DEV),
                    torch.zeros(w.T, w.H // 2, dtype=torch.bfloat16, device=DEV)),
                   (torch.zeros(w.T, 2 * w.H, dtype=torch.bfloat16, device=DEV)[:, ::2], None),
                   (torch.zeros(w.T, w.H, dtype=torch.bfloat16), None)]:
        with pytest.raises(ValueError):
            layer.forward(x, out)
    with pytest.raises(ValueError):
        moe.combine(torch.zeros(w.T * w.k - 1, w.H, dtype=torch.bfloat16, device=DEV),
                    torch.zeros(w.T * w.k, dtype=torch.int32, device=DEV),
                    torch.zeros(w.T, w.k, dtype=torch.float32, device=DEV))
    assert moe.launch_count() == n0
    assert moe.check_error() == 0
