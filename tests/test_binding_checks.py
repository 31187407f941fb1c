"""Host-side argument checks of the Python binding (no GPU needed).

The library trusts the sizes it is given, so the binding checks every tensor
against the layout in include/moe.h before passing its pointer on.  The
checks look at dtype and shape first and placement last.  So on a machine
without a GPU, a wrong shape raises its own error, and a correctly shaped
host tensor gets as far as the "must live on a CUDA device" error.  No
library call is reached here.
"""
import pytest
import torch

import workloads as wl

CUDA_ONLY = "must live on a CUDA device"


@pytest.fixture(scope="module")
def capi():
    from int4_routed_expert_fp32_gb300.build import build
    build()
    from int4_routed_expert_fp32_gb300 import capi as c
    return c


def bf16(*shape):
    return torch.zeros(*shape, dtype=torch.bfloat16)


def i32(*shape):
    return torch.zeros(*shape, dtype=torch.int32)


def f32(*shape):
    return torch.zeros(*shape, dtype=torch.float32)


def experts(E, D, I, **override):
    ex = {"gate_packed": i32(E, I, D // 8), "gate_scale": bf16(E, I, D // 32),
          "up_packed": i32(E, I, D // 8), "up_scale": bf16(E, I, D // 32),
          "down_packed": i32(E, D, I // 8), "down_scale": bf16(E, D, I // 32)}
    ex.update(override)
    return ex


def raises(match, fn, *args, **kwargs):
    with pytest.raises(ValueError, match=match):
        fn(*args, **kwargs)


def test_route(capi):
    w = wl.WORKLOADS["tiny"]
    x = wl.gen_x(w)
    W, b = wl.gen_router(w)
    raises(CUDA_ONLY, capi.route, x, W, b, w.k)             # generator outputs pass the checks
    raises("w_router: expected shape", capi.route, x, W[:, :-8], b, w.k)
    raises("bias: expected shape", capi.route, x, W, b[:-1], w.k)
    raises("x: expected torch.bfloat16", capi.route, x.float(), W, b, w.k)
    raises("w_router: expected torch.float32", capi.route, x, W.to(torch.bfloat16), b, w.k)
    raises("x must be contiguous", capi.route, bf16(256, 16).t(), W, b, w.k)


@pytest.mark.parametrize("fn", ["dispatch", "dispatch_noalloc"])
def test_dispatch(capi, fn):
    f = getattr(capi, fn)
    raises(CUDA_ONLY, f, i32(16, 2), bf16(16, 256), 8)
    raises("x: expected shape", f, i32(16, 2), bf16(15, 256), 8)   # fewer rows than tokens
    raises("topk_idx: expected torch.int32", f, torch.zeros(16, 2, dtype=torch.int64),
           bf16(16, 256), 8)


def test_expert_ffn(capi):
    E, D, I, rows = 4, 256, 128, 40
    raises(CUDA_ONLY, capi.expert_ffn, bf16(rows, D), None, i32(E + 1), experts(E, D, I))
    raises(CUDA_ONLY, capi.expert_ffn, torch.zeros(rows, D, dtype=torch.int8), f32(rows),
           i32(E + 1), experts(E, D, I), 8)
    raises(CUDA_ONLY, capi.expert_ffn, torch.zeros(rows, D, dtype=torch.float16), None,
           i32(E + 1), experts(E, D, I), 16, pairs=True)
    raises("offsets: expected shape", capi.expert_ffn, bf16(rows, D), None, i32(E), experts(E, D, I))
    raises("x_scale is required", capi.expert_ffn, torch.zeros(rows, D, dtype=torch.int8), None,
           i32(E + 1), experts(E, D, I), 8)
    raises("x_scale: expected shape", capi.expert_ffn, torch.zeros(rows, D, dtype=torch.int8),
           f32(rows - 1), i32(E + 1), experts(E, D, I), 8)
    raises("x: expected torch.float16", capi.expert_ffn, bf16(rows, D), None, i32(E + 1),
           experts(E, D, I), 16, pairs=True)
    raises("down_scale: expected shape", capi.expert_ffn, bf16(rows, D), None, i32(E + 1),
           experts(E, D, I, down_scale=bf16(E, D, I // 64)))
    raises("up_packed: expected shape", capi.expert_ffn, bf16(rows, D), None, i32(E + 1),
           experts(E, D, I, up_packed=i32(E, I, D // 16)))
    raises("gate_scale is required", capi.expert_ffn, bf16(rows, D), None, i32(E + 1),
           experts(E, D, I, gate_scale=None))


def test_int4_linear(capi):
    E, K, N, rows = 3, 256, 64, 10
    raises(CUDA_ONLY, capi.int4_linear, bf16(rows, K), None, i32(E + 1), i32(E, N, K // 8),
           bf16(E, N, K // 32))
    raises("w_packed: expected shape", capi.int4_linear, bf16(rows, K), None, i32(E + 1),
           i32(E, N, K // 16), bf16(E, N, K // 32))
    raises("w_scale: expected shape", capi.int4_linear, bf16(rows, K), None, i32(E + 1),
           i32(E, N, K // 8), bf16(E, N + 1, K // 32))
    raises("x: expected torch.int8", capi.int4_linear, bf16(rows, K), f32(rows), i32(E + 1),
           i32(E, N, K // 8), bf16(E, N, K // 32), 8)


def test_combine_linear_rmsnorm_quantisers(capi):
    T, k, D = 6, 3, 128
    raises(CUDA_ONLY, capi.combine, bf16(T * k, D), i32(T * k), f32(T, k))
    raises("y_sorted: expected shape", capi.combine, bf16(T * k - 1, D), i32(T * k), f32(T, k))
    raises("inv_row: expected 18 entries", capi.combine, bf16(T * k, D), i32(T * k - 1), f32(T, k))
    raises(CUDA_ONLY, capi.linear_bf16, bf16(5, 64), bf16(32, 64))
    raises("w: expected shape", capi.linear_bf16, bf16(5, 64), bf16(32, 96))
    raises(CUDA_ONLY, capi.rmsnorm, bf16(5, 64), bf16(64), 1e-6)
    raises("gain: expected shape", capi.rmsnorm, bf16(5, 64), bf16(32), 1e-6)
    raises("v: expected shape", capi.quantize_rows, bf16(64))
    raises(CUDA_ONLY, capi.quantize_int4, bf16(3, 8, 64))
    raises(CUDA_ONLY, capi.quantize_int8, bf16(3, 8, 64))


def test_shared_expert(capi):
    T, H, I = 4, 128, 64
    raises(CUDA_ONLY, capi.shared_expert, bf16(T, H), bf16(I, H), bf16(I, H), bf16(H, I))
    raises(CUDA_ONLY, capi.shared_expert, bf16(T, H), bf16(I, H), bf16(I, H), bf16(H, I),
           bf16(T, H))
    raises("down_w: expected shape", capi.shared_expert, bf16(T, H), bf16(I, H), bf16(I, H),
           bf16(I, H))
    raises("up_w: expected shape", capi.shared_expert, bf16(T, H), bf16(I, H), bf16(I + 1, H),
           bf16(H, I))
    raises("out: expected shape", capi.shared_expert, bf16(T, H), bf16(I, H), bf16(I, H),
           bf16(H, I), bf16(T - 1, H))


def _layer_weights(H, E, I, L=0, Is=0):
    D = L if L else H
    w = {"router_w": f32(E, H), "router_bias": f32(E), **experts(E, D, I)}
    if L:
        w.update({"lat_down": bf16(L, H), "lat_norm": bf16(L), "lat_up": bf16(H, L)})
    if Is:
        w.update({"shared_gate": bf16(Is, H), "shared_up": bf16(Is, H), "shared_down": bf16(H, Is)})
    return w


def test_layer_weights(capi):
    T, H, E, k, I, L, Is = 8, 256, 6, 2, 128, 128, 64
    Layer = capi.MoeLayer
    raises(CUDA_ONLY, Layer, T, H, E, k, I, _layer_weights(H, E, I))
    raises(CUDA_ONLY, Layer, T, H, E, k, I, _layer_weights(H, E, I, L=L), L=L)
    raises(CUDA_ONLY, Layer, T, H, E, k, I, _layer_weights(H, E, I, Is=Is), I_shared=Is)
    w = _layer_weights(H, E, I, L=L)
    w["lat_norm"] = None                        # the latent norm is optional
    raises(CUDA_ONLY, Layer, T, H, E, k, I, w, L=L)
    for name, bad in [("router_w", f32(E, H + 32)), ("router_w", f32(E + 1, H)),
                      ("router_bias", f32(E + 1)), ("down_scale", bf16(E, H, I // 64))]:
        w = _layer_weights(H, E, I)
        w[name] = bad
        raises(f"{name}: expected shape", Layer, T, H, E, k, I, w)
    # the experts take the latent width when L > 0
    w = _layer_weights(H, E, I, L=L)
    w.update(experts(E, H, I))
    raises("gate_packed: expected shape", Layer, T, H, E, k, I, w, L=L)
    w = _layer_weights(H, E, I, L=L)
    del w["lat_up"]
    raises("lat_up is required", Layer, T, H, E, k, I, w, L=L)
    w = _layer_weights(H, E, I, Is=Is)
    w["shared_down"] = bf16(Is, H)
    raises("shared_down: expected shape", Layer, T, H, E, k, I, w, I_shared=Is)
    raises("shared_gate is required", Layer, T, H, E, k, I, _layer_weights(H, E, I), I_shared=Is)
    w = _layer_weights(H, E, I)
    w["router_b"] = f32(E)
    raises("unknown weight names", Layer, T, H, E, k, I, w)


def test_layer_forward_buffers(capi, monkeypatch):
    """x and out of forward / forward_host must be bf16 [T, H]; a layer is
    built on host tensors with the placement check and the workspace faked."""
    monkeypatch.setattr(capi, "_placed", lambda **t: torch.device("cpu"))
    monkeypatch.setattr(capi, "_ws", lambda n, d: torch.empty(1))
    monkeypatch.setattr(capi.lib, "moe_workspace_size", lambda cfg: 1)
    T, H, E, k, I = 8, 256, 6, 2, 128
    layer = capi.MoeLayer(T, H, E, k, I, _layer_weights(H, E, I))
    raises("x: expected shape", layer.forward, bf16(T - 1, H))
    raises("x: expected torch.bfloat16", layer.forward, f32(T, H))
    raises("out: expected shape", layer.forward, bf16(T, H), bf16(T, H - 64))
    raises("x_host: expected torch.bfloat16", layer.forward_host, f32(T, H), bf16(T, H))
    raises("out_host: expected shape", layer.forward_host, bf16(T, H), bf16(2 * T, H))
    raises("x_host must be contiguous", layer.forward_host, bf16(H, T).t(), bf16(T, H))
