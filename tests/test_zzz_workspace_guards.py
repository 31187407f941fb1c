"""Guard words around every buffer the layer writes.

compute-sanitizer is not available on the pool, so out-of-bounds writes are
looked for directly. The layer is called through the C ABI with a workspace
and an output that each sit between guard regions filled with a known byte
pattern. After the call every guard byte must be unchanged, and so must the
input. The input is checked too, since the library only reads it.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl
from tests._helpers import conditioned_attempts, device_weights

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
GUARD = 1 << 16        # bytes on each side of the workspace (a multiple of 256)
PATTERN = 0xA5


@pytest.fixture(scope="module")
def moe():
    from int4_routed_expert_fp32_gb300.build import build
    build()
    import int4_routed_expert_fp32_gb300 as m
    torch.cuda.set_device(DEV)
    assert m.check_error() == 0
    yield m
    assert m.check_error() == 0


CASES = {
    "tiny": wl.WORKLOADS["tiny"],
    "ragged_exact": wl.workload("tiny", name="ragged", T=77, H=512, E=40, k=6, I=192, seed=3,
                                act_bits=8),
    "small_latent": wl.workload("tiny", name="small_latent", T=50, H=512, L=256, E=16, k=4,
                                I=128, seed=9, norm_gain_std=0.1),
    "small_adversarial": wl.workload("tiny", name="small_adv", T=60, H=512, E=16, k=4, I=192,
                                     seed=10, act_bits=8, routing="adversarial"),
    "multi_chunk": wl.workload("tiny", name="multi", T=200, H=256, E=4, k=2, I=128, seed=13),
    "one_token": wl.workload("tiny", name="one", T=1, H=256, E=8, k=2, I=128, seed=12),
}


@pytest.mark.parametrize("case", list(CASES))
def test_layer_writes_stay_inside_workspace_and_output(moe, case):
    w = CASES[case]
    capi = moe.capi
    x = wl.gen_x(w, attempts=conditioned_attempts(w)).to(DEV)
    layer = capi.MoeLayer(w.T, w.H, w.E, w.k, w.I, device_weights(w, DEV), L=w.L,
                          act_bits=w.act_bits, renorm=w.renorm, eps=w.eps)
    need = int(capi.lib.moe_workspace_size(ctypes.byref(layer.cfg)))
    ws = torch.full((GUARD + need + GUARD,), PATTERN, dtype=torch.uint8, device=DEV)
    gr = 4  # guard rows above and below the output
    out = torch.empty(gr + w.T + gr, w.H, dtype=torch.bfloat16, device=DEV)
    out.view(torch.uint8).fill_(PATTERN)
    x_before = x.clone()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = capi.lib.moe_layer_forward(ctypes.byref(layer.cfg), ctypes.byref(layer.wstruct),
                                    ctypes.c_void_p(x.data_ptr()),
                                    ctypes.c_void_p(out[gr].data_ptr()),
                                    ctypes.c_void_p(ws.data_ptr() + GUARD), need, stream)
    assert rc == capi.MOE_OK
    assert moe.check_error() == 0
    ws_h = ws.cpu().numpy()
    assert np.all(ws_h[:GUARD] == PATTERN), "write before the workspace"
    assert np.all(ws_h[GUARD + need:] == PATTERN), "write past the end of the workspace"
    out_h = out.view(torch.uint8).cpu().numpy().reshape(-1)
    row = w.H * 2
    assert np.all(out_h[:gr * row] == PATTERN), "write before the output"
    assert np.all(out_h[(gr + w.T) * row:] == PATTERN), "write past the end of the output"
    assert torch.equal(x, x_before), "the input was modified"
    # the guarded call computed the same output as a plain one
    assert torch.equal(out[gr:gr + w.T], layer.forward(x))
