"""The dispatch entry point that allocates nothing (moe_dispatch_noalloc).

Some host programs cannot give this library a workspace: a plugin whose host
owns every device allocation and passes it only its inputs and outputs, or a
runtime that forbids allocating once it serves.  For them the dispatch has a
variant whose scratch is a fixed array in the library's device data.  Its
results must be those of the workspace version, bit for bit, on repeated
calls (the array keeps the previous call's contents).  This file is collected
last so that a run stopping at the first failure has run every other test.
"""
import numpy as np
import pytest
import torch

from tests._helpers import random_topk

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def moe():
    from int4_routed_expert_fp32_gb300.build import build
    build()
    import int4_routed_expert_fp32_gb300 as m
    torch.cuda.set_device(DEV)
    assert m.check_error() == 0
    return m


def _case(T, E, k, D, seed, hot=False):
    rng = np.random.default_rng(seed)
    p = None
    if hot:
        p = np.arange(1, E + 1, dtype=np.float64) ** -1.1
    idx = torch.from_numpy(random_topk(T, E, k, rng, hot=p)).to(DEV)
    x = torch.from_numpy(rng.normal(size=(T, D)).astype(np.float32)).to(torch.bfloat16).to(DEV)
    return idx, x


@pytest.mark.parametrize("act_bits", [16, 8])
def test_noalloc_dispatch_equals_workspace_dispatch_twice(moe, act_bits):
    cases = [(77, 40, 6, 192, 1, False), (8192, 384, 8, 256, 2, True), (5, 16, 3, 64, 3, False)]
    for T, E, k, D, seed, hot in cases:
        idx, x = _case(T, E, k, D, seed, hot)
        ref = moe.dispatch(idx, x, E, act_bits)
        for _ in range(2):   # the second call starts from the first call's scratch contents
            got = moe.dispatch_noalloc(idx, x, E, act_bits)
            assert moe.check_error() == 0
            for name, t in ref.items():
                if t is None:
                    assert got[name] is None
                    continue
                assert torch.equal(got[name], t), (T, E, k, name)


def test_noalloc_rejects_sizes_beyond_its_scratch(moe):
    # ceil(T/32)*E + T*k over 524288 ints: refused on the host, nothing launched
    T, E, k = 40000, 384, 8
    n = None
    rc = moe.lib.moe_dispatch_noalloc(n, n, T, 64, E, k, 16, n, n, n, n, n, n, n, n)
    assert rc == moe.capi.MOE_ERR_INVALID   # null outputs are caught first
    import ctypes
    v = ctypes.c_void_p
    idx = torch.zeros(1, dtype=torch.int32, device=DEV)
    x = torch.zeros(8, 64, dtype=torch.bfloat16, device=DEV)
    i, xp = v(idx.data_ptr()), v(x.data_ptr())
    stream = v(torch.cuda.current_stream().cuda_stream)
    # valid-looking pointers: only the size check can refuse the call
    rc = moe.lib.moe_dispatch_noalloc(i, xp, T, 64, E, k, 16, i, i, i, i, i, xp, None, stream)
    assert rc == moe.capi.MOE_ERR_WORKSPACE
