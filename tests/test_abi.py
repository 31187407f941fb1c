"""The C-ABI library: it builds for sm_103a, loads without a GPU, exports every
symbol that include/moe.h declares, and rejects bad arguments on the host
before any CUDA call (no compute is launched here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def capi():
    from int4_routed_expert_fp32_gb300.build import build
    build()
    from int4_routed_expert_fp32_gb300 import capi as c
    return c


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine",
                     "moe_layer_forward", "moe_workspace_size", "moe_check_error"]:
        assert required in names


def test_every_declared_symbol_is_exported_and_bound(capi):
    for name in declared_functions():
        assert hasattr(capi.lib, name), name
        assert name in capi.SIGNATURES, f"{name} has no ctypes signature"
    assert set(capi.SIGNATURES) == set(declared_functions())


def _header_struct_fields(name):
    """Field names, in order, of ``typedef struct name { ... } name;`` in moe.h."""
    import re
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        text = f.read()
    body = re.search(r"typedef struct %s \{(.*?)\} %s;" % (name, name), text, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    return [re.findall(r"(\w+)\s*$", d.strip())[0] for d in body.split(";") if d.strip()]


def test_struct_layouts_match_header(capi):
    cfg = _header_struct_fields("moe_config")
    wts = _header_struct_fields("moe_weights")
    assert [n for n, _ in capi.MoeConfig._fields_] == cfg
    assert [n for n, _ in capi.MoeWeights._fields_] == wts
    assert ctypes.sizeof(capi.MoeConfig) == len(cfg) * 4            # int32 / float fields
    assert ctypes.sizeof(capi.MoeWeights) == len(wts) * ctypes.sizeof(ctypes.c_void_p)


def test_status_strings(capi):
    assert capi.status_string(0) == "MOE_OK"
    assert capi.status_string(-5) == "MOE_ERR_TIMEOUT"
    assert capi.lib.moe_version().decode().startswith("int4-routed-moe")


def test_workspace_sizes_are_host_only(capi):
    cfg = capi.MoeConfig(32, 7168, 384, 8, 2048, 0, 16, 1, 1e-6)
    n = capi.lib.moe_workspace_size(ctypes.byref(cfg))
    # at least the sorted activations and expert outputs (256 rows x 7168 bf16 each)
    assert n >= 2 * 256 * 7168 * 2
    cfg8 = capi.MoeConfig(32, 7168, 384, 8, 2048, 0, 8, 1, 1e-6)
    assert capi.lib.moe_workspace_size(ctypes.byref(cfg8)) > 0
    assert capi.lib.moe_route_workspace_size(32, 7168, 384) >= 32 * 384 * 4
    assert capi.lib.moe_expert_ffn_workspace_size(384, 7168, 2048, 256, 16) >= 256 * 2048 * 2


def test_argument_errors_return_before_any_launch(capi):
    L = capi.lib
    n = None
    launches = capi.launch_count()
    # null pointers
    assert L.moe_route(n, n, n, 4, 64, 8, 2, 1, n, n, n, 0, n) == capi.MOE_ERR_INVALID
    # unsupported shapes
    assert L.moe_route(n, n, n, 4, 100, 8, 2, 1, n, n, n, 0, n) == capi.MOE_ERR_UNSUPPORTED
    assert L.moe_route(n, n, n, 4, 64, 8, 9, 1, n, n, n, 0, n) == capi.MOE_ERR_UNSUPPORTED
    assert L.moe_dispatch(n, n, 4, 64, 8, 2, 12, n, n, n, n, n, n, n, n, 0, n) == capi.MOE_ERR_UNSUPPORTED
    assert L.moe_expert_ffn(n, n, n, 8, 96, 128, 8, n, n, n, n, n, n, 16, n, n, 0, n) == \
        capi.MOE_ERR_UNSUPPORTED
    assert L.moe_expert_ffn(n, n, n, 8, 128, 128, 8, n, n, n, n, n, n, 16, n, n, 0, n) == \
        capi.MOE_ERR_INVALID
    assert L.moe_combine(n, n, n, 4, 64, 2, n, n) == capi.MOE_ERR_INVALID
    assert L.moe_linear_bf16(n, n, 4, 64, 48, n, n) == capi.MOE_ERR_UNSUPPORTED
    assert L.moe_rmsnorm(n, n, 4, 64, -1.0, n, n) == capi.MOE_ERR_INVALID
    assert L.moe_wait_selftest(10, n) == capi.MOE_ERR_INVALID
    assert L.moe_layer_forward(n, n, n, n, n, 0, n) == capi.MOE_ERR_INVALID
    cfg = capi.MoeConfig(4, 64, 8, 2, 64, 0, 16, 1, 1e-6)
    w = capi.MoeWeights()
    assert L.moe_layer_forward(ctypes.byref(cfg), ctypes.byref(w), n, n, n, 0, n) == capi.MOE_ERR_INVALID
    bad = capi.MoeConfig(4, 64, 8, 2, 64, 0, 4, 1, 1e-6)
    assert L.moe_layer_forward(ctypes.byref(bad), ctypes.byref(w), n, n, n, 0, n) == \
        capi.MOE_ERR_UNSUPPORTED
    # router preparation and the layer pipe
    assert L.moe_router_prepare(n, 8, 64, n, n) == capi.MOE_ERR_INVALID
    assert L.moe_router_prepare(n, 0, 64, n, n) == capi.MOE_ERR_INVALID
    pipe = ctypes.c_void_p(1)
    assert L.moe_layer_pipe_create(ctypes.byref(cfg), ctypes.byref(w), n, 0, n,
                                   ctypes.byref(pipe)) == capi.MOE_ERR_INVALID
    assert pipe.value is None  # NULL on every error
    assert L.moe_layer_pipe_create(ctypes.byref(bad), ctypes.byref(w), n, 0, n,
                                   ctypes.byref(pipe)) == capi.MOE_ERR_UNSUPPORTED
    assert L.moe_layer_pipe_submit(n, n, n, n) == capi.MOE_ERR_INVALID
    assert L.moe_layer_pipe_join(n, n) == capi.MOE_ERR_INVALID
    L.moe_layer_pipe_destroy(n)  # NULL is ignored
    assert L.moe_expert_ffn_pairs_bounded(n, n, n, 8, 128, 128, 8, -1, n, n, n, n, n, n, 16, n, n,
                                          0, n) == capi.MOE_ERR_INVALID
    assert L.moe_layer_pipe_workspace_size(ctypes.byref(cfg)) == \
        L.moe_workspace_size(ctypes.byref(cfg)) + 4 * 512  # two slots of x and out, 4 x 64 bf16
    assert capi.launch_count() == launches


def test_workspace_too_small_is_reported(capi):
    # non-null but fake pointers: the size check comes before any use
    fake = ctypes.c_void_p(0x10000)
    rc = capi.lib.moe_route(fake, fake, fake, 4, 64, 8, 2, 1, fake, fake, fake, 16, None)
    assert rc == capi.MOE_ERR_WORKSPACE


def test_last_cuda_error_is_named_per_thread(capi):
    import threading
    import torch
    if torch.cuda.is_available():
        pytest.skip("needs a host without a usable CUDA device")
    # without a device the runtime refuses the synchronisation: MOE_ERR_CUDA,
    # and the runtime error behind it is named for this thread only
    assert capi.lib.moe_check_error(None) == capi.MOE_ERR_CUDA
    name = capi.last_cuda_error()
    assert name.startswith("cudaError") and name != "cudaSuccess"
    assert name in str(capi.MoeError("moe_check_error", capi.MOE_ERR_CUDA))
    seen = []
    t = threading.Thread(target=lambda: seen.append(capi.last_cuda_error()))
    t.start()
    t.join()
    assert seen == ["cudaSuccess"]


def test_missing_library_fails_loudly(tmp_path):
    """A copy of the package without libmoe.so imports, but its first use of
    any binding name raises ImportError: there is no CPU fallback."""
    import shutil
    import subprocess
    import sys
    src = os.path.join(ROOT, "int4_routed_expert_fp32_gb300")
    dst = tmp_path / "int4_routed_expert_fp32_gb300"
    dst.mkdir()
    for name in os.listdir(src):
        if name.endswith(".py"):
            shutil.copy(os.path.join(src, name), dst / name)
    code = (
        "import int4_routed_expert_fp32_gb300 as m\n"
        "for name in ('MoeLayer', 'route', 'expert_ffn', 'lib'):\n"
        "    try:\n"
        "        getattr(m, name)\n"
        "    except ImportError as e:\n"
        "        assert 'libmoe.so is missing' in str(e), e\n"
        "    else:\n"
        "        raise SystemExit(name + ' did not fail')\n"
        "print('ok')\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=tmp_path, capture_output=True, text=True,
                       env={**os.environ, "PYTHONPATH": str(tmp_path)}, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


def test_header_is_plain_c_and_links(capi, tmp_path):
    """include/moe.h compiles as strict C99 and a C program links against
    libmoe.so and calls it: the entry points that need no GPU answer, and
    argument errors come back before any CUDA call."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_moe.c"
    src.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "moe.h"

int main(void) {
  moe_config cfg;
  moe_weights w;
  memset(&cfg, 0, sizeof cfg);
  memset(&w, 0, sizeof w);
  cfg.T = 4; cfg.H = 64; cfg.E = 8; cfg.k = 2; cfg.I = 64; cfg.act_bits = 16; cfg.renorm = 1;
  if (moe_workspace_size(&cfg) == 0) return 1;
  if (moe_layer_forward(&cfg, &w, NULL, NULL, NULL, 0, NULL) != MOE_ERR_INVALID) return 2;
  if (moe_route(NULL, NULL, NULL, 4, 64, 8, 2, 1, NULL, NULL, NULL, 0, NULL) != MOE_ERR_INVALID)
    return 3;
  if (strcmp(moe_status_string(MOE_ERR_TIMEOUT), "MOE_ERR_TIMEOUT") != 0) return 4;
  printf("%s\n", moe_version());
  return 0;
}
''')
    from int4_routed_expert_fp32_gb300.build import LIB_PATH
    libdir = os.path.dirname(LIB_PATH)
    exe = tmp_path / "use_moe"
    r = subprocess.run([cc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror",
                        "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                        "-L", libdir, "-l:libmoe.so", "-Wl,-rpath," + libdir],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, (run.returncode, run.stderr)
    assert run.stdout.startswith("int4-routed-moe")
