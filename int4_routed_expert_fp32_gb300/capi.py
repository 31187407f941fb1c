"""ctypes binding of ``libmoe.so`` (declared in ``include/moe.h``).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Output tensors and workspaces are allocated with torch (device
memory) and passed as raw pointers; calls are enqueued on torch's current CUDA
stream.  Importing this module fails loudly when the library is missing -- there
is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int, c_int32, c_int64, c_size_t, c_void_p
from typing import Dict, Optional

import torch

from .build import LIB_PATH

MOE_OK = 0
MOE_ERR_INVALID = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_WORKSPACE = -3
MOE_ERR_CUDA = -4
MOE_ERR_TIMEOUT = -5


class MoeError(RuntimeError):
    def __init__(self, name: str, code: int):
        what = status_string(code)
        if code == MOE_ERR_CUDA:
            what += f": {last_cuda_error()}"
        super().__init__(f"{name} returned {code} ({what})")
        self.code = code


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", c_int32), ("H", c_int32), ("E", c_int32), ("k", c_int32), ("I", c_int32),
                ("L", c_int32), ("act_bits", c_int32), ("renorm", c_int32), ("eps", c_float),
                ("I_shared", c_int32)]


class MoeWeights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in (
        "router_w", "router_bias", "gate_packed", "gate_scale", "up_packed", "up_scale",
        "down_packed", "down_scale", "lat_down", "lat_norm", "lat_up", "shared_gate", "shared_up",
        "shared_down", "router_w_terms")]


# name -> (restype, argtypes); mirrors include/moe.h
SIGNATURES = {
    "moe_route_workspace_size": (c_size_t, [c_int, c_int, c_int]),
    "moe_route": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                          c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_dispatch_workspace_size": (c_size_t, [c_int, c_int, c_int]),
    "moe_dispatch": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_void_p,
                             c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                             c_size_t, c_void_p]),
    "moe_dispatch_pairs": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                                   c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                   c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_dispatch_noalloc": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                                     c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_void_p, c_void_p]),
    "moe_expert_ffn_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "moe_expert_ffn": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                               c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int,
                               c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_expert_ffn_pairs_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "moe_expert_ffn_pairs": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                     c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_int, c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_int4_linear_workspace_size": (c_size_t, [c_int, c_int, c_int]),
    "moe_int4_linear": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_int4_linear_partials_workspace_size": (c_size_t, [c_int, c_int, c_int]),
    "moe_int4_linear_partials": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                         c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_void_p,
                                         c_size_t, c_void_p]),
    "moe_int4_linear_stall_selftest": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int,
                                               c_int, c_void_p, c_void_p, c_int, c_int, c_int,
                                               c_int64, c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_quantize_rows": (c_int, [c_void_p, c_int, c_int, c_void_p, c_void_p, c_void_p]),
    "moe_quantize_int4": (c_int, [c_void_p, c_int, c_int, c_void_p, c_void_p, c_void_p]),
    "moe_quantize_int8": (c_int, [c_void_p, c_int, c_int, c_void_p, c_void_p, c_void_p]),
    "moe_quantize_rows_int16": (c_int, [c_void_p, c_int, c_int, c_void_p, c_void_p, c_void_p]),
    "moe_int4_linear_int16_workspace_size": (c_size_t, [c_int, c_int, c_int]),
    "moe_int4_linear_int16": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_void_p,
                                      c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                      c_void_p]),
    "moe_shared_expert_workspace_size": (c_size_t, [c_int, c_int, c_int]),
    "moe_shared_expert": (c_int, [c_void_p, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p,
                                  c_int, c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_combine": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p]),
    "moe_linear_bf16": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p]),
    "moe_rmsnorm": (c_int, [c_void_p, c_void_p, c_int, c_int, c_float, c_void_p, c_void_p]),
    "moe_workspace_size": (c_size_t, [POINTER(MoeConfig)]),
    "moe_layer_forward": (c_int, [POINTER(MoeConfig), POINTER(MoeWeights), c_void_p, c_void_p,
                                  c_void_p, c_size_t, c_void_p]),
    "moe_layer_graph_create": (c_int, [POINTER(MoeConfig), POINTER(MoeWeights), c_void_p, c_void_p,
                                       c_int, c_void_p, c_size_t, c_void_p,
                                       POINTER(c_void_p)]),
    "moe_layer_graph_launch": (c_int, [c_void_p, c_void_p]),
    "moe_layer_graph_destroy": (None, [c_void_p]),
    "moe_layer_pipe_workspace_size": (c_size_t, [POINTER(MoeConfig)]),
    "moe_layer_pipe_create": (c_int, [POINTER(MoeConfig), POINTER(MoeWeights), c_void_p, c_size_t,
                                      c_void_p, POINTER(c_void_p)]),
    "moe_layer_pipe_submit": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p]),
    "moe_layer_pipe_join": (c_int, [c_void_p, c_void_p]),
    "moe_layer_pipe_destroy": (None, [c_void_p]),
    "moe_layer_forward_host": (c_int, [POINTER(MoeConfig), POINTER(MoeWeights), c_void_p, c_void_p,
                                       c_void_p, c_size_t, c_void_p]),
    "moe_check_error": (c_int, [c_void_p]),
    "moe_wait_selftest": (c_int, [c_int64, c_void_p]),
    "moe_status_string": (ctypes.c_char_p, [c_int]),
    "moe_last_cuda_error": (ctypes.c_char_p, []),
    "moe_version": (ctypes.c_char_p, []),
    "moe_launch_count": (ctypes.c_uint64, []),
    "moe_set_tc_pair": (c_int, [c_int]),
    "moe_router_prepare": (c_int, [c_void_p, c_int, c_int, c_void_p, c_void_p]),
    "moe_expert_ffn_pairs_bounded": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int,
                                             c_int, c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                                             c_void_p, c_void_p, c_int, c_void_p, c_void_p,
                                             c_size_t, c_void_p]),
}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                          "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def status_string(code: int) -> str:
    return lib.moe_status_string(code).decode()


def last_cuda_error() -> str:
    """Name of the CUDA runtime error behind this thread's last MOE_ERR_CUDA."""
    return lib.moe_last_cuda_error().decode()


def launch_count() -> int:
    """Kernels the library has launched in this process so far."""
    return int(lib.moe_launch_count())


def set_tc_pair(enable: bool) -> bool:
    """Run the act_bits 16 tensor-core GEMMs on CTA pairs (True, the default)
    or on the one-CTA kernels (False); returns the previous setting."""
    return bool(lib.moe_set_tc_pair(1 if enable else 0))


def _check(name: str, rc: int) -> None:
    if rc != MOE_OK:
        raise MoeError(name, rc)


def _p(t: Optional[torch.Tensor]):
    return None if t is None else c_void_p(t.data_ptr())


def _stream():
    return c_void_p(torch.cuda.current_stream().cuda_stream)


def _ws(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _arg(name: str, t: Optional[torch.Tensor], shape=None, dtype=None) -> torch.Tensor:
    """Check one tensor argument against the layout its C entry point reads
    (``include/moe.h``) before its pointer is passed on: the library trusts
    the sizes it is given, so a short or strided buffer would be read or
    written out of bounds.  ``shape`` entries of None match any size.  Only
    metadata is checked here; ``_placed`` checks where the tensors live."""
    if t is None:
        raise ValueError(f"{name} is required")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    if shape is not None and (t.dim() != len(shape) or any(
            want is not None and int(got) != int(want) for got, want in zip(t.shape, shape))):
        want = tuple("*" if w is None else int(w) for w in shape)
        raise ValueError(f"{name}: expected shape {want}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _placed(**tensors: Optional[torch.Tensor]) -> torch.device:
    """Every given tensor (None skipped) lives on the current CUDA device, the
    one whose stream the call is enqueued on; returns that device."""
    dev = None
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must live on a CUDA device")
        if dev is None:
            dev = torch.device("cuda", torch.cuda.current_device())
        if t.device != dev:
            raise ValueError(f"{name} is on {t.device}; the call runs on {dev}")
    return dev


EXPERT_NAMES = ("gate_packed", "gate_scale", "up_packed", "up_scale", "down_packed", "down_scale")


def _experts(experts: Dict[str, torch.Tensor], E: int, D: int, I: int) -> None:
    """Gate/up [E, I, D/8] + [E, I, D/32]; down [E, D, I/8] + [E, D, I/32]."""
    for proj, (N, K) in (("gate", (I, D)), ("up", (I, D)), ("down", (D, I))):
        _arg(f"{proj}_packed", experts.get(f"{proj}_packed"), (E, N, K // 8), torch.int32)
        _arg(f"{proj}_scale", experts.get(f"{proj}_scale"), (E, N, K // 32), torch.bfloat16)


# ------------------------------------------------------------------ stages

def route(x: torch.Tensor, w_router: torch.Tensor, bias: torch.Tensor, k: int, renorm: bool = True):
    """topk_idx int32 [T, k], topk_w fp32 [T, k] for bf16 x [T, H]."""
    T, H = _arg("x", x, (None, None), torch.bfloat16).shape
    E = _arg("w_router", w_router, (None, H), torch.float32).shape[0]
    _arg("bias", bias, (E,), torch.float32)
    dev = _placed(x=x, w_router=w_router, bias=bias)
    idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    ws = _ws(lib.moe_route_workspace_size(T, H, E), dev)
    _check("moe_route", lib.moe_route(_p(x), _p(w_router), _p(bias), T, H, E, k, int(renorm),
                                      _p(idx), _p(w), _p(ws), ws.numel(), _stream()))
    return idx, w


def _dispatch_out(T: int, k: int, D: int, E: int, act_bits: int, pairs: bool, dev):
    R = T * k
    xdt = torch.int8 if act_bits == 8 else (torch.float16 if pairs else torch.bfloat16)
    return {
        "counts": torch.empty(E, dtype=torch.int32, device=dev),
        "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
        "row_token": torch.empty(R, dtype=torch.int32, device=dev),
        "row_slot": torch.empty(R, dtype=torch.int32, device=dev),
        "inv_row": torch.empty(R, dtype=torch.int32, device=dev),
        "x_sorted": torch.empty(R, D, dtype=xdt, device=dev),
        "x_scale": torch.empty(R, dtype=torch.float32, device=dev) if act_bits == 8 else None,
    }


def _dispatch_args(topk_idx: torch.Tensor, x: torch.Tensor):
    """T, k, D and the device of topk_idx int32 [T, k] and x bf16 [T, D]."""
    T, k = _arg("topk_idx", topk_idx, (None, None), torch.int32).shape
    D = _arg("x", x, (T, None), torch.bfloat16).shape[1]
    return T, k, D, _placed(topk_idx=topk_idx, x=x)


def dispatch(topk_idx: torch.Tensor, x: torch.Tensor, E: int, act_bits: int = 16,
             pairs: bool = False) -> Dict[str, torch.Tensor]:
    """Counts, offsets, the stable expert-major permutation and the gathered
    rows (pairs=True: moe_dispatch_pairs, rows in the expert kernels' pair
    order, fp16 or int8)."""
    T, k, D, dev = _dispatch_args(topk_idx, x)
    out = _dispatch_out(T, k, D, E, act_bits, pairs, dev)
    ws = _ws(lib.moe_dispatch_workspace_size(T, E, k), dev)
    name = "moe_dispatch_pairs" if pairs else "moe_dispatch"
    _check(name, getattr(lib, name)(
        _p(topk_idx), _p(x), T, D, E, k, act_bits, _p(out["counts"]), _p(out["offsets"]),
        _p(out["row_token"]), _p(out["row_slot"]), _p(out["inv_row"]), _p(out["x_sorted"]),
        _p(out["x_scale"]), _p(ws), ws.numel(), _stream()))
    return out


def dispatch_noalloc(topk_idx: torch.Tensor, x: torch.Tensor, E: int,
                     act_bits: int = 16) -> Dict[str, torch.Tensor]:
    """moe_dispatch without a workspace: the library's fixed device scratch is
    used instead (for callers that cannot allocate device memory; calls must
    not overlap on the GPU)."""
    T, k, D, dev = _dispatch_args(topk_idx, x)
    out = _dispatch_out(T, k, D, E, act_bits, False, dev)
    _check("moe_dispatch_noalloc", lib.moe_dispatch_noalloc(
        _p(topk_idx), _p(x), T, D, E, k, act_bits, _p(out["counts"]), _p(out["offsets"]),
        _p(out["row_token"]), _p(out["row_slot"]), _p(out["inv_row"]), _p(out["x_sorted"]),
        _p(out["x_scale"]), _stream()))
    return out


def _rows_args(x: torch.Tensor, x_scale: Optional[torch.Tensor], offsets: torch.Tensor,
               act_bits: int, dtype16, E: int) -> Optional[torch.Tensor]:
    """Expert-sorted rows x (int8 with act_bits 8, else ``dtype16``), their
    fp32 scales (act_bits 8 only; returned, None otherwise) and the E + 1
    segment offsets."""
    rows = _arg("x", x, (None, None), torch.int8 if act_bits == 8 else dtype16).shape[0]
    _arg("offsets", offsets, (E + 1,), torch.int32)
    if act_bits != 8:
        return None
    return _arg("x_scale", x_scale, (rows,), torch.float32)


def expert_ffn(x_sorted: torch.Tensor, x_scale: Optional[torch.Tensor], offsets: torch.Tensor,
               experts: Dict[str, torch.Tensor], act_bits: int = 16,
               pairs: bool = False, max_rows_per_expert: Optional[int] = None) -> torch.Tensor:
    """y_sorted bf16 [rows, D] = down(SiLU(gate(x)) * up(x)) per expert segment
    (pairs=True: moe_expert_ffn_pairs on rows from dispatch(..., pairs=True);
    with max_rows_per_expert, moe_expert_ffn_pairs_bounded)."""
    E, I = _arg("gate_packed", experts.get("gate_packed"), (None, None, None), torch.int32).shape[:2]
    x_scale = _rows_args(x_sorted, x_scale, offsets, act_bits,
                         torch.float16 if pairs else torch.bfloat16, E)
    rows, D = x_sorted.shape
    _experts(experts, E, D, I)
    dev = _placed(x_sorted=x_sorted, x_scale=x_scale, offsets=offsets,
                  **{n: experts[n] for n in EXPERT_NAMES})
    y = torch.empty(rows, D, dtype=torch.bfloat16, device=dev)
    name = "moe_expert_ffn_pairs" if pairs else "moe_expert_ffn"
    ws = _ws(getattr(lib, name + "_workspace_size")(E, D, I, rows, act_bits), dev)
    wargs = (_p(experts["gate_packed"]), _p(experts["gate_scale"]), _p(experts["up_packed"]),
             _p(experts["up_scale"]), _p(experts["down_packed"]), _p(experts["down_scale"]),
             act_bits, _p(y), _p(ws), ws.numel(), _stream())
    if max_rows_per_expert is not None:
        if not pairs:
            raise ValueError("max_rows_per_expert needs pairs=True")
        _check("moe_expert_ffn_pairs_bounded", lib.moe_expert_ffn_pairs_bounded(
            _p(x_sorted), _p(x_scale), _p(offsets), E, D, I, rows, int(max_rows_per_expert),
            *wargs))
        return y
    _check(name, getattr(lib, name)(_p(x_sorted), _p(x_scale), _p(offsets), E, D, I, rows, *wargs))
    return y


def int4_linear(x: torch.Tensor, x_scale: Optional[torch.Tensor], offsets: torch.Tensor,
                w_packed: torch.Tensor, w_scale: torch.Tensor, act_bits: int = 16) -> torch.Tensor:
    """fp32 [rows, N] = x W_e^T per expert segment (one grouped PackedInt4Linear)."""
    E, N = _arg("w_packed", w_packed, (None, None, None), torch.int32).shape[:2]
    x_scale = _rows_args(x, x_scale, offsets, act_bits, torch.bfloat16, E)
    rows, K = x.shape
    _arg("w_packed", w_packed, (E, N, K // 8), torch.int32)
    _arg("w_scale", w_scale, (E, N, K // 32), torch.bfloat16)
    dev = _placed(x=x, x_scale=x_scale, offsets=offsets, w_packed=w_packed, w_scale=w_scale)
    out = torch.empty(rows, N, dtype=torch.float32, device=dev)
    ws = _ws(lib.moe_int4_linear_workspace_size(E, K, rows), dev)
    _check("moe_int4_linear", lib.moe_int4_linear(
        _p(x), _p(x_scale), _p(offsets), E, K, N, rows, _p(w_packed), _p(w_scale), act_bits,
        _p(out), _p(ws), ws.numel(), _stream()))
    return out


def int4_linear_partials(x: torch.Tensor, x_scale: torch.Tensor, offsets: torch.Tensor,
                         w_packed: torch.Tensor, w_scale: torch.Tensor, kernel: int):
    """Exact-mode grouped int4 linear on one chosen kernel (0: stream,
    1: tensor cores), for tests: (out fp32 [rows, N], partials int32
    [rows, N, K/32], the integer partial of every 32-column weight group)."""
    E, N = _arg("w_packed", w_packed, (None, None, None), torch.int32).shape[:2]
    x_scale = _rows_args(x, x_scale, offsets, 8, torch.bfloat16, E)
    rows, K = x.shape
    _arg("w_packed", w_packed, (E, N, K // 8), torch.int32)
    _arg("w_scale", w_scale, (E, N, K // 32), torch.bfloat16)
    dev = _placed(x=x, x_scale=x_scale, offsets=offsets, w_packed=w_packed, w_scale=w_scale)
    out = torch.empty(rows, N, dtype=torch.float32, device=dev)
    partials = torch.empty(rows, N, K // 32, dtype=torch.int32, device=dev)
    ws = _ws(lib.moe_int4_linear_partials_workspace_size(E, K, rows), dev)
    _check("moe_int4_linear_partials", lib.moe_int4_linear_partials(
        _p(x), _p(x_scale), _p(offsets), E, K, N, rows, _p(w_packed), _p(w_scale), kernel,
        _p(out), _p(partials), _p(ws), ws.numel(), _stream()))
    return out, partials


def int4_linear_stall_selftest(x: torch.Tensor, x_scale: Optional[torch.Tensor],
                               offsets: torch.Tensor, w_packed: torch.Tensor, w_scale: torch.Tensor,
                               act_bits: int, kernel: int, stall_stage: int, limit_ns: int) -> None:
    """Run int4_linear on a kernel build whose producer stops before stage
    ``stall_stage`` (tests of the exit paths; the device records
    MOE_ERR_TIMEOUT, read with check_error())."""
    E, N = _arg("w_packed", w_packed, (None, None, None), torch.int32).shape[:2]
    x_scale = _rows_args(x, x_scale, offsets, act_bits, torch.bfloat16, E)
    rows, K = x.shape
    _arg("w_packed", w_packed, (E, N, K // 8), torch.int32)
    _arg("w_scale", w_scale, (E, N, K // 32), torch.bfloat16)
    dev = _placed(x=x, x_scale=x_scale, offsets=offsets, w_packed=w_packed, w_scale=w_scale)
    out = torch.empty(rows, N, dtype=torch.float32, device=dev)
    ws = _ws(lib.moe_int4_linear_workspace_size(E, K, rows), dev)
    _check("moe_int4_linear_stall_selftest", lib.moe_int4_linear_stall_selftest(
        _p(x), _p(x_scale), _p(offsets), E, K, N, rows, _p(w_packed), _p(w_scale), act_bits,
        kernel, stall_stage, limit_ns, _p(out), _p(ws), ws.numel(), _stream()))


def quantize_rows(v: torch.Tensor):
    """Per-row int8 quantisation: (q int8 [R, C], scale fp32 [R])."""
    R, C = _arg("v", v, (None, None), torch.bfloat16).shape
    dev = _placed(v=v)
    q = torch.empty(R, C, dtype=torch.int8, device=dev)
    s = torch.empty(R, dtype=torch.float32, device=dev)
    _check("moe_quantize_rows", lib.moe_quantize_rows(_p(v), R, C, _p(q), _p(s), _stream()))
    return q, s


def quantize_int4(w: torch.Tensor):
    """bf16 weight [..., N, K] -> (packed int32 [..., N, K/8], bf16 scale [..., N, K/32])."""
    if _arg("w", w, None, torch.bfloat16).dim() < 1:
        raise ValueError("w: expected at least one dimension")
    dev = _placed(w=w)
    K = w.shape[-1]
    rows = w.numel() // K if K else 0
    packed = torch.empty(*w.shape[:-1], K // 8, dtype=torch.int32, device=dev)
    scale = torch.empty(*w.shape[:-1], K // 32, dtype=torch.bfloat16, device=dev)
    _check("moe_quantize_int4", lib.moe_quantize_int4(_p(w), rows, K, _p(packed), _p(scale),
                                                      _stream()))
    return packed, scale


def quantize_int8(w: torch.Tensor):
    """bf16 weight [..., N, K] -> (int8 codes [..., N, K], bf16 scale [..., N, K/32])."""
    if _arg("w", w, None, torch.bfloat16).dim() < 1:
        raise ValueError("w: expected at least one dimension")
    dev = _placed(w=w)
    K = w.shape[-1]
    rows = w.numel() // K if K else 0
    q = torch.empty(*w.shape, dtype=torch.int8, device=dev)
    scale = torch.empty(*w.shape[:-1], K // 32, dtype=torch.bfloat16, device=dev)
    _check("moe_quantize_int8", lib.moe_quantize_int8(_p(w), rows, K, _p(q), _p(scale),
                                                      _stream()))
    return q, scale


def quantize_rows_int16(v: torch.Tensor):
    """Per-row symmetric int16 codes of bf16 v [R, C]: (int16 [R, C], fp32 scale [R])."""
    R, C = _arg("v", v, (None, None), torch.bfloat16).shape
    dev = _placed(v=v)
    q = torch.empty(R, C, dtype=torch.int16, device=dev)
    scale = torch.empty(R, dtype=torch.float32, device=dev)
    _check("moe_quantize_rows_int16", lib.moe_quantize_rows_int16(_p(v), R, C, _p(q), _p(scale),
                                                                  _stream()))
    return q, scale


def int4_linear_int16(x: torch.Tensor, offsets: torch.Tensor, w_packed: torch.Tensor,
                      w_scale: torch.Tensor, partials: bool = False):
    """fp32 [rows, N] = x W_e^T per expert segment under the int16/int64
    reading of act_bits 16 (per-row int16 codes, exact group partials); with
    partials=True also the int32 partials [rows, N, K/32]."""
    E, N = _arg("w_packed", w_packed, (None, None, None), torch.int32).shape[:2]
    rows, K = _arg("x", x, (None, None), torch.bfloat16).shape
    _arg("offsets", offsets, (E + 1,), torch.int32)
    _arg("w_packed", w_packed, (E, N, K // 8), torch.int32)
    _arg("w_scale", w_scale, (E, N, K // 32), torch.bfloat16)
    dev = _placed(x=x, offsets=offsets, w_packed=w_packed, w_scale=w_scale)
    out = torch.empty(rows, N, dtype=torch.float32, device=dev)
    part = torch.empty(rows, N, K // 32, dtype=torch.int32, device=dev) if partials else None
    ws = _ws(lib.moe_int4_linear_int16_workspace_size(E, K, rows), dev)
    _check("moe_int4_linear_int16", lib.moe_int4_linear_int16(
        _p(x), _p(offsets), E, K, N, rows, _p(w_packed), _p(w_scale), _p(out), _p(part),
        _p(ws), ws.numel(), _stream()))
    return (out, part) if partials else out


def shared_expert(x: torch.Tensor, gate_w: torch.Tensor, up_w: torch.Tensor,
                  down_w: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """out (+)= down(SiLU(gate x) * up x) with bf16 weights; a new output when
    ``out`` is None, else added to it in place."""
    T, H = _arg("x", x, (None, None), torch.bfloat16).shape
    I = _arg("gate_w", gate_w, (None, H), torch.bfloat16).shape[0]
    _arg("up_w", up_w, (I, H), torch.bfloat16)
    _arg("down_w", down_w, (H, I), torch.bfloat16)
    acc = out is not None
    if acc:
        _arg("out", out, (T, H), torch.bfloat16)
    dev = _placed(x=x, gate_w=gate_w, up_w=up_w, down_w=down_w, out=out)
    if not acc:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    ws = _ws(lib.moe_shared_expert_workspace_size(T, H, I), dev)
    _check("moe_shared_expert", lib.moe_shared_expert(
        _p(x), T, H, I, _p(gate_w), _p(up_w), _p(down_w), int(acc), _p(out), _p(ws), ws.numel(),
        _stream()))
    return out


def combine(y_sorted: torch.Tensor, inv_row: torch.Tensor, topk_w: torch.Tensor) -> torch.Tensor:
    """out bf16 [T, D] = sum over the k slots of topk_w * y_sorted[inv_row]."""
    T, k = _arg("topk_w", topk_w, (None, None), torch.float32).shape
    D = _arg("y_sorted", y_sorted, (T * k, None), torch.bfloat16).shape[1]
    if _arg("inv_row", inv_row, None, torch.int32).numel() != T * k:
        raise ValueError(f"inv_row: expected {T * k} entries, got {inv_row.numel()}")
    dev = _placed(y_sorted=y_sorted, inv_row=inv_row, topk_w=topk_w)
    out = torch.empty(T, D, dtype=torch.bfloat16, device=dev)
    _check("moe_combine", lib.moe_combine(_p(y_sorted), _p(inv_row), _p(topk_w), T, D, k, _p(out),
                                          _stream()))
    return out


def linear_bf16(x: torch.Tensor, w: torch.Tensor) -> torch.Tensor:
    """y bf16 [M, N] = x [M, K] w^T, w bf16 [N, K]."""
    M, K = _arg("x", x, (None, None), torch.bfloat16).shape
    N = _arg("w", w, (None, K), torch.bfloat16).shape[0]
    dev = _placed(x=x, w=w)
    y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    _check("moe_linear_bf16", lib.moe_linear_bf16(_p(x), _p(w), M, N, K, _p(y), _stream()))
    return y


def rmsnorm(x: torch.Tensor, gain: torch.Tensor, eps: float) -> torch.Tensor:
    """Row-wise RMSNorm of bf16 x [M, N] with bf16 gain [N]."""
    M, N = _arg("x", x, (None, None), torch.bfloat16).shape
    _arg("gain", gain, (N,), torch.bfloat16)
    _placed(x=x, gain=gain)
    y = torch.empty_like(x)
    _check("moe_rmsnorm", lib.moe_rmsnorm(_p(x), _p(gain), M, N, float(eps), _p(y), _stream()))
    return y


def check_error() -> int:
    """Synchronise the current stream and return (and clear) the device status word."""
    return lib.moe_check_error(_stream())


def wait_selftest(limit_ns: int) -> None:
    _check("moe_wait_selftest", lib.moe_wait_selftest(int(limit_ns), _stream()))


def router_prepare(w_router: torch.Tensor) -> torch.Tensor:
    """The three bf16 terms [3, E, H] of the fp32 router weight (their sum is
    w_router exactly), for MoeLayer's tensor-core router."""
    E, H = _arg("w_router", w_router, (None, None), torch.float32).shape
    dev = _placed(w_router=w_router)
    terms = torch.empty(3, E, H, dtype=torch.bfloat16, device=dev)
    _check("moe_router_prepare", lib.moe_router_prepare(_p(w_router), E, H, _p(terms), _stream()))
    return terms


# ------------------------------------------------------------------ layer

class MoeLayer:
    """One routed int4 MoE layer: configuration, device weights and a workspace."""

    def __init__(self, T: int, H: int, E: int, k: int, I: int, weights: Dict[str, torch.Tensor],
                 L: int = 0, act_bits: int = 16, renorm: bool = True, eps: float = 1e-6,
                 I_shared: int = 0, prepare_router: bool = True):
        """prepare_router: from T = 512 on, split the router weight into its
        bf16 terms once here (moe_router_prepare) rather than on every call."""
        self.cfg = MoeConfig(T, H, E, k, I, L, act_bits, int(renorm), eps, I_shared)
        _check_layer_weights(weights, H, E, I, L, I_shared)
        self.device = _placed(**{n: t for n, t in weights.items() if t is not None})
        weights = dict(weights)
        if prepare_router and T >= 512 and weights.get("router_w_terms") is None:
            weights["router_w_terms"] = router_prepare(weights["router_w"])
        self.weights = weights
        self.wstruct = MoeWeights(*[_p(weights.get(n)) for n, _ in MoeWeights._fields_])
        self.ws = _ws(lib.moe_workspace_size(ctypes.byref(self.cfg)), self.device)

    def forward(self, x: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
        shape = (self.cfg.T, self.cfg.H)
        _arg("x", x, shape, torch.bfloat16)
        if out is not None:
            _arg("out", out, shape, torch.bfloat16)
        dev = _placed(x=x, out=out)
        if dev != self.device:
            raise ValueError(f"x is on {dev}; the layer's weights are on {self.device}")
        if out is None:
            out = torch.empty_like(x)
        _check("moe_layer_forward", lib.moe_layer_forward(
            ctypes.byref(self.cfg), ctypes.byref(self.wstruct), _p(x), _p(out), _p(self.ws),
            self.ws.numel(), _stream()))
        return out

    def forward_host(self, x_host: torch.Tensor, out_host: torch.Tensor) -> None:
        """x_host / out_host: CPU bf16 [T, H] (pinned for asynchronous copies)."""
        shape = (self.cfg.T, self.cfg.H)
        for name, t in (("x_host", x_host), ("out_host", out_host)):
            if _arg(name, t, shape, torch.bfloat16).is_cuda:
                raise ValueError(f"{name} must be a host tensor")
        _check("moe_layer_forward_host", lib.moe_layer_forward_host(
            ctypes.byref(self.cfg), ctypes.byref(self.wstruct), _p(x_host), _p(out_host),
            _p(self.ws), self.ws.numel(), _stream()))

    def graph(self, x: torch.Tensor, out: torch.Tensor, host: bool = False) -> "LayerGraph":
        """The forward call (forward_host with host=True: pinned CPU buffers)
        on exactly these buffers, captured once as a CUDA graph (on a side
        stream: the legacy default stream cannot capture); LayerGraph.launch()
        replays it on the current stream."""
        shape = (self.cfg.T, self.cfg.H)
        _arg("x", x, shape, torch.bfloat16)
        _arg("out", out, shape, torch.bfloat16)
        if host:
            for name, t in (("x", x), ("out", out)):
                if t.is_cuda or not t.is_pinned():
                    raise ValueError(f"{name} must be a pinned host tensor")
        elif _placed(x=x, out=out) != self.device:
            raise ValueError("x and out must be on the layer's device")
        handle = c_void_p()
        cur = torch.cuda.current_stream(self.device)
        side = torch.cuda.Stream(self.device)
        side.wait_stream(cur)
        with torch.cuda.stream(side):
            rc = lib.moe_layer_graph_create(
                ctypes.byref(self.cfg), ctypes.byref(self.wstruct), _p(x), _p(out), int(host),
                _p(self.ws), self.ws.numel(), _stream(), ctypes.byref(handle))
        cur.wait_stream(side)
        _check("moe_layer_graph_create", rc)
        return LayerGraph(handle, (self, x, out))

    def pipe(self) -> "LayerPipe":
        """Pipelined calls on pinned host buffers (see LayerPipe); the pipe has
        its own workspace, so it can run beside this layer's other calls."""
        ws = _ws(lib.moe_layer_pipe_workspace_size(ctypes.byref(self.cfg)), self.device)
        handle = c_void_p()
        cur = torch.cuda.current_stream(self.device)
        side = torch.cuda.Stream(self.device)
        side.wait_stream(cur)
        with torch.cuda.stream(side):
            rc = lib.moe_layer_pipe_create(ctypes.byref(self.cfg), ctypes.byref(self.wstruct),
                                           _p(ws), ws.numel(), _stream(), ctypes.byref(handle))
        cur.wait_stream(side)
        _check("moe_layer_pipe_create", rc)
        return LayerPipe(handle, (self, ws), (self.cfg.T, self.cfg.H))


class LayerPipe:
    """Pipelined layer calls on pinned host buffers (moe_layer_pipe_*): the
    copies of one call overlap the compute of its neighbours.  Submit every
    call from the same current stream; join() makes it wait for the output
    copies of the calls submitted so far."""

    def __init__(self, handle: c_void_p, keep, shape):
        self._h = handle
        self._keep = keep
        self._shape = shape
        self._pending = []  # host buffers of calls not yet joined

    def submit(self, x_host: torch.Tensor, out_host: torch.Tensor) -> None:
        if not self._h:
            raise ValueError("the pipe was closed")
        for name, t in (("x_host", x_host), ("out_host", out_host)):
            _arg(name, t, self._shape, torch.bfloat16)
            if t.is_cuda or not t.is_pinned():
                raise ValueError(f"{name} must be a pinned host tensor")
        _check("moe_layer_pipe_submit",
               lib.moe_layer_pipe_submit(self._h, _p(x_host), _p(out_host), _stream()))
        self._pending.append((x_host, out_host))

    def join(self) -> None:
        if not self._h:
            raise ValueError("the pipe was closed")
        _check("moe_layer_pipe_join", lib.moe_layer_pipe_join(self._h, _stream()))
        # the buffers stay referenced until the stream has passed the join
        self._joined = self._pending
        self._pending = []

    def close(self) -> None:
        if self._h:
            lib.moe_layer_pipe_destroy(self._h)
            self._h = c_void_p()
            self._pending = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class LayerGraph:
    """A captured layer call (moe_layer_graph_*); keeps its layer and buffers alive."""

    def __init__(self, handle: c_void_p, keep):
        self._h = handle
        self._keep = keep

    def launch(self) -> None:
        if not self._h:
            raise ValueError("the graph was closed")
        _check("moe_layer_graph_launch", lib.moe_layer_graph_launch(self._h, _stream()))

    def close(self) -> None:
        if self._h:
            lib.moe_layer_graph_destroy(self._h)
            self._h = c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _check_layer_weights(w: Dict[str, torch.Tensor], H: int, E: int, I: int, L: int,
                         I_shared: int) -> None:
    """Every pointer of moe_weights against the layout the configuration
    implies (the experts read the latent width L when L > 0)."""
    bf16 = torch.bfloat16
    extra = set(w) - {n for n, _ in MoeWeights._fields_}
    if extra:
        raise ValueError(f"unknown weight names: {sorted(extra)}")
    _arg("router_w", w.get("router_w"), (E, H), torch.float32)
    _arg("router_bias", w.get("router_bias"), (E,), torch.float32)
    _experts(w, E, L if L else H, I)
    if L:
        _arg("lat_down", w.get("lat_down"), (L, H), bf16)
        _arg("lat_up", w.get("lat_up"), (H, L), bf16)
        if w.get("lat_norm") is not None:
            _arg("lat_norm", w["lat_norm"], (L,), bf16)
    if I_shared:
        _arg("shared_gate", w.get("shared_gate"), (I_shared, H), bf16)
        _arg("shared_up", w.get("shared_up"), (I_shared, H), bf16)
        _arg("shared_down", w.get("shared_down"), (H, I_shared), bf16)
    if w.get("router_w_terms") is not None:
        _arg("router_w_terms", w["router_w_terms"], (3, E, H), bf16)
