"""Seeded synthetic inputs for the routed int4 mixture-of-experts layer.

This module is shared by the fp64 oracle (tests) and by the GPU harness (tests,
bench).  It holds none of the layer's arithmetic: it only draws numbers.  All
randomness comes from one counter-based integer hash (``mix32`` below, the
"lowbias32" finaliser published by C. Wellons), so any slice of any tensor can
be regenerated on its own, on the CPU or on a CUDA device, with identical bits:

* integer data (packed int4 words) is the hash output itself;
* bf16 scales are ``lo + (hi - lo) * u`` with ``u = (word >> 8) / 2**24``,
  evaluated as two IEEE float32 operations and rounded to bf16 (RNE);
* normal draws use Box-Muller on two hashed uniforms in float64 on the CPU.

Shapes follow the Kimi K2.5 donor-reference page ("What the archive contains":
384 routed experts, 8 selected; "Tensor-pattern discrepancy": hidden width
7,168) and the Kimi K3 latent up-projection page (latent width 3,584).  The
intermediate widths (2,048; 1,024 latent) and value distributions are the
workload definitions this library is measured on.

Routing structure that cannot be drawn blindly -- tokens re-drawn until the
k-th and (k+1)-th router scores differ by at least 1e-3, and the prefill bias
that gives a Zipf(1.1) expert load -- is stored as data in
``calibration.json`` (written by ``oracle/calibrate_workloads.py``); this module
only reads it.
"""
from __future__ import annotations

import json
import math
import os
from dataclasses import dataclass, field, replace
from typing import Dict, Optional

import numpy as np
import torch

MASK32 = 0xFFFFFFFF

# stream tags (arbitrary distinct constants)
TAG_X = 0x11
TAG_ROUTER_W = 0x21
TAG_ROUTER_B = 0x22
TAG_EXPERT_PERM = 0x23
TAG_GATE = 0x31
TAG_UP = 0x32
TAG_DOWN = 0x33
TAG_GATE_SCALE = 0x41
TAG_UP_SCALE = 0x42
TAG_DOWN_SCALE = 0x43
TAG_LAT_DOWN = 0x51
TAG_LAT_UP = 0x52
TAG_LAT_NORM = 0x53


def _mul32(x, c):
    """(x * c) mod 2**32 for 0 <= x, c < 2**32 without leaving int64 range.

    Works on Python ints and on int64 torch tensors (CPU or CUDA)."""
    lo = x & 0xFFFF
    hi = x >> 16
    return (lo * c + (((hi * c) & 0xFFFF) << 16)) & MASK32


def mix32(x):
    """lowbias32 integer hash: a bijection on [0, 2**32)."""
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def stream_key(seed: int, tag: int, a: int = 0, b: int = 0) -> int:
    """Key of one independent random stream (pure Python ints)."""
    k = mix32((seed & MASK32) ^ 0x9E3779B9)
    k = mix32(k ^ (tag & MASK32))
    k = mix32(k ^ (a & MASK32))
    k = mix32(k ^ (b & MASK32))
    return k


def _mix32_np(x: np.ndarray) -> np.ndarray:
    """mix32 on uint32 numpy arrays (multiplication wraps modulo 2**32)."""
    x = x ^ (x >> np.uint32(16))
    x = x * np.uint32(0x7FEB352D)
    x = x ^ (x >> np.uint32(15))
    x = x * np.uint32(0x846CA68B)
    x = x ^ (x >> np.uint32(16))
    return x


def words(key, start: int, count: int, device="cpu") -> torch.Tensor:
    """``count`` hashed 32-bit words of stream ``key`` from counter ``start``.

    ``key`` is an int (result [count]) or an int64 tensor of keys [R] (result
    [R, count], row r being stream key[r]).  Values are int64 in [0, 2**32).
    The CPU path evaluates the same hash with numpy uint32 arithmetic."""
    if str(device) == "cpu" and start + count <= 2 ** 32:
        i = np.arange(start, start + count, dtype=np.uint64).astype(np.uint32)
        if isinstance(key, torch.Tensor):
            i = i[None, :] ^ key.numpy().astype(np.uint32)[:, None]
        else:
            i = i ^ np.uint32(key)
        with np.errstate(over="ignore"):
            w = _mix32_np(_mix32_np(i) ^ np.uint32(0x5BD1E995))
        return torch.from_numpy(w.astype(np.int64))
    i = torch.arange(start, start + count, dtype=torch.int64, device=device)
    if isinstance(key, torch.Tensor):
        i = i[None, :] ^ key.to(device=device, dtype=torch.int64)[:, None]
    else:
        i = i ^ key
    return mix32(mix32(i) ^ 0x5BD1E995)


def _uniform24(w: torch.Tensor) -> torch.Tensor:
    return (w >> 8)  # integer in [0, 2**24)


def _box_muller(w: torch.Tensor) -> torch.Tensor:
    """float64 normals from word pairs along the last axis (cosine branch)."""
    u1 = (_uniform24(w[..., 0]).to(torch.float64) + 1.0) * (2.0 ** -24)  # (0, 1]
    u2 = _uniform24(w[..., 1]).to(torch.float64) * (2.0 ** -24)  # [0, 1)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def normals(key: int, count: int, std: float = 1.0, start: int = 0) -> torch.Tensor:
    """``count`` float64 N(0, std**2) draws (CPU) of stream ``key``."""
    w = words(key, 2 * start, 2 * count).view(count, 2)
    return _box_muller(w) * std


def normal_rows(keys, count: int, std: float = 1.0, chunk: int = 512) -> torch.Tensor:
    """float64 [R, count]: row r holds the first ``count`` normals of stream keys[r]
    (identical to ``normals(keys[r], count, std)``)."""
    keys = torch.as_tensor(list(keys), dtype=torch.int64)
    out = torch.empty(len(keys), count, dtype=torch.float64)
    for r0 in range(0, len(keys), chunk):
        kk = keys[r0:r0 + chunk]
        w = words(kk, 0, 2 * count).view(len(kk), count, 2)
        out[r0:r0 + chunk] = _box_muller(w) * std
    return out


def uniform_bf16(key: int, count: int, lo: float, hi: float, start: int = 0,
                 device="cpu") -> torch.Tensor:
    """``count`` bf16 draws from U(lo, hi): two float32 ops then RNE to bf16."""
    u = _uniform24(words(key, start, count, device)).to(torch.float32) * (2.0 ** -24)
    span = torch.tensor(hi - lo, dtype=torch.float32, device=device)
    base = torch.tensor(lo, dtype=torch.float32, device=device)
    v = torch.add(torch.mul(u, span), base)
    return v.to(torch.bfloat16)


def as_int32(w: torch.Tensor) -> torch.Tensor:
    """Reinterpret words in [0, 2**32) as two's-complement int32."""
    if w.device.type == "cpu":
        return torch.from_numpy(w.numpy().astype(np.uint32).view(np.int32))
    return (w - ((w >> 31) << 32)).to(torch.int32)


@dataclass(frozen=True)
class Workload:
    """One layer configuration plus the recipe of its synthetic inputs."""
    name: str
    T: int            # tokens
    H: int            # hidden width (input and output of the layer)
    E: int            # routed experts
    k: int            # experts selected per token
    I: int            # expert intermediate width
    L: int = 0        # latent width (0: no latent projections)
    act_bits: int = 16
    renorm: bool = True
    eps: float = 1e-6
    seed: int = 0
    x_std: float = 1.0
    router_std: float = 0.02
    bias_std: float = 0.01
    scale_lo: float = 0.002
    scale_hi: float = 0.01
    latent_std: float = 0.02
    norm_gain_std: float = 0.0   # RMSNorm gain = 1 + N(0, std); 0 gives ones
    routing: str = "uniform"     # "uniform" | "zipf" | "adversarial"
    zipf_s: float = 1.1
    zipf_dead: int = 16          # experts that receive no token under "zipf"
    adversarial_bias: float = 2.0

    @property
    def D(self) -> int:
        """Width the experts see (latent width when the latent path is on)."""
        return self.L if self.L else self.H

    @property
    def rows(self) -> int:
        """Number of dispatched (token, expert) pairs."""
        return self.T * self.k


WORKLOADS: Dict[str, Workload] = {
    # small case the oracle finishes in seconds
    "tiny": Workload("tiny", T=16, H=256, E=8, k=2, I=128, scale_lo=0.005, scale_hi=0.02),
    # one decode step of a K2.5-shaped layer
    "decode": Workload("decode", T=32, H=7168, E=384, k=8, I=2048),
    # prefill with a Zipf(1.1) expert load and some idle experts
    "prefill": Workload("prefill", T=8192, H=7168, E=384, k=8, I=2048, routing="zipf"),
    # K3-style latent MoE: 7168 -> 3584 -> experts -> RMSNorm -> 7168
    "latent": Workload("latent", T=2048, H=7168, E=384, k=8, I=1024, L=3584),
    # act_bits=8 exact mode, every token routed to the same 8 experts
    "exact": Workload("exact", T=1024, H=7168, E=384, k=8, I=2048, act_bits=8,
                      routing="adversarial"),
}

_CALIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "calibration.json")
_calib_cache: Optional[dict] = None


def calibration() -> dict:
    """Stored routing calibration (resample counters, prefill bias)."""
    global _calib_cache
    if _calib_cache is None:
        if os.path.exists(_CALIB_PATH):
            with open(_CALIB_PATH) as f:
                _calib_cache = json.load(f)
        else:
            _calib_cache = {}
    return _calib_cache


def resample_counts(w: Workload) -> Dict[int, int]:
    """Token -> number of re-draws recorded for this workload (default 0)."""
    c = calibration().get(w.name, {})
    return {int(t): int(a) for t, a in c.get("resample", {}).items()}


# ----------------------------------------------------------------------------
# generators
# ----------------------------------------------------------------------------

def gen_x(w: Workload, tokens=None, attempts: Optional[Dict[int, int]] = None) -> torch.Tensor:
    """Layer input x, bf16 [T, H] (or the listed ``tokens`` rows), CPU.

    Token t is drawn from stream (seed, X, t, a_t) where a_t is its recorded
    re-draw count."""
    if attempts is None:
        attempts = resample_counts(w)
    toks = range(w.T) if tokens is None else list(tokens)
    keys = [stream_key(w.seed, TAG_X, int(t), attempts.get(int(t), 0)) for t in toks]
    if not keys:
        return torch.empty(0, w.H, dtype=torch.bfloat16)
    return normal_rows(keys, w.H, w.x_std).to(torch.float32).to(torch.bfloat16)


def gen_x_token(w: Workload, t: int, attempt: int) -> torch.Tensor:
    """One token row drawn with an explicit re-draw counter, bf16 [H]."""
    key = stream_key(w.seed, TAG_X, t, attempt)
    return normals(key, w.H, w.x_std).to(torch.float32).to(torch.bfloat16)


def expert_permutation(w: Workload) -> torch.Tensor:
    """A seeded permutation of expert ids (used to place hot/cold experts)."""
    return torch.argsort(words(stream_key(w.seed, TAG_EXPERT_PERM), 0, w.E), stable=True)


def gen_router(w: Workload):
    """Router weight fp32 [E, H] ~ N(0, router_std) and correction bias fp32 [E].

    "uniform": bias ~ N(0, bias_std).
    "adversarial": the first ``k`` experts of the seeded permutation get
      ``adversarial_bias`` added, so that every token selects them.
    "zipf": the bias stored in the calibration file (float32 bit patterns)."""
    W = normal_rows([stream_key(w.seed, TAG_ROUTER_W, e) for e in range(w.E)], w.H,
                    w.router_std).to(torch.float32)
    b = normals(stream_key(w.seed, TAG_ROUTER_B), w.E, w.bias_std).to(torch.float32)
    if w.routing == "adversarial":
        chosen = expert_permutation(w)[: w.k]
        b[chosen] += w.adversarial_bias
    elif w.routing == "zipf":
        bits = calibration().get(w.name, {}).get("bias_bits")
        if bits is not None:
            b = torch.tensor(bits, dtype=torch.int64).to(torch.int32).view(torch.float32).clone()
    return W, b


def _packed(w: Workload, tag: int, e: int, rows: int, cols: int, device) -> torch.Tensor:
    n_words = rows * cols // 8
    return as_int32(words(stream_key(w.seed, tag, e), 0, n_words, device)).view(rows, cols // 8)


def _scales(w: Workload, tag: int, e: int, rows: int, cols: int, device) -> torch.Tensor:
    n = rows * cols // 32
    return uniform_bf16(stream_key(w.seed, tag, e), n, w.scale_lo, w.scale_hi,
                        device=device).view(rows, cols // 32)


def gen_expert(w: Workload, e: int, device="cpu") -> dict:
    """Packed int4 weights and bf16 group-32 scales of expert ``e``.

    gate/up: packed int32 [I, D/8], scale bf16 [I, D/32];
    down:    packed int32 [D, I/8], scale bf16 [D, I/32]."""
    D, I = w.D, w.I
    return {
        "gate_packed": _packed(w, TAG_GATE, e, I, D, device),
        "gate_scale": _scales(w, TAG_GATE_SCALE, e, I, D, device),
        "up_packed": _packed(w, TAG_UP, e, I, D, device),
        "up_scale": _scales(w, TAG_UP_SCALE, e, I, D, device),
        "down_packed": _packed(w, TAG_DOWN, e, D, I, device),
        "down_scale": _scales(w, TAG_DOWN_SCALE, e, D, I, device),
    }


def gen_experts(w: Workload, device="cpu") -> dict:
    """All experts stacked: packed [E, N, K/8] int32, scales [E, N, K/32] bf16.

    Generated expert by expert directly on ``device``."""
    D, I, E = w.D, w.I, w.E
    out = {
        "gate_packed": torch.empty(E, I, D // 8, dtype=torch.int32, device=device),
        "gate_scale": torch.empty(E, I, D // 32, dtype=torch.bfloat16, device=device),
        "up_packed": torch.empty(E, I, D // 8, dtype=torch.int32, device=device),
        "up_scale": torch.empty(E, I, D // 32, dtype=torch.bfloat16, device=device),
        "down_packed": torch.empty(E, D, I // 8, dtype=torch.int32, device=device),
        "down_scale": torch.empty(E, D, I // 32, dtype=torch.bfloat16, device=device),
    }
    for e in range(E):
        ex = gen_expert(w, e, device)
        for name, t in ex.items():
            out[name][e].copy_(t)
    return out


def gen_latent(w: Workload):
    """Latent projections: down bf16 [L, H], RMSNorm gain bf16 [L], up bf16 [H, L]."""
    if not w.L:
        return None
    L, H = w.L, w.H
    down = normal_rows([stream_key(w.seed, TAG_LAT_DOWN, r) for r in range(L)], H,
                       w.latent_std).to(torch.float32).to(torch.bfloat16)
    up = normal_rows([stream_key(w.seed, TAG_LAT_UP, r) for r in range(H)], L,
                     w.latent_std).to(torch.float32).to(torch.bfloat16)
    if w.norm_gain_std > 0:
        g = 1.0 + normals(stream_key(w.seed, TAG_LAT_NORM), L, w.norm_gain_std)
    else:
        g = torch.ones(L, dtype=torch.float64)
    return {"lat_down": down, "lat_norm": g.to(torch.float32).to(torch.bfloat16), "lat_up": up}


def workload(base: str, **overrides) -> Workload:
    """Workload ``base`` with fields replaced (test shapes; ``name`` may be replaced too)."""
    return replace(WORKLOADS[base], **overrides)
