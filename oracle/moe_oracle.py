"""fp64 CPU oracle: routing, sorted dispatch, int4 unpack/dequantisation, the
gated expert MLP, the top-k combine, the latent wrap and the act_bits=8 mode.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Page references:

* "Kimi exact-generator adaptation" page -- sections "The proposed substitution"
  and "Sources & provenance" (routed experts use PackedInt4Linear for gate, up
  and down with buffers weight_packed / weight_scale, group size 32, act_bits
  16 by default or 8, "int64 exact int4 MAC"); section "The preserved forward
  form" (down applied to the activated gate times up).
* "Kimi K2.5 donor reference" page -- equations "MoEGate.forward: logits",
  "Independent sigmoid scores for the router", "Bias the choice of experts
  while retaining original affinities", "MoEGate.forward: ( , topk idx)",
  "MoEGate.forward: topk weight", "Normalize the selected routing affinities",
  "DeepSeek MoE.moe_infer: tokens per expert", "DeepSeek MoE.moe_infer: sorted
  tokens", "Sum the selected expert outputs with their routing weights",
  "SwiGLU-style gated feed-forward projection", and the three RMSNorm
  equations ("RMSNorm mean square ...", "Normalize by the root mean square",
  "Apply learned per-feature RMSNorm gains"); section "Quantization and source
  boundaries" (packed int4 routed experts, BF16 scales, F32 router bias).
* "Kimi K3 latent up-projection" page -- the KimiSparseMoeBlock listing
  (forward: router on the full width, then down-projection, moe_infer, norm,
  up-projection; moe_infer: one-hot counts, argsort, gather, per-expert loop,
  scatter back, fp32 weighted sum) and the "Latent up-projection" shapes.

Readings where the pages are silent:
  - one expert group, so group-limited masking is the identity;
  - rank by s + b, weight by the unbiased s; ties go to the lower expert id;
  - argsort is stable (rows of one expert ascend by token id);
  - nibble j (bits 4j..4j+3) of packed word i is column 8i+j, two's complement;
  - act_bits=16: bf16 activations times exactly dequantised weights;
  - the int16/int64 reading of act_bits=16 (quantize_rows_int16,
    int4_linear_int16): the int8 steps with 32767, integer group partials;
  - the weight quantisers (four and eight bits, group 32): scale =
    bf16(max|w| / 7 or / 127), codes = clamp(rint(w / scale)) in IEEE float32;
  - act_bits=8: per-row symmetric int8, scale = max|v|/127 and
    q = clamp(rint(v/scale), -127, 127), all in IEEE float32; weight-group
    integer partials are exact; the input of every int4 linear is its bf16
    value (module dtype);
  - RMSNorm eps 1e-6 and the latent norm on.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, Mapping, Optional

import numpy as np

GROUP = 32          # columns per weight scale
RENORM_EPS = 1e-20  # stabiliser of the top-k renormalisation
Q8_MAX = 127        # symmetric int8 activation range


# ----------------------------------------------------------------------------
# number formats
# ----------------------------------------------------------------------------

def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact: a bf16 is the top half of a float32)."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f32_to_bf16_bits(v) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest, ties to even (finite inputs)."""
    u = np.ascontiguousarray(np.asarray(v, dtype=np.float32)).view(np.uint32).astype(np.uint64)
    bias = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return ((u + bias) >> np.uint64(16)).astype(np.uint16)


def round_bf16(v) -> np.ndarray:
    """Value of ``v`` after storage in a bf16 tensor (via float32), as float64."""
    return bf16_bits_to_f64(f32_to_bf16_bits(np.asarray(v, dtype=np.float64).astype(np.float32)))


# ----------------------------------------------------------------------------
# PackedInt4Linear storage
# ----------------------------------------------------------------------------

def unpack_int4(packed) -> np.ndarray:
    """int32 [..., K/8] -> int8 [..., K].

    Word i holds columns 8i..8i+7; column 8i+j is nibble j (bits 4j..4j+3),
    a two's-complement value in [-8, 7]."""
    w = np.ascontiguousarray(np.asarray(packed, dtype=np.int32)).view(np.uint32)
    shifts = (np.arange(8, dtype=np.uint32) * np.uint32(4))
    nib = ((w[..., None] >> shifts) & np.uint32(0xF)).astype(np.int16)
    val = np.where(nib >= 8, nib - 16, nib).astype(np.int8)
    return val.reshape(*w.shape[:-1], w.shape[-1] * 8)


def pack_int4(q) -> np.ndarray:
    """int [..., K] with values in [-8, 7] -> int32 [..., K/8] (inverse of unpack_int4)."""
    q = np.asarray(q, dtype=np.int64)
    if q.shape[-1] % 8:
        raise ValueError("K must be a multiple of 8")
    if q.size and (q.min() < -8 or q.max() > 7):
        raise ValueError("int4 values must lie in [-8, 7]")
    nib = (q & 0xF).astype(np.uint32).reshape(*q.shape[:-1], q.shape[-1] // 8, 8)
    w = np.zeros(nib.shape[:-1], dtype=np.uint32)
    for j in range(8):
        w |= nib[..., j] << np.uint32(4 * j)
    return w.view(np.int32)


def dequantize(packed, scale_bits) -> np.ndarray:
    """W[n, c] = q[n, c] * scale[n, c // 32] in float64 (exact)."""
    q = unpack_int4(packed).astype(np.float64)
    s = bf16_bits_to_f64(scale_bits)
    if q.shape[-1] != s.shape[-1] * GROUP:
        raise ValueError("scale must have K/32 columns")
    return q * np.repeat(s, GROUP, axis=-1)


# ----------------------------------------------------------------------------
# router
# ----------------------------------------------------------------------------

def sigmoid(z) -> np.ndarray:
    """Independent per-expert sigmoid 1/(1+exp(-z))."""
    return 1.0 / (1.0 + np.exp(-np.asarray(z, dtype=np.float64)))


@dataclass
class Route:
    idx: np.ndarray     # int64 [T, k], slots in descending ranking score
    weight: np.ndarray  # float64 [T, k]
    s: np.ndarray       # float64 [T, E] sigmoid affinities
    r: np.ndarray       # float64 [T, E] ranking scores s + b


def router_scores(x, w_router, bias):
    """Logits z = x W^T, affinities s = sigmoid(z), ranking scores r = s + b."""
    z = np.asarray(x, dtype=np.float64) @ np.asarray(w_router, dtype=np.float64).T
    s = sigmoid(z)
    r = s + np.asarray(bias, dtype=np.float64)[None, :]
    return z, s, r


def select_topk(r, k: int) -> np.ndarray:
    """Indices of the k largest r per row, descending; equal scores keep the lower index first."""
    order = np.argsort(-np.asarray(r), axis=-1, kind="stable")
    return order[:, :k]


def route(x, w_router, bias, k: int, renorm: bool = True) -> Route:
    """Top-k routing: rank by the biased score, weight by the unbiased affinity,
    optionally divide by (sum of the selected affinities + 1e-20)."""
    _, s, r = router_scores(x, w_router, bias)
    idx = select_topk(r, k)
    w = np.take_along_axis(s, idx, axis=1)
    if renorm:
        w = w / (w.sum(axis=1, keepdims=True) + RENORM_EPS)
    return Route(idx=idx, weight=w, s=s, r=r)


def topk_gap(r, k: int) -> np.ndarray:
    """Per row: k-th largest minus (k+1)-th largest ranking score (inf if k == E)."""
    r = np.asarray(r, dtype=np.float64)
    if k >= r.shape[1]:
        return np.full(r.shape[0], np.inf)
    srt = -np.sort(-r, axis=1)
    return srt[:, k - 1] - srt[:, k]


# ----------------------------------------------------------------------------
# sorted dispatch (the moe_infer structure)
# ----------------------------------------------------------------------------

@dataclass
class Dispatch:
    counts: np.ndarray     # int64 [E]   tokens per expert
    offsets: np.ndarray    # int64 [E+1] exclusive prefix of counts
    row_token: np.ndarray  # int64 [T*k] token of each expert-sorted row
    row_slot: np.ndarray   # int64 [T*k] top-k slot of each row
    inv_row: np.ndarray    # int64 [T*k] flat (t*k + j) -> row


def dispatch(idx, E: int) -> Dispatch:
    """One-hot counts, stable argsort of the flattened expert ids, and its inverse."""
    idx = np.asarray(idx, dtype=np.int64)
    T, k = idx.shape
    onehot = np.zeros((T, E), dtype=np.int64)
    onehot[np.arange(T)[:, None], idx] = 1
    counts = onehot.sum(axis=0)
    order = np.argsort(idx.reshape(-1), kind="stable")
    inv_row = np.empty(T * k, dtype=np.int64)
    inv_row[order] = np.arange(T * k, dtype=np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    return Dispatch(counts=counts, offsets=offsets, row_token=order // k,
                    row_slot=order % k, inv_row=inv_row)


# ----------------------------------------------------------------------------
# act_bits = 8
# ----------------------------------------------------------------------------

def quantize_rows_int8(v):
    """Per-row symmetric int8 quantisation, every step in IEEE float32.

    a = max|v| (exact); scale = a / 127 (RN); q = clamp(rint(v / scale), -127, 127)
    with rint rounding half to even.  A zero row gives scale 0 and q = 0."""
    v = np.asarray(v, dtype=np.float32)
    amax = np.max(np.abs(v), axis=-1)
    scale = (amax / np.float32(Q8_MAX)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint(v / scale[..., None])
    q = np.where(scale[..., None] > 0, q, np.float32(0))
    q = np.clip(q, -Q8_MAX, Q8_MAX).astype(np.int8)
    return q, scale


Q4_MAX = 7           # symmetric int4 weight range used by the quantiser


def quantize_weight_int4(w):
    """bf16 weight [N, K] -> (packed int32 [N, K/8], bf16 scale bits [N, K/32]).

    The conversion the "Kimi exact-generator adaptation" page names (section
    "The proposed substitution": the to_exact path calls ExactLinear.from_weight
    with a four-bit choice and group size 32; the page gives no rounding
    rule).  Reading, per row and 32-column group, every step in IEEE float32:
    a = max|w| (exact); s = bf16(a / 7) (the division rounded to nearest, then
    rounded to bf16, ties to even); q = clamp(rint(w / s), -8, 7) with the
    stored (bf16) s and rint rounding half to even; s = 0 gives q = 0.  The
    values are packed as in ``pack_int4``."""
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    if K % GROUP:
        raise ValueError("K must be a multiple of 32")
    g = w.reshape(N, K // GROUP, GROUP)
    amax = np.max(np.abs(g), axis=-1)
    s_bits = f32_to_bf16_bits((amax / np.float32(Q4_MAX)).astype(np.float32))
    s = (s_bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint(g / s[..., None])
    q = np.where(s[..., None] > 0, q, np.float32(0))
    q = np.clip(q, -8, Q4_MAX).astype(np.int64).reshape(N, K)
    return pack_int4(q), s_bits


Q8W_MAX = 127       # symmetric int8 weight range used by the 8-bit quantiser


def quantize_weight_int8(w):
    """bf16 weight [N, K] -> (int8 codes [N, K], bf16 scale bits [N, K/32]).

    The eight-bit choice of the conversion the "Kimi exact-generator
    adaptation" page names (section "The proposed substitution":
    ExactLinear.from_weight with "four-bit or eight-bit choices and a group
    size of 32"; no rounding rule is given).  The reading of the four-bit
    quantiser with 127 in place of 7, per row and 32-column group, every step
    in IEEE float32: a = max|w| (exact); s = bf16(a / 127) (the division
    rounded to nearest, then to bf16, ties to even); q = clamp(rint(w / s),
    -127, 127) with the stored s and rint rounding half to even; s = 0 gives
    q = 0.  Codes are stored one per byte in column order."""
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    if K % GROUP:
        raise ValueError("K must be a multiple of 32")
    g = w.reshape(N, K // GROUP, GROUP)
    amax = np.max(np.abs(g), axis=-1)
    s_bits = f32_to_bf16_bits((amax / np.float32(Q8W_MAX)).astype(np.float32))
    s = (s_bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint(g / s[..., None])
    q = np.where(s[..., None] > 0, q, np.float32(0))
    q = np.clip(q, -Q8W_MAX, Q8W_MAX).astype(np.int8).reshape(N, K)
    return q, s_bits


def int4_group_partials(qx, packed) -> np.ndarray:
    """Exact integer partial sums P[r, n, g] = sum_{c in group g} qx[r, c] * qw[n, c].

    Computed as a float64 matrix product of integer-valued operands: every
    product and partial sum is an integer of magnitude <= 32*8*127 < 2**53, so
    the result is exact; it is returned as int64.  The whole-K bound
    K*8*127 < 2**31 is asserted as the int32 accumulator bound."""
    qx = np.asarray(qx, dtype=np.int64)
    qw = unpack_int4(packed).astype(np.int64)
    R, K = qx.shape
    N = qw.shape[0]
    if K * 8 * Q8_MAX >= 2 ** 31:
        raise ValueError("K*8*127 must stay below 2**31")
    G = K // GROUP
    qx3 = qx.reshape(R, G, GROUP).astype(np.float64).transpose(1, 0, 2)   # [G, R, 32]
    qw3 = qw.reshape(N, G, GROUP).astype(np.float64).transpose(1, 2, 0)   # [G, 32, N]
    P = np.matmul(qx3, qw3).transpose(1, 2, 0)                            # [R, N, G]
    Pi = np.rint(P).astype(np.int64)
    assert np.all(np.abs(Pi) <= GROUP * 8 * Q8_MAX)
    return Pi


# ----------------------------------------------------------------------------
# PackedInt4Linear and the gated expert
# ----------------------------------------------------------------------------

def int4_linear(u, packed, scale_bits, act_bits: int = 16, row_chunk: int = 64) -> np.ndarray:
    """y = u W^T for one PackedInt4Linear, float64 [R, N].

    act_bits=16: u (bf16 values) times the exactly dequantised W.
    act_bits=8:  u quantised per row to int8 (scale sx); integer partials P per
                 weight group; y[r, n] = sx[r] * sum_g scale[n, g] * P[r, n, g]."""
    u = np.asarray(u, dtype=np.float64)
    if act_bits == 16:
        return u @ dequantize(packed, scale_bits).T
    if act_bits != 8:
        raise ValueError("act_bits must be 16 or 8")
    s = bf16_bits_to_f64(scale_bits)  # [N, G]
    out = np.empty((u.shape[0], s.shape[0]), dtype=np.float64)
    for r0 in range(0, u.shape[0], row_chunk):
        qx, sx = quantize_rows_int8(u[r0:r0 + row_chunk].astype(np.float32))
        P = int4_group_partials(qx, packed)
        out[r0:r0 + row_chunk] = sx.astype(np.float64)[:, None] * np.einsum("rng,ng->rn", P, s)
    return out


# ----------------------------------------------------------------------------
# the int16 / int64 reading of act_bits = 16
# ----------------------------------------------------------------------------

Q16_MAX = 32767      # symmetric int16 activation range


def quantize_rows_int16(v):
    """Per-row symmetric int16 quantisation, every step in IEEE float32.

    The alternative reading of act_bits=16 (the exact-generator page's
    "int64 exact int4 MAC" with 16-bit activations): the int8 quantiser's
    steps with 32767 in place of 127.  a = max|v| (exact); scale = a / 32767
    (RN); q = clamp(rint(v / scale), -32767, 32767) with rint rounding half to
    even.  A zero row gives scale 0 and q = 0."""
    v = np.asarray(v, dtype=np.float32)
    amax = np.max(np.abs(v), axis=-1)
    scale = (amax / np.float32(Q16_MAX)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q16 = np.rint(v / scale[..., None])
    q16 = np.where(scale[..., None] > 0, q16, np.float32(0))
    q16 = np.clip(q16, -Q16_MAX, Q16_MAX).astype(np.int16)
    return q16, scale


def int16_group_partials(q16, packed) -> np.ndarray:
    """Exact integer partial sums P[r, n, g] = sum_{c in group g} q16[r, c] * qw[n, c].

    |P| <= 32 * 8 * 32767 < 2**23 per group, so the float64 matrix product of
    the integer operands is exact; returned as int64.  The whole-K bound
    K * 8 * 32767 < 2**31 (an int32 accumulator over all of K) is asserted."""
    q16 = np.asarray(q16, dtype=np.int64)
    qw = unpack_int4(packed).astype(np.int64)
    R, K = q16.shape
    N = qw.shape[0]
    if K * 8 * Q16_MAX >= 2 ** 31:
        raise ValueError("K*8*32767 must stay below 2**31")
    G = K // GROUP
    a = q16.reshape(R, G, GROUP).astype(np.float64).transpose(1, 0, 2)   # [G, R, 32]
    b = qw.reshape(N, G, GROUP).astype(np.float64).transpose(1, 2, 0)    # [G, 32, N]
    P = np.rint(np.matmul(a, b).transpose(1, 2, 0)).astype(np.int64)     # [R, N, G]
    assert np.all(np.abs(P) <= GROUP * 8 * Q16_MAX)
    return P


def int4_linear_int16(u, packed, scale_bits, row_chunk: int = 64) -> np.ndarray:
    """y = u W^T under the int16/int64 reading of act_bits=16, float64 [R, N]:
    u quantised per row to int16 (scale sx), integer partials P per weight
    group, y[r, n] = sx[r] * sum_g scale[n, g] * P[r, n, g]."""
    u = np.asarray(u, dtype=np.float64)
    s = bf16_bits_to_f64(scale_bits)  # [N, G]
    out = np.empty((u.shape[0], s.shape[0]), dtype=np.float64)
    for r0 in range(0, u.shape[0], row_chunk):
        q16, sx = quantize_rows_int16(u[r0:r0 + row_chunk].astype(np.float32))
        P = int16_group_partials(q16, packed)
        out[r0:r0 + row_chunk] = sx.astype(np.float64)[:, None] * np.einsum("rng,ng->rn", P, s)
    return out


def silu(g) -> np.ndarray:
    return np.asarray(g, dtype=np.float64) * sigmoid(g)


def expert_ffn(u, ex: Mapping[str, np.ndarray], act_bits: int = 16) -> np.ndarray:
    """down( SiLU(gate(u)) * up(u) ) with three PackedInt4Linear projections.

    ``ex`` holds gate/up/down ``*_packed`` (int32) and ``*_scale`` (bf16 bits)."""
    u = np.asarray(u, dtype=np.float64)
    if act_bits == 8:
        u = round_bf16(u)
    g = int4_linear(u, ex["gate_packed"], ex["gate_scale"], act_bits)
    up = int4_linear(u, ex["up_packed"], ex["up_scale"], act_bits)
    h = silu(g) * up
    if act_bits == 8:
        h = round_bf16(h)
    return int4_linear(h, ex["down_packed"], ex["down_scale"], act_bits)


def shared_expert(x, gate_bits, up_bits, down_bits) -> np.ndarray:
    """The always-active shared expert: down( SiLU(gate(x)) * up(x) ) with bf16
    nn.Linear weights and no bias, on the full-width input ("Kimi K3 latent
    up-projection" page, KimiSparseMoeBlock listing: ``self.shared_experts =
    KimiMLP(...)`` of moe_intermediate_size * num_shared_experts features and
    ``y = y + self.shared_experts(identity)``; "Kimi K2.5 donor reference"
    page, "Add an always-active shared expert"; the exact-generator page keeps
    shared experts as ordinary bf16 linear modules).

    gate_bits, up_bits bf16 bits [I, H]; down_bits [H, I].  The intermediate h
    is stored in bf16 (the module's dtype) before the down projection; the
    rest is fp64."""
    x = np.asarray(x, dtype=np.float64)
    g = x @ bf16_bits_to_f64(gate_bits).T
    u = x @ bf16_bits_to_f64(up_bits).T
    h = round_bf16(silu(g) * u)
    return h @ bf16_bits_to_f64(down_bits).T


def rmsnorm(v, gain_bits, eps: float) -> np.ndarray:
    """v / sqrt(mean(v**2) + eps) * gain, over the last axis."""
    v = np.asarray(v, dtype=np.float64)
    ms = np.mean(v * v, axis=-1, keepdims=True)
    return v / np.sqrt(ms + eps) * bf16_bits_to_f64(gain_bits)


# ----------------------------------------------------------------------------
# the layer
# ----------------------------------------------------------------------------

ExpertSource = Callable[[int], Mapping[str, np.ndarray]]


@dataclass
class LayerParams:
    k: int
    renorm: bool
    act_bits: int
    w_router: np.ndarray          # float32/float64 [E, H]
    bias: np.ndarray              # [E]
    expert: ExpertSource          # e -> dict of packed/scale arrays
    E: int
    lat_down: Optional[np.ndarray] = None   # bf16 bits [L, H]
    lat_norm: Optional[np.ndarray] = None   # bf16 bits [L] (None: no norm)
    lat_up: Optional[np.ndarray] = None     # bf16 bits [H, L]
    eps: float = 1e-6
    shared_gate: Optional[np.ndarray] = None  # bf16 bits [Is, H] (None: no shared expert)
    shared_up: Optional[np.ndarray] = None    # bf16 bits [Is, H]
    shared_down: Optional[np.ndarray] = None  # bf16 bits [H, Is]


def add_shared(out, x, p: "LayerParams") -> np.ndarray:
    """Routed output plus the shared expert on the full-width x (when present)."""
    if p.shared_gate is None:
        return out
    return out + shared_expert(x, p.shared_gate, p.shared_up, p.shared_down)


def expert_input(x, p: LayerParams) -> np.ndarray:
    """What the experts see: x itself, or its latent down-projection."""
    x = np.asarray(x, dtype=np.float64)
    if p.lat_down is None:
        return x
    return x @ bf16_bits_to_f64(p.lat_down).T


def latent_out(y, p: LayerParams) -> np.ndarray:
    """Latent wrap after the routed sum: optional RMSNorm, then the up-projection."""
    if p.lat_up is None:
        return y
    if p.lat_norm is not None:
        y = rmsnorm(y, p.lat_norm, p.eps)
    return y @ bf16_bits_to_f64(p.lat_up).T


def moe_forward(x, p: LayerParams, tokens=None) -> np.ndarray:
    """Per-token definition: out[t] = sum over the selected experts of
    weight * expert(u[t]); the router sees the full-width x.

    ``tokens`` restricts the evaluation to those rows (the result has one row
    per listed token); routing of a token depends on that token only."""
    x = np.asarray(x, dtype=np.float64)
    rows = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens)
    xs = x[rows]
    rt = route(xs, p.w_router, p.bias, p.k, p.renorm)
    u = expert_input(xs, p)
    out = np.zeros_like(u)
    cache = {}
    for i in range(xs.shape[0]):
        for j in range(p.k):
            e = int(rt.idx[i, j])
            if e not in cache:
                cache[e] = p.expert(e)
            out[i] += rt.weight[i, j] * expert_ffn(u[i:i + 1], cache[e], p.act_bits)[0]
    return add_shared(latent_out(out, p), xs, p)


@dataclass
class SortedResult:
    out: np.ndarray
    route: Route
    disp: Dispatch
    y_sorted: np.ndarray   # float64 [T*k, D] expert outputs in sorted-row order


def moe_forward_sorted(x, p: LayerParams) -> SortedResult:
    """The moe_infer structure: count, stable sort, gather, loop over experts
    (skipping idle ones), scatter back, weighted sum over the k slots."""
    x = np.asarray(x, dtype=np.float64)
    T = x.shape[0]
    rt = route(x, p.w_router, p.bias, p.k, p.renorm)
    u = expert_input(x, p)
    d = dispatch(rt.idx, p.E)
    sorted_u = u[d.row_token]
    outs = np.zeros_like(sorted_u)
    for e in range(p.E):
        a, b = int(d.offsets[e]), int(d.offsets[e + 1])
        if a == b:
            continue
        outs[a:b] = expert_ffn(sorted_u[a:b], p.expert(e), p.act_bits)
    new_x = outs[d.inv_row]                      # new_x[t*k + j] = outs[row of (t, j)]
    y = (new_x.reshape(T, p.k, -1) * rt.weight[:, :, None]).sum(axis=1)
    return SortedResult(out=add_shared(latent_out(y, p), x, p), route=rt, disp=d, y_sorted=outs)
