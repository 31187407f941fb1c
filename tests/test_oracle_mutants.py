"""Planted mistakes in the oracle, on the CPU: the pins must reject each one.

Each mutant below is one plausible slip in the fp64 oracle: a wrong sign, an
off-by-one index, a transposed operand, a dropped term, a wrong rounding or
a step in the wrong order.  The test compiles the oracle's source with that
one change applied, points the pins of ``test_oracle_pins.py`` at the
result, and requires that at least one pin fails.  A control run with the
unchanged source requires that all of them pass, so that the harness itself
is shown to run the pins.  Nothing here touches the GPU or the library.
"""
import importlib.util
import inspect
import os
import sys
import types

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ORACLE_PATH = os.path.join(os.path.dirname(HERE), "oracle", "moe_oracle.py")
PINS_PATH = os.path.join(HERE, "test_oracle_pins.py")
GOLDEN = os.path.join(HERE, "golden")

with open(ORACLE_PATH) as _f:
    SOURCE = _f.read()

# (id, the mistake, text of the oracle, the text that replaces it)
MUTANTS = [
    # number formats
    ("bf16_shift", "bf16 bits widened with the wrong shift",
     "astype(np.uint16).astype(np.uint32) << np.uint32(16)",
     "astype(np.uint16).astype(np.uint32) << np.uint32(15)"),
    ("bf16_ties_away", "bf16 rounding with ties away from zero",
     "bias = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)", "bias = np.uint64(0x8000)"),
    ("bf16_truncate", "bf16 rounding by truncation",
     "bias = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)", "bias = np.uint64(0)"),
    # int4 storage
    ("nibble_order", "nibbles read most-significant first",
     "shifts = (np.arange(8, dtype=np.uint32) * np.uint32(4))",
     "shifts = ((7 - np.arange(8, dtype=np.uint32)) * np.uint32(4))"),
    ("nibble_unsigned", "nibbles read as unsigned",
     "val = np.where(nib >= 8, nib - 16, nib).astype(np.int8)", "val = nib.astype(np.int8)"),
    ("nibble_sign_off_by_one", "code 8 (-8) read as +8",
     "np.where(nib >= 8, nib - 16, nib)", "np.where(nib > 8, nib - 16, nib)"),
    ("pack_drops_sign", "sign bit dropped when packing",
     "nib = (q & 0xF)", "nib = (q & 0x7)"),
    ("scale_interleaved", "scale of column c taken from group c mod G",
     "q * np.repeat(s, GROUP, axis=-1)", "q * np.tile(s, GROUP)"),
    # router
    ("sigmoid_sign", "sigmoid written with exp(+z)",
     "np.exp(-np.asarray(z, dtype=np.float64))", "np.exp(np.asarray(z, dtype=np.float64))"),
    ("rank_by_logit", "experts ranked by logit plus bias",
     "r = s + np.asarray(bias", "r = z + np.asarray(bias"),
    ("bias_sign", "bias subtracted from the ranking score",
     "r = s + np.asarray(bias", "r = s - np.asarray(bias"),
    ("weight_by_biased", "weights taken from the biased score",
     "w = np.take_along_axis(s, idx, axis=1)", "w = np.take_along_axis(r, idx, axis=1)"),
    ("renorm_eps", "stabiliser 1e-6 instead of 1e-20",
     "RENORM_EPS = 1e-20", "RENORM_EPS = 1e-6"),
    ("renorm_skipped", "renormalisation never applied",
     "if renorm:\n        w = w /", "if False:\n        w = w /"),
    ("topk_ascending", "the k smallest scores selected",
     "np.argsort(-np.asarray(r), axis=-1", "np.argsort(np.asarray(r), axis=-1"),
    ("topk_window_shifted", "top-k window off by one",
     "return order[:, :k]", "return order[:, 1:k + 1]"),
    ("ties_to_higher", "equal scores go to the higher expert id",
     'order = np.argsort(-np.asarray(r), axis=-1, kind="stable")',
     'order = np.asarray(r).shape[-1] - 1 - np.argsort(-np.asarray(r)[..., ::-1], axis=-1, kind="stable")'),
    ("gap_off_by_one", "gap taken between the (k-1)-th and k-th scores",
     "srt[:, k - 1] - srt[:, k]", "srt[:, k - 2] - srt[:, k - 1]"),
    ("gap_k_equals_E", "no gap case when k equals E",
     "if k >= r.shape[1]:", "if k > r.shape[1]:"),
    ("renorm_ignores_flag", "renormalisation applied with renorm off",
     "    if renorm:\n        w = w /", "    if True:\n        w = w /"),
    ("router_on_latent", "the router fed the latent input",
     "    rt = route(xs, p.w_router, p.bias, p.k, p.renorm)\n    u = expert_input(xs, p)",
     "    u = expert_input(xs, p)\n    rt = route(u, p.w_router, p.bias, p.k, p.renorm)"),
    ("token_subset_ignored", "the token subset ignored",
     "rows = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens)",
     "rows = np.arange(x.shape[0])"),
    # sorted dispatch
    ("scan_inclusive", "offsets from an inclusive scan",
     "offsets[1:] = np.cumsum(counts)", "offsets[:-1] = np.cumsum(counts)"),
    ("flatten_transposed", "top-k ids flattened slot-major",
     'np.argsort(idx.reshape(-1), kind="stable")', 'np.argsort(idx.T.reshape(-1), kind="stable")'),
    ("inverse_not_inverted", "the sort order used as its own inverse",
     "inv_row[order] = np.arange(T * k, dtype=np.int64)", "inv_row[:] = order"),
    ("token_from_remainder", "row token taken as order mod k",
     "row_token=order // k,", "row_token=order % k,"),
    ("unstable_sort", "an unstable sort of the expert ids",
     'np.argsort(idx.reshape(-1), kind="stable")', 'np.argsort(idx.reshape(-1), kind="quicksort")'),
    ("single_row_experts_skipped", "sorted path skipping experts with one row",
     "        if a == b:\n            continue", "        if b - a < 2:\n            continue"),
    # act_bits = 8 activation quantiser
    ("q8_divisor_128", "activation scale max/128",
     "(amax / np.float32(Q8_MAX))", "(amax / np.float32(128))"),
    ("q8_truncate", "activation codes truncated instead of rounded",
     "q = np.rint(v / scale[..., None])", "q = np.trunc(v / scale[..., None])"),
    ("q8_in_float64", "activation quantiser evaluated in float64",
     "    v = np.asarray(v, dtype=np.float32)\n    amax = np.max(np.abs(v), axis=-1)\n    scale = (amax / np.float32(Q8_MAX))",
     "    v = np.asarray(v, dtype=np.float64)\n    amax = np.max(np.abs(v), axis=-1)\n    scale = (amax / np.float32(Q8_MAX))"),
    ("q8_clip_126", "activation codes clamped to +-126",
     "q = np.clip(q, -Q8_MAX, Q8_MAX)", "q = np.clip(q, -Q8_MAX + 1, Q8_MAX - 1)"),
    ("q16_divisor_32768", "int16 activation scale max/32768",
     "(amax / np.float32(Q16_MAX))", "(amax / np.float32(32768))"),
    ("q16_truncate", "int16 activation codes truncated instead of rounded",
     "q16 = np.rint(v / scale[..., None])", "q16 = np.trunc(v / scale[..., None])"),
    ("q16_in_float64", "int16 activation quantiser evaluated in float64",
     "    v = np.asarray(v, dtype=np.float32)\n    amax = np.max(np.abs(v), axis=-1)\n    scale = (amax / np.float32(Q16_MAX))",
     "    v = np.asarray(v, dtype=np.float64)\n    amax = np.max(np.abs(v), axis=-1)\n    scale = (amax / np.float32(Q16_MAX))"),
    ("q16_partials_group_16", "int16 partials over groups of 16 columns",
     "a = q16.reshape(R, G, GROUP)", "a = q16.reshape(R, G, GROUP)[:, :, ::-1]"),
    ("int32_bound_loosened", "accumulator bound checked against 2^32",
     "if K * 8 * Q8_MAX >= 2 ** 31:", "if K * 8 * Q8_MAX > 2 ** 32:"),
    ("q8_row_scale_dropped", "activation row scale left out of the output",
     "P = int4_group_partials(qx, packed)\n        out[r0:r0 + row_chunk] = sx.astype(np.float64)[:, None] * np.einsum",
     "P = int4_group_partials(qx, packed)\n        out[r0:r0 + row_chunk] = np.einsum"),
    ("partials_group_strided", "weight groups taken as strided columns",
     "qw3 = qw.reshape(N, G, GROUP).astype(np.float64).transpose(1, 2, 0)",
     "qw3 = qw.reshape(N, GROUP, G).astype(np.float64).transpose(2, 1, 0)"),
    # int4 weight quantiser
    ("q4_divisor_8", "weight scale max/8",
     "(amax / np.float32(Q4_MAX))", "(amax / np.float32(8))"),
    ("q4_unrounded_scale", "weight codes from the scale before its bf16 rounding",
     "q = np.rint(g / s[..., None])\n    q = np.where(s[..., None] > 0, q, np.float32(0))\n    q = np.clip(q, -8, Q4_MAX)",
     "q = np.rint(g / (amax / np.float32(Q4_MAX))[..., None])\n    q = np.where(s[..., None] > 0, q, np.float32(0))\n    q = np.clip(q, -8, Q4_MAX)"),
    ("q4_truncate", "weight codes truncated instead of rounded",
     "q = np.rint(g / s[..., None])\n    q = np.where(s[..., None] > 0, q, np.float32(0))\n    q = np.clip(q, -8, Q4_MAX)",
     "q = np.trunc(g / s[..., None])\n    q = np.where(s[..., None] > 0, q, np.float32(0))\n    q = np.clip(q, -8, Q4_MAX)"),
    ("q4_zero_group_unguarded", "a zero group divided by its zero scale",
     "q = np.where(s[..., None] > 0, q, np.float32(0))\n    q = np.clip(q, -8, Q4_MAX)",
     "pass\n    q = np.clip(q, -8, Q4_MAX)"),
    ("q8w_divisor_128", "8-bit weight scale max/128",
     "f32_to_bf16_bits((amax / np.float32(Q8W_MAX)).astype(np.float32))",
     "f32_to_bf16_bits((amax / np.float32(128)).astype(np.float32))"),
    ("q8w_unrounded_scale", "8-bit weight codes from the scale before its bf16 rounding",
     "    s = (s_bits.astype(np.uint32) << np.uint32(16)).view(np.float32)\n    with np.errstate(divide=\"ignore\", invalid=\"ignore\"):\n        q = np.rint(g / s[..., None])\n    q = np.where(s[..., None] > 0, q, np.float32(0))\n    q = np.clip(q, -Q8W_MAX",
     "    s = (amax / np.float32(Q8W_MAX)).astype(np.float32)\n    with np.errstate(divide=\"ignore\", invalid=\"ignore\"):\n        q = np.rint(g / s[..., None])\n    q = np.where(s[..., None] > 0, q, np.float32(0))\n    q = np.clip(q, -Q8W_MAX"),
    ("q8w_truncate", "8-bit weight codes truncated instead of rounded",
     "        q = np.rint(g / s[..., None])\n    q = np.where(s[..., None] > 0, q, np.float32(0))\n    q = np.clip(q, -Q8W_MAX",
     "        q = np.trunc(g / s[..., None])\n    q = np.where(s[..., None] > 0, q, np.float32(0))\n    q = np.clip(q, -Q8W_MAX"),
    ("q8w_group_of_16", "8-bit weight groups of 16 columns",
     "    g = w.reshape(N, K // GROUP, GROUP)\n    amax = np.max(np.abs(g), axis=-1)\n    s_bits = f32_to_bf16_bits((amax / np.float32(Q8W_MAX))",
     "    g = w.reshape(N, K // 16, 16)\n    amax = np.max(np.abs(g), axis=-1)\n    s_bits = f32_to_bf16_bits((amax / np.float32(Q8W_MAX))"),
    ("pack_range_unchecked", "out-of-range codes packed silently",
     "if q.size and (q.min() < -8 or q.max() > 7):", "if False:"),
    # expert
    ("silu_sign", "SiLU written as g * sigmoid(-g)",
     "return np.asarray(g, dtype=np.float64) * sigmoid(g)",
     "return np.asarray(g, dtype=np.float64) * sigmoid(-np.asarray(g, dtype=np.float64))"),
    ("gate_up_swapped", "SiLU applied to up instead of gate",
     "h = silu(g) * up", "h = g * silu(up)"),
    ("exact_h_unrounded", "exact-mode h not rounded to its bf16 value",
     "    if act_bits == 8:\n        h = round_bf16(h)", "    if False:\n        h = round_bf16(h)"),
    ("exact_u_unrounded", "exact-mode expert input not rounded to its bf16 value",
     "    if act_bits == 8:\n        u = round_bf16(u)", "    if False:\n        u = round_bf16(u)"),
    # shared expert
    ("shared_h_unrounded", "shared-expert h kept in fp64",
     "h = round_bf16(silu(g) * u)", "h = silu(g) * u"),
    ("shared_gate_up_swapped", "shared-expert SiLU applied to up",
     "h = round_bf16(silu(g) * u)", "h = round_bf16(g * silu(u))"),
    ("shared_down_rows_reversed", "shared down projection rows reversed",
     "return h @ bf16_bits_to_f64(down_bits).T", "return h @ bf16_bits_to_f64(down_bits).T[::-1]"),
    ("shared_never_added", "the shared expert left out of the layer",
     "if p.shared_gate is None:\n        return out", "if True:\n        return out"),
    ("shared_on_expert_input", "the shared expert fed the experts' (latent) input",
     "return add_shared(latent_out(out, p), xs, p)", "return add_shared(latent_out(out, p), u, p)"),
    # RMSNorm and the latent wrap
    ("rms_eps_outside_sqrt", "eps added outside the square root",
     "v / np.sqrt(ms + eps)", "v / (np.sqrt(ms) + eps)"),
    ("rms_mean_abs", "mean |v| squared instead of the mean square",
     "ms = np.mean(v * v, axis=-1, keepdims=True)", "ms = np.mean(np.abs(v), axis=-1, keepdims=True) ** 2"),
    ("rms_over_rows", "mean square taken over the rows instead of the features",
     "ms = np.mean(v * v, axis=-1, keepdims=True)", "ms = np.mean(v * v, axis=0, keepdims=True)"),
    ("latent_norm_skipped", "the latent RMSNorm left out",
     "    if p.lat_norm is not None:\n        y = rmsnorm(y, p.lat_norm, p.eps)",
     "    if False:\n        y = rmsnorm(y, p.lat_norm, p.eps)"),
    ("rms_gain_dropped", "RMSNorm gain left out",
     "np.sqrt(ms + eps) * bf16_bits_to_f64(gain_bits)", "np.sqrt(ms + eps)"),
    ("latent_down_untransposed", "lat_down applied as [H, L]",
     "return x @ bf16_bits_to_f64(p.lat_down).T", "return x @ bf16_bits_to_f64(p.lat_down)"),
    ("norm_after_up", "RMSNorm applied after the up-projection",
     "        y = rmsnorm(y, p.lat_norm, p.eps)\n    return y @ bf16_bits_to_f64(p.lat_up).T",
     "        return rmsnorm(y @ bf16_bits_to_f64(p.lat_up).T, p.lat_norm, p.eps)\n"
     "    return y @ bf16_bits_to_f64(p.lat_up).T"),
    # the layer
    ("combine_first_slot_weight", "every slot weighted by the first slot's weight",
     "out[i] += rt.weight[i, j] *", "out[i] += rt.weight[i, 0] *"),
    ("sorted_slots_reversed", "sorted path pairs rows with reversed slots",
     "rt.weight[:, :, None]).sum(axis=1)", "rt.weight[:, ::-1, None]).sum(axis=1)"),
    ("sorted_scatter_forward", "sorted path scatters with the sort order, not its inverse",
     "new_x = outs[d.inv_row]", "new_x = outs[np.argsort(d.inv_row)]"),
]


def _compile(src: str) -> types.ModuleType:
    """The oracle module built from ``src`` (registered only while it runs,
    which its dataclasses need)."""
    name = "_oracle_under_mutation"
    mod = types.ModuleType(name)
    mod.__file__ = ORACLE_PATH
    sys.modules[name] = mod
    try:
        exec(compile(src, ORACLE_PATH, "exec"), mod.__dict__)
    finally:
        sys.modules.pop(name, None)
    return mod


def _pins(oracle_mod: types.ModuleType) -> types.ModuleType:
    """A fresh copy of the pin module (fresh random draws) whose ``O`` is ``oracle_mod``."""
    spec = importlib.util.spec_from_file_location("_pins_under_mutation", PINS_PATH)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.O = oracle_mod
    return mod


def _cases(pins: types.ModuleType):
    """(name, function, keyword arguments) of every pin, parametrisations expanded."""
    tests = [(n, f) for n, f in vars(pins).items() if n.startswith("test_") and callable(f)]
    tests.sort(key=lambda nf: inspect.getsourcelines(nf[1])[1])
    for name, fn in tests:
        combos = [{}]
        for mark in getattr(fn, "pytestmark", []):
            if mark.name != "parametrize":
                continue
            argnames, argvalues = mark.args[0], mark.args[1]
            names = [a.strip() for a in argnames.split(",")] if isinstance(argnames, str) else list(argnames)
            combos = [{**c, **dict(zip(names, v if len(names) > 1 else (v,)))}
                      for c in combos for v in argvalues]
        for c in combos:
            if "golden_dir" in inspect.signature(fn).parameters:
                c = {**c, "golden_dir": GOLDEN}
            yield f"{name}{sorted(c.items()) if c else ''}", fn, c


def _failing_pins(src: str, stop_at_first: bool) -> list:
    failed = []
    with np.errstate(all="ignore"):
        mod = _compile(src)
        for name, fn, kwargs in _cases(_pins(mod)):
            try:
                fn(**kwargs)
            # an assertion, the mistake breaking a shape, or a pytest.raises
            # that saw no exception (pytest's Failed is not an Exception)
            except (Exception, pytest.fail.Exception) as e:
                failed.append(f"{name}: {type(e).__name__}")
                if stop_at_first:
                    break
    return failed


def test_harness_runs_every_pin_and_all_pass_unchanged():
    n = sum(1 for _ in _cases(_pins(_compile(SOURCE))))
    assert n >= 40
    assert _failing_pins(SOURCE, stop_at_first=False) == []


def test_mutants_are_distinct_and_apply_once():
    assert len({m[0] for m in MUTANTS}) == len(MUTANTS)
    for ident, _, old, new in MUTANTS:
        assert SOURCE.count(old) == 1, ident
        assert old != new, ident


@pytest.mark.parametrize("ident,what,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_mutant(ident, what, old, new):
    assert SOURCE.count(old) == 1, f"{ident}: the mutated text no longer occurs once"
    assert _failing_pins(SOURCE.replace(old, new), stop_at_first=True), f"no pin rejects: {what}"
