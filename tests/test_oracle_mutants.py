"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in a fresh copy of the oracle: a sign, an index,
a dropped rounding, a transposed operand, a wrong constant or tie rule.  The
copy is built from the oracle's own source with that one edit, in memory; the
installed oracle is not touched.  The pins of tests/test_oracle_*.py then run
against the copy, and at least one of them must fail.  The unquantised
accuracy comparison is context, not a pin, and is left out.
"""

import os
import sys
import types

import pytest

import test_oracle_codec
import test_oracle_linear
import test_oracle_moe
import test_oracle_router

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE = os.path.join(ROOT, "oracle")
PIN_MODULES = (test_oracle_codec, test_oracle_moe, test_oracle_router, test_oracle_linear)
NOT_PINS = {"test_accuracy_against_unquantized_moe_matches_pages_order"}

# (oracle module, exact source text, replacement)
MUTANTS = {
    # codec
    "e4m3 exponent bias 8": ("nvfp4", "out[nrm] = ((E + 7) << 3) | f8", "out[nrm] = ((E + 8) << 3) | f8"),
    "e4m3 subnormals truncated": ("nvfp4", "out[sub] = np.rint(a[sub] * 2.0**9)",
                                  "out[sub] = np.floor(a[sub] * 2.0**9)"),
    "nibbles swapped": ("nvfp4", "(c[..., 0::2] | (c[..., 1::2] << 4))",
                        "(c[..., 1::2] | (c[..., 0::2] << 4))"),
    "bf16 keeps 7 bits": ("nvfp4", "np.rint(m * 256.0), e - 8", "np.rint(m * 128.0), e - 7"),
    "bf16 truncates": ("nvfp4", "np.rint(m * 256.0), e - 8", "np.trunc(m * 256.0), e - 8"),
    "block scale over 4": ("nvfp4", "(amax_b * gs) / np.float32(6.0)", "(amax_b * gs) / np.float32(4.0)"),
    "global scale 448 / amax": ("nvfp4", "GLOBAL_SCALE_NUMERATOR = 448.0 * 6.0",
                                "GLOBAL_SCALE_NUMERATOR = 448.0"),
    "encode factor halved": ("nvfp4", "enc = np.where(nz, gs / np.where(nz, sd, np.float32(1))",
                             "enc = np.where(nz, np.float32(0.5) * gs / np.where(nz, sd, np.float32(1))"),
    "zero block keeps codes": ("nvfp4", "codes[~nz] = 0", "pass"),
    "e2m1 tie 2.5 rounds up": ("nvfp4", "+ (a > 2.5)", "+ (a >= 2.5)"),
    "e2m1 tie 0.75 rounds down": ("nvfp4", "+ (a >= 0.75)", "+ (a > 0.75)"),
    "e2m1 sign dropped": ("nvfp4", "return (mag | (np.signbit(x).astype(np.uint8) << 3))",
                          "return (mag | (np.zeros_like(mag) << 3))"),
    "dequantise multiplies by gs": ("nvfp4", "* sd / np.float64(gs)).reshape(rows, K)",
                                    "* sd * np.float64(gs)).reshape(rows, K)"),
    "scales of the next block": ("nvfp4", "sd = _SCALE_TABLE[np.asarray(scales, dtype=np.uint8)][..., None]",
                                 "sd = np.roll(_SCALE_TABLE[np.asarray(scales, dtype=np.uint8)], -1, axis=-1)[..., None]"),
    # route, GEMM, SiLU, combine
    "route order descending": ("moe", "slots = np.nonzero(flat == e)[0]",
                               "slots = np.nonzero(flat == e)[0][::-1]"),
    "always one pad more": ("moe", "padded = (counts + pad - 1) // pad * pad",
                            "padded = (counts // pad + 1) * pad"),
    "id 0 skipped": ("moe", "for e in flat[flat >= 0]:", "for e in flat[flat > 0]:"),
    "silu sign": ("moe", "return g / (1.0 + np.exp(-g))", "return g / (1.0 + np.exp(g))"),
    "silu on up": ("moe", "hu = silu(v[:, :I]) * v[:, I:]", "hu = v[:, :I] * silu(v[:, I:])"),
    "h not rounded": ("moe", "hv = bf16_round(hu)", "hv = hu"),
    "h amax before rounding": ("moe", "amax = max(amax, float(np.max(np.abs(hv))))",
                               "amax = max(amax, float(np.max(np.abs(hu))))"),
    "gate takes the up scale": ("moe", 'w["w13_scales"][:I], w["w13_gs"][0])',
                                'w["w13_scales"][:I], w["w13_gs"][1])'),
    "combine weight index": ("moe", "acc = acc + w[t, j] * y[r]", "acc = acc + w[t, 0] * y[r]"),
    "gather by slot modulo k": ("moe", "valid = rt.row_src >= 0\n    a_codes[valid] = xq_codes[rt.row_src[valid] // k]\n"
                                "    a_scales[valid] = xq_scales[rt.row_src[valid] // k]\n\n    h, amax_h_own, h64",
                                "valid = rt.row_src >= 0\n    a_codes[valid] = xq_codes[rt.row_src[valid] % k]\n"
                                "    a_scales[valid] = xq_scales[rt.row_src[valid] % k]\n\n    h, amax_h_own, h64"),
    "sample ignores the batch's amax of x": ("moe", "quantize(x, amax=amax_x)", "quantize(x)"),
    "sample ignores the batch's amax of h": ("moe", "    if amax_h is None:\n        amax_h = amax_h_own",
                                             "    amax_h = amax_h_own"),
    "expert rows shifted by one": ("moe", "out[r0:r0 + m] = ahat[r0:r0 + m] @ wm.T",
                                   "out[r0:r0 + m] = np.roll(ahat, 1, axis=0)[r0:r0 + m] @ wm.T"),
    "combine not rounded": ("moe", "    out = bf16_round(out64)\n", "    out = out64\n"),
    "unquantised forward unweighted": ("moe", "out[t] += w[t, j] * (d_w @ hv)", "out[t] += d_w @ hv"),
    "shared h with its own scale": ("moe", "hs_codes, hs_scales, _, _ = quantize(h_s.astype(np.float32), amax=amax_h)",
                                    "hs_codes, hs_scales, _, _ = quantize(h_s.astype(np.float32))"),
    "shared amax from routed rows only": ("moe", "amax_h = np.float32(max(float(amax_r), float(np.max(np.abs(h_s))) if T else 0.0))",
                                          "amax_h = np.float32(amax_r)"),
    # router
    "ties to the higher index": ("router", "np.lexsort((idx, -score), axis=-1)",
                                 "np.lexsort((-idx, -score), axis=-1)"),
    "lowest scores selected": ("router", "np.lexsort((idx, -score), axis=-1)",
                               "np.lexsort((idx, score), axis=-1)"),
    "softmax of biased scores": ("router", "sel = np.take_along_axis(lg, ids, axis=1)",
                                 "sel = np.take_along_axis(score, ids, axis=1)"),
    "shared expert weight 1/(k+1)": ("router", "w = np.concatenate([w, np.ones((T, 1))], axis=1)",
                                     "w = np.concatenate([w, np.full((T, 1), 1.0 / (k + 1))], axis=1)"),
    # dense linear
    "linear output columns reversed": ("linear", "out = xhat @ what.T", "out = xhat @ what.T[:, ::-1]"),
    "linear ignores the given amax": ("linear", "quantize(x, amax=amax)", "quantize(x)"),
    "linear output not rounded": ("linear", "return (bf16_round(out) if round_bf16 else out), inter",
                                  "return out, inter"),
}


def _mutated_oracle(module, old, new):
    """A fresh `oracle` package object whose `module` has `old` replaced."""
    saved = {k: v for k, v in sys.modules.items() if k == "oracle" or k.startswith("oracle.")}
    pkg = types.ModuleType("oracle")
    pkg.__path__ = [ORACLE]
    pkg.__package__ = "oracle"
    try:
        for k in saved:
            del sys.modules[k]
        sys.modules["oracle"] = pkg
        for name in ("nvfp4", "moe", "router", "linear"):
            path = os.path.join(ORACLE, name + ".py")
            with open(path) as f:
                src = f.read()
            if name == module:
                assert src.count(old) == 1, f"{old!r} must occur once in oracle/{name}.py"
                src = src.replace(old, new)
            m = types.ModuleType(f"oracle.{name}")
            m.__package__ = "oracle"
            m.__file__ = path
            sys.modules[m.__name__] = m
            exec(compile(src, path, "exec"), m.__dict__)
            setattr(pkg, name, m)
        init = os.path.join(ORACLE, "__init__.py")
        with open(init) as f:
            exec(compile(f.read(), init, "exec"), pkg.__dict__)
    finally:
        for k in [k for k in sys.modules if k == "oracle" or k.startswith("oracle.")]:
            del sys.modules[k]
        sys.modules.update(saved)
    return pkg


def _first_failing_pin(pkg, monkeypatch):
    for mod in PIN_MODULES:
        for name, value in (("oracle", pkg), ("q", pkg.nvfp4), ("router_topk", pkg.router_topk)):
            if hasattr(mod, name):
                monkeypatch.setattr(mod, name, value)
    for mod in PIN_MODULES:
        for name in sorted(vars(mod)):
            if name.startswith("test_") and name not in NOT_PINS:
                try:
                    getattr(mod, name)()
                except AssertionError:
                    return f"{mod.__name__}.{name}"
    return None


def test_the_unmutated_copy_passes_every_pin(monkeypatch):
    assert _first_failing_pin(_mutated_oracle(None, "", ""), monkeypatch) is None


@pytest.mark.parametrize("case", sorted(MUTANTS))
def test_a_planted_mistake_fails_a_pin(case, monkeypatch):
    pkg = _mutated_oracle(*MUTANTS[case])
    assert _first_failing_pin(pkg, monkeypatch) is not None, f"no pin catches: {case}"
