"""Shared helpers of the GPU parity tests."""

import numpy as np
import torch

# Tolerance for floating-point GEMM / combine outputs against the float64 oracle:
# relative L2 error and max |error| relative to the rms of the expected output.
REL_L2 = 2e-3
MAX_ABS_OF_RMS = 1e-2


def assert_close(got, want, rel_l2=REL_L2, max_abs_of_rms=MAX_ABS_OF_RMS, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if want.size == 0:
        return 0.0, 0.0
    nrm = np.linalg.norm(want)
    err = np.linalg.norm(got - want) / nrm if nrm > 0 else np.linalg.norm(got)
    rms = np.sqrt(np.mean(want ** 2))
    mae = np.max(np.abs(got - want))
    assert err <= rel_l2, f"{what}: rel-L2 {err:.3e} > {rel_l2}"
    assert mae <= max_abs_of_rms * rms, f"{what}: max-abs {mae:.3e} > {max_abs_of_rms}*rms ({rms:.3e})"
    return err, mae / rms if rms > 0 else 0.0


def bf16_half_ulp(v):
    """Half a bf16 ulp at |v| (bf16 keeps 8 significant bits)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.ldexp(1.0, (e - 8).astype(np.int64)), 0.0)


def assert_close_bf16(got, want_f64, rel_l2=REL_L2, max_abs_of_rms=MAX_ABS_OF_RMS, what=""):
    """A bf16 output against the oracle's value before its final bf16 rounding.

    The bound of assert_close applies to |got - want| minus the half ulp that
    rounding the exact value to bf16 may add by itself: two correct programs
    whose sums straddle a bf16 rounding midpoint differ by one whole ulp, which
    for outputs above ~2.6 rms is more than 1e-2 rms.
    """
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want_f64, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if want.size == 0:
        return 0.0, 0.0
    # relative L2 against the oracle's own bf16 output (both sides rounded once)
    want_bf16 = bf16_round(want)
    nrm = np.linalg.norm(want_bf16)
    err = np.linalg.norm(got - want_bf16) / nrm if nrm > 0 else np.linalg.norm(got)
    rms = np.sqrt(np.mean(want ** 2))
    excess = np.maximum(np.abs(got - want) - bf16_half_ulp(want), 0.0)
    mae = float(np.max(excess))
    assert err <= rel_l2, f"{what}: rel-L2 {err:.3e} > {rel_l2}"
    assert mae <= max_abs_of_rms * rms, \
        f"{what}: max-abs beyond half an ulp {mae:.3e} > {max_abs_of_rms}*rms ({rms:.3e})"
    return err, mae / rms if rms > 0 else 0.0


def bf16_round(x):
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 256.0), e - 8)


def _rows_np(t, rows):
    """Rows of a (device or host) tensor or array as float64 / uint8 NumPy."""
    if isinstance(t, torch.Tensor):
        sel = t[torch.as_tensor(np.asarray(rows, dtype=np.int64), device=t.device)]
        if sel.dtype == torch.bfloat16:
            sel = sel.float()
        a = sel.cpu().numpy()
    else:
        a = np.asarray(t)[np.asarray(rows, dtype=np.int64)]
    return a.astype(np.float64) if a.dtype.kind == "f" else a


def _scalar(v):
    return v.item() if isinstance(v, torch.Tensor) else float(v)


def check_forward(fwd, out, inter, experts, ids, topk_weights, tokens=None, what=""):
    """The GPU forward against the oracle's forward, token by token.

    ``inter`` holds the oracle's intermediates for the checked tokens: the
    whole batch (``tokens`` None), or the sample ``tokens`` run through the
    oracle with the whole batch's global amax values (``oracle.forward(...,
    amax_x=..., amax_h=...)``).  ``ids`` / ``topk_weights`` are the whole
    batch's routing inputs.

    The L1 output h is rounded to bf16 and then re-quantised to NVFP4; both
    are decisions.  The GPU accumulates L1 in fp32 and the oracle in float64,
    so a few h values can land one bf16 ulp apart, and an NVFP4 code or block
    scale of h decided from such a value can differ; that step is a
    discontinuity of the method, not an error of either side.  So:
      * h of every checked slot meets the stated tolerance against the
        oracle's h before its bf16 rounding (assert_close_bf16), and at most
        1e-3 of those h elements differ from the oracle's rounded h;
      * every requantised block whose codes or scale differ contains such an
        h difference, and at most 1 % of the checked tokens (at least one)
        own one;
      * the output of every other token meets the stated tolerance against the
        oracle's value before its final rounding (assert_close_bf16);
      * each token that owns a flip is recomputed from the forward's own h
        (check_sampled_tokens: its requantised rows bit-exact given the
        forward's amax(h), then the oracle's L2 and combine), so no token goes
        unchecked.
    """
    v = fwd.intermediates()
    ids = np.asarray(ids)
    w = np.asarray(topk_weights)
    T, k = ids.shape
    tokens = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    rt = inter["routing"]  # the oracle's routing of the checked tokens
    got_all = bf16_to_np(out)
    got = got_all[tokens]
    slot_gpu = _rows_np(v["slot_dst"], np.arange(T * k)).astype(np.int64).reshape(T, k)
    g_rows = slot_gpu[tokens].reshape(-1)
    o_rows = np.asarray(rt.slot_dst, dtype=np.int64).reshape(-1)
    assert np.array_equal(g_rows >= 0, o_rows >= 0), f"{what}: skipped slots differ"
    sel = o_rows >= 0
    slot_tok = np.repeat(np.arange(tokens.size), k)[sel]  # index into tokens
    g_rows, o_rows = g_rows[sel], o_rows[sel]
    if g_rows.size == 0:
        assert_close_bf16(got, inter["out_f64"], what=what)
        return
    h_gpu = _rows_np(v["h"], g_rows)
    h_or = inter["h"][o_rows]
    assert_close_bf16(h_gpu, inter["h_f64"][o_rows], what=what + " h")
    diff = h_gpu != h_or
    assert diff.sum() <= max(1, 1e-3 * diff.size), f"{what}: {diff.sum()} h diffs"
    hq = _rows_np(v["hq_codes"], g_rows)
    hs = _rows_np(v["hq_sf"], g_rows)
    n, I = h_or.shape
    code_flip = (hq != inter["hq_codes"][o_rows]).reshape(n, I // 16, 8).any(axis=2)
    scale_flip = hs != inter["hq_scales"][o_rows]
    block_flip = code_flip | scale_flip
    h_block_diff = diff.reshape(n, I // 16, 16).any(axis=2)
    assert np.all(h_block_diff[block_flip]), f"{what}: a requant flip without an h difference"
    flip_tok = np.unique(slot_tok[block_flip.any(axis=1)])
    assert flip_tok.size <= max(1, 0.01 * tokens.size), f"{what}: {flip_tok.size} tokens with flips"
    keep = np.ones(tokens.size, dtype=bool)
    keep[flip_tok] = False
    assert_close_bf16(got[keep], inter["out_f64"][keep], what=what)
    if flip_tok.size:
        check_sampled_tokens(experts, ids, w, slot_gpu.reshape(-1), v["h"], v["hq_codes"],
                             v["hq_sf"], _scalar(v["gs_h"]), _scalar(v["amax_h"]), got_all,
                             tokens[flip_tok], what=what + " (tokens with a requant flip)")
    assert np.all(np.isfinite(got))


def to_np(t):
    return t.detach().cpu().numpy()


def bf16_to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


class NumpyExperts:
    """Expert set over in-memory NumPy weights (the oracle's protocol)."""

    def __init__(self, ws, d, I):
        self.ws, self.d, self.I = ws, d, I
        self.num_experts = len(ws)

    def __getitem__(self, e):
        return self.ws[e]


def random_experts(rng, E, d, I, oracle_q):
    """Quantise random float weights with the oracle; returns (NumpyExperts,
    stacked dict of torch CPU tensors in the library's row-major layout)."""
    ws = []
    for _ in range(E):
        g = (rng.standard_normal((I, d)) * 0.05).astype(np.float32)
        u = (rng.standard_normal((I, d)) * 0.05).astype(np.float32)
        dn = (rng.standard_normal((d, I)) * 0.05).astype(np.float32)
        gc, gsc, ggs, _ = oracle_q.quantize(g)
        uc, usc, ugs, _ = oracle_q.quantize(u)
        dc, dsc, dgs, _ = oracle_q.quantize(dn)
        ws.append(dict(w13_codes=np.concatenate([gc, uc]), w13_scales=np.concatenate([gsc, usc]),
                       w13_gs=np.array([ggs, ugs], np.float32), w2_codes=dc, w2_scales=dsc,
                       w2_gs=np.float32(dgs)))
    stacked = dict(
        w13_codes=torch.from_numpy(np.stack([w["w13_codes"] for w in ws])),
        w13_scales=torch.from_numpy(np.stack([w["w13_scales"] for w in ws])),
        w13_gs=torch.from_numpy(np.stack([w["w13_gs"] for w in ws])),
        w2_codes=torch.from_numpy(np.stack([w["w2_codes"] for w in ws])),
        w2_scales=torch.from_numpy(np.stack([w["w2_scales"] for w in ws])),
        w2_gs=torch.from_numpy(np.array([w["w2_gs"] for w in ws], np.float32)),
    )
    return NumpyExperts(ws, d, I), stacked


def bf16_tensor(rng, shape, scale=1.0):
    x = torch.from_numpy((rng.standard_normal(shape) * scale).astype(np.float32))
    return x.to(torch.bfloat16)


def check_sampled_tokens(experts, ids, topk_weights, slot_dst, h, hq_codes, hq_sf, gs_h, amax_h,
                         out, tokens, what=""):
    """Sampled output tokens of a forward, recomputed one by one from its own h.

    For each routed row of a sampled token: the row's requantised codes and
    scales must equal the oracle's quantisation of that h row with the
    forward's amax(h) (row-local given the global scale, so bit-exact); then
    the oracle's L2 (float64 on dequantised operands) and the weighted sum
    over the token's slots give the value its bf16 output must meet
    (assert_close_bf16).  Needs only the token's k rows and experts, so it
    runs at any size.
    """
    from oracle import nvfp4 as q

    k = ids.shape[1]
    gs_h = np.float32(gs_h)
    amax_h = np.float32(amax_h)
    w2 = {}
    want = np.zeros((len(tokens), out.shape[1]))
    for i, t in enumerate(tokens):
        for j in range(k):
            r = int(slot_dst[int(t) * k + j])
            if r < 0:
                continue
            hc, hs, hg, _ = q.quantize(_rows_np(h, [r]).astype(np.float32), amax=amax_h)
            assert hg == gs_h, f"{what}: gs_h {gs_h!r} vs {hg!r}"
            assert np.array_equal(_rows_np(hq_codes, [r])[0], hc[0]), \
                f"{what}: requantised codes of row {r}"
            assert np.array_equal(_rows_np(hq_sf, [r])[0], hs[0]), \
                f"{what}: requantised scales of row {r}"
            e = int(ids[t, j])
            if e not in w2:
                ew = experts[e]
                w2[e] = q.dequantize(ew["w2_codes"], ew["w2_scales"], ew["w2_gs"])
            y = (q.dequantize(hc, hs, hg) @ w2[e].T)[0]
            want[i] += np.float64(topk_weights[t, j]) * y
    assert_close_bf16(np.asarray(out)[np.asarray(tokens)], want, what=what + " sampled tokens")


# ---------------------------------------------------------------------------
# BFP16 (the forward's storage of y): a NumPy model of the encoding, in the
# float32 decisions the epilogue takes, to check the GPU bytes and to bound
# the error the format adds.  Groups are 16 rows x 8 columns; values are
# stored as u = rint(v * 2^-s) + 32768.
# ---------------------------------------------------------------------------
BFP16_NONFINITE = 127


def bfp16_exponents(v32, valid=None):
    """Per group of 16 rows x 8 columns of a float32 [rows, n] array (rows a
    multiple of 16, n of 8), over the group's written rows (``valid``,
    default all): s = max(floor(log2 max|v|) - 14, -126), plus one when
    max|v| * 2^-s >= 32767.5; 0 when they are all zero, 127 when they hold
    Inf or NaN."""
    v32 = np.asarray(v32, dtype=np.float32)
    rows, n = v32.shape
    bits = v32.view(np.uint32) & np.uint32(0x7FFFFFFF)
    if valid is not None:
        bits = np.where(np.asarray(valid)[:, None], bits, np.uint32(0))
    bits = bits.reshape(rows // 16, 16, n // 8, 8).max(axis=(1, 3))
    be = (bits >> 23).astype(np.int64)
    s = np.maximum(np.where(be == 0, -127, be - 127) - 14, -126)
    m = bits.view(np.float32).astype(np.float64)
    s = np.where(np.ldexp(m, -s) >= 32767.5, s + 1, s)
    s = np.where(bits == 0, 0, s)
    return np.where(bits >= 0x7F800000, BFP16_NONFINITE, s).astype(np.int8)


def _expand(s, rows):
    """Exponents [rows/16, n/8] -> per element [rows, n]."""
    return np.repeat(np.repeat(np.asarray(s, dtype=np.int64), 16, axis=0), 8, axis=1)[:rows]


def bfp16_encode(v32, valid=None):
    """(stored uint16 values u [rows, n], int8 exponents s [rows/16, n/8]) of
    a float32 array; rows outside ``valid`` are encoded with their group's
    exponent but take no part in choosing it."""
    v32 = np.asarray(v32, dtype=np.float32)
    s = bfp16_exponents(v32, valid)
    se = _expand(s, v32.shape[0])
    nonfin = se == BFP16_NONFINITE
    scaled = np.ldexp(v32.astype(np.float64), np.where(nonfin, 0, -se))  # exact
    with np.errstate(invalid="ignore", over="ignore"):
        q = np.rint(np.where(nonfin, 0.0, scaled))
        rows_ok = np.ones(q.shape[0], bool) if valid is None else np.asarray(valid)
        assert np.all(np.abs(q[rows_ok]) <= 32767)  # by the choice of s
        u = (np.clip(q, -32768, 32767) + 32768).astype(np.uint16)  # rows outside `valid`: any bits
        half = v32.astype(np.float16).view(np.uint16)  # used only in non-finite groups
    return np.where(nonfin, half, u).astype(np.uint16), s


def bfp16_decode(u, s):
    """float64 values of a BFP16 matrix (u [rows, n], s [rows/16, n/8])."""
    u = np.asarray(u, dtype=np.uint16)
    se = _expand(s, u.shape[0])
    nonfin = se == BFP16_NONFINITE
    val = np.ldexp(u.astype(np.float64) - 32768.0, np.where(nonfin, 0, se))
    with np.errstate(invalid="ignore"):
        return np.where(nonfin, u.view(np.float16).astype(np.float64), val)


def bfp16_split(buf, rows, ld):
    """(u [rows, ld], s [ceil(rows/16), ld/8]) NumPy views of a BFP16 matrix
    held in a uint8 buffer."""
    b = np.asarray(buf.cpu().numpy() if isinstance(buf, torch.Tensor) else buf, dtype=np.uint8)
    g = (rows + 15) // 16
    u = b[:rows * ld * 2].view(np.uint16).reshape(rows, ld)
    s = b[rows * ld * 2:rows * ld * 2 + g * (ld // 8)].view(np.int8).reshape(g, ld // 8)
    return u, s
