"""Pins for the oracle's routing, grouped GEMM and forward (CPU only).

Checks against hand-computed routing, a brute-force per-slot forward written
with scalar loops, lossless closed forms where the GEMMs must equal a plain
float64 matmul, and invariants (conservation, relabelling, zero-token
experts, finiteness, quantise/scatter commuting, one-hot weights).
"""

import math

import numpy as np
import pytest

import oracle
from oracle import nvfp4 as q


class Experts:
    """Minimal expert set over in-memory NumPy weights."""

    def __init__(self, ws, d, I):
        self.ws, self.d, self.I = ws, d, I
        self.num_experts = len(ws)

    def __getitem__(self, e):
        return self.ws[e]


def _rand_experts(rng, E, d, I):
    ws = []
    for _ in range(E):
        g = (rng.standard_normal((I, d)) * 0.05).astype(np.float32)
        u = (rng.standard_normal((I, d)) * 0.05).astype(np.float32)
        dn = (rng.standard_normal((d, I)) * 0.05).astype(np.float32)
        gc, gsc, ggs, _ = q.quantize(g)
        uc, usc, ugs, _ = q.quantize(u)
        dc, dsc, dgs, _ = q.quantize(dn)
        ws.append(dict(w13_codes=np.concatenate([gc, uc]), w13_scales=np.concatenate([gsc, usc]),
                       w13_gs=np.array([ggs, ugs], np.float32), w2_codes=dc, w2_scales=dsc,
                       w2_gs=np.float32(dgs)))
    return Experts(ws, d, I)


def _softmax_rows(z):
    z = z - z.max(1, keepdims=True)
    e = np.exp(z)
    return (e / e.sum(1, keepdims=True)).astype(np.float32)


def test_route_hand_example():
    ids = np.array([[1, 0], [1, 1], [-1, 0]])
    r = oracle.route(ids, 3, pad=1)
    assert r.counts.tolist() == [2, 3, 0]
    assert r.offsets.tolist() == [0, 2, 5, 5]
    assert r.padded_offsets.tolist() == [0, 2, 5, 5]
    # expert 0 gets slots 1, 5; expert 1 gets slots 0, 2, 3
    assert r.row_src.tolist() == [1, 5, 0, 2, 3]
    assert r.slot_dst.tolist() == [2, 0, 3, 4, -1, 1]
    r4 = oracle.route(ids, 3, pad=4)
    assert r4.padded_offsets.tolist() == [0, 4, 8, 8]
    assert r4.row_src.tolist() == [1, 5, -1, -1, 0, 2, 3, -1]
    assert r4.slot_dst.tolist() == [4, 0, 5, 6, -1, 1]


def test_route_invariants_random():
    rng = np.random.default_rng(4)
    for E, T, k, pad in [(16, 50, 4, 1), (16, 50, 4, 32), (7, 1, 3, 128), (384, 8, 6, 32)]:
        ids = rng.integers(-1, E, (T, k))
        r = oracle.route(ids, E, pad)
        valid = ids.reshape(-1) >= 0
        assert r.counts.sum() == valid.sum()  # conservation
        assert np.all(r.padded_offsets[1:] - r.padded_offsets[:-1] ==
                      -(-r.counts // pad) * pad)  # zero stays zero
        # slot_dst and row_src are inverse on valid slots
        s = np.nonzero(valid)[0]
        assert np.array_equal(r.row_src[r.slot_dst[s]], s)
        assert np.all(r.slot_dst[~valid] == -1)
        # each expert's rows hold exactly its slots, ascending
        for e in range(E):
            rows = r.row_src[r.padded_offsets[e]:r.padded_offsets[e] + r.counts[e]]
            assert np.array_equal(rows, np.nonzero(ids.reshape(-1) == e)[0])
        assert (r.row_src == -1).sum() == r.padded_offsets[-1] - r.counts.sum()


def test_route_rejects_out_of_range_id():
    with pytest.raises(ValueError):
        oracle.route(np.array([[0, 3]]), 3)


def test_grouped_gemm_lossless_equals_plain_matmul():
    # Operands exactly on the NVFP4 grid (see the lossless codec test), so the
    # grouped GEMM must equal x @ W.T of the original float arrays.
    rng = np.random.default_rng(5)
    E, d, I, T, k = 3, 64, 32, 6, 2

    def grid_tensor(rows, K):
        g = np.array([0, .5, 1, 1.5, 2, 3, 4, -.5, -1, -2, -3, -4])
        v = rng.choice(g, (rows, K // 16, 16))
        v[:, :, 0] = 6.0
        sd = 2.0 ** rng.integers(-2, 6, (rows, K // 16, 1))
        return (v * sd / 1024.0).reshape(rows, K).astype(np.float32)

    ws, dense = [], []
    for _ in range(E):
        w13 = grid_tensor(2 * I, d)
        w2 = grid_tensor(d, I)
        c13, s13, g13, _ = q.quantize(w13, amax=2.625)
        c2, s2, g2, _ = q.quantize(w2, amax=2.625)
        ws.append(dict(w13_codes=c13, w13_scales=s13, w13_gs=np.array([g13, g13], np.float32),
                       w2_codes=c2, w2_scales=s2, w2_gs=g2))
        dense.append((w13.astype(np.float64), w2.astype(np.float64)))
    ex = Experts(ws, d, I)
    x = grid_tensor(T, d)
    ids = np.array([[0, 2], [2, 2], [1, 0], [0, -1], [2, 1], [1, 2]])
    rt = oracle.route(ids, E, pad=4)
    R = rt.padded_offsets[-1]
    xc, xs, xg, _ = q.quantize(x, amax=2.625)
    a_c = np.zeros((R, d // 2), np.uint8)
    a_s = np.zeros((R, d // 16), np.uint8)
    v = rt.row_src >= 0
    a_c[v] = xc[rt.row_src[v] // k]
    a_s[v] = xs[rt.row_src[v] // k]
    out = oracle.grouped_gemm(a_c, a_s, xg, ex, "w13", rt, "f32")
    for s in range(T * k):
        e = ids.reshape(-1)[s]
        if e < 0:
            continue
        want = dense[e][0] @ x[s // k].astype(np.float64)
        assert np.array_equal(out[rt.slot_dst[s]], want)
    # L2 of a lossless activation equally matches
    hq = grid_tensor(R, I)
    hc, hs, hg, _ = q.quantize(hq, amax=2.625)
    y = oracle.grouped_gemm(hc, hs, hg, ex, "w2", rt, "f32")
    for e in range(E):
        r0, m = rt.padded_offsets[e], rt.counts[e]
        assert np.array_equal(y[r0:r0 + m], hq[r0:r0 + m].astype(np.float64) @ dense[e][1].T)
    assert np.all(np.isnan(y[~v]))


def _brute_force_forward(x, ids, w, ex):
    """Per-slot forward with scalar loops and no permutation."""
    T, k = ids.shape
    d, I = ex.d, ex.I
    xc, xs, xg, _ = q.quantize(x)
    xh = q.dequantize(xc, xs, xg)
    hs = {}
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            if e < 0:
                continue
            we = ex[e]
            gate = q.dequantize(we["w13_codes"][:I], we["w13_scales"][:I], we["w13_gs"][0])
            up = q.dequantize(we["w13_codes"][I:], we["w13_scales"][I:], we["w13_gs"][1])
            h = np.empty(I)
            for i in range(I):
                g = math.fsum(xh[t, c] * gate[i, c] for c in range(d))
                u = math.fsum(xh[t, c] * up[i, c] for c in range(d))
                h[i] = g / (1.0 + math.exp(-g)) * u
            hs[(t, j)] = q.bf16_round(h)
    keys = sorted(hs)
    H = np.stack([hs[key] for key in keys]) if keys else np.zeros((0, I))
    amax = np.float32(np.max(np.abs(H))) if keys else np.float32(0)
    hc, hsc, hg, _ = q.quantize(H.astype(np.float32), amax=amax)
    hh = q.dequantize(hc, hsc, hg)
    out = np.zeros((T, d))
    for n, (t, j) in enumerate(keys):
        we = ex[ids[t, j]]
        down = q.dequantize(we["w2_codes"], we["w2_scales"], we["w2_gs"])
        y = np.array([math.fsum(hh[n, i] * down[c, i] for i in range(I)) for c in range(d)])
        out[t] += float(w[t, j]) * y
    return q.bf16_round(out)


def test_forward_matches_brute_force_4_tokens_2_experts():
    rng = np.random.default_rng(6)
    d, I, T, k, E = 32, 16, 4, 2, 2
    ex = _rand_experts(rng, E, d, I)
    x = q.bf16_round(rng.standard_normal((T, d)) * 0.5).astype(np.float32)
    ids = np.array([[0, 1], [1, 0], [1, -1], [0, 0]])
    w = _softmax_rows(rng.standard_normal((T, k)))
    got = oracle.forward(x, ids, w, ex, pad=1)
    want = _brute_force_forward(x, ids, w, ex)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12 * np.abs(want).max())
    got32 = oracle.forward(x, ids, w, ex, pad=32)
    assert np.array_equal(got, got32)  # padding changes nothing


def test_unquantized_forward_matches_scalar_loops():
    """The accuracy comparison point (float64 x and h, nothing rounded)
    against scalar loops with math.fsum and math.exp on a tiny case."""
    rng = np.random.default_rng(8)
    d, I, T, k, E = 16, 16, 3, 2, 3
    ex = _rand_experts(rng, E, d, I)
    x = rng.standard_normal((T, d)) * 0.7
    ids = np.array([[0, 2], [2, -1], [1, 1]])
    w = _softmax_rows(rng.standard_normal((T, k)))
    got = oracle.forward_unquantized(x, ids, w, ex)
    want = np.zeros((T, d))
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j])
            if e < 0:
                continue
            we = ex[e]
            gate = q.dequantize(we["w13_codes"][:I], we["w13_scales"][:I], we["w13_gs"][0])
            up = q.dequantize(we["w13_codes"][I:], we["w13_scales"][I:], we["w13_gs"][1])
            down = q.dequantize(we["w2_codes"], we["w2_scales"], we["w2_gs"])
            h = []
            for i in range(I):
                g = math.fsum(x[t, c] * gate[i, c] for c in range(d))
                u = math.fsum(x[t, c] * up[i, c] for c in range(d))
                h.append(g / (1.0 + math.exp(-g)) * u)
            for c in range(d):
                want[t, c] += float(w[t, j]) * math.fsum(h[i] * down[c, i] for i in range(I))
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12 * np.abs(want).max())


def test_forward_invariant_to_expert_relabelling():
    rng = np.random.default_rng(7)
    d, I, T, k, E = 64, 32, 12, 3, 5
    ex = _rand_experts(rng, E, d, I)
    x = q.bf16_round(rng.standard_normal((T, d)) * 0.3).astype(np.float32)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    w = _softmax_rows(rng.standard_normal((T, k)))
    base = oracle.forward(x, ids, w, ex, pad=8)
    perm = rng.permutation(E)  # new label of old expert e is perm[e]
    inv = np.argsort(perm)
    ex2 = Experts([ex[inv[e]] for e in range(E)], d, I)
    assert np.array_equal(oracle.forward(x, perm[ids], w, ex2, pad=8), base)


def test_zero_token_expert_contributes_nothing_and_output_finite():
    rng = np.random.default_rng(8)
    d, I, T, k, E = 64, 32, 10, 2, 4
    ex = _rand_experts(rng, E, d, I)
    x = q.bf16_round(rng.standard_normal((T, d)) * 0.3).astype(np.float32)
    ids = rng.integers(0, E, (T, k))
    w = _softmax_rows(rng.standard_normal((T, k)))
    base = oracle.forward(x, ids, w, ex, pad=4)
    assert np.all(np.isfinite(base))
    # add an expert whose block scales are all E4M3 NaN; nobody routes to it
    poison = dict(ex[0])
    poison["w13_scales"] = np.full_like(poison["w13_scales"], 0x7F)
    poison["w2_scales"] = np.full_like(poison["w2_scales"], 0x7F)
    ex2 = Experts(list(ex.ws) + [poison], d, I)
    assert np.array_equal(oracle.forward(x, ids, w, ex2, pad=4), base)


def test_quantise_then_scatter_equals_scatter_then_quantise():
    rng = np.random.default_rng(9)
    x = q.bf16_round(rng.standard_normal((20, 64))).astype(np.float32)
    ids = rng.integers(-1, 5, (20, 3))
    rt = oracle.route(ids, 5, pad=8)
    c, s, g, amax = q.quantize(x)
    v = rt.row_src >= 0
    src = rt.row_src[v] // 3
    c2, s2, g2, _ = q.quantize(x[src], amax=amax)
    assert g2 == g
    assert np.array_equal(c[src], c2) and np.array_equal(s[src], s2)


def test_one_hot_topk_weight_selects_one_expert():
    rng = np.random.default_rng(10)
    d, I, T, k, E = 32, 32, 3, 2, 3
    ex = _rand_experts(rng, E, d, I)
    x = q.bf16_round(rng.standard_normal((T, d)) * 0.3).astype(np.float32)
    ids = np.array([[0, 1], [2, 0], [1, 2]])
    w1 = np.array([[1, 0], [1, 0], [1, 0]], np.float32)
    out, inter = oracle.forward(x, ids, w1, ex, return_intermediates=True)
    rt = inter["routing"]
    for t in range(T):
        assert np.array_equal(out[t], q.bf16_round(inter["y"][rt.slot_dst[t * k]]))


def test_accuracy_against_unquantized_moe_matches_pages_order():
    # The pages report cosine 0.988 for their NVFP4 MoE against a BF16
    # reference.  With synthetic weights the same order of agreement must hold;
    # a dropped term, a wrong sign or a transposed operand in the quantised
    # path destroys it.
    from nvfp4_block_scaled_topk_gb300 import inputs

    cfg = inputs.CONFIGS["tiny"]
    x = inputs.make_activations(cfg).float().numpy()
    ids, w = inputs.make_routing(cfg)
    ex = inputs.ExpertSet(cfg)
    out = oracle.forward(x, ids.numpy(), w.numpy(), ex, pad=32)
    ref = oracle.forward_unquantized(x, ids.numpy(), w.numpy(), ex)
    cos = float((out * ref).sum() / np.linalg.norm(out) / np.linalg.norm(ref))
    assert 0.97 < cos < 0.9999


def test_shared_expert_dense_equals_one_more_routed_expert():
    """The dense shared-expert formulation (one matrix product over all
    tokens) equals running the shared expert as expert E that every token
    visits with weight 1 through the routed machinery."""
    rng = np.random.default_rng(41)
    E, d, I, T, k = 5, 64, 128, 11, 2
    ex = _rand_experts(rng, E + 1, d, I)
    x = (rng.standard_normal((T, d)) * 0.5).astype(np.float32)
    ids = rng.integers(-1, E, (T, k))
    ids[4] = -1  # a token with no routed slot still gets the shared expert
    w = _softmax_rows(rng.standard_normal((T, k)))
    ids_x = np.concatenate([ids, np.full((T, 1), E)], 1)
    w_x = np.concatenate([w, np.ones((T, 1), np.float32)], 1)
    # as drawn, then with the shared expert's gate and up 4x larger so that
    # its h holds the amax of the intermediate (the scale both parts share)
    for boost in (1.0, 4.0):
        shared = dict(ex.ws[E], w13_gs=(ex.ws[E]["w13_gs"] / np.float32(boost)).astype(np.float32))
        full = Experts(ex.ws[:E] + [shared], d, I)
        out_d, out64_d = oracle.forward_with_shared(x, ids, w, Experts(ex.ws[:E], d, I), shared,
                                                    pad=4)
        out_x, inter = oracle.forward(x, ids_x, w_x, full, pad=4, return_intermediates=True)
        scale = np.abs(out64_d).max()
        assert np.allclose(out64_d, inter["out_f64"], rtol=0, atol=1e-12 * scale)
        assert np.array_equal(out_d, out_x)
        assert np.any(out64_d[4] != 0)
        rt = inter["routing"]
        r0, r1 = int(rt.padded_offsets[E]), int(rt.padded_offsets[E] + rt.counts[E])
        shared_amax = np.float32(np.abs(inter["h"][r0:r1]).max())
        assert (shared_amax == inter["amax_h"]) == (boost > 1)


def test_token_sample_with_the_batch_global_scales_reproduces_the_batch():
    """A token's output depends on the rest of the batch only through the two
    global scales (one per tensor): the forward over a sample of the tokens,
    given the whole batch's amax of x and of h, equals the whole batch's
    forward on those tokens (bit for bit after the bf16 rounding); measured
    over the sample alone, the
    scales (and so the outputs) differ, because the sample leaves out the
    token holding the batch's amax."""
    rng = np.random.default_rng(11)
    d, I, T, k, E = 64, 32, 16, 2, 4
    ex = _rand_experts(rng, E, d, I)
    x = q.bf16_round(rng.standard_normal((T, d)) * 0.3).astype(np.float32)
    x[5, 3] = 4.0  # the batch's amax of x sits in token 5
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    w = _softmax_rows(rng.standard_normal((T, k)))
    full, inter = oracle.forward(x, ids, w, ex, pad=8, return_intermediates=True)
    sample = np.array([0, 2, 3, 9, 14])
    sub, sub_inter = oracle.forward(x[sample], ids[sample], w[sample], ex, pad=8,
                                    return_intermediates=True, amax_x=inter["amax_x"],
                                    amax_h=inter["amax_h"])
    assert sub_inter["gs_x"] == inter["gs_x"] and sub_inter["gs_h"] == inter["gs_h"]
    assert np.array_equal(sub, full[sample])
    # float64 sums agree to BLAS blocking order
    np.testing.assert_allclose(sub_inter["out_f64"], inter["out_f64"][sample], rtol=0,
                               atol=1e-12 * np.abs(inter["out_f64"]).max())
    own = oracle.forward(x[sample], ids[sample], w[sample], ex, pad=8)
    assert not np.array_equal(own, full[sample])
