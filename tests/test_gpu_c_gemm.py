"""megamoe_grouped_gemm (tcgen05 block-scaled NVFP4) against the oracle's
float64 grouped GEMM on identical NVFP4 operands: the fp32 epilogue, the
BFP16 epilogue (the forward's storage of y; bit-exact against the model of
tests/helpers.py applied to the fp32 epilogue's output) and the fused
SiLU(gate)*up -> bf16 + amax epilogue, over every token tile, with ragged
per-expert counts, zero-token experts and several tiles per expert; the
combine over fp32 and over BFP16 y."""

import numpy as np
import pytest
import torch

import oracle
from oracle import nvfp4 as q
from helpers import (assert_close, assert_close_bf16, bf16_tensor, bfp16_decode, bfp16_encode,
                     bfp16_split, random_experts)

pytestmark = pytest.mark.gpu


def _setup(seed, E, d, I, counts, pad=32):
    rng = np.random.default_rng(seed)
    ex, stacked = random_experts(rng, E, d, I, q)
    ids = np.concatenate([np.full(c, e) for e, c in enumerate(counts)])
    rng.shuffle(ids)
    ids = ids.reshape(-1, 1)
    rt = oracle.route(ids, E, pad)
    R = int(rt.padded_offsets[-1])
    return rng, ex, stacked, rt, R


def _quantised_rows(rng, rt, R, K, scale):
    """Activations already in padded-row order, quantised by the oracle."""
    x = bf16_tensor(rng, (R, K), scale).float().numpy()
    valid = rt.row_src >= 0
    x[~valid] = 0
    c, s, g, _ = q.quantize(x)
    return x, c, s, g


def _dev_weights(stacked, which, megamoe):
    if which == "w13":
        E, N, hk = stacked["w13_codes"].shape
        codes = megamoe.pack_weight_codes(
            stacked["w13_codes"].reshape(E * N, hk).cuda(), N // 2).view(E, N, hk)
        sc = megamoe.swizzle_scales(stacked["w13_scales"].reshape(E * N, hk // 8).cuda())
        gs = stacked["w13_gs"].cuda()
    else:
        E, N, hk = stacked["w2_codes"].shape
        codes = megamoe.pack_weight_codes(
            stacked["w2_codes"].reshape(E * N, hk).cuda()).view(E, N, hk)
        sc = megamoe.swizzle_scales(stacked["w2_scales"].reshape(E * N, hk // 8).cuda())
        gs = stacked["w2_gs"].cuda()
    return codes, sc, gs


COUNTS = [37, 0, 1, 130, 64, 0, 5, 260]


# 256: token-major tiles (128 tokens x 256 weight rows)
@pytest.mark.parametrize("tile_n", [32, 64, 128, 256])
def test_grouped_gemm_f32_epilogue(cuda_lib, tile_n):
    from nvfp4_block_scaled_topk_gb300 import megamoe

    E, d, I = len(COUNTS), 512, 256  # L2 shape: N = d = 512, K = I = 256
    rng, ex, stacked, rt, R = _setup(30 + tile_n, E, d, I, COUNTS)
    a, ac, asc, ag = _quantised_rows(rng, rt, R, I, 0.5)
    wcodes, wsc, wgs = _dev_weights(stacked, "w2", megamoe)
    act_sf = torch.from_numpy(np.ascontiguousarray(asc))
    out, _ = megamoe.grouped_gemm(
        torch.from_numpy(ac).cuda(), act_sf.cuda(), torch.tensor([float(ag)], dtype=torch.float32).cuda(), wcodes, wsc, wgs,
        torch.from_numpy(rt.offsets.astype(np.int32)).cuda(),
        torch.from_numpy(rt.padded_offsets.astype(np.int32)).cuda(), megamoe.EPI_F32,
        tile_n=tile_n)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    want = oracle.grouped_gemm(ac, asc, ag, ex, "w2", rt, "f32")
    v = rt.row_src >= 0
    err, _ = assert_close(got[v], want[v], what=f"f32 tile {tile_n}")
    assert err < 1e-5  # identical operands: only fp32 accumulation differs
    assert np.all(np.isnan(got[~v]))  # padding rows untouched


def _gemm(megamoe, ac, asc, ag, wcodes, wsc, wgs, rt, epi, tile_n):
    out, amax = megamoe.grouped_gemm(
        torch.from_numpy(ac).cuda(), torch.from_numpy(np.ascontiguousarray(asc)).cuda(),
        torch.tensor([float(ag)], dtype=torch.float32).cuda(), wcodes, wsc, wgs,
        torch.from_numpy(rt.offsets.astype(np.int32)).cuda(),
        torch.from_numpy(rt.padded_offsets.astype(np.int32)).cuda(), epi, tile_n=tile_n)
    torch.cuda.synchronize()
    return out, amax


def _check_bfp16(buf, f32_out, rt, R, n, want64, what):
    """A BFP16 output against the model's encoding of the fp32 epilogue's
    output on the same operands (bit-exact), untouched padding rows, and the
    decoded values against the oracle."""
    qv, sv = bfp16_split(buf, R, n)
    v = rt.row_src >= 0
    g = v[::16]  # 16-row groups holding valid rows (they come first in an expert)
    q_want, s_want = bfp16_encode(f32_out, v)
    assert np.array_equal(sv[g], s_want[g]), what
    assert np.array_equal(qv[v], q_want[v]), what
    assert np.all(qv[~v] == 0xFFFF) and np.all(sv[~g] == -1), what  # 0xFF fill untouched
    assert_close(bfp16_decode(qv, sv)[v], want64[v], what=what)


@pytest.mark.parametrize("tile_n", [32, 64, 128, 256])
def test_grouped_gemm_bfp16_epilogue(cuda_lib, tile_n):
    """EPI_BFP16: the bytes are the BFP16 encoding of the fp32 epilogue's
    values (the same fp32 accumulators times alpha) at the same weights-on-M
    tile (tile 256 runs as 128)."""
    from nvfp4_block_scaled_topk_gb300 import megamoe

    E, d, I = len(COUNTS), 512, 256
    rng, ex, stacked, rt, R = _setup(130 + tile_n, E, d, I, COUNTS)
    a, ac, asc, ag = _quantised_rows(rng, rt, R, I, 0.5)
    wcodes, wsc, wgs = _dev_weights(stacked, "w2", megamoe)
    f32, _ = _gemm(megamoe, ac, asc, ag, wcodes, wsc, wgs, rt, megamoe.EPI_F32, min(tile_n, 128))
    buf, _ = _gemm(megamoe, ac, asc, ag, wcodes, wsc, wgs, rt, megamoe.EPI_BFP16, tile_n)
    want = oracle.grouped_gemm(ac, asc, ag, ex, "w2", rt, "f32")
    _check_bfp16(buf, f32.cpu().numpy(), rt, R, d, want, f"bfp16 tile {tile_n}")


@pytest.mark.parametrize("tile_n", [32, 64, 128, 256])
def test_grouped_gemm_silu_mul_epilogue(cuda_lib, tile_n):
    from nvfp4_block_scaled_topk_gb300 import megamoe

    E, d, I = len(COUNTS), 512, 256  # L1 shape: N = 2I = 512, K = d = 512
    rng, ex, stacked, rt, R = _setup(40 + tile_n, E, d, I, COUNTS)
    a, ac, asc, ag = _quantised_rows(rng, rt, R, d, 0.5)
    wcodes, wsc, wgs = _dev_weights(stacked, "w13", megamoe)
    act_sf = torch.from_numpy(np.ascontiguousarray(asc))
    out, amax = megamoe.grouped_gemm(
        torch.from_numpy(ac).cuda(), act_sf.cuda(), torch.tensor([float(ag)], dtype=torch.float32).cuda(), wcodes, wsc, wgs,
        torch.from_numpy(rt.offsets.astype(np.int32)).cuda(),
        torch.from_numpy(rt.padded_offsets.astype(np.int32)).cuda(), megamoe.EPI_SILU_MUL,
        tile_n=tile_n)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    want, want_amax = oracle.grouped_gemm(ac, asc, ag, ex, "w13", rt, "silu_mul")
    gu = oracle.grouped_gemm(ac, asc, ag, ex, "w13", rt, "f32")
    v = rt.row_src >= 0
    h64 = oracle.silu(gu[v][:, :I]) * gu[v][:, I:]
    assert_close_bf16(got[v], h64, what=f"silu tile {tile_n}")
    # bf16 outputs: all but a few rounding-boundary cases are identical
    assert np.mean(got[v] == want[v]) > 0.99
    assert abs(amax.item() - float(want_amax)) <= 2 ** -7 * float(want_amax)


def test_grouped_gemm_real_shape_one_expert_per_token(cuda_lib):
    """d = 7168, I = 2048 (the MegaMoE expert shape) with decode-like counts."""
    from nvfp4_block_scaled_topk_gb300 import megamoe

    E, d, I = 3, 7168, 2048
    counts = [1, 0, 3]
    rng, ex, stacked, rt, R = _setup(50, E, d, I, counts)
    a, ac, asc, ag = _quantised_rows(rng, rt, R, d, 0.09)
    wcodes, wsc, wgs = _dev_weights(stacked, "w13", megamoe)
    act_sf = torch.from_numpy(np.ascontiguousarray(asc))
    out, amax = megamoe.grouped_gemm(
        torch.from_numpy(ac).cuda(), act_sf.cuda(), torch.tensor([float(ag)], dtype=torch.float32).cuda(), wcodes, wsc, wgs,
        torch.from_numpy(rt.offsets.astype(np.int32)).cuda(),
        torch.from_numpy(rt.padded_offsets.astype(np.int32)).cuda(), megamoe.EPI_SILU_MUL,
        tile_n=32)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    gu = oracle.grouped_gemm(ac, asc, ag, ex, "w13", rt, "f32")
    v = rt.row_src >= 0
    h64 = oracle.silu(gu[v][:, :I]) * gu[v][:, I:]
    assert_close_bf16(got[v], h64, what="real shape")


@pytest.mark.parametrize("T,k,d", [(64, 2, 256), (8, 6, 7168), (333, 6, 1024)])
def test_combine_matches_oracle(cuda_lib, T, k, d):
    from nvfp4_block_scaled_topk_gb300 import megamoe

    rng = np.random.default_rng(60 + T)
    rows = T * k + 40
    y = (rng.standard_normal((rows, d)) * 0.03).astype(np.float32)
    slot_dst = rng.permutation(rows)[:T * k].astype(np.int32)
    slot_dst[rng.random(T * k) < 0.1] = -1  # skipped slots
    w = rng.random((T, k)).astype(np.float32)
    out = megamoe.combine(torch.from_numpy(y).cuda(), torch.from_numpy(slot_dst).cuda(),
                          torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    want64 = oracle.combine(y.astype(np.float64), w, slot_dst, round_bf16=False)
    assert_close_bf16(out.float().cpu().numpy(), want64, what="combine")


@pytest.mark.parametrize("T,k,d", [(64, 2, 256), (8, 6, 7168), (333, 6, 1024)])
def test_combine_bfp16_matches_oracle(cuda_lib, T, k, d):
    """The combine over a BFP16 y: each element decoded exactly, so against
    the oracle's combine of the decoded values; huge groups; a group holding
    NaN or Inf (exponent 127) passes its values through to the output."""
    from nvfp4_block_scaled_topk_gb300 import megamoe

    rng = np.random.default_rng(160 + T)
    rows = (T * k + 40 + 15) // 16 * 16
    y = (rng.standard_normal((rows, d)) * np.exp(rng.uniform(-8, 8, (rows, 1)))).astype(np.float32)
    slot_dst = rng.permutation(rows)[:T * k].astype(np.int32)
    slot_dst[rng.random(T * k) < 0.1] = -1  # skipped slots
    w = rng.random((T, k)).astype(np.float32)
    qv, sv = bfp16_encode(y)
    buf = np.concatenate([qv.reshape(-1).view(np.uint8), sv.reshape(-1).view(np.uint8)])
    out = megamoe.combine_bfp16(torch.from_numpy(buf).cuda(), rows, d,
                                torch.from_numpy(slot_dst).cuda(), torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    assert (sv != 0).any() and (np.diff(sv, axis=0) != 0).any()  # exponents vary by group
    want64 = oracle.combine(bfp16_decode(qv, sv), w, slot_dst, round_bf16=False)
    assert_close_bf16(out.float().cpu().numpy(), want64, what="combine bfp16")
    # groups of huge values (exponents 100 and above take the general decode)
    yh = y.copy()
    yh[:16] = (rng.standard_normal((16, d)) * 2.0 ** 115).astype(np.float32)
    qh, sh = bfp16_encode(yh)
    assert sh[0].min() >= 100
    buf = np.concatenate([qh.reshape(-1).view(np.uint8), sh.reshape(-1).view(np.uint8)])
    out = megamoe.combine_bfp16(torch.from_numpy(buf).cuda(), rows, d,
                                torch.from_numpy(slot_dst).cuda(), torch.from_numpy(w).cuda())
    want64 = oracle.combine(bfp16_decode(qh, sh), w, slot_dst, round_bf16=False)
    huge = np.isin(slot_dst.reshape(T, k), np.arange(16)).any(axis=1)
    assert huge.any()
    assert_close_bf16(out.float().cpu().numpy()[huge], want64[huge], what="combine bfp16 huge")
    # slot indices at or past y_rows are skipped like -1 (not read)
    far = slot_dst.copy()
    far[::3] = np.where(far[::3] >= 0, rows + far[::3], far[::3])
    near = np.where(far >= rows, -1, far).astype(np.int32)
    out = megamoe.combine_bfp16(torch.from_numpy(buf).cuda(), rows, d,
                                torch.from_numpy(far).cuda(), torch.from_numpy(w).cuda())
    want64 = oracle.combine(bfp16_decode(qh, sh), w, near, round_bf16=False)
    small = ~np.isin(near.reshape(T, k), np.arange(16)).any(axis=1)
    assert_close_bf16(out.float().cpu().numpy()[small], want64[small], what="combine bfp16 far")
    # a NaN in one group of one routed row reaches exactly that token's group
    t = int(np.nonzero((slot_dst.reshape(T, k) >= 0).any(axis=1))[0][0])
    j = int(np.nonzero(slot_dst.reshape(T, k)[t] >= 0)[0][0])
    r = int(slot_dst[t * k + j])
    y[r, 33] = np.nan
    qv, sv = bfp16_encode(y)
    assert sv[r // 16, 33 // 8] == 127
    buf = np.concatenate([qv.reshape(-1).view(np.uint8), sv.reshape(-1).view(np.uint8)])
    out = megamoe.combine_bfp16(torch.from_numpy(buf).cuda(), rows, d,
                                torch.from_numpy(slot_dst).cuda(),
                                torch.from_numpy(w).cuda()).float().cpu().numpy()
    bad = np.isnan(out)
    assert bad[t, 33] and bad.sum() == 1


def test_pack_weight_codes_layout(cuda_lib):
    from nvfp4_block_scaled_topk_gb300 import megamoe

    rng = np.random.default_rng(70)
    rows, K = 512, 768
    c = rng.integers(0, 256, (rows, K // 2), dtype=np.uint8)
    got = megamoe.pack_weight_codes(torch.from_numpy(c).cuda()).cpu().numpy().reshape(-1)
    # 128-byte swizzle inside a block: 16-byte chunk j of row i lands at j ^ (i % 8)
    i = np.arange(128)[:, None]
    j = np.arange(8)[None, :]
    src_chunk = j ^ (i % 8)  # the chunk stored at position j of row i

    def swz(blocks):  # [..., 128 rows, 128 bytes] -> swizzled
        ch = blocks.reshape(blocks.shape[:-1] + (8, 16))
        return np.take_along_axis(ch, np.broadcast_to(src_chunk[..., None], ch.shape), -2
                                  ).reshape(blocks.shape)

    # blocks of 128 rows x 128 bytes, ordered [rows/128][K/256]
    want = swz(c.reshape(rows // 128, 128, K // 256, 128).transpose(0, 2, 1, 3)).reshape(-1)
    assert np.array_equal(got, want)
    # a hand-checked byte: row 3, chunk 1 of block (0, 0) sits at chunk 1 ^ 3 = 2
    assert np.array_equal(got[3 * 128 + 2 * 16: 3 * 128 + 3 * 16], c[3, 16:32])
    # gate/up pairing: groups of 2H rows, [group][H/128][K/256][gate, up]
    H = 128
    got = megamoe.pack_weight_codes(torch.from_numpy(c).cuda(), H).cpu().numpy().reshape(-1)
    want = swz(c.reshape(rows // (2 * H), 2, H // 128, 128, K // 256, 128)
               .transpose(0, 2, 4, 1, 3, 5)).reshape(-1)
    assert np.array_equal(got, want)


def _hist_experts(E, d, I, seed):
    """Experts drawn like the workloads' (NVFP4 bytes from the fixed
    histograms), with edge blocks planted in every matrix: all-zero block
    scales (0x00), subnormal block scales (0x01..0x07), and blocks holding
    the largest codes (+-6).  Returns (NumpyExperts, stacked torch dict)."""
    from nvfp4_block_scaled_topk_gb300 import inputs
    from helpers import NumpyExperts

    cfg = inputs.MoEConfig("gemm_edges", E, 1, d, I, 1, "uniform", seed=seed)
    rng = np.random.default_rng(seed)
    ws = []
    for e in range(E):
        w = {k: v.numpy().copy() for k, v in inputs.make_expert(cfg, e).items()}
        for cname, sname in (("w13_codes", "w13_scales"), ("w2_codes", "w2_scales")):
            sc, co = w[sname], w[cname]
            n = sc.size // 50
            flat = rng.choice(sc.size, size=3 * n, replace=False)
            sc.reshape(-1)[flat[:n]] = 0
            sc.reshape(-1)[flat[n:2 * n]] = rng.integers(1, 8, size=n)
            rows, blk = np.unravel_index(flat[2 * n:], sc.shape)
            for r, b in zip(rows, blk):
                co[r, 8 * b:8 * b + 8] = rng.choice([0x77, 0xFF, 0x7F, 0xF7], size=8)
        w["w2_gs"] = np.float32(w["w2_gs"][0])
        ws.append(w)
    stacked = dict(
        w13_codes=torch.from_numpy(np.stack([w["w13_codes"] for w in ws])),
        w13_scales=torch.from_numpy(np.stack([w["w13_scales"] for w in ws])),
        w13_gs=torch.from_numpy(np.stack([w["w13_gs"] for w in ws])),
        w2_codes=torch.from_numpy(np.stack([w["w2_codes"] for w in ws])),
        w2_scales=torch.from_numpy(np.stack([w["w2_scales"] for w in ws])),
        w2_gs=torch.from_numpy(np.array([w["w2_gs"] for w in ws], np.float32)),
    )
    return NumpyExperts(ws, d, I), stacked


def _edge_rows(rng, rt, R, K):
    """Token rows (padded-row order) ~ N(0, 0.09) with one outlier at 8 and,
    in some rows, an all-zero block and a block small enough (1e-4) for a
    subnormal block scale; quantised by the oracle."""
    x = bf16_tensor(rng, (R, K), 0.09).float().numpy()
    valid = np.nonzero(rt.row_src >= 0)[0]
    x[valid[0], 5] = 8.0
    for r in valid[::7]:
        b = rng.integers(0, K // 16, size=2)
        x[r, 16 * b[0]:16 * b[0] + 16] = 0.0
        x[r, 16 * b[1]:16 * b[1] + 16] = bf16_tensor(rng, (16,), 1e-4).float().numpy()
    x[rt.row_src < 0] = 0
    c, s, g, _ = q.quantize(x)
    assert (s[valid] == 0).any() and ((s[valid] > 0) & (s[valid] < 8)).any()
    return c, s, g


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("which", ["w13", "w2"])
def test_grouped_gemm_real_shape_prefill_tiles(cuda_lib, which, tile_n):
    """The prefill path's GEMM configurations: token tiles of 128, and
    token-major tiles (128 tokens x 256 weight rows), at the MegaMoE shapes
    (L1: K = 7168, 28 K steps; L2: K = 2048, 8 K steps, so the stage ring
    wraps many times), experts holding several, one and no token tiles with
    ragged tails, and edge blocks in weights and activations."""
    from nvfp4_block_scaled_topk_gb300 import megamoe

    E, d, I = 4, 7168, 2048
    counts = [300, 0, 129, 1]
    rng = np.random.default_rng(90)
    ex, stacked = _hist_experts(E, d, I, seed=91)
    ids = np.concatenate([np.full(c, e) for e, c in enumerate(counts)])
    rng.shuffle(ids)
    rt = oracle.route(ids.reshape(-1, 1), E, 32)
    R = int(rt.padded_offsets[-1])
    K = d if which == "w13" else I
    ac, asc, ag = _edge_rows(rng, rt, R, K)
    wcodes, wsc, wgs = _dev_weights(stacked, which, megamoe)
    if which == "w2":
        wgs = wgs.view(-1, 1)
    epi = megamoe.EPI_SILU_MUL if which == "w13" else megamoe.EPI_F32
    out, amax = megamoe.grouped_gemm(
        torch.from_numpy(ac).cuda(), torch.from_numpy(np.ascontiguousarray(asc)).cuda(),
        torch.tensor([float(ag)], dtype=torch.float32).cuda(), wcodes, wsc, wgs,
        torch.from_numpy(rt.offsets.astype(np.int32)).cuda(),
        torch.from_numpy(rt.padded_offsets.astype(np.int32)).cuda(), epi, tile_n=tile_n)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    v = rt.row_src >= 0
    if which == "w13":
        gu = oracle.grouped_gemm(ac, asc, ag, ex, "w13", rt, "f32")
        h64 = oracle.silu(gu[v][:, :I]) * gu[v][:, I:]
        assert_close_bf16(got[v], h64, what=f"L1 tile {tile_n}")
        want_h, want_amax = oracle.grouped_gemm(ac, asc, ag, ex, "w13", rt, "silu_mul")
        assert np.mean(got[v] == want_h[v]) > 0.99
        assert abs(amax.item() - float(want_amax)) <= 2 ** -7 * float(want_amax)
    else:
        want = oracle.grouped_gemm(ac, asc, ag, ex, "w2", rt, "f32")
        err, _ = assert_close(got[v], want[v], what=f"L2 tile {tile_n}")
        assert err < 1e-5  # identical operands: only fp32 accumulation differs
        assert np.all(np.isnan(got[~v]))  # padding rows untouched
        if tile_n == 128:  # the forward's L2: BFP16 of the same values
            buf, _ = _gemm(megamoe, ac, asc, ag, wcodes, wsc, wgs, rt, megamoe.EPI_BFP16, 128)
            _check_bfp16(buf, out.cpu().numpy(), rt, R, d, want, "L2 bfp16 tile 128")
