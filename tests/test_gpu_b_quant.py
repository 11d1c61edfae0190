"""megamoe_quantize_nvfp4 against the oracle's quantiser: bit-exact codes,
block scales (both layouts), amax and global scale, including the routed
gather, padding rows, the requantisation mode and the E2M1/E4M3 corner
cases."""

import numpy as np
import pytest
import torch

import oracle
from oracle import nvfp4 as q
from nvfp4_block_scaled_topk_gb300 import inputs, megamoe
from helpers import bf16_tensor

pytestmark = pytest.mark.gpu


def _gpu_quant(x, layout, **kw):
    codes, scales, amax, gs = megamoe.quantize_nvfp4(x.cuda(), scale_layout=layout, **kw)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy(), amax.item(), gs.item()


def _check_plain(x):
    xf = x.float().numpy()
    wc, ws, wg, wa = q.quantize(xf)
    for layout in (megamoe.SCALES_ROWMAJOR, megamoe.SCALES_MMA):
        c, s, a, g = _gpu_quant(x, layout)
        assert np.float32(a) == wa and np.float32(g) == wg
        assert np.array_equal(c, wc)
        if layout == megamoe.SCALES_MMA:
            s = q.unswizzle_scales(s, xf.shape[0], xf.shape[1] // 16)
        assert np.array_equal(s, ws)


@pytest.mark.parametrize("name", ["tiny", "decode", "decode1", "prefill"])
def test_quant_bit_exact_on_workload_activations(cuda_lib, name):
    _check_plain(inputs.make_activations(inputs.CONFIGS[name]))


def test_quant_bit_exact_wide_dynamic_range(cuda_lib):
    # per-block magnitudes spanning 2^-40 .. 2^8: subnormal and zero block
    # scales, saturating scales, and blocks of exact zeros
    rng = np.random.default_rng(20)
    rows, K = 96, 512
    mag = np.exp2(rng.uniform(-40, 8, (rows, K // 16, 1)))
    x = rng.standard_normal((rows, K // 16, 16)) * mag
    x[5, 3] = 0.0
    x[7] = -0.0
    x = torch.from_numpy(x.reshape(rows, K).astype(np.float32)).to(torch.bfloat16)
    _check_plain(x)


def test_quant_e2m1_encoder_on_every_bf16_value_in_range(cuda_lib):
    # gs = 1 (amax 2688) and every block holds a 6, so its scale is exactly 1
    # and enc = 1: the codes are the E2M1 rounding of the raw values, which
    # here are every bf16 value in [-8, 8] plus the grid midpoints and -0.
    pos = torch.arange(0, 0x4101, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float()
    vals = torch.cat([pos, -pos, torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.0])])
    vals = vals[torch.isfinite(vals) & (vals.abs() <= 8)]
    n = vals.numel()
    per = 15
    blocks = -(-n // per)
    x = torch.zeros(blocks, 16)
    x[:, 0] = 6.0
    flat = torch.zeros(blocks * per)
    flat[:n] = vals
    x[:, 1:] = flat.view(blocks, per)
    x = x.reshape(-1, 64)
    pad_rows = torch.zeros(1, 64)
    pad_rows[0, 0] = 2688.0
    x = torch.cat([x, pad_rows]).to(torch.bfloat16)
    _check_plain(x)


@pytest.mark.parametrize("name,pad", [("tiny", 32), ("tiny", 128), ("decode", 32), ("slice", 128),
                                      ("prefill", 32)])
def test_quant_routed_gather_with_zero_padding(cuda_lib, name, pad):
    cfg = inputs.CONFIGS[name]
    x = inputs.make_activations(cfg)
    ids, _ = inputs.make_routing(cfg)
    r = megamoe.route_permute(ids.cuda(), cfg.E, pad)
    rt = oracle.route(ids.numpy(), cfg.E, pad)
    R = int(rt.padded_offsets[-1])
    cap = r["row_src"].numel()
    live = r["padded_offsets"][cfg.E:]
    c, s, a, g = _gpu_quant(x, megamoe.SCALES_MMA, slot_dst=r["slot_dst"], k=cfg.k,
                            row_src=r["row_src"], live_rows=live, out_rows=cap)
    wc, ws, wg, wa = q.quantize(x.float().numpy())
    want_c = np.zeros((R, cfg.d // 2), np.uint8)
    want_s = np.zeros((R, cfg.d // 16), np.uint8)
    v = rt.row_src >= 0
    want_c[v] = wc[rt.row_src[v] // cfg.k]
    want_s[v] = ws[rt.row_src[v] // cfg.k]
    assert np.float32(a) == wa and np.float32(g) == wg
    assert np.array_equal(c[:R], want_c)
    assert np.array_equal(q.unswizzle_scales(s, cap, cfg.d // 16)[:R], want_s)


@pytest.mark.parametrize("rows", [200, 3000])  # one and four 16-element blocks per thread
def test_requant_mode_given_amax_zeroes_padding_rows(cuda_lib, rows):
    rng = np.random.default_rng(21)
    K = 1024
    h = bf16_tensor(rng, (rows, K), 0.01)
    row_src = np.arange(rows, dtype=np.int32)
    row_src[rng.random(rows) < 0.3] = -1
    valid = row_src >= 0
    hf = h.float().numpy()
    amax = np.float32(np.abs(hf[valid]).max())
    wc, ws, wg, _ = q.quantize(hf, amax=amax)
    wc[~valid] = 0
    ws[~valid] = 0
    amax_t = torch.tensor([amax], device="cuda")
    live = torch.tensor([rows], dtype=torch.int32, device="cuda")
    for layout in (megamoe.SCALES_ROWMAJOR, megamoe.SCALES_MMA):
        c, s, a, g = _gpu_quant(h, layout, amax_in=amax_t,
                                row_src=torch.from_numpy(row_src).cuda(), live_rows=live)
        assert np.float32(g) == wg
        assert np.array_equal(c, wc)
        if layout == megamoe.SCALES_MMA:
            s = q.unswizzle_scales(s, rows, K // 16)
        assert np.array_equal(s, ws)


def test_swizzle_matches_oracle_layout(cuda_lib):
    rng = np.random.default_rng(22)
    s = rng.integers(0, 256, (300, 32), dtype=np.uint8)
    got = megamoe.swizzle_scales(torch.from_numpy(s).cuda()).cpu().numpy()
    assert np.array_equal(got, q.swizzle_scales(s))


def test_nonfinite_input_sets_status(cuda_lib):
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    x[2, 7] = float("inf")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    megamoe.quantize_nvfp4(x.cuda(), status=status)
    torch.cuda.synchronize()
    assert status.item() & megamoe.DEV_NONFINITE
