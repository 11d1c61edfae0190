"""Thin ctypes binding over the C ABI in ``include/megamoe.h``.

Argument marshalling only: torch tensors supply device pointers, torch's
current CUDA stream is passed as the stream, and every step of the forward
runs in the library's CUDA kernels.  There is no CPU or PyTorch fallback: if
the library is missing, ``load()`` raises.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmegamoe.so")

OK = 0
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported shape",
                3: "workspace too small", 4: "CUDA error", 5: "device reported an error"}
DEV_BAD_EXPERT_ID = 0x1
DEV_NONFINITE = 0x2
DEV_TIMEOUT = 0x4
SCALES_ROWMAJOR = 0
SCALES_MMA = 1
EPI_F32 = 0
EPI_SILU_MUL = 1
EPI_BF16 = 2
EPI_BFP16 = 3  # BFP16: uint16 values, then one int8 exponent per 16 rows x 8 columns

#: every function the header declares, with (restype, argtypes)
_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
SIGNATURES = {
    "megamoe_status_string": (ctypes.c_char_p, [_I]),
    "megamoe_max_padded_rows": (_I64, [_I, _I, _I, _I]),
    "megamoe_route_permute": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _I64, _P, _P, _P]),
    "megamoe_quantize_nvfp4": (_I, [_P, _I64, _I, _I64, _P, _I, _P, _P, _I64, _P, _P, _P, _P, _P,
                                    _I, _P, _P]),
    "megamoe_swizzle_scales": (_I, [_P, _I64, _I, _P, _P]),
    "megamoe_pack_weight_codes": (_I, [_P, _I64, _I, _I, _P, _P]),
    "megamoe_grouped_gemm": (_I, [_P, _P, _P, _I64, _P, _P, _P, _I, _I, _I, _P, _P, _I, _P, _I64,
                                  _P, _I, ctypes.c_double, _P, _P]),
    "megamoe_combine": (_I, [_P, _I64, _P, _P, _I, _I, _I, _P, _P]),
    "megamoe_combine_bfp16": (_I, [_P, _I64, _I64, _P, _P, _I, _I, _I, _P, _P]),
    "megamoe_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "megamoe_forward": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _SZ, _P]),
    "megamoe_read_status": (_I, [_P, _P, _P]),
    "megamoe_forward_static": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _P]),
    "megamoe_set_wait_limit_ns": (None, [ctypes.c_uint64]),
    "megamoe_set_fused_requant": (None, [_I]),
    "megamoe_linear_workspace_size": (_SZ, [_I64, _I, _I]),
    "megamoe_router_topk": (_I, [_P, _I64, _I, _I64, _P, _I, _I, _P, _P, _P]),
    "megamoe_forward_from_logits": (_I, [_P, _P, _P, _I64, _P, _I, _I, _I, _I, _I, _P, _P, _SZ,
                                         _P]),
    "megamoe_linear_nvfp4": (_I, [_P, _I64, _I, _I64, _P, _P, _P, _I, _I, _P, _I64, _P, _SZ, _P]),
    "megamoe_ep_forward_begin": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _SZ, _P]),
    "megamoe_ep_forward_end": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "megamoe_round_bf16": (_I, [_P, _I64, _P, _P]),
    "megamoe_forward_scan_stages": (_I, [_P, _I, _I, _I, _P, _P, _SZ, _P, _P]),
}
STAGE_XQ_SCALE = 0x01
STAGE_H = 0x02
STAGE_HQ_SCALE = 0x04
STAGE_Y = 0x08
STAGE_OUT = 0x10


class MegaMoEError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn}: {STATUS_NAMES.get(code, code)} ({code})")
        self.code = code


class CWeights(ctypes.Structure):
    _fields_ = [("num_experts", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("intermediate", ctypes.c_int32), ("w13_codes", _P), ("w13_scales", _P),
                ("w13_gs", _P), ("w2_codes", _P), ("w2_scales", _P), ("w2_gs", _P)]


_LIB = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the C-ABI library (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def _check(fn, code):
    if code != OK:
        raise MegaMoEError(fn, code)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _on_current_device(t, name):
    # the library launches on the current device and its stream
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, the current CUDA device is "
                         f"cuda:{torch.cuda.current_device()}")


def _dev(t, dtype, name):
    if not (t.is_cuda and t.dtype == dtype and t.is_contiguous()):
        raise TypeError(f"{name} must be a contiguous CUDA {dtype} tensor")
    _on_current_device(t, name)


def _dev_rows(t, dtype, name):
    """A CUDA matrix whose rows may be strided (unit stride along columns)."""
    if not (t.is_cuda and t.dtype == dtype and t.dim() == 2 and (t.stride(1) == 1 or t.shape[1] <= 1)):
        raise TypeError(f"{name} must be a CUDA {dtype} matrix with unit column stride")
    _on_current_device(t, name)


def max_padded_rows(T, k, E, pad):
    return int(load().megamoe_max_padded_rows(T, k, E, pad))


def workspace_size(T, k, E, d, I, pad):
    return int(load().megamoe_workspace_size(T, k, E, d, I, pad))


def set_wait_limit_ns(ns: int):
    """Bound of the grouped GEMM's pipeline waits (0 restores 4 s)."""
    load().megamoe_set_wait_limit_ns(int(ns))


def set_fused_requant(enable: bool):
    """Requantise h inside the L1 GEMM kernel (True) or in its own kernel
    after it (False, the default and the faster)."""
    load().megamoe_set_fused_requant(1 if enable else 0)


def status_string(code):
    return load().megamoe_status_string(code).decode()


# --------------------------------------------------------------------------
# the four steps and the forward
# --------------------------------------------------------------------------
def route_permute(topk_ids: torch.Tensor, E: int, pad: int = 1, status=None):
    """Bucket slots by expert; returns a dict of device int32 tensors."""
    _dev(topk_ids, torch.int32, "topk_ids")
    T, k = topk_ids.shape
    dev = topk_ids.device
    cap = max_padded_rows(T, k, E, pad)
    r = dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
             offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
             padded_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
             row_src=torch.empty(max(cap, 1), dtype=torch.int32, device=dev),
             slot_dst=torch.empty(max(T * k, 1), dtype=torch.int32, device=dev))
    _check("megamoe_route_permute", load().megamoe_route_permute(
        _p(topk_ids), T, k, E, pad, _p(r["counts"]), _p(r["offsets"]), _p(r["padded_offsets"]),
        _p(r["row_src"]), cap, _p(r["slot_dst"]), _p(status), _stream()))
    r["row_src"] = r["row_src"][:cap]
    r["slot_dst"] = r["slot_dst"][:T * k]
    return r


def router_topk(logits: torch.Tensor, k: int, bias=None, shared_expert: int = -1):
    """(topk_ids int32 [T, k_out], topk_weights float32 [T, k_out]) from fp32
    logits [T, E]: top-k of logits + bias, softmax of the selected logits,
    plus a weight-1 column of ``shared_expert`` when it is >= 0."""
    _dev(logits, torch.float32, "logits")
    T, E = logits.shape
    if logits.stride(1) != 1:
        raise ValueError("logits must have unit stride along experts")
    if bias is not None:
        _dev(bias, torch.float32, "bias")
    k_out = k + (1 if shared_expert >= 0 else 0)
    ids = torch.empty(T, k_out, dtype=torch.int32, device=logits.device)
    w = torch.empty(T, k_out, dtype=torch.float32, device=logits.device)
    _check("megamoe_router_topk", load().megamoe_router_topk(
        _p(logits), T, E, logits.stride(0), _p(bias), k, shared_expert, _p(ids), _p(w), _stream()))
    return ids, w


def sf_atom_bytes(rows, K):
    return (rows + 127) // 128 * 128 * (K // 16)


def quantize_nvfp4(x: torch.Tensor, amax_in=None, slot_dst=None, k=1, row_src=None,
                   live_rows=None, out_rows=None, scale_layout=SCALES_ROWMAJOR, status=None):
    """bf16 [rows, K] -> (codes [out_rows, K/2] u8, scales u8, amax f32[1], gs f32[1])."""
    _dev(x, torch.bfloat16, "x")
    rows, K = x.shape
    dev = x.device
    if out_rows is None:
        out_rows = rows
    codes = torch.empty(max(out_rows, 1), K // 2, dtype=torch.uint8, device=dev)
    if scale_layout == SCALES_MMA:
        scales = torch.empty(max(sf_atom_bytes(out_rows, K), 1), dtype=torch.uint8, device=dev)
    else:
        scales = torch.empty(max(out_rows, 1), K // 16, dtype=torch.uint8, device=dev)
    amax = torch.empty(1, dtype=torch.float32, device=dev)
    gs = torch.empty(1, dtype=torch.float32, device=dev)
    _check("megamoe_quantize_nvfp4", load().megamoe_quantize_nvfp4(
        _p(x), rows, K, K, _p(slot_dst), k, _p(row_src), _p(live_rows), out_rows, _p(amax_in),
        _p(amax), _p(gs), _p(codes), _p(scales), scale_layout, _p(status), _stream()))
    if scale_layout != SCALES_MMA:
        scales = scales[:out_rows]
    return codes[:out_rows], scales, amax, gs


def swizzle_scales(scales: torch.Tensor) -> torch.Tensor:
    """Row-major [rows, K/16] E4M3 bytes -> atom layout (weight preparation)."""
    _dev(scales, torch.uint8, "scales")
    rows, nb = scales.shape
    K = nb * 16
    dst = torch.empty((rows + 127) // 128 * 128 * nb, dtype=torch.uint8, device=scales.device)
    _check("megamoe_swizzle_scales",
           load().megamoe_swizzle_scales(_p(scales), rows, K, _p(dst), _stream()))
    return dst


def pack_weight_codes(codes: torch.Tensor, half_rows: int = 0) -> torch.Tensor:
    """Row-major [rows, K/2] E2M1 codes -> tile-major layout (weight preparation);
    half_rows = I pairs the gate and up blocks of W13."""
    _dev(codes, torch.uint8, "codes")
    rows, half = codes.shape
    dst = torch.empty_like(codes)
    _check("megamoe_pack_weight_codes", load().megamoe_pack_weight_codes(
        _p(codes), rows, half * 2, half_rows, _p(dst), _stream()))
    return dst


def bfp16_bytes(rows: int, ld: int) -> int:
    """Bytes of a BFP16 [rows, ld] matrix: uint16 values, then int8 exponents
    (one per 16 rows x 8 columns)."""
    return rows * ld * 2 + (rows + 15) // 16 * (ld // 8)


def grouped_gemm(act_codes, act_scales, act_gs, w_codes_packed, w_scales_mma, w_gs, offsets,
                 padded_offsets, epilogue=EPI_F32, tile_n=0, expected_tokens=0.0, out=None,
                 out_amax=None, status=None):
    """Grouped block-scaled GEMM; returns (out, out_amax).  ``w_codes_packed``
    is [E, N, K/2]-shaped in the tile-major layout of pack_weight_codes.  For
    EPI_BFP16 ``out`` is the uint8 buffer of a BFP16 [act_rows, N] matrix
    (bfp16_bytes(act_rows, N) bytes)."""
    act_rows, half_k = act_codes.shape
    E, N, _ = w_codes_packed.shape
    w_codes = w_codes_packed
    K = half_k * 2
    dev = act_codes.device
    width = N // 2 if epilogue == EPI_SILU_MUL else N
    if epilogue == EPI_BFP16:
        if out is None:  # all-ones bytes wherever nothing is written
            out = torch.full((bfp16_bytes(max(act_rows, 1), width),), 255, dtype=torch.uint8,
                             device=dev)
        if out.dtype != torch.uint8 or out.numel() < bfp16_bytes(act_rows, width):
            raise ValueError("out must be a uint8 buffer of bfp16_bytes(act_rows, N) bytes")
        ld_out = width
    else:
        dt = torch.float32 if epilogue == EPI_F32 else torch.bfloat16
        if out is None:
            out = torch.full((max(act_rows, 1), width), float("nan"), dtype=dt, device=dev)
        # the library writes act_rows rows of ld_out elements of this type
        if (out.dtype != dt or out.dim() != 2 or out.shape[0] < act_rows or out.shape[1] < width
                or out.stride(1) != 1 or out.device != dev):
            raise ValueError(f"out must be a {dt} tensor of at least [{act_rows}, {width}] "
                             "with unit column stride on the activations' device")
        ld_out = out.stride(0)
    if out_amax is None and epilogue == EPI_SILU_MUL:
        out_amax = torch.empty(1, dtype=torch.float32, device=dev)
    _check("megamoe_grouped_gemm", load().megamoe_grouped_gemm(
        _p(act_codes), _p(act_scales), _p(act_gs), act_rows, _p(w_codes), _p(w_scales_mma),
        _p(w_gs), E, N, K, _p(offsets), _p(padded_offsets), epilogue, _p(out), ld_out,
        _p(out_amax), tile_n, float(expected_tokens), _p(status), _stream()))
    if epilogue == EPI_BFP16:
        return out, out_amax
    return out[:act_rows], out_amax


@dataclass
class LinearWeights:
    """A dense NVFP4 weight [N, K] prepared for megamoe_linear_nvfp4: codes
    packed tile-major, block scales in the atom layout, global scale on the
    device."""

    N: int
    K: int
    codes: torch.Tensor
    scales: torch.Tensor  # atom layout
    gs: torch.Tensor  # [1] float32

    @classmethod
    def prepare(cls, codes: torch.Tensor, scales: torch.Tensor, gs) -> "LinearWeights":
        """From row-major codes [N, K/2], scales [N, K/16] and the global scale."""
        N, half_k = codes.shape
        gs_t = torch.as_tensor([float(gs)], dtype=torch.float32, device=codes.device)
        return cls(N, half_k * 2, pack_weight_codes(codes.contiguous()),
                   swizzle_scales(scales.contiguous()), gs_t)


def linear_workspace_size(T: int, K: int, N: int) -> int:
    return int(load().megamoe_linear_workspace_size(T, K, N))


def linear_nvfp4(x: torch.Tensor, w: LinearWeights, out_dtype=EPI_BF16, out=None, ws=None):
    """out [T, N] = NVFP4(x, gs from the measured amax of x) @ w.T, in bf16
    (EPI_BF16) or float32 (EPI_F32).  Returns (out, ws); ws holds amax, gs_x
    and the status word at bytes 0, 4 and 8."""
    _dev_rows(x, torch.bfloat16, "x")
    T, K = x.shape
    if K != w.K:
        raise ValueError("x and w disagree on K")
    need = linear_workspace_size(T, K, w.N)
    if ws is None:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    dt = torch.float32 if out_dtype == EPI_F32 else torch.bfloat16
    if out is None:
        out = torch.empty(T, w.N, dtype=dt, device=x.device)
    _dev_rows(out, dt, "out")
    _check("megamoe_linear_nvfp4", load().megamoe_linear_nvfp4(
        _p(x), T, K, x.stride(0), _p(w.codes), _p(w.scales), _p(w.gs), w.N, out_dtype, _p(out),
        out.stride(0), _p(ws), ws.numel(), _stream()))
    return out, ws


def combine(y, slot_dst, topk_weights, out=None):
    """bf16 [T, d] = sum_j w[t, j] * y[slot_dst[t*k+j]]."""
    T, k = topk_weights.shape
    d = y.shape[1]
    if out is None:
        out = torch.empty(T, d, dtype=torch.bfloat16, device=y.device)
    _check("megamoe_combine", load().megamoe_combine(
        _p(y), y.stride(0), _p(slot_dst), _p(topk_weights), T, k, d, _p(out), _stream()))
    return out


def combine_bfp16(y_buf, y_rows: int, d: int, slot_dst, topk_weights, out=None):
    """The combine over a BFP16 y [y_rows, d] held in the uint8 buffer y_buf."""
    T, k = topk_weights.shape
    if y_buf.dtype != torch.uint8 or y_buf.numel() < bfp16_bytes(y_rows, d):
        raise ValueError("y_buf must be a uint8 buffer of bfp16_bytes(y_rows, d) bytes")
    if out is None:
        out = torch.empty(T, d, dtype=torch.bfloat16, device=y_buf.device)
    _check("megamoe_combine_bfp16", load().megamoe_combine_bfp16(
        _p(y_buf), d, y_rows, _p(slot_dst), _p(topk_weights), T, k, d, _p(out), _stream()))
    return out


@dataclass
class Weights:
    """Device NVFP4 expert weights, prepared for the library (codes packed
    tile-major, scales swizzled into the atom layout)."""

    E: int
    d: int
    I: int
    w13_codes: torch.Tensor
    w13_scales: torch.Tensor  # atom layout
    w13_gs: torch.Tensor
    w2_codes: torch.Tensor
    w2_scales: torch.Tensor  # atom layout
    w2_gs: torch.Tensor

    @classmethod
    def prepare(cls, w: dict) -> "Weights":
        """From row-major stacked weights (w13_codes [E, 2I, d/2], w13_scales
        [E, 2I, d/16], w13_gs [E, 2], w2_codes [E, d, I/2], w2_scales
        [E, d, I/16], w2_gs [E]) on the GPU: swizzle the block scales once."""
        E, I2, half_d = w["w13_codes"].shape
        d, I = half_d * 2, I2 // 2
        s13 = swizzle_scales(w["w13_scales"].reshape(E * I2, d // 16))
        s2 = swizzle_scales(w["w2_scales"].reshape(E * d, I // 16))
        c13 = pack_weight_codes(w["w13_codes"].reshape(E * I2, d // 2), I).view(E, I2, d // 2)
        c2 = pack_weight_codes(w["w2_codes"].reshape(E * d, I // 2)).view(E, d, I // 2)
        return cls(E, d, I, c13, s13, w["w13_gs"].contiguous(), c2, s2,
                   w["w2_gs"].reshape(E).contiguous())

    def shard(self, first: int, count: int) -> "Weights":
        """Experts [first, first + count) as their own weight set (views: each
        expert's packed codes and atom-layout scales are contiguous)."""
        if first < 0 or count < 1 or first + count > self.E:
            raise ValueError("expert range out of bounds")
        r13 = 2 * self.I * (self.d // 16)  # scale bytes of one expert's W13
        r2 = self.d * (self.I // 16)
        return Weights(count, self.d, self.I, self.w13_codes[first:first + count],
                       self.w13_scales[first * r13:(first + count) * r13],
                       self.w13_gs[first:first + count], self.w2_codes[first:first + count],
                       self.w2_scales[first * r2:(first + count) * r2],
                       self.w2_gs[first:first + count])

    def cstruct(self) -> CWeights:
        return CWeights(self.E, self.d, self.I, self.w13_codes.data_ptr(),
                        self.w13_scales.data_ptr(), self.w13_gs.data_ptr(),
                        self.w2_codes.data_ptr(), self.w2_scales.data_ptr(),
                        self.w2_gs.data_ptr())


class Forward:
    """megamoe_forward with a reusable workspace for one (T, k, pad) shape."""

    def __init__(self, weights: Weights, T: int, k: int, pad: int = 32, device=None):
        self.w = weights
        self.cw = weights.cstruct()
        self.T, self.k, self.pad = T, k, pad
        dev = device or weights.w13_codes.device
        self.ws_bytes = workspace_size(T, k, weights.E, weights.d, weights.I, pad)
        self.ws = torch.empty(self.ws_bytes + 256, dtype=torch.uint8, device=dev)
        base = self.ws.data_ptr()
        self.ws_off = (-base) % 256
        self.out = torch.empty(max(T, 1), weights.d, dtype=torch.bfloat16, device=dev)

    @property
    def ws_ptr(self):
        return ctypes.c_void_p(self.ws.data_ptr() + self.ws_off)

    def status_tensor(self):
        return self.ws[self.ws_off:self.ws_off + 4].view(torch.int32)

    def __call__(self, x, topk_ids, topk_weights, out=None):
        _dev(x, torch.bfloat16, "x")
        _dev(topk_ids, torch.int32, "topk_ids")
        _dev(topk_weights, torch.float32, "topk_weights")
        out = self.out if out is None else out
        _check("megamoe_forward", load().megamoe_forward(
            ctypes.byref(self.cw), _p(x), _p(topk_ids), _p(topk_weights), self.T, self.k,
            self.pad, _p(out), self.ws_ptr, self.ws_bytes, _stream()))
        return out[:self.T]

    def from_logits(self, x, logits, k: int, bias=None, shared_expert: int = -1, out=None):
        """megamoe_forward_from_logits: the router (top-k of logits + bias,
        softmax of the selected logits, plus ``shared_expert`` with weight 1
        when >= 0) then the forward; this object's k must be k (+1 with a
        shared expert)."""
        _dev(x, torch.bfloat16, "x")
        _dev(logits, torch.float32, "logits")
        if bias is not None:
            _dev(bias, torch.float32, "bias")
        if self.k != k + (1 if shared_expert >= 0 else 0):
            raise ValueError("Forward was built for a different number of slots")
        out = self.out if out is None else out
        _check("megamoe_forward_from_logits", load().megamoe_forward_from_logits(
            ctypes.byref(self.cw), _p(x), _p(logits), logits.stride(0), _p(bias),
            logits.shape[1], k, shared_expert, self.T, self.pad, _p(out), self.ws_ptr,
            self.ws_bytes, _stream()))
        return out[:self.T]

    def read_status(self) -> int:
        bits = ctypes.c_uint32(0)
        code = load().megamoe_read_status(self.ws_ptr, ctypes.byref(bits), _stream())
        if code not in (OK, 5):
            raise MegaMoEError("megamoe_read_status", code)
        return int(bits.value)

    def scan_stages(self, out=None) -> int:
        """megamoe_forward_scan_stages after the last call: the STAGE_* bits of
        every stage whose valid rows hold a non-finite value (synchronises)."""
        out = self.out if out is None else out
        flags = torch.empty(1, dtype=torch.int32, device=self.ws.device)
        _check("megamoe_forward_scan_stages", load().megamoe_forward_scan_stages(
            ctypes.byref(self.cw), self.T, self.k, self.pad, _p(out), self.ws_ptr, self.ws_bytes,
            _p(flags), _stream()))
        return int(flags.item()) & 0xFFFFFFFF

    def intermediates(self):
        """Views into the workspace (for debugging and stage-level tests)."""
        return _carve_views(self.ws, self.ws_off, self.T, self.k, self.w.E, self.w.d, self.w.I,
                            self.pad)


class ShardForward:
    """The two halves of the forward on one expert-parallel shard
    (megamoe_ep_forward_begin / _end): the shard's weights hold experts
    [expert_base, expert_base + weights.E) of num_experts_total; x, ids and
    weights are the whole layer's T tokens (global ids)."""

    def __init__(self, weights: Weights, expert_base: int, num_experts_total: int, T: int, k: int,
                 pad: int = 32, device=None):
        self.w = weights
        self.cw = weights.cstruct()
        self.base, self.E_total = expert_base, num_experts_total
        self.T, self.k, self.pad = T, k, pad
        dev = device or weights.w13_codes.device
        self.ws_bytes = workspace_size(T, k, weights.E, weights.d, weights.I, pad)
        self.ws = torch.empty(self.ws_bytes + 256, dtype=torch.uint8, device=dev)
        self.ws_off = (-self.ws.data_ptr()) % 256
        self.partial = torch.empty(max(T, 1), weights.d, dtype=torch.float32, device=dev)

    @property
    def ws_ptr(self):
        return ctypes.c_void_p(self.ws.data_ptr() + self.ws_off)

    def amax_h(self) -> torch.Tensor:
        """The shard's amax(h) after begin(): a device float [1] view into the
        workspace, to be replaced by the maximum over all shards."""
        return self.ws[self.ws_off + 12:self.ws_off + 16].view(torch.float32)

    def begin(self, x, topk_ids) -> torch.Tensor:
        _dev(x, torch.bfloat16, "x")
        _dev(topk_ids, torch.int32, "topk_ids")
        _check("megamoe_ep_forward_begin", load().megamoe_ep_forward_begin(
            ctypes.byref(self.cw), _p(x), _p(topk_ids), self.T, self.k, self.base, self.E_total,
            self.pad, self.ws_ptr, self.ws_bytes, _stream()))
        return self.amax_h()

    def end(self, topk_weights) -> torch.Tensor:
        """fp32 [T, d]: this shard's share of the output, before rounding."""
        _dev(topk_weights, torch.float32, "topk_weights")
        _check("megamoe_ep_forward_end", load().megamoe_ep_forward_end(
            ctypes.byref(self.cw), _p(topk_weights), self.T, self.k, self.E_total, self.pad,
            _p(self.partial), self.ws_ptr, self.ws_bytes, _stream()))
        return self.partial[:self.T]

    def read_status(self) -> int:
        bits = ctypes.c_uint32(0)
        code = load().megamoe_read_status(self.ws_ptr, ctypes.byref(bits), _stream())
        if code not in (OK, 5):
            raise MegaMoEError("megamoe_read_status", code)
        return int(bits.value)

    def intermediates(self):
        return _carve_views(self.ws, self.ws_off, self.T, self.k, self.w.E, self.w.d, self.w.I,
                            self.pad)


def round_bf16(x: torch.Tensor, out=None) -> torch.Tensor:
    """bf16 copy of a float32 CUDA tensor (round to nearest even), by the library."""
    _dev(x, torch.float32, "x")
    if out is None:
        out = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
    _check("megamoe_round_bf16", load().megamoe_round_bf16(_p(x), x.numel(), _p(out), _stream()))
    return out


def forward_static(weights: Weights, x, topk_ids, topk_weights, pad: int = 32, out=None,
                   status_out=None):
    """megamoe_forward_static: the forward with the library's fixed internal
    workspace (no allocation by the library; for small batches)."""
    _dev(x, torch.bfloat16, "x")
    _dev(topk_ids, torch.int32, "topk_ids")
    _dev(topk_weights, torch.float32, "topk_weights")
    T, k = topk_ids.shape
    if out is None:
        out = torch.empty(max(T, 1), weights.d, dtype=torch.bfloat16, device=x.device)
    cw = weights.cstruct()
    _check("megamoe_forward_static", load().megamoe_forward_static(
        ctypes.byref(cw), _p(x), _p(topk_ids), _p(topk_weights), T, k, pad, _p(out),
        _p(status_out), _stream()))
    return out[:T]


def _carve_views(ws, off, T, k, E, d, I, pad):
    """Mirror of the workspace layout (every region 256-byte aligned)."""
    rows = max_padded_rows(T, k, E, pad)
    views = {}
    cur = off

    def take(name, nbytes):
        nonlocal cur
        views[name] = ws[cur:cur + nbytes]
        cur += -(-nbytes // 256) * 256

    take("hdr", 256)
    take("counts", 4 * E)
    take("offsets", 4 * (E + 1))
    take("padded_offsets", 4 * (E + 1))
    take("slot_dst", 4 * T * k)
    take("row_src", 4 * rows)
    take("xq_codes", rows * (d // 2))
    take("xq_sf", rows * (d // 16))
    take("h", rows * I * 2)
    take("hq_codes", rows * (I // 2))
    take("hq_sf", rows * (I // 16))
    take("y", bfp16_bytes(rows, d))  # BFP16: uint16 values, then exponents
    hdr = views.pop("hdr")
    v = {
        "status": hdr[0:4].view(torch.int32),
        "amax_x": hdr[4:8].view(torch.float32),
        "gs_x": hdr[8:12].view(torch.float32),
        "amax_h": hdr[12:16].view(torch.float32),
        "gs_h": hdr[16:20].view(torch.float32),
        "counts": views["counts"].view(torch.int32),
        "offsets": views["offsets"].view(torch.int32),
        "padded_offsets": views["padded_offsets"].view(torch.int32),
        "slot_dst": views["slot_dst"].view(torch.int32),
        "row_src": views["row_src"].view(torch.int32),
        "xq_codes": views["xq_codes"].view(rows, d // 2),
        "xq_sf": views["xq_sf"].view(rows, d // 16),
        "h": views["h"].view(torch.bfloat16).view(rows, I),
        "hq_codes": views["hq_codes"].view(rows, I // 2),
        "hq_sf": views["hq_sf"].view(rows, I // 16),
        "y": views["y"][:rows * d * 2].view(torch.int16).view(rows, d),  # uint16 bits
        "y_exp": views["y"][rows * d * 2:].view(torch.int8).view((rows + 15) // 16, d // 8),
        "y_buf": views["y"],
        "rows": rows,
    }
    return v
