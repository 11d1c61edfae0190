"""The C-ABI library loads, exports what include/megamoe.h declares, and its
host-side logic (size helpers, argument checks) behaves, all without a GPU."""

import ctypes
import os
import re

import pytest

import __graft_entry__
from nvfp4_block_scaled_topk_gb300 import megamoe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return megamoe.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "megamoe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(megamoe_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary_calls():
    names = _declared_functions()
    for n in ("megamoe_route_permute", "megamoe_quantize_nvfp4", "megamoe_grouped_gemm",
              "megamoe_forward", "megamoe_workspace_size", "megamoe_read_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert names == sorted(megamoe.SIGNATURES)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert megamoe.status_string(0) == "ok"
    assert megamoe.status_string(3) == "workspace too small"
    assert megamoe.status_string(99) == "unknown status"


def test_max_padded_rows(lib):
    assert megamoe.max_padded_rows(8, 6, 384, 32) == 48 + 48 * 31
    assert megamoe.max_padded_rows(4096, 6, 384, 32) == 24576 + 384 * 31
    assert megamoe.max_padded_rows(0, 6, 384, 128) == 0
    assert megamoe.max_padded_rows(1, 6, 48, 1) == 6
    assert megamoe.max_padded_rows(-1, 6, 48, 1) == 0


def test_workspace_size_is_aligned_and_monotone(lib):
    a = megamoe.workspace_size(8, 6, 384, 7168, 2048, 32)
    b = megamoe.workspace_size(16, 6, 384, 7168, 2048, 32)
    assert a > 0 and a % 256 == 0 and b > a
    assert megamoe.workspace_size(8, 0, 384, 7168, 2048, 32) == 0


def test_argument_errors_return_before_any_device_work(lib):
    P = None
    # route: E = 0, E too large, k too large, capacity too small
    assert lib.megamoe_route_permute(P, 1, 1, 0, 1, P, P, P, P, 0, P, P, P) == 1
    assert lib.megamoe_route_permute(P, 1, 1, 2000, 1, P, P, P, P, 0, P, P, P) == 2
    assert lib.megamoe_route_permute(P, 1, 17, 8, 1, P, P, P, P, 0, P, P, P) == 2
    # padded rows beyond int32: 2^24 slots + 1024 experts padded to 2^21
    assert megamoe.max_padded_rows(1 << 20, 16, 1024, 1 << 21) >= 1 << 31
    assert lib.megamoe_route_permute(P, 1 << 20, 16, 1024, 1 << 21, P, P, P, P, 0, P, P,
                                     P) == 2
    fake = ctypes.c_void_p(256)
    assert lib.megamoe_route_permute(fake, 4, 2, 8, 32, fake, fake, fake, fake, 10, fake, P,
                                     P) == 1
    # quantise: K not a multiple of 64, bad layout, missing gs
    assert lib.megamoe_quantize_nvfp4(fake, 4, 48, 48, P, 1, P, P, 4, P, fake, fake, fake, fake,
                                      0, P, P) == 2
    assert lib.megamoe_quantize_nvfp4(fake, 4, 64, 64, P, 1, P, P, 4, P, fake, fake, fake, fake,
                                      7, P, P) == 1
    assert lib.megamoe_quantize_nvfp4(fake, 4, 64, 64, P, 1, P, P, 4, P, fake, P, fake, fake,
                                      0, P, P) == 1
    # grouped GEMM: bad epilogue, K not a multiple of 256, bad tile
    assert lib.megamoe_grouped_gemm(fake, fake, fake, 8, fake, fake, fake, 2, 256, 256, fake,
                                    fake, 9, fake, 256, P, 0, 0.0, P, P) == 1
    assert lib.megamoe_grouped_gemm(fake, fake, fake, 8, fake, fake, fake, 2, 256, 128, fake,
                                    fake, 0, fake, 256, P, 0, 0.0, P, P) == 2
    assert lib.megamoe_grouped_gemm(fake, fake, fake, 8, fake, fake, fake, 2, 256, 256, fake,
                                    fake, 0, fake, 256, P, 48, 0.0, P, P) == 1
    # combine: d not a multiple of 4; BFP16 combine: d not a multiple of 32, y_rows < 0
    assert lib.megamoe_combine(fake, 6, fake, fake, 2, 2, 6, fake, P) == 2
    assert lib.megamoe_combine_bfp16(fake, 48, 8, fake, fake, 2, 2, 48, fake, P) == 2
    assert lib.megamoe_combine_bfp16(fake, 64, -1, fake, fake, 2, 2, 64, fake, P) == 1
    # forward: no weights; pad not a multiple of 32; workspace too small
    assert lib.megamoe_forward(P, fake, fake, fake, 1, 1, 32, fake, fake, 1 << 30, P) == 1
    w = megamoe.CWeights(8, 256, 512, 256, 256, 256, 256, 256, 256)
    assert lib.megamoe_forward(ctypes.byref(w), fake, fake, fake, 4, 2, 16, fake, fake,
                               1 << 30, P) == 2
    assert lib.megamoe_forward(ctypes.byref(w), fake, fake, fake, 4, 2, 32, fake, fake, 16,
                               P) == 3
    w_bad = megamoe.CWeights(8, 200, 512, 256, 256, 256, 256, 256, 256)
    assert lib.megamoe_forward(ctypes.byref(w_bad), fake, fake, fake, 4, 2, 32, fake, fake,
                               1 << 30, P) == 2


def test_argument_errors_of_the_router_linear_and_layer_calls(lib):
    P = None
    fake = ctypes.c_void_p(256)
    # router: k = 0, k > E, ld < E, E too large
    assert lib.megamoe_router_topk(fake, 4, 8, 8, P, 0, -1, fake, fake, P) == 1
    assert lib.megamoe_router_topk(fake, 4, 8, 8, P, 9, -1, fake, fake, P) == 1
    assert lib.megamoe_router_topk(fake, 4, 8, 4, P, 2, -1, fake, fake, P) == 1
    assert lib.megamoe_router_topk(fake, 4, 2000, 2000, P, 2, -1, fake, fake, P) == 2
    # dense linear: K not a multiple of 256, N not a multiple of 128, bad
    # output type, short workspace
    ws = lib.megamoe_linear_workspace_size(8, 512, 256)
    assert ws > 0
    assert lib.megamoe_linear_nvfp4(fake, 8, 128, 128, fake, fake, fake, 256, 2, fake, 256, fake,
                                    1 << 30, P) == 2
    assert lib.megamoe_linear_nvfp4(fake, 8, 512, 512, fake, fake, fake, 200, 2, fake, 256, fake,
                                    1 << 30, P) == 2
    assert lib.megamoe_linear_nvfp4(fake, 8, 512, 512, fake, fake, fake, 256, 1, fake, 256, fake,
                                    1 << 30, P) == 1
    assert lib.megamoe_linear_nvfp4(fake, 8, 512, 512, fake, fake, fake, 256, 2, fake, 256, fake,
                                    ws - 1, P) == 3
    # layer from logits: shared expert inside the routed range or beyond the
    # weights, more logits than experts, k_out above 16
    w = megamoe.CWeights(9, 256, 512, 256, 256, 256, 256, 256, 256)
    assert lib.megamoe_forward_from_logits(ctypes.byref(w), fake, fake, 8, P, 8, 2, 3, 4, 32,
                                           fake, fake, 1 << 30, P) == 1
    assert lib.megamoe_forward_from_logits(ctypes.byref(w), fake, fake, 8, P, 8, 2, 9, 4, 32,
                                           fake, fake, 1 << 30, P) == 1
    assert lib.megamoe_forward_from_logits(ctypes.byref(w), fake, fake, 10, P, 10, 2, -1, 4, 32,
                                           fake, fake, 1 << 30, P) == 1
    w16 = megamoe.CWeights(40, 256, 512, 256, 256, 256, 256, 256, 256)
    assert lib.megamoe_forward_from_logits(ctypes.byref(w16), fake, fake, 32, P, 32, 16, 33, 4,
                                           32, fake, fake, 1 << 30, P) == 2


def test_missing_library_fails_loudly(monkeypatch):
    # no CPU or PyTorch fallback: without the built library every call raises
    monkeypatch.setattr(megamoe, "_LIB", None)
    missing = os.path.join(ROOT, "nvfp4_block_scaled_topk_gb300", "no_such_libmegamoe.so")
    with pytest.raises(RuntimeError, match="missing"):
        megamoe.load(missing)
    monkeypatch.setattr(megamoe, "LIB_PATH", missing)
    monkeypatch.setattr(megamoe.load, "__defaults__", (missing,))
    with pytest.raises(RuntimeError, match="missing"):
        megamoe.max_padded_rows(8, 6, 384, 32)


def _c_to_ctypes(decl):
    """ctypes type of one C parameter or return type of the header."""
    import ctypes as C

    t = " ".join(decl.replace("*", " * ").split())
    if "*" in t:
        return C.c_char_p if t == "const char *" else C.c_void_p
    t = t.replace("const ", "")
    table = {"int": C.c_int, "int32_t": C.c_int32, "int64_t": C.c_int64, "size_t": C.c_size_t,
             "double": C.c_double, "uint64_t": C.c_uint64, "megamoe_status": C.c_int,
             "megamoe_stream_t": C.c_void_p, "void": None}
    return table[t]


def test_binding_signatures_match_the_header_types():
    src = open(os.path.join(ROOT, "include", "megamoe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    protos = re.findall(r"([A-Za-z_][\w\s\*]*?)\s*\b(megamoe_[a-z_0-9]+)\s*\(([^)]*)\)\s*;", src)
    assert len(protos) == len(megamoe.SIGNATURES)
    for ret, name, params in protos:
        ret = ret.split("\n")[-1].strip()
        want_args = []
        for p in params.split(","):
            p = " ".join(p.split())
            if p in ("", "void"):
                continue
            typ = re.sub(r"\b[A-Za-z_]\w*$", "", p).strip()  # drop the parameter name
            want_args.append(_c_to_ctypes(typ))
        res, args = megamoe.SIGNATURES[name]
        assert res == _c_to_ctypes(ret), (name, ret)
        assert args == want_args, name


def test_weights_struct_matches_the_header():
    src = open(os.path.join(ROOT, "include", "megamoe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    body = re.search(r"typedef struct megamoe_weights\s*\{(.*?)\}\s*megamoe_weights;", src, re.S).group(1)
    fields = []
    for decl in body.split(";"):
        decl = " ".join(decl.split())
        if not decl:
            continue
        name = re.search(r"([A-Za-z_]\w*)$", decl).group(1)
        fields.append((name, _c_to_ctypes(decl[: -len(name)])))
    got = [(n, t) for n, t in megamoe.CWeights._fields_]
    assert got == fields


@pytest.mark.parametrize("T,k,E,d,I,pad", [(8, 6, 384, 7168, 2048, 32), (64, 2, 8, 256, 512, 128),
                                           (1, 1, 1, 256, 256, 32), (4096, 6, 384, 7168, 2048, 32)])
def test_stage_views_mirror_the_workspace_layout(lib, T, k, E, d, I, pad):
    """The binding's views of the forward's stages lie where the library
    carves them: the same regions in the same order and sizes, each 256-byte
    aligned, and the library's size is those regions plus its two
    router-output regions (no split-K planes unless asked for) and, from
    16384 slots on, the multi-block routing's per-block histograms (256
    blocks x E ints)."""
    import torch

    size = megamoe.workspace_size(T, k, E, d, I, pad)
    ws = torch.empty(size, dtype=torch.uint8, device="meta")
    v = megamoe._carve_views(ws, 0, T, k, E, d, I, pad)
    rows = megamoe.max_padded_rows(T, k, E, pad)
    regions = [("counts", 4 * E), ("offsets", 4 * (E + 1)), ("padded_offsets", 4 * (E + 1)),
               ("slot_dst", 4 * T * k), ("row_src", 4 * rows), ("xq_codes", rows * d // 2),
               ("xq_sf", rows * d // 16), ("h", rows * I * 2), ("hq_codes", rows * I // 2),
               ("hq_sf", rows * I // 16), ("y_buf", rows * d * 2 + (rows + 15) // 16 * (d // 8))]
    a256 = lambda n: -(-n // 256) * 256
    off = 256  # the status word and the scalars
    for name, nbytes in regions:
        t = v[name]
        assert t.storage_offset() * t.element_size() == off, name
        assert t.numel() * t.element_size() == nbytes, name
        if name == "y_buf":  # BFP16: the uint16 values, then one exponent per 16 x 8
            y, ye = v["y"], v["y_exp"]
            assert y.storage_offset() * 2 == off and tuple(y.shape) == (rows, d)
            assert ye.storage_offset() == off + rows * d * 2
            assert tuple(ye.shape) == ((rows + 15) // 16, d // 8)
        off = a256(off + nbytes)
    hist = 4 * 256 * E if T * k >= 16384 else 0
    assert size == off + 2 * a256(4 * T * k) + a256(hist)


def test_plain_c_program_compiles_links_and_calls_the_host_helpers(lib):
    """The boundary is plain C: a C99 program includes the header, links
    against the library, references every declared call and runs the
    host-only helpers and an argument check (no device work)."""
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = _declared_functions()
    refs = ",\n    ".join(f"(void (*)(void)){n}" for n in names)
    prog = f"""
#include <stdio.h>
#include <string.h>
#include "megamoe.h"
static void (*const every_call[])(void) = {{
    {refs}
}};
int main(void) {{
  size_t i;
  for (i = 0; i < sizeof every_call / sizeof every_call[0]; ++i)
    if (!every_call[i]) return 10;
  if (megamoe_max_padded_rows(8, 6, 384, 32) != 48 + 48 * 31) return 1;
  if (megamoe_workspace_size(8, 6, 384, 7168, 2048, 32) % 256 != 0) return 2;
  if (strcmp(megamoe_status_string(MEGAMOE_ERR_WORKSPACE_TOO_SMALL), "workspace too small"))
    return 3;
  if (megamoe_route_permute(NULL, 1, 1, 0, 1, NULL, NULL, NULL, NULL, 0, NULL, NULL, NULL) !=
      MEGAMOE_ERR_INVALID_ARG)
    return 4;
  puts("ok");
  return 0;
}}
"""
    out_dir = os.path.join(ROOT, "_build", "c_consumer")
    os.makedirs(out_dir, exist_ok=True)
    src = os.path.join(out_dir, "consumer.c")
    exe = os.path.join(out_dir, "consumer")
    with open(src, "w") as f:
        f.write(prog)
    libdir = os.path.dirname(megamoe.LIB_PATH)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I",
                        os.path.join(ROOT, "include"), src, "-o", exe, "-L", libdir, "-lmegamoe",
                        f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)


def test_alignment_errors_return_before_any_device_work(lib):
    P = None
    a16 = ctypes.c_void_p(4096)
    odd = ctypes.c_void_p(4096 + 4)  # 4-byte but not 16-byte aligned
    # quantise: ld not a multiple of 8; x or codes misaligned
    assert lib.megamoe_quantize_nvfp4(a16, 4, 64, 68, P, 1, P, P, 4, P, a16, a16, a16, a16,
                                      0, P, P) == 2
    assert lib.megamoe_quantize_nvfp4(odd, 4, 64, 64, P, 1, P, P, 4, P, a16, a16, a16, a16,
                                      0, P, P) == 2
    assert lib.megamoe_quantize_nvfp4(a16, 4, 64, 64, P, 1, P, P, 4, P, a16, a16, odd, a16,
                                      0, P, P) == 2
    # combine: y misaligned
    assert lib.megamoe_combine(odd, 8, a16, a16, 2, 2, 8, a16, P) == 2
    # grouped GEMM: output rows not on 16-byte boundaries (bf16 ld of 4); a
    # BFP16 ld that does not hold whole 32-column exponent groups
    assert lib.megamoe_grouped_gemm(a16, a16, a16, 8, a16, a16, a16, 1, 256, 256, a16, a16, 2,
                                    a16, 260, P, 0, 0.0, P, P) == 2
    assert lib.megamoe_grouped_gemm(a16, a16, a16, 8, a16, a16, a16, 1, 256, 256, a16, a16, 3,
                                    a16, 272, P, 0, 0.0, P, P) == 2
    # BFP16 combine: y misaligned
    assert lib.megamoe_combine_bfp16(odd, 64, 8, a16, a16, 2, 2, 64, a16, P) == 2
    # forward: x misaligned; workspace not 256-byte aligned
    w = megamoe.CWeights(8, 256, 512, 4096, 4096, 4096, 4096, 4096, 4096)
    assert lib.megamoe_forward(ctypes.byref(w), odd, a16, a16, 4, 2, 32, a16, a16, 1 << 30,
                               P) == 2
    assert lib.megamoe_forward(ctypes.byref(w), a16, a16, a16, 4, 2, 32, a16, odd, 1 << 30,
                               P) == 1


def test_binding_refuses_an_output_buffer_that_does_not_fit_the_epilogue():
    """megamoe.grouped_gemm checks the output's type and size against the
    epilogue before anything is launched: an fp32 epilogue into a narrower
    buffer (the BFP16 y's int16 view) or a too-short one is an error, not a
    write past the buffer."""
    import pytest
    import torch

    E, N, K, rows = 2, 256, 256, 64
    act = torch.zeros(rows, K // 2, dtype=torch.uint8)
    sf = torch.zeros(rows, K // 16, dtype=torch.uint8)
    w = torch.zeros(E, N, K // 2, dtype=torch.uint8)
    ws = torch.zeros(E * N, K // 16, dtype=torch.uint8)
    gs = torch.ones(E)
    offs = torch.zeros(E + 1, dtype=torch.int32)
    for bad in (torch.zeros(rows, N, dtype=torch.int16), torch.zeros(rows - 1, N),
                torch.zeros(rows, N - 4)):
        with pytest.raises(ValueError):
            megamoe.grouped_gemm(act, sf, gs[:1], w, ws, gs, offs, offs, megamoe.EPI_F32, out=bad)
    with pytest.raises(ValueError):  # BFP16 wants the byte buffer of bfp16_bytes(rows, N)
        megamoe.grouped_gemm(act, sf, gs[:1], w, ws, gs, offs, offs, megamoe.EPI_BFP16,
                             out=torch.zeros(megamoe.bfp16_bytes(rows, N) - 1, dtype=torch.uint8))


def test_library_sources_call_no_device_allocator():
    """The library allocates and frees no device memory: every buffer,
    workspace included, is the caller's (megamoe_forward_static uses a
    file-scope device array).  No allocator or free call appears in the
    code of any library source (comments stripped)."""
    import glob
    csrc = os.path.join(ROOT, "nvfp4_block_scaled_topk_gb300", "csrc")
    calls = re.compile(r"\b(cudaMalloc\w*|cudaFree\w*|cudaHostAlloc|cuMemAlloc\w*|cuMemFree\w*|"
                       r"cuMemCreate|cuMemHostAlloc|cudaMemPoolCreate|cuMemPoolCreate)\s*\(")
    files = sorted(glob.glob(os.path.join(csrc, "*.cu")) + glob.glob(os.path.join(csrc, "*.cuh"))
                   + glob.glob(os.path.join(csrc, "*.h")))
    assert files
    for f in files:
        with open(f) as fh:
            code = re.sub(r"/\*.*?\*/", "", fh.read(), flags=re.S)
        code = re.sub(r"//[^\n]*", "", code)
        found = calls.findall(code)
        assert not found, f"{os.path.basename(f)} calls {sorted(set(found))}"
