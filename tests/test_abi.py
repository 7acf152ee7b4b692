"""CPU checks of the C-ABI library: it builds for sm_103a, loads without a GPU,
exports every entry point include/libmoe.h declares, and rejects bad host
arguments before touching CUDA.  No compute call is made here."""
import ctypes
import os
import re
import subprocess

import pytest

from token_dispatch_grouped_router_gb300 import build as B
from token_dispatch_grouped_router_gb300 import libmoe as LM

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "libmoe.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return LM.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 17
    out = subprocess.run(["nm", "-D", "--defined-only", LM.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (moe_[a-z0-9_]+)\b", out))
    for n in names:
        assert n in exported, n
        assert n in LM.SIGNATURES, n
        assert getattr(lib, n) is not None
    # and nothing exported that the header does not declare
    assert exported == set(names)


def test_status_strings_and_version(lib):
    for st in (0, -1, -2, -3, -4):
        assert lib.moe_status_string(st)
    assert lib.moe_status_string(123).startswith(b"unknown")
    assert lib.moe_version() == 100


def test_workspace_size_grows_with_the_problem(lib):
    small = lib.moe_workspace_size(512, 8, 2, 256, 512)
    big = lib.moe_workspace_size(32768, 128, 4, 2048, 1024)
    assert 256 <= small < big
    # route-map scratch: per-chunk histograms + one rank per routed slot
    R = 32768 * 4
    assert big >= 256 + (R // 1024) * 128 * 4 + R * 4
    assert lib.moe_workspace_size(-1, 8, 2, 256, 512) == 0


def test_host_argument_checks_return_before_any_cuda_call(lib):
    NULL = None
    fake = ctypes.c_void_p(0x1000)   # aligned, never dereferenced: checks fail first
    # k out of range / k > E
    assert lib.moe_router_topk(fake, 4, 8, 0, fake, fake, NULL) == -1
    assert lib.moe_router_topk(fake, 4, 8, 9, fake, fake, NULL) == -1
    assert lib.moe_router_topk(fake, 4, 2000, 2, fake, fake, NULL) == -1
    # null or misaligned pointers
    assert lib.moe_router_topk(NULL, 4, 8, 2, fake, fake, NULL) == -1
    assert lib.moe_router_topk(ctypes.c_void_p(0x1001), 4, 8, 2, fake, fake, NULL) == -1
    assert lib.moe_dispatch_rows(fake, 4, 12, 2, fake, fake, NULL) == -1        # d % 8
    # grouped GEMMs need d, h multiples of 64
    assert lib.moe_grouped_swiglu_fwd(fake, fake, 8, 4, 96, 128, fake, fake, fake, fake, fake,
                                      fake, fake, fake, 1 << 20, NULL) == -2
    # workspace too small / missing
    assert lib.moe_grouped_swiglu_fwd(fake, fake, 8, 4, 128, 128, fake, fake, fake, fake, fake,
                                      fake, fake, fake, 16, NULL) == -3
    assert lib.moe_expert_offsets(fake, 4, 2, 8, fake, fake, fake, fake, NULL, 0, NULL) == -3
    assert lib.moe_expert_offsets(fake, 1024, 2, 8, fake, fake, fake, fake, fake, 300, NULL) == -3
    assert lib.moe_get_status(NULL, NULL, NULL) == -3
    # T = 0 is a no-op that succeeds without launching anything
    before = lib.moe_launch_count()
    assert lib.moe_router_topk(NULL, 0, 8, 2, NULL, NULL, NULL) == 0
    assert lib.moe_combine(NULL, NULL, NULL, 0, 2, 256, NULL, NULL) == 0
    assert lib.moe_launch_count() == before


def test_binding_fails_loudly_without_the_library(tmp_path):
    saved = LM._lib
    try:
        LM._lib = None
        with pytest.raises(RuntimeError, match="not found"):
            LM.load(str(tmp_path / "missing.so"))
    finally:
        LM._lib = saved


def test_wgrad_workspace_holds_the_per_expert_descriptors(lib):
    # five 128-byte TMA descriptors per expert after the 256-byte status word,
    # the tile plan ((8 + 2E) int32) after them
    for E in (1, 8, 128, 1024):
        # + the weight-gradient GEMM's fp32 partial tiles (80 x 256 x 256)
        assert lib.moe_workspace_size(16, E, 1, 64, 64) >= 256 + 640 * E + (8 + 2 * E) * 4 + 80 * 256 * 256 * 4
    fake = ctypes.c_void_p(0x1000)
    args = lambda ws, n: (fake, fake, 64, 128, 128, 128, fake, fake, fake, fake, fake, fake,
                          fake, ws, n, None)
    need = lib.moe_workspace_size(16, 128, 4, 128, 128)
    # too small for 128 experts' descriptors (but larger than the status word)
    assert lib.moe_grouped_swiglu_bwd_wgrad(*args(fake, 256 + 640 * 127)) == -3
    # the descriptors fit, the tile plan does not
    assert lib.moe_grouped_swiglu_bwd_wgrad(*args(fake, 256 + 640 * 128 + (8 + 2 * 128) * 4 - 4)) == -3
    # descriptors must sit on 128-byte boundaries
    assert lib.moe_grouped_swiglu_bwd_wgrad(*args(ctypes.c_void_p(0x1010), need)) == -1


def test_router_and_mxfp8_additions_check_arguments_on_the_host(lib):
    NULL = None
    fake = ctypes.c_void_p(0x1000)
    big = 1 << 30
    # tensor-core router: d must give 16-byte rows of x; a workspace is required
    assert lib.moe_router_logits_tc(fake, fake, NULL, 64, 12, 8, fake, fake, big, NULL) == -2
    assert lib.moe_router_logits_tc(fake, fake, NULL, 64, 16, 8, fake, NULL, 0, NULL) == -3
    assert lib.moe_router_logits_tc(fake, fake, NULL, 64, 16, 2000, fake, fake, big, NULL) == -1
    # ... and the scratch for the three bf16 parts of W_r (6 E ceil(d/64)*64 bytes)
    assert lib.moe_router_logits_tc(fake, fake, NULL, 64, 2048, 128, fake, fake,
                                    256 + 6 * 128 * 2048 - 1, NULL) == -3
    # router backward through the top-k: d % 8, k <= E, workspace size
    assert lib.moe_router_logits_bwd_topk(fake, fake, fake, fake, fake, fake, 64, 12, 8, 2,
                                          fake, fake, NULL, fake, big, NULL) == -2
    assert lib.moe_router_logits_bwd_topk(fake, fake, fake, fake, fake, fake, 64, 16, 4, 8,
                                          fake, fake, NULL, fake, big, NULL) == -1
    assert lib.moe_router_logits_bwd_topk(fake, fake, fake, fake, fake, fake, 64, 16, 8, 2,
                                          fake, fake, NULL, fake, 300, NULL) == -3
    # its scratch lies past the weight-gradient GEMM's part of the workspace
    # (descriptors, tile plan, fp32 partial tiles), so that part alone is too small
    E = 8
    plan = -(-(256 + 640 * E) // 256) * 256 + (8 + 2 * E) * 4
    wgrad_part = -(-plan // 256) * 256 + 80 * 256 * 256 * 4
    assert lib.moe_workspace_size(64, E, 2, 16, 64) > wgrad_part
    assert lib.moe_router_logits_bwd_topk(fake, fake, fake, fake, fake, fake, 64, 16, E, 2,
                                          fake, fake, NULL, fake, wgrad_part, NULL) == -3
    # MXFP8: dequantise needs K % 32, the fp32-master quantiser N % 128
    assert lib.moe_mxfp8_dequantize_rows(fake, fake, 4, 48, fake, NULL) == -2
    assert lib.moe_mxfp8_dequantize_rows(fake, NULL, 4, 64, fake, NULL) == -1
    assert lib.moe_mxfp8_quantize_weights_f32(fake, 2, 64, 96, fake, fake, NULL) == -2
    # T = 0 / rows = 0 launch nothing
    before = lib.moe_launch_count()
    assert lib.moe_router_logits_tc(NULL, NULL, NULL, 0, 16, 8, NULL, fake, big, NULL) == 0
    assert lib.moe_mxfp8_dequantize_rows(NULL, NULL, 0, 64, NULL, NULL) == 0
    assert lib.moe_launch_count() == before


def test_capacity_calls_check_arguments_on_the_host(lib):
    NULL = None
    fake = ctypes.c_void_p(0x1000)
    big = 1 << 30
    before = lib.moe_launch_count()
    # capacity below 1, E*C beyond int32, missing outputs, short workspace
    assert lib.moe_expert_offsets_capacity(fake, 64, 2, 8, 0, fake, fake, fake, fake, NULL,
                                           fake, big, NULL) == -1
    assert lib.moe_expert_offsets_capacity(fake, 64, 2, 8, 1 << 29, fake, fake, fake, fake, NULL,
                                           fake, big, NULL) == -1
    assert lib.moe_expert_offsets_capacity(fake, 64, 2, 8, 20, fake, fake, fake, NULL, NULL,
                                           fake, big, NULL) == -1
    assert lib.moe_expert_offsets_capacity(fake, 64, 2, 8, 20, fake, fake, fake, fake,
                                           ctypes.c_void_p(0x1004), fake, big, NULL) == -1
    assert lib.moe_expert_offsets_capacity(fake, 64, 2, 8, 20, fake, fake, fake, fake, NULL,
                                           NULL, 0, NULL) == -3
    assert lib.moe_expert_offsets_capacity(fake, 64, 2, 8, 20, fake, fake, fake, fake, NULL,
                                           fake, 300, NULL) == -3
    # padded dispatch / combine / combine backward: sizes and pointers
    assert lib.moe_dispatch_rows_capacity(fake, 4, 12, 2, fake, fake, 8, 4, fake, NULL) == -1
    assert lib.moe_dispatch_rows_capacity(fake, 4, 16, 2, fake, NULL, 8, 4, fake, NULL) == -1
    assert lib.moe_dispatch_rows_capacity(fake, 4, 16, 2, fake, fake, 8, 0, fake, NULL) == -1
    assert lib.moe_combine_capacity(fake, 8, 0, fake, NULL, 4, 2, 16, fake, NULL) == -1
    assert lib.moe_combine_capacity(fake, 8, 4, fake, ctypes.c_void_p(0x1004), 4, 2, 16, fake,
                                    NULL) == -1
    assert lib.moe_combine_bwd_capacity(fake, fake, 8, 4, fake, NULL, fake, 4, 2, 16, fake, fake,
                                        NULL) == -1
    # T = 0: the padded combine does nothing
    assert lib.moe_combine_capacity(NULL, 8, 4, NULL, NULL, 0, 2, 16, NULL, NULL) == 0
    assert lib.moe_launch_count() == before


def test_mxfp8_atom_and_dgrad_calls_check_arguments_on_the_host(lib):
    NULL = None
    fake = ctypes.c_void_p(0x1000)
    odd4 = ctypes.c_void_p(0x1002)          # not 4-byte aligned
    big = 1 << 34
    before = lib.moe_launch_count()
    # atom sizes: zero unless d and h are multiples of 128
    assert lib.moe_mxfp8_weight_atom_bytes(2, 96, 128) == 0
    assert lib.moe_mxfp8_dx_weight_atom_bytes(2, 128, 64) == 0
    # per expert: ceil(h/96) up tiles x d/128 k-blocks + ceil(d/192) down tiles x h/128, 2 atoms each
    assert lib.moe_mxfp8_weight_atom_bytes(2, 256, 384) == 2 * (4 * 2 + 2 * 3) * 2 * 512
    assert lib.moe_mxfp8_dx_weight_atom_bytes(2, 256, 384) == 2 * 2 * 6 * 2 * 512
    # weight atoms: sizes, scale-table alignment
    assert lib.moe_mxfp8_weight_scale_atoms(fake, fake, fake, 2, 96, 128, fake, NULL) == -2
    assert lib.moe_mxfp8_weight_scale_atoms(odd4, fake, fake, 2, 128, 128, fake, NULL) == -1
    assert lib.moe_mxfp8_dx_weight_scale_atoms(fake, NULL, 2, 128, 128, fake, NULL) == -1
    assert lib.moe_mxfp8_dx_weight_scale_atoms(fake, fake, 0, 128, 128, fake, NULL) == -1
    # the MXFP8 dgrad: sizes, experts, workspace, pointers
    args = lambda R, E, d, h, ws, n, s1=fake: (fake, s1, fake, fake, fake, R, E, d, h, fake, fake,  # noqa: E731
                                             fake, fake, ws, n, NULL)
    assert lib.moe_grouped_swiglu_bwd_dx_mxfp8(*args(64, 2, 192, 128, fake, big)) == -2
    assert lib.moe_grouped_swiglu_bwd_dx_mxfp8(*args(64, 800, 128, 128, fake, big)) == -2
    assert lib.moe_grouped_swiglu_bwd_dx_mxfp8(*args(64, 2, 128, 128, NULL, 0)) == -3
    assert lib.moe_grouped_swiglu_bwd_dx_mxfp8(*args(64, 2, 128, 128, fake, 4096)) == -3
    assert lib.moe_grouped_swiglu_bwd_dx_mxfp8(*args(64, 2, 128, 128, fake, big, s1=odd4)) == -1
    # the MXFP8 forward checks its workspace for the activation scale atoms
    fwd = (fake, fake, fake, 64, 2, 128, 128, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake)
    assert lib.moe_grouped_swiglu_fwd_mxfp8(*fwd, fake, 4096, NULL) == -3
    # R = 0 launches nothing
    assert lib.moe_grouped_swiglu_bwd_dx_mxfp8(*args(0, 2, 128, 128, fake, big)) == 0
    assert lib.moe_launch_count() == before


def test_the_header_alone_serves_a_c_program(lib, tmp_path):
    # a plain C caller: compiled with gcc against include/libmoe.h, linked to
    # libmoe.so, host-side calls only (no CUDA call is reached)
    import shutil
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "c_abi", "host_checks.c")
    exe = str(tmp_path / "host_checks")
    libdir = os.path.dirname(LM.LIB_PATH)
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), src, "-o", exe,
                    "-L", libdir, "-lmoe", "-Wl,-rpath," + libdir], check=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
