"""The C-ABI library loads, exports every entry point include/nvfp4.h
declares (and the measurement library every entry point of
include/nvfp4_probe.h), and rejects bad arguments before launching anything
(no GPU needed: every case here fails the host-side checks)."""
import ctypes
import os
import re

import pytest
import torch

import nvfp4_block_scaled_28_b300 as nv
from nvfp4_block_scaled_28_b300 import _native as N

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4.h")
PROBE_HEADER = os.path.join(ROOT, "include", "nvfp4_probe.h")


def declared_functions(path=HEADER, macro="NVFP4_API"):
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(macro + r"\s+[\w\s\*]+?\b(nvfp4_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from nvfp4_block_scaled_28_b300 import build
    build.build()
    return N.load()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("nvfp4_quantize", "nvfp4_quantize_weight", "nvfp4_linear", "nvfp4_gemm",
                 "nvfp4_global_scale", "nvfp4_device_error"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(N.SIGNATURES), "binding and header disagree"


def test_probe_library_is_separate_and_exports_its_header():
    from nvfp4_block_scaled_28_b300 import build
    build.build_probe()
    probe = N.load_probe()
    names = declared_functions(PROBE_HEADER, "NVFP4_PROBE_API")
    assert names == sorted(N.PROBE_SIGNATURES)
    for name in names:
        assert hasattr(probe, name), name
    # the product library carries no measurement probe
    product = N.load()
    for name in names:
        assert not hasattr(product, name), name
    assert "nvfp4_mma_peak_probe" not in declared_functions()


def test_debug_library_exports_the_same_abi():
    """The bounds-checking debug build (loaded with NVFP4_B300_DEBUG=1) is a
    separate file with every entry point of include/nvfp4.h."""
    from nvfp4_block_scaled_28_b300 import build
    build.build()
    dbg = ctypes.CDLL(build.DEBUG_LIB_PATH)
    for name in declared_functions():
        assert hasattr(dbg, name), name
    dbg.nvfp4_status_string.restype = ctypes.c_char_p
    assert dbg.nvfp4_status_string(7).decode() == "NVFP4_ERR_BOUNDS"
    assert build.DEBUG_LIB_PATH != build.LIB_PATH


def test_every_header_is_checked():
    import glob
    assert sorted(os.path.basename(h) for h in glob.glob(os.path.join(ROOT, "include", "*.h"))) \
        == ["nvfp4.h", "nvfp4_probe.h"]


def test_status_strings(lib):
    for code, name in [(0, "NVFP4_OK"), (1, "NVFP4_ERR_INVALID_ARG"), (2, "NVFP4_ERR_MISALIGNED"),
                       (3, "NVFP4_ERR_UNSUPPORTED_SHAPE"), (4, "NVFP4_ERR_WORKSPACE_TOO_SMALL"),
                       (5, "NVFP4_ERR_CUDA"), (6, "NVFP4_ERR_TIMEOUT"), (7, "NVFP4_ERR_BOUNDS"),
                       (99, "NVFP4_ERR_UNKNOWN")]:
        assert lib.nvfp4_status_string(code).decode() == name


def test_sf_bytes(lib):
    assert lib.nvfp4_sf_bytes(300, 256, 0) == 300 * 16
    assert lib.nvfp4_sf_bytes(300, 256, 1) == 384 * 16
    assert lib.nvfp4_sf_bytes(128, 64, 1) == 128 * 4
    assert lib.nvfp4_sf_bytes(3, 40, 0) == 0  # K % 16
    assert lib.nvfp4_sf_bytes(3, 48, 1) == 0  # K % 64
    assert lib.nvfp4_sf_bytes(-1, 64, 0) == 0


# fake, never-dereferenced addresses: every call below fails its checks first
A16 = 0x10000
ODD = 0x10001


def test_quantize_argument_checks(lib):
    q = lib.nvfp4_quantize
    assert q(A16, 4, 40, 40, A16, A16, A16, 0, None) == N.ERR_UNSUPPORTED_SHAPE  # K % 16
    assert q(A16, 4, 48, 48, A16, A16, A16, 1, None) == N.ERR_UNSUPPORTED_SHAPE  # K % 64 (tile)
    assert q(ODD, 4, 64, 64, A16, A16, A16, 0, None) == N.ERR_MISALIGNED
    assert q(A16, 4, 64, 60, A16, A16, A16, 0, None) == N.ERR_INVALID_ARG  # ld < cols
    assert q(A16, 4, 64, 68, A16, A16, A16, 0, None) == N.ERR_MISALIGNED  # ld % 8
    assert q(A16, 4, 64, 64, None, A16, A16, 0, None) == N.ERR_INVALID_ARG  # g
    assert q(A16, 4, 64, 64, A16, None, A16, 0, None) == N.ERR_INVALID_ARG  # q
    assert q(A16, 4, 64, 64, A16, A16, A16, 7, None) == N.ERR_INVALID_ARG  # layout
    assert q(A16, -1, 64, 64, A16, A16, A16, 0, None) == N.ERR_INVALID_ARG
    assert q(None, 4, 64, 64, A16, A16, A16, 0, None) == N.ERR_INVALID_ARG


def test_gemm_argument_checks(lib):
    g = lib.nvfp4_gemm
    args = lambda **kw: [kw.get("Aq", A16), kw.get("As", A16), A16, kw.get("Bq", A16), A16, A16,
                         kw.get("M", 128), kw.get("N", 256), kw.get("K", 512), kw.get("Y", A16),
                         kw.get("ldy", 256), None, 0, None]
    assert g(*args(K=320)) == N.ERR_UNSUPPORTED_SHAPE
    assert g(*args(K=0)) == N.ERR_INVALID_ARG
    assert g(*args(Aq=ODD)) == N.ERR_MISALIGNED
    assert g(*args(Y=A16 + 1)) == N.ERR_MISALIGNED
    assert g(*args(ldy=100)) == N.ERR_INVALID_ARG
    assert g(*args(Bq=None)) == N.ERR_INVALID_ARG
    assert g(*args(M=-3)) == N.ERR_INVALID_ARG


def test_linear_argument_checks(lib):
    f = lib.nvfp4_linear
    base = dict(X=A16, M=64, K=512, ldx=512, Wq=A16, Ws=A16, gw=A16, N=128, Y=A16, ldy=128,
                gx=None, mode=0, ws=A16 * 16, wsb=1 << 30)
    call = lambda **kw: f(*[{**base, **kw}[k] for k in base], None)
    assert call(mode=3) == N.ERR_INVALID_ARG
    assert call(K=448, ldx=448) == N.ERR_UNSUPPORTED_SHAPE
    assert call(wsb=16) == N.ERR_WORKSPACE_TOO_SMALL
    assert call(ws=A16 + 16) == N.ERR_MISALIGNED
    assert call(ws=None) == N.ERR_INVALID_ARG
    assert call(X=ODD) == N.ERR_MISALIGNED
    need = lib.nvfp4_linear_workspace_bytes(64, 128, 512, 0)
    assert need >= 64 * 256 + 512 * 128 // 16


def test_python_binding_rejects_packed_fp4_as_bf16():
    """The "nvfp4-gemma4" page (section 4) reports a crash from packed FP4
    weights read as bfloat16 with half the columns; the binding refuses
    such tensors before any launch."""
    X = torch.zeros(4, 512, dtype=torch.bfloat16)
    Wq_as_bf16 = torch.zeros(128, 256, dtype=torch.bfloat16)
    Ws = torch.zeros(128, 32, dtype=torch.uint8)
    g = torch.ones(1)
    with pytest.raises(ValueError, match="uint8 packed FP4"):
        nv.nvfp4_linear(X, Wq_as_bf16, Ws, g)
    Wq_half_rows = torch.zeros(64, 256, dtype=torch.uint8)
    with pytest.raises(ValueError, match="shape"):
        nv.nvfp4_linear(X, Wq_half_rows.view(128, 128), Ws, g)
    with pytest.raises(ValueError, match="bfloat16"):
        nv.nvfp4_linear(X.float(), torch.zeros(128, 256, dtype=torch.uint8), Ws, g)
    with pytest.raises(ValueError, match="scale bytes"):
        nv.nvfp4_linear(X, torch.zeros(128, 256, dtype=torch.uint8),
                        torch.zeros(128, 16, dtype=torch.uint8), g)


def test_mma_peak_probe_argument_checks():
    p = N.load_probe().nvfp4_mma_peak_probe
    assert p(1, 8, 8, A16, None) == N.ERR_INVALID_ARG   # no such variant
    assert p(1, 8, 7, A16, None) == N.ERR_INVALID_ARG   # pair variant needs 2 CTAs
    assert p(1, 8, -1, A16, None) == N.ERR_INVALID_ARG
    assert p(1, 6, 0, A16, None) == N.ERR_INVALID_ARG   # iters not a multiple of 4
    assert p(1, 12, 2, A16, None) == N.ERR_INVALID_ARG  # two warps: multiple of 8
    assert p(0, 8, 0, A16, None) == N.ERR_INVALID_ARG
    assert p(1, 8, 0, None, None) == N.ERR_INVALID_ARG
    assert p(1, 8, 0, A16 + 4, None) == N.ERR_MISALIGNED


def test_select_gemm_kernel_checks(lib):
    assert lib.nvfp4_debug_select_gemm_kernel(2) == N.ERR_INVALID_ARG
    assert lib.nvfp4_debug_select_gemm_kernel(-1) == N.ERR_INVALID_ARG
    for k in (1, 0):
        assert lib.nvfp4_debug_select_gemm_kernel(k) == N.OK
    assert lib.nvfp4_debug_capture_fused_operand(2) == N.ERR_INVALID_ARG
    assert lib.nvfp4_debug_capture_fused_operand(0) == N.OK


def test_linear_bias_requant_argument_checks(lib):
    f = lib.nvfp4_linear_bias_requant
    base = dict(X=A16, M=256, K=512, ldx=512, Wq=A16, Ws=A16, gw=A16, N=512, bias=A16, Y=A16,
                ldy=512, gy=A16, Yq=A16, Ys=A16, gx=None, ws=A16 * 16, wsb=1 << 30)
    call = lambda **kw: f(*[{**base, **kw}[k] for k in base], None)
    # above 128 rows the epilogue is in the CTA-pair kernel only
    assert lib.nvfp4_debug_select_gemm_kernel(1) == N.OK
    try:
        assert call(M=256) == N.ERR_UNSUPPORTED_SHAPE
    finally:
        assert lib.nvfp4_debug_select_gemm_kernel(0) == N.OK
    assert call(N=384, ldy=384) == N.ERR_UNSUPPORTED_SHAPE  # N % 256
    assert call(K=448, ldx=448) == N.ERR_UNSUPPORTED_SHAPE  # K % 256
    assert call(Y=None, gy=None, Yq=None, Ys=None) == N.ERR_INVALID_ARG  # no output at all
    assert call(Ys=None) == N.ERR_INVALID_ARG            # requant outputs all or none
    assert call(gy=None) == N.ERR_INVALID_ARG
    assert call(ldy=100) == N.ERR_INVALID_ARG
    assert call(bias=A16 + 8) == N.ERR_MISALIGNED         # bias read 16 bytes at a time
    assert call(Yq=A16 + 8) == N.ERR_MISALIGNED
    assert call(gy=ODD) == N.ERR_MISALIGNED
    assert call(wsb=16) == N.ERR_WORKSPACE_TOO_SMALL
    assert call(ws=A16 + 16) == N.ERR_MISALIGNED
    assert call(M=0) == N.OK and call(N=0, ldy=0) == N.OK  # empty: nothing launched


def test_linear_bias_requant_dynamic_argument_checks(lib):
    f = lib.nvfp4_linear_bias_requant_dynamic
    base = dict(X=A16, M=256, K=512, ldx=512, Wq=A16, Ws=A16, gw=A16, N=512, bias=A16, Y=A16,
                ldy=512, gy=A16, Yq=A16, Ys=A16, gx=None, ws=A16 * 16, wsb=1 << 30)
    call = lambda **kw: f(*[{**base, **kw}[k] for k in base], None)
    assert call(gy=None) == N.ERR_INVALID_ARG            # g_y_out is always written
    assert call(gy=None, M=0) == N.ERR_INVALID_ARG
    assert call(Y=None) == N.ERR_INVALID_ARG             # Y is required (read back)
    assert call(Yq=None) == N.ERR_INVALID_ARG
    assert call(Ys=None) == N.ERR_INVALID_ARG
    assert call(Y=A16 + 8) == N.ERR_MISALIGNED           # the quantizer reads Y 16 bytes at a time
    assert call(ldy=516) == N.ERR_MISALIGNED
    assert call(ldy=100) == N.ERR_INVALID_ARG
    assert call(N=384, ldy=384) == N.ERR_UNSUPPORTED_SHAPE
    assert call(K=448, ldx=448) == N.ERR_UNSUPPORTED_SHAPE
    assert call(gy=ODD) == N.ERR_MISALIGNED
    assert call(gy=ODD, M=0) == N.ERR_MISALIGNED
    assert call(bias=A16 + 8) == N.ERR_MISALIGNED
    assert call(Yq=A16 + 8) == N.ERR_MISALIGNED
    assert call(wsb=16) == N.ERR_WORKSPACE_TOO_SMALL
    assert call(ws=A16 + 16) == N.ERR_MISALIGNED
    assert lib.nvfp4_debug_select_gemm_kernel(1) == N.OK
    try:
        assert call(M=256) == N.ERR_UNSUPPORTED_SHAPE
    finally:
        assert lib.nvfp4_debug_select_gemm_kernel(0) == N.OK


def test_linear_grouped_argument_checks(lib):
    import ctypes
    f = lib.nvfp4_linear_grouped

    def call(ns, groups=None, **kw):
        arr = (ctypes.c_int64 * max(1, len(ns)))(*ns)
        base = dict(X=A16, M=64, K=512, ldx=512, Wq=A16, Ws=A16, gw=A16,
                    gn=ctypes.cast(arr, ctypes.c_void_p), G=len(ns) if groups is None else groups,
                    Y=A16, ldy=sum(ns), gx=None, mode=0, ws=A16 * 16, wsb=1 << 30)
        base.update(kw)
        return f(*base.values(), None)

    assert call([256, 256], gn=None) == N.ERR_INVALID_ARG
    assert call([256], groups=0) == N.ERR_INVALID_ARG
    assert call([256] * 9) == N.ERR_INVALID_ARG            # at most 8 groups
    assert call([256, 0]) == N.ERR_INVALID_ARG
    assert call([256, 128]) == N.ERR_UNSUPPORTED_SHAPE     # multiples of 256
    assert call([256, 512], ldy=512) == N.ERR_INVALID_ARG  # ldy < sum
    assert call([256, 512], mode=2) == N.ERR_INVALID_ARG
    assert call([256, 512], wsb=16) == N.ERR_WORKSPACE_TOO_SMALL
    assert call([256, 512], M=0) == N.OK


def test_quantize_select_argument_checks(lib):
    f = lib.nvfp4_quantize_select
    assert f(A16, 4, 64, 64, A16, 3, A16, A16, 0, None) == N.ERR_INVALID_ARG   # no such rule
    assert f(A16, 4, 64, 64, A16, -1, A16, A16, 0, None) == N.ERR_INVALID_ARG
    assert f(A16, 4, 40, 40, A16, 2, A16, A16, 0, None) == N.ERR_UNSUPPORTED_SHAPE  # K % 16
    assert f(ODD, 4, 64, 64, A16, 1, A16, A16, 0, None) == N.ERR_MISALIGNED
    assert f(A16, 4, 64, 64, None, 1, A16, A16, 0, None) == N.ERR_INVALID_ARG   # no g
    assert f(A16, 0, 64, 64, A16, 2, A16, A16, 0, None) == N.OK                 # empty


def test_linear_lora_argument_checks(lib):
    f = lib.nvfp4_linear_lora
    base = dict(X=A16, M=256, K=512, ldx=512, Wq=A16, Ws=A16, gw=A16, N=256, la=A16, lb=A16,
                r=32, s=1.0, Y=A16, ldy=256, gx=None, ws=A16 * 16, wsb=1 << 30)
    call = lambda **kw: f(*[{**base, **kw}[k] for k in base], None)
    assert call(M=128) == N.ERR_UNSUPPORTED_SHAPE          # the CTA-pair kernel: M > 128
    assert call(r=24) == N.ERR_UNSUPPORTED_SHAPE           # r in 16, 32, 48, 64
    assert call(r=128) == N.ERR_UNSUPPORTED_SHAPE
    assert call(K=448, ldx=448) == N.ERR_UNSUPPORTED_SHAPE
    assert call(s=float("nan")) == N.ERR_INVALID_ARG
    assert call(la=None) == N.ERR_INVALID_ARG
    assert call(lb=A16 + 8) == N.ERR_MISALIGNED
    assert call(wsb=16) == N.ERR_WORKSPACE_TOO_SMALL
    assert call(M=0) == N.OK
    need = lib.nvfp4_linear_lora_workspace_bytes(256, 256, 512, 32)
    assert need >= lib.nvfp4_linear_workspace_bytes(256, 256, 512, 0) + 256 * 32 * 2


def test_library_is_built_from_the_current_sources():
    """A library older than any of its sources would test stale code: the
    artifact's own time stamp is compared with every source (no stamp files)."""
    from nvfp4_block_scaled_28_b300 import build
    assert build.up_to_date(), "the library is older than its sources: rebuild it"


def test_block_count_limit_keeps_indices_32_bit(lib):
    """Tensors of 2^28 or more 16-element blocks are rejected before any
    launch (the kernels' 32-bit block and vector indices, plus the grid
    strides added ahead of their bounds tests, stay below 2^32). Just below
    the limit the shape passes and the next check (a null global scale)
    fails instead."""
    limit = 1 << 28
    rows, cols = 1 << 14, (limit // (1 << 14)) * 16   # exactly 2^28 blocks
    q = lib.nvfp4_quantize
    assert q(A16, rows, cols, cols, A16, A16, A16, 0, None) == N.ERR_UNSUPPORTED_SHAPE
    assert q(A16, rows - 1, cols, cols, None, A16, A16, 0, None) == N.ERR_INVALID_ARG
    assert lib.nvfp4_global_scale(A16, rows, cols, cols, A16, None) == N.ERR_UNSUPPORTED_SHAPE
    assert lib.nvfp4_global_scale(A16, rows - 1, cols, cols, None, None) == N.ERR_INVALID_ARG
    lin = lib.nvfp4_linear
    K = cols
    assert lin(A16, rows, K, K, A16, A16, A16, 256, A16, 256, None, 0, A16 * 16, 1 << 62,
               None) == N.ERR_UNSUPPORTED_SHAPE
    # M x N beyond the output limit
    assert lib.nvfp4_gemm(A16, A16, A16, A16, A16, A16, 1 << 21, 1 << 21, 256, A16, 1 << 21,
                          None, 0, None) == N.ERR_UNSUPPORTED_SHAPE
