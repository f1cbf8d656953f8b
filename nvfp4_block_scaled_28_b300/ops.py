"""Thin PyTorch binding over the C ABI (argument marshalling only).

Each function checks dtypes, shapes, devices and contiguity, allocates the
outputs it returns with torch (device memory is torch's job here), and calls
the C entry point of the same name on the current CUDA stream. All
arithmetic happens in the library's CUDA kernels.

The checks guard the failure the "nvfp4-gemma4" page reports in section 4:
a packed FP4 tensor read as bfloat16 has half the columns it should, so
every packed operand is checked for dtype uint8 and shape (rows, K/2), and
every scale tensor for its exact byte count.
"""
from __future__ import annotations

import torch

from . import _native as N

SF_ROW_MAJOR = N.SF_ROW_MAJOR
SF_MMA_128x4 = N.SF_MMA_128x4
LINEAR_UNFUSED = N.LINEAR_UNFUSED
LINEAR_FUSED = N.LINEAR_FUSED
SCALE_ABSMAX = N.SCALE_ABSMAX
SCALE_FOUR_OVER_SIX = N.SCALE_FOUR_OVER_SIX
SCALE_MSE = N.SCALE_MSE
NVFP4Error = N.NVFP4Error


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _require(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def _check_cuda(*ts) -> None:
    for t in ts:
        if t is not None:
            _require(t.is_cuda, "tensors must be on a CUDA device")


def _check_bf16_2d(x: torch.Tensor, name: str) -> None:
    _require(x.dtype == torch.bfloat16, "%s must be bfloat16, got %s" % (name, x.dtype))
    _require(x.dim() == 2, "%s must be 2-D" % name)
    _require(x.stride(1) == 1, "%s must have unit stride along K" % name)


def _check_codes(q: torch.Tensor, rows: int, K: int, name: str) -> None:
    _require(q.dtype == torch.uint8, "%s must be uint8 packed FP4, got %s" % (name, q.dtype))
    _require(tuple(q.shape) == (rows, K // 2),
             "%s must have shape (%d, %d) (two FP4 codes per byte), got %s"
             % (name, rows, K // 2, tuple(q.shape)))
    _require(q.is_contiguous(), "%s must be contiguous" % name)


def _check_scales(s: torch.Tensor, rows: int, K: int, layout: int, name: str) -> None:
    _require(s.dtype in (torch.uint8, torch.float8_e4m3fn),
             "%s must be uint8 or float8_e4m3fn, got %s" % (name, s.dtype))
    _require(s.is_contiguous(), "%s must be contiguous" % name)
    need = sf_bytes(rows, K, layout)
    _require(s.numel() == need, "%s must hold %d scale bytes for (%d rows, K=%d), got %d"
             % (name, need, rows, K, s.numel()))


def _check_g(g: torch.Tensor, name: str) -> None:
    _require(g.dtype == torch.float32 and g.numel() >= 1, "%s must be a float32 tensor" % name)


def sf_bytes(rows: int, K: int, layout: int) -> int:
    return int(N.load().nvfp4_sf_bytes(rows, K, layout))


def sf_shape(rows: int, K: int, layout: int):
    if layout == SF_ROW_MAJOR:
        return (rows, K // 16)
    return ((rows + 127) // 128 * 128, K // 16)


def nvfp4_global_scale(X: torch.Tensor, g: torch.Tensor | None = None) -> torch.Tensor:
    """Decode-direction global scale amax(|X|) / (6 * 448) as a 1-element
    float32 device tensor (1.0 for an all-zero X)."""
    _check_bf16_2d(X, "X")
    _check_cuda(X)
    if g is None:
        g = torch.empty(1, dtype=torch.float32, device=X.device)
    _check_g(g, "g")
    N.check("nvfp4_global_scale", N.load().nvfp4_global_scale(
        _ptr(X), X.shape[0], X.shape[1], X.stride(0), _ptr(g), _stream()))
    return g


def nvfp4_quantize(X: torch.Tensor, g: torch.Tensor, sf_layout: int = SF_ROW_MAJOR,
                   q: torch.Tensor | None = None, sf: torch.Tensor | None = None,
                   rule: int = SCALE_ABSMAX):
    """Quantize bfloat16 X (rows, K) to packed E2M1 codes (rows, K/2) uint8
    and E4M3 block scales (uint8 bytes) in ``sf_layout``; ``rule`` picks the
    block scale (absmax, four-over-six or MSE)."""
    _check_bf16_2d(X, "X")
    _check_g(g, "g")
    _check_cuda(X, g)
    rows, K = X.shape
    _require(K % 16 == 0, "K must be a multiple of 16")
    if q is None:
        q = torch.empty((rows, K // 2), dtype=torch.uint8, device=X.device)
    if sf is None:
        sf = torch.empty(sf_shape(rows, K, sf_layout), dtype=torch.uint8, device=X.device)
    _check_codes(q, rows, K, "q")
    _check_scales(sf, rows, K, sf_layout, "sf")
    if rule == SCALE_ABSMAX:
        N.check("nvfp4_quantize", N.load().nvfp4_quantize(
            _ptr(X), rows, K, X.stride(0), _ptr(g), _ptr(q), _ptr(sf), sf_layout, _stream()))
    else:
        N.check("nvfp4_quantize_select", N.load().nvfp4_quantize_select(
            _ptr(X), rows, K, X.stride(0), _ptr(g), rule, _ptr(q), _ptr(sf), sf_layout,
            _stream()))
    return q, sf


def nvfp4_quantize_weight(W: torch.Tensor, sf_layout: int = SF_MMA_128x4,
                          rule: int = SCALE_ABSMAX):
    """Offline weight quantization: returns (Wq (N, K/2) uint8, Ws scales,
    g_w 1-element float32); ``rule`` picks the block scale."""
    _check_bf16_2d(W, "W")
    _check_cuda(W)
    rows, K = W.shape
    if rule != SCALE_ABSMAX:
        g = nvfp4_global_scale(W)
        Wq, Ws = nvfp4_quantize(W, g, sf_layout, rule=rule)
        return Wq, Ws, g
    Wq = torch.empty((rows, K // 2), dtype=torch.uint8, device=W.device)
    Ws = torch.empty(sf_shape(rows, K, sf_layout), dtype=torch.uint8, device=W.device)
    g = torch.empty(1, dtype=torch.float32, device=W.device)
    N.check("nvfp4_quantize_weight", N.load().nvfp4_quantize_weight(
        _ptr(W), rows, K, W.stride(0), _ptr(Wq), _ptr(Ws), _ptr(g), sf_layout, _stream()))
    return Wq, Ws, g


def nvfp4_sf_to_mma_layout(sf_row_major: torch.Tensor, rows: int, K: int) -> torch.Tensor:
    _check_scales(sf_row_major, rows, K, SF_ROW_MAJOR, "sf_row_major")
    _check_cuda(sf_row_major)
    out = torch.empty(sf_shape(rows, K, SF_MMA_128x4), dtype=torch.uint8,
                      device=sf_row_major.device)
    N.check("nvfp4_sf_to_mma_layout", N.load().nvfp4_sf_to_mma_layout(
        _ptr(sf_row_major), rows, K, _ptr(out), _stream()))
    return out


def gemm_workspace_bytes(M: int, Nn: int, K: int) -> int:
    return int(N.load().nvfp4_gemm_workspace_bytes(M, Nn, K))


def linear_workspace_bytes(M: int, Nn: int, K: int, mode: int = LINEAR_UNFUSED) -> int:
    return int(N.load().nvfp4_linear_workspace_bytes(M, Nn, K, mode))


def nvfp4_gemm(Aq, As, g_a, Bq, Bs, g_b, K: int, Y: torch.Tensor | None = None,
               workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Block-scaled FP4 GEMM, scales in the 128x4 tile layout:
    Y (M, N) bfloat16 = g_a g_b (A_hat @ B_hat^T)."""
    M, Nn = Aq.shape[0], Bq.shape[0]
    _check_codes(Aq, M, K, "Aq")
    _check_codes(Bq, Nn, K, "Bq")
    _check_scales(As, M, K, SF_MMA_128x4, "As")
    _check_scales(Bs, Nn, K, SF_MMA_128x4, "Bs")
    _check_g(g_a, "g_a")
    _check_g(g_b, "g_b")
    _check_cuda(Aq, As, g_a, Bq, Bs, g_b, Y, workspace)
    if Y is None:
        Y = torch.empty((M, Nn), dtype=torch.bfloat16, device=Aq.device)
    _check_bf16_2d(Y, "Y")
    _require(tuple(Y.shape) == (M, Nn), "Y must have shape (%d, %d)" % (M, Nn))
    need = gemm_workspace_bytes(M, Nn, K)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=Aq.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    N.check("nvfp4_gemm", N.load().nvfp4_gemm(
        _ptr(Aq), _ptr(As), _ptr(g_a), _ptr(Bq), _ptr(Bs), _ptr(g_b), M, Nn, K,
        _ptr(Y), Y.stride(0), _ptr(workspace), ws_bytes, _stream()))
    return Y


def _default_mode(mode, workspace) -> int:
    """With no mode given: the fused decode kernel where it applies (it
    produces the same Y, but leaves no quantized X in the workspace), unless
    the caller passes a workspace, whose contents it may then read."""
    if mode is not None:
        return mode
    return LINEAR_FUSED if workspace is None else LINEAR_UNFUSED


def nvfp4_linear(X: torch.Tensor, Wq: torch.Tensor, Ws: torch.Tensor, g_w: torch.Tensor,
                 g_x: torch.Tensor | None = None, mode: int | None = None,
                 Y: torch.Tensor | None = None,
                 workspace: torch.Tensor | None = None) -> torch.Tensor:
    """NVFP4 linear layer: Y = bf16(quant(X) @ dequant(Wq, Ws, g_w)^T), the
    activation quantized on the fly (g_x computed from X when None).
    ``mode`` None: LINEAR_FUSED when no workspace is passed (the one-kernel
    decode path for M <= 8, K <= 6144; the same sequence otherwise), else
    LINEAR_UNFUSED."""
    mode = _default_mode(mode, workspace)
    _check_bf16_2d(X, "X")
    M, K = X.shape
    Nn = Wq.shape[0]
    _check_codes(Wq, Nn, K, "Wq")
    _check_scales(Ws, Nn, K, SF_MMA_128x4, "Ws")
    _check_g(g_w, "g_w")
    if g_x is not None:
        _check_g(g_x, "g_x")
    _check_cuda(X, Wq, Ws, g_w, g_x, Y, workspace)
    if Y is None:
        Y = torch.empty((M, Nn), dtype=torch.bfloat16, device=X.device)
    _check_bf16_2d(Y, "Y")
    _require(tuple(Y.shape) == (M, Nn), "Y must have shape (%d, %d)" % (M, Nn))
    need = linear_workspace_bytes(M, Nn, K, mode)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=X.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    N.check("nvfp4_linear", N.load().nvfp4_linear(
        _ptr(X), M, K, X.stride(0), _ptr(Wq), _ptr(Ws), _ptr(g_w), Nn, _ptr(Y), Y.stride(0),
        _ptr(g_x), mode, _ptr(workspace), ws_bytes, _stream()))
    return Y


def pack_weight_groups(weights):
    """Stack quantized weights [(Wq, Ws, g_w), ...] (scales in the 128x4 tile
    layout, rows a multiple of 256 each) into the operands of
    nvfp4_linear_grouped: (Wq, Ws, g_w (G,), group_n). A one-time copy."""
    _require(1 <= len(weights) <= 8, "1 to 8 weight groups")
    K = weights[0][0].shape[1] * 2
    for Wq, Ws, g in weights:
        n = Wq.shape[0]
        _require(n % 256 == 0, "each group's rows must be a multiple of 256, got %d" % n)
        _check_codes(Wq, n, K, "Wq")
        _check_scales(Ws, n, K, SF_MMA_128x4, "Ws")
        _check_g(g, "g_w")
    Wq = torch.cat([w[0] for w in weights], 0)
    Ws = torch.cat([w[1].view(torch.uint8).reshape(w[0].shape[0], K // 16) for w in weights], 0)
    g = torch.cat([w[2].reshape(-1)[:1] for w in weights], 0)
    return Wq, Ws, g, [int(w[0].shape[0]) for w in weights]


def nvfp4_linear_grouped(X: torch.Tensor, Wq: torch.Tensor, Ws: torch.Tensor,
                         g_w: torch.Tensor, group_n, g_x: torch.Tensor | None = None,
                         mode: int | None = None, Y: torch.Tensor | None = None,
                         workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Several projections of the same X in one call (X quantized once, one
    GEMM launch), group g with its own global scale g_w[g]; Y's columns are
    the groups' outputs side by side (see pack_weight_groups). ``mode`` as
    in nvfp4_linear."""
    import ctypes

    mode = _default_mode(mode, workspace)
    _check_bf16_2d(X, "X")
    M, K = X.shape
    group_n = [int(n) for n in group_n]
    Nn = sum(group_n)
    _check_codes(Wq, Nn, K, "Wq")
    _check_scales(Ws, Nn, K, SF_MMA_128x4, "Ws")
    _require(g_w.dtype == torch.float32 and g_w.numel() == len(group_n) and g_w.is_contiguous(),
             "g_w must be a contiguous float32 tensor with one scale per group")
    if g_x is not None:
        _check_g(g_x, "g_x")
    _check_cuda(X, Wq, Ws, g_w, g_x, Y, workspace)
    if Y is None:
        Y = torch.empty((M, Nn), dtype=torch.bfloat16, device=X.device)
    _check_bf16_2d(Y, "Y")
    _require(tuple(Y.shape) == (M, Nn), "Y must have shape (%d, %d)" % (M, Nn))
    need = linear_workspace_bytes(M, Nn, K, mode)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=X.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    ns = (ctypes.c_int64 * len(group_n))(*group_n)
    N.check("nvfp4_linear_grouped", N.load().nvfp4_linear_grouped(
        _ptr(X), M, K, X.stride(0), _ptr(Wq), _ptr(Ws), _ptr(g_w),
        ctypes.cast(ns, ctypes.c_void_p), len(group_n), _ptr(Y), Y.stride(0), _ptr(g_x), mode,
        _ptr(workspace), ws_bytes, _stream()))
    return Y


def nvfp4_linear_lora(X: torch.Tensor, Wq: torch.Tensor, Ws: torch.Tensor, g_w: torch.Tensor,
                      lora_A: torch.Tensor, lora_B: torch.Tensor, lora_scale: float,
                      g_x: torch.Tensor | None = None, Y: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None) -> torch.Tensor:
    """NVFP4 linear with a run-time LoRA correction lora_scale * (X A^T) B^T
    (A: (r, K), B: (N, r) bfloat16, r in 16/32/48/64) on the unquantized
    activation; the down projection is computed in the quantization pass."""
    _check_bf16_2d(X, "X")
    M, K = X.shape
    Nn = Wq.shape[0]
    _check_codes(Wq, Nn, K, "Wq")
    _check_scales(Ws, Nn, K, SF_MMA_128x4, "Ws")
    _check_g(g_w, "g_w")
    if g_x is not None:
        _check_g(g_x, "g_x")
    r = lora_A.shape[0]
    _require(lora_A.dtype == torch.bfloat16 and tuple(lora_A.shape) == (r, K)
             and lora_A.is_contiguous(), "lora_A must be a contiguous bfloat16 (r, K) tensor")
    _require(lora_B.dtype == torch.bfloat16 and tuple(lora_B.shape) == (Nn, r)
             and lora_B.is_contiguous(), "lora_B must be a contiguous bfloat16 (N, r) tensor")
    _check_cuda(X, Wq, Ws, g_w, g_x, lora_A, lora_B, Y, workspace)
    if Y is None:
        Y = torch.empty((M, Nn), dtype=torch.bfloat16, device=X.device)
    _check_bf16_2d(Y, "Y")
    _require(tuple(Y.shape) == (M, Nn), "Y must have shape (%d, %d)" % (M, Nn))
    need = int(N.load().nvfp4_linear_lora_workspace_bytes(M, Nn, K, r))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=X.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    N.check("nvfp4_linear_lora", N.load().nvfp4_linear_lora(
        _ptr(X), M, K, X.stride(0), _ptr(Wq), _ptr(Ws), _ptr(g_w), Nn, _ptr(lora_A),
        _ptr(lora_B), r, float(lora_scale), _ptr(Y), Y.stride(0), _ptr(g_x), _ptr(workspace),
        ws_bytes, _stream()))
    return Y


def nvfp4_linear_noalloc(X: torch.Tensor, Wq: torch.Tensor, Ws: torch.Tensor,
                         g_w: torch.Tensor, g_x: torch.Tensor | None = None,
                         Y: torch.Tensor | None = None) -> torch.Tensor:
    """nvfp4_linear without a caller-provided workspace: the library keeps
    the scratch in a fixed 16 MiB device array of its own, for callers that
    cannot allocate device memory. Calls that overlap on the GPU race on
    that array."""
    _check_bf16_2d(X, "X")
    M, K = X.shape
    Nn = Wq.shape[0]
    _check_codes(Wq, Nn, K, "Wq")
    _check_scales(Ws, Nn, K, SF_MMA_128x4, "Ws")
    _check_g(g_w, "g_w")
    if g_x is not None:
        _check_g(g_x, "g_x")
    _check_cuda(X, Wq, Ws, g_w, g_x, Y)
    if Y is None:
        Y = torch.empty((M, Nn), dtype=torch.bfloat16, device=X.device)
    _check_bf16_2d(Y, "Y")
    _require(tuple(Y.shape) == (M, Nn), "Y must have shape (%d, %d)" % (M, Nn))
    N.check("nvfp4_linear_noalloc", N.load().nvfp4_linear_noalloc(
        _ptr(X), M, K, X.stride(0), _ptr(Wq), _ptr(Ws), _ptr(g_w), Nn, _ptr(Y), Y.stride(0),
        _ptr(g_x), _stream()))
    return Y


def nvfp4_linear_bias_requant(X: torch.Tensor, Wq: torch.Tensor, Ws: torch.Tensor,
                              g_w: torch.Tensor, g_y: torch.Tensor | None,
                              bias: torch.Tensor | None = None, g_x: torch.Tensor | None = None,
                              store_y: bool = True, Y: torch.Tensor | None = None,
                              Yq: torch.Tensor | None = None, Ys: torch.Tensor | None = None,
                              workspace: torch.Tensor | None = None):
    """nvfp4_linear with the bias add and the NVFP4 re-quantization of the
    bfloat16 output fused into the GEMM epilogue. Returns (Y, Yq, Ys):
    Y is None when store_y is False; Yq (M, N/2) codes and Ys tile-layout
    scales of Y under the global scale g_y are None when g_y is None."""
    _check_bf16_2d(X, "X")
    M, K = X.shape
    Nn = Wq.shape[0]
    _check_codes(Wq, Nn, K, "Wq")
    _check_scales(Ws, Nn, K, SF_MMA_128x4, "Ws")
    _check_g(g_w, "g_w")
    if g_x is not None:
        _check_g(g_x, "g_x")
    if g_y is not None:
        _check_g(g_y, "g_y")
    if bias is not None:
        _require(bias.dtype == torch.bfloat16 and tuple(bias.shape) == (Nn,)
                 and bias.is_contiguous(), "bias must be a contiguous bfloat16 vector of %d" % Nn)
    _check_cuda(X, Wq, Ws, g_w, g_x, g_y, bias, Y, Yq, Ys, workspace)
    if store_y:
        if Y is None:
            Y = torch.empty((M, Nn), dtype=torch.bfloat16, device=X.device)
        _check_bf16_2d(Y, "Y")
        _require(tuple(Y.shape) == (M, Nn), "Y must have shape (%d, %d)" % (M, Nn))
    else:
        Y = None
    if g_y is not None:
        if Yq is None:
            Yq = torch.empty((M, Nn // 2), dtype=torch.uint8, device=X.device)
        if Ys is None:
            Ys = torch.empty(sf_shape(M, Nn, SF_MMA_128x4), dtype=torch.uint8, device=X.device)
        _check_codes(Yq, M, Nn, "Yq")
        _check_scales(Ys, M, Nn, SF_MMA_128x4, "Ys")
    else:
        Yq = Ys = None
    need = linear_workspace_bytes(M, Nn, K, LINEAR_UNFUSED)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=X.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    N.check("nvfp4_linear_bias_requant", N.load().nvfp4_linear_bias_requant(
        _ptr(X), M, K, X.stride(0), _ptr(Wq), _ptr(Ws), _ptr(g_w), Nn, _ptr(bias), _ptr(Y),
        Nn if Y is None else Y.stride(0), _ptr(g_y), _ptr(Yq), _ptr(Ys), _ptr(g_x),
        _ptr(workspace), ws_bytes, _stream()))
    return Y, Yq, Ys


def nvfp4_linear_bias_requant_dynamic(X: torch.Tensor, Wq: torch.Tensor, Ws: torch.Tensor,
                                      g_w: torch.Tensor, bias: torch.Tensor | None = None,
                                      g_x: torch.Tensor | None = None,
                                      Y: torch.Tensor | None = None,
                                      g_y: torch.Tensor | None = None,
                                      Yq: torch.Tensor | None = None,
                                      Ys: torch.Tensor | None = None,
                                      workspace: torch.Tensor | None = None):
    """nvfp4_linear_bias_requant with the output's global scale computed from
    the output (the GEMM epilogue folds max |y| into g_y). Returns
    (Y, g_y, Yq, Ys)."""
    _check_bf16_2d(X, "X")
    M, K = X.shape
    Nn = Wq.shape[0]
    _check_codes(Wq, Nn, K, "Wq")
    _check_scales(Ws, Nn, K, SF_MMA_128x4, "Ws")
    _check_g(g_w, "g_w")
    if g_x is not None:
        _check_g(g_x, "g_x")
    if bias is not None:
        _require(bias.dtype == torch.bfloat16 and tuple(bias.shape) == (Nn,)
                 and bias.is_contiguous(), "bias must be a contiguous bfloat16 vector of %d" % Nn)
    _check_cuda(X, Wq, Ws, g_w, g_x, bias, Y, g_y, Yq, Ys, workspace)
    if Y is None:
        Y = torch.empty((M, Nn), dtype=torch.bfloat16, device=X.device)
    _check_bf16_2d(Y, "Y")
    _require(tuple(Y.shape) == (M, Nn), "Y must have shape (%d, %d)" % (M, Nn))
    if g_y is None:
        g_y = torch.empty(1, dtype=torch.float32, device=X.device)
    _check_g(g_y, "g_y")
    if Yq is None:
        Yq = torch.empty((M, Nn // 2), dtype=torch.uint8, device=X.device)
    if Ys is None:
        Ys = torch.empty(sf_shape(M, Nn, SF_MMA_128x4), dtype=torch.uint8, device=X.device)
    _check_codes(Yq, M, Nn, "Yq")
    _check_scales(Ys, M, Nn, SF_MMA_128x4, "Ys")
    need = linear_workspace_bytes(M, Nn, K, LINEAR_UNFUSED)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=X.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    N.check("nvfp4_linear_bias_requant_dynamic", N.load().nvfp4_linear_bias_requant_dynamic(
        _ptr(X), M, K, X.stride(0), _ptr(Wq), _ptr(Ws), _ptr(g_w), Nn, _ptr(bias), _ptr(Y),
        Y.stride(0), _ptr(g_y), _ptr(Yq), _ptr(Ys), _ptr(g_x), _ptr(workspace), ws_bytes,
        _stream()))
    return Y, g_y, Yq, Ys


def nvfp4_device_error(clear: bool = True) -> int:
    """Synchronize and return the device-side status (OK or ERR_TIMEOUT)."""
    return int(N.load().nvfp4_device_error(1 if clear else 0))


def nvfp4_debug_set_fault_injection(mode: int, timeout_us: int = 0) -> None:
    N.check("nvfp4_debug_set_fault_injection",
            N.load().nvfp4_debug_set_fault_injection(mode, timeout_us))
