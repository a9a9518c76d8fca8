"""Thin Python binding of libmxmoe.so: argument marshalling only.

Each function has the name of the C entry point it calls, takes CUDA torch
tensors, allocates its outputs with torch (device memory is PyTorch's job),
checks dtypes/shapes/contiguity, and passes raw pointers plus the current
CUDA stream.  Every step of the computation runs in the library's kernels.
"""

from __future__ import annotations

import ctypes as C

import torch

from . import _lib


def _ptr(t):
    return C.c_void_p(t.data_ptr()) if t is not None else C.c_void_p(0)


def _stream():
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def _need(t, name, dtype, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name}: expected {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _u8(t):
    return t.view(torch.uint8) if t.dtype in (torch.float8_e4m3fn, torch.int8) else t


def mx_quantize_3d(w: torch.Tensor):
    """bf16 [E, N, K] (or [N, K]) -> (e4m3 payload uint8 same shape, e8m0 scales uint8 [.., ceil(K/32)]).

    K % 16 == 0; with K % 32 == 16 each row ends in a partial block of 16."""
    _need(w, "w", torch.bfloat16)
    shape = tuple(w.shape)
    if w.dim() == 2:
        E, (N, K) = 1, shape
    elif w.dim() == 3:
        E, N, K = shape
    else:
        raise ValueError("w must be 2D or 3D")
    q = torch.empty(shape, dtype=torch.uint8, device=w.device)
    s = torch.empty(shape[:-1] + ((K + 31) // 32 if K % 16 == 0 else 0,), dtype=torch.uint8,
                    device=w.device)
    _lib.check("mx_quantize_3d", _lib.load().mx_quantize_3d(
        _ptr(w), E, N, K, _ptr(q), _ptr(s), _stream()))
    return q, s


def mx_quantize_fp4_3d(w: torch.Tensor):
    """bf16 [E, N, K] (or [N, K]) -> (packed MXFP4 uint8 [.., K/2], e8m0 scales uint8 [.., K/32]).

    W4A8 weights: e2m1 elements, two per byte (element 2i in the low nibble)."""
    _need(w, "w", torch.bfloat16)
    shape = tuple(w.shape)
    if w.dim() == 2:
        E, (N, K) = 1, shape
    elif w.dim() == 3:
        E, N, K = shape
    else:
        raise ValueError("w must be 2D or 3D")
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    q = torch.empty(shape[:-1] + (K // 2,), dtype=torch.uint8, device=w.device)
    s = torch.empty(shape[:-1] + (K // 32,), dtype=torch.uint8, device=w.device)
    _lib.check("mx_quantize_fp4_3d", _lib.load().mx_quantize_fp4_3d(
        _ptr(w), E, N, K, _ptr(q), _ptr(s), _stream()))
    return q, s


def _route(x, logits, k, renormalize, quant):
    _need(x, "x", torch.bfloat16, 2)
    _need(logits, "logits", torch.float32, 2)
    T, H = x.shape
    E = logits.shape[1]
    if logits.shape[0] != T:
        raise ValueError("x and logits disagree on T")
    dev = x.device
    M = T * k
    L = _lib.load()
    ws_bytes = L.moe_route_quant_mxfp8_workspace_size(T, E)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    out = dict(
        topk_ids=torch.empty(T, k, dtype=torch.int32, device=dev),
        topk_w=torch.empty(T, k, dtype=torch.float32, device=dev),
        sorted_to_src=torch.empty(M, dtype=torch.int32, device=dev),
        src_to_sorted=torch.empty(M, dtype=torch.int32, device=dev),
        expert_counts=torch.empty(E, dtype=torch.int64, device=dev),
        expert_offsets=torch.empty(E + 1, dtype=torch.int64, device=dev),
    )
    common = (_ptr(out["topk_ids"]), _ptr(out["topk_w"]), _ptr(out["sorted_to_src"]),
              _ptr(out["src_to_sorted"]), _ptr(out["expert_counts"]),
              _ptr(out["expert_offsets"]), _ptr(ws), ws.numel(), _stream())
    if quant:
        out["xq"] = torch.empty(M, H, dtype=torch.uint8, device=dev)
        out["xs"] = torch.empty(M, H // 32, dtype=torch.uint8, device=dev)
        _lib.check("moe_route_quant_mxfp8", L.moe_route_quant_mxfp8(
            _ptr(x), _ptr(logits), T, H, E, k, int(bool(renormalize)), _ptr(out["xq"]),
            _ptr(out["xs"]), *common))
    else:
        out["xp"] = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
        _lib.check("moe_route_permute_bf16", L.moe_route_permute_bf16(
            _ptr(x), _ptr(logits), T, H, E, k, int(bool(renormalize)), _ptr(out["xp"]), *common))
    return out


def moe_route_quant_mxfp8(x, logits, k: int, renormalize: bool = True) -> dict:
    """Routing + permutation with the MX activation quant fused (quant_mode=3)."""
    return _route(x, logits, k, renormalize, True)


def moe_route_permute_bf16(x, logits, k: int, renormalize: bool = True) -> dict:
    """Routing + permutation writing bf16 expanded rows (two-step comparator)."""
    return _route(x, logits, k, renormalize, False)


def grouped_gemm_swiglu_quant_mxfp8(xq, xs, w13q, w13s, expert_offsets):
    """gmm1 + SwiGLU + requant -> (aq uint8 [M, I], as uint8 [M, I/32])."""
    xq, w13q = _u8(xq), _u8(w13q)
    _need(xq, "xq", torch.uint8, 2)
    _need(xs, "xs", torch.uint8, 2)
    _need(w13q, "w13q", torch.uint8, 3)
    _need(w13s, "w13s", torch.uint8, 3)
    _need(expert_offsets, "expert_offsets", torch.int64, 1)
    M, H = xq.shape
    E, N2, _ = w13q.shape
    I = N2 // 2
    if expert_offsets.numel() != E + 1:
        raise ValueError("expert_offsets must have E+1 entries")
    aq = torch.empty(M, I, dtype=torch.uint8, device=xq.device)
    as_ = torch.empty(M, I // 32, dtype=torch.uint8, device=xq.device)
    _lib.check("grouped_gemm_swiglu_quant_mxfp8", _lib.load().grouped_gemm_swiglu_quant_mxfp8(
        _ptr(xq), _ptr(xs), _ptr(w13q), _ptr(w13s), _ptr(expert_offsets), M, E, H, I,
        _ptr(aq), _ptr(as_), _stream()))
    return aq, as_


def grouped_gemm_mxfp8(aq, as_, w2q, w2s, expert_offsets):
    """gmm2 -> y bf16 [M, H]."""
    aq, w2q = _u8(aq), _u8(w2q)
    _need(aq, "aq", torch.uint8, 2)
    _need(as_, "as", torch.uint8, 2)
    _need(w2q, "w2q", torch.uint8, 3)
    _need(w2s, "w2s", torch.uint8, 3)
    _need(expert_offsets, "expert_offsets", torch.int64, 1)
    M, I = aq.shape
    E, H, _ = w2q.shape
    y = torch.empty(M, H, dtype=torch.bfloat16, device=aq.device)
    _lib.check("grouped_gemm_mxfp8", _lib.load().grouped_gemm_mxfp8(
        _ptr(aq), _ptr(as_), _ptr(w2q), _ptr(w2s), _ptr(expert_offsets), M, E, I, H, _ptr(y),
        _stream()))
    return y


def moe_finalize_routing(y, topk_w, src_to_sorted, k: int):
    """Weighted top-k combine -> out bf16 [T, H]."""
    _need(y, "y", torch.bfloat16, 2)
    _need(topk_w, "topk_w", torch.float32, 2)
    _need(src_to_sorted, "src_to_sorted", torch.int32, 1)
    T = topk_w.shape[0]
    H = y.shape[1]
    out = torch.empty(T, H, dtype=torch.bfloat16, device=y.device)
    _lib.check("moe_finalize_routing", _lib.load().moe_finalize_routing(
        _ptr(y), _ptr(topk_w), _ptr(src_to_sorted), T, k, H, _ptr(out), _stream()))
    return out


def moe_forward_mxfp8_workspace_size(T: int, H: int, E: int, k: int, I: int) -> int:
    return int(_lib.load().moe_forward_mxfp8_workspace_size(T, H, E, k, I))


def moe_forward_mxfp8(x, logits, w13q, w13s, w2q, w2s, k: int, renormalize: bool = True,
                      out=None, workspace=None):
    """The whole expert forward on the current stream -> out bf16 [T, H]."""
    w13q, w2q = _u8(w13q), _u8(w2q)
    _need(x, "x", torch.bfloat16, 2)
    _need(logits, "logits", torch.float32, 2)
    for t, n in ((w13q, "w13q"), (w13s, "w13s"), (w2q, "w2q"), (w2s, "w2s")):
        _need(t, n, torch.uint8, 3)
    T, H = x.shape
    E, N2, _ = w13q.shape
    I = N2 // 2
    ws_bytes = moe_forward_mxfp8_workspace_size(T, H, E, k, I)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=x.device)
    _lib.check("moe_forward_mxfp8", _lib.load().moe_forward_mxfp8(
        _ptr(x), _ptr(logits), _ptr(w13q), _ptr(w13s), _ptr(w2q), _ptr(w2s), T, H, E, k, I,
        int(bool(renormalize)), _ptr(out), _ptr(workspace), workspace.numel(), _stream()))
    return out


def mx_scales_to_mma_layout(scale, K: int):
    """e8m0 scales [E, N, ceil(K/32)] (or [N, ceil(K/32)]) -> the tensor-core layout.

    The result has shape [.., ceil(N/128)*128, ceil(K/128)*4] (the input's
    shape when N and K are multiples of 128); it is an opaque byte array."""
    _need(scale, "scale", torch.uint8)
    if scale.dim() == 2:
        E, N = 1, scale.shape[0]
    elif scale.dim() == 3:
        E, N = scale.shape[0], scale.shape[1]
    else:
        raise ValueError("scale must be 2D or 3D")
    tiled = (-(-N // 128) * 128, -(-K // 128) * 4)
    out = torch.empty(tuple(scale.shape[:-2]) + tiled, dtype=torch.uint8, device=scale.device)
    _lib.check("mx_scales_to_mma_layout", _lib.load().mx_scales_to_mma_layout(
        _ptr(scale), E, N, K, _ptr(out), _stream()))
    return out


def moe_forward_mxfp8_mma_scales(x, logits, w13q, w13s_mma, w2q, w2s_mma, k: int,
                                 renormalize: bool = True, out=None, workspace=None):
    """moe_forward_mxfp8 with weight scales already in the tensor-core layout."""
    w13q, w2q = _u8(w13q), _u8(w2q)
    _need(x, "x", torch.bfloat16, 2)
    _need(logits, "logits", torch.float32, 2)
    for t, n in ((w13q, "w13q"), (w13s_mma, "w13s_mma"), (w2q, "w2q"), (w2s_mma, "w2s_mma")):
        _need(t, n, torch.uint8, 3)
    T, H = x.shape
    E, N2, _ = w13q.shape
    I = N2 // 2
    ws_bytes = moe_forward_mxfp8_workspace_size(T, H, E, k, I)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=x.device)
    _lib.check("moe_forward_mxfp8_mma_scales", _lib.load().moe_forward_mxfp8_mma_scales(
        _ptr(x), _ptr(logits), _ptr(w13q), _ptr(w13s_mma), _ptr(w2q), _ptr(w2s_mma), T, H, E, k, I,
        int(bool(renormalize)), _ptr(out), _ptr(workspace), workspace.numel(), _stream()))
    return out


def moe_forward_w4a8_mma_scales(x, logits, w13p, w13s_mma, w2p, w2s_mma, k: int,
                                renormalize: bool = True, out=None, workspace=None):
    """The W4A8 layer: packed MXFP4 expert weights (mx_quantize_fp4_3d) with
    their scales in the tensor-core layout, MXFP8 activations."""
    return _fp4_layer("moe_forward_w4a8_mma_scales", x, logits, w13p, w13s_mma, w2p, w2s_mma, k,
                      renormalize, out, workspace)


def moe_forward_w4a4_mma_scales(x, logits, w13p, w13s_mma, w2p, w2s_mma, k: int,
                                renormalize: bool = True, out=None, workspace=None):
    """The W4A4 layer: packed MXFP4 expert weights, and each grouped GEMM's
    input quantized to MXFP4 on the device (the routed hidden states, and
    the SwiGLU output)."""
    return _fp4_layer("moe_forward_w4a4_mma_scales", x, logits, w13p, w13s_mma, w2p, w2s_mma, k,
                      renormalize, out, workspace)


def _fp4_layer(fn, x, logits, w13p, w13s_mma, w2p, w2s_mma, k, renormalize, out, workspace):
    _need(x, "x", torch.bfloat16, 2)
    _need(logits, "logits", torch.float32, 2)
    for t, n in ((w13p, "w13p"), (w13s_mma, "w13s_mma"), (w2p, "w2p"), (w2s_mma, "w2s_mma")):
        _need(t, n, torch.uint8, 3)
    T, H = x.shape
    E, N2, _ = w13p.shape
    I = N2 // 2
    if w13p.shape[2] * 2 != H or w2p.shape[2] * 2 != I:
        raise ValueError("w13p / w2p must be packed [E, 2I, H/2] / [E, H, I/2]")
    ws_bytes = moe_forward_mxfp8_workspace_size(T, H, E, k, I)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=x.device)
    _lib.check(fn, getattr(_lib.load(), fn)(
        _ptr(x), _ptr(logits), _ptr(w13p), _ptr(w13s_mma), _ptr(w2p), _ptr(w2s_mma), T, H, E, k, I,
        int(bool(renormalize)), _ptr(out), _ptr(workspace), workspace.numel(), _stream()))
    return out


def moe_forward_mxfp8_host_workspace_size(T: int, H: int, E: int, k: int, I: int,
                                          n_chunks: int = 0) -> int:
    return int(_lib.load().moe_forward_mxfp8_host_workspace_size(T, H, E, k, I, n_chunks))


def moe_forward_mxfp8_host(x_host, logits_host, w13q, w13s_mma, w2q, w2s_mma, k: int,
                           renormalize: bool = True, out_host=None, n_chunks: int = 0,
                           workspace=None, chunks=None):
    """The layer on host (CPU, ideally pinned) tensors, copies overlapped with compute.

    Weights and their MMA-layout scales are CUDA tensors.  Returns out_host
    (bf16 [T, H] on the host); it is complete once the current stream is.
    `chunks` (a list of token counts summing to T) selects an explicit chunk
    plan (moe_forward_mxfp8_host_plan); otherwise `n_chunks` (0 = default plan).
    """
    w13q, w2q = _u8(w13q), _u8(w2q)
    for t, n in ((x_host, "x_host"), (logits_host, "logits_host")):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous host tensor")
    if x_host.dtype != torch.bfloat16 or logits_host.dtype != torch.float32:
        raise TypeError("x_host must be bf16 and logits_host fp32")
    for t, n in ((w13q, "w13q"), (w13s_mma, "w13s_mma"), (w2q, "w2q"), (w2s_mma, "w2s_mma")):
        _need(t, n, torch.uint8, 3)
    T, H = x_host.shape
    E, N2, _ = w13q.shape
    I = N2 // 2
    if out_host is None:
        out_host = torch.empty(T, H, dtype=torch.bfloat16, pin_memory=True)
    if chunks is not None:
        plan = (C.c_int32 * len(chunks))(*[int(c) for c in chunks])
        need = moe_forward_mxfp8_host_workspace_size(max(chunks), H, E, k, I, 1)
    else:
        need = moe_forward_mxfp8_host_workspace_size(T, H, E, k, I, n_chunks)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=w13q.device)
    if chunks is not None:
        _lib.check("moe_forward_mxfp8_host_plan", _lib.load().moe_forward_mxfp8_host_plan(
            _ptr(x_host), _ptr(logits_host), _ptr(w13q), _ptr(w13s_mma), _ptr(w2q), _ptr(w2s_mma),
            T, H, E, k, I, int(bool(renormalize)), _ptr(out_host), C.cast(plan, C.c_void_p),
            len(chunks), _ptr(workspace), workspace.numel(), _stream()))
    else:
        _lib.check("moe_forward_mxfp8_host", _lib.load().moe_forward_mxfp8_host(
            _ptr(x_host), _ptr(logits_host), _ptr(w13q), _ptr(w13s_mma), _ptr(w2q), _ptr(w2s_mma),
            T, H, E, k, I, int(bool(renormalize)), _ptr(out_host), int(n_chunks),
            _ptr(workspace), workspace.numel(), _stream()))
    return out_host


def device_status(clear: bool = True) -> int:
    """The library's device status word (synchronizes the device)."""
    v = C.c_int32(0)
    _lib.check("mxmoe_get_device_status", _lib.load().mxmoe_get_device_status(C.byref(v), int(clear)))
    return int(v.value)


def layer_profile_enable(enable=True) -> None:
    """Record CUDA events between the layer call's kernels (instrumentation):
    True / 1 = every boundary, "gemm1" / 2 = only around gmm1 (the other
    boundaries keep their overlapped launches), False / 0 = off."""
    mode = 2 if enable == "gemm1" else int(enable)
    _lib.check("mxmoe_layer_profile_enable", _lib.load().mxmoe_layer_profile_enable(mode))


def layer_profile_read() -> dict:
    """Per-kernel milliseconds of the last profiled layer call (synchronizes)."""
    arr = (C.c_float * 5)()
    _lib.check("mxmoe_layer_profile_read", _lib.load().mxmoe_layer_profile_read(arr, 5))
    keys = ("weight_scale_layout", "route_quant", "gemm1_swiglu_quant", "gemm2", "finalize")
    return dict(zip(keys, (float(v) for v in arr)))


def linear_profile_read() -> dict:
    """Per-kernel milliseconds of the last profiled dense-linear call (synchronizes)."""
    arr = (C.c_float * 3)()
    _lib.check("mxmoe_layer_profile_read", _lib.load().mxmoe_layer_profile_read(arr, 3))
    return dict(zip(("weight_scale_layout", "act_quant", "gemm"), (float(v) for v in arr)))


def set_gemm_2sm(mode="auto") -> None:
    """Grouped-GEMM kernel choice: False/0 = 1-SM kernel, True/1 = 2-SM kernel
    (cta_group::2) for the layer's 256-wide tiles, "auto"/2 (the default) =
    2-SM for grouped GEMM2 when it has at least 512 rows per expert on
    average and for grouped GEMM1 at 1024.  Both kernels give the same bytes."""
    m = 2 if mode == "auto" else int(mode)
    _lib.load().mxmoe_set_gemm_2sm(m)


def set_gemm_chain(enable: bool = True) -> None:
    """Small MXFP8 batches (at most 32 tokens): both grouped GEMMs in one
    persistent kernel (True, the default) or one kernel each (False).  Both
    give the same bytes; with one kernel the layer profile reports the pair's
    time as gmm1's and 0 for gmm2."""
    _lib.load().mxmoe_set_gemm_chain(1 if enable else 0)


def set_wait_limit_cycles(cycles: int) -> None:
    _lib.load().mxmoe_set_wait_limit_cycles(int(cycles))


def moe_router_gate_topk(x, gate, k: int, renormalize: bool = True, logits=False) -> dict:
    """The router gate GEMM fused with softmax top-k: bf16 x [T, H] and bf16
    gate [E, H] -> topk_ids int32 [T, k], topk_w fp32 [T, k] (and the fp32
    logits [T, E] when ``logits``)."""
    _need(x, "x", torch.bfloat16, 2)
    _need(gate, "gate", torch.bfloat16, 2)
    T, H = x.shape
    E = gate.shape[0]
    if gate.shape[1] != H:
        raise ValueError(f"gate is {tuple(gate.shape)}, x has H = {H}")
    dev = x.device
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    lg = torch.empty(T, E, dtype=torch.float32, device=dev) if logits else None
    _lib.check("moe_router_gate_topk", _lib.load().moe_router_gate_topk(
        _ptr(x), _ptr(gate), T, H, E, k, int(bool(renormalize)), _ptr(lg), _ptr(ids), _ptr(w),
        _stream()))
    out = dict(topk_ids=ids, topk_w=w)
    if logits:
        out["logits"] = lg
    return out


def mx_dequantize_bf16_2d(q, scale):
    """e4m3 [N, K] (uint8 codes) + e8m0 [N, K/32] -> bf16 [N, K] (the offline
    MXFP8 router gate, dequantized once at load)."""
    q = _u8(q)
    _need(q, "q", torch.uint8, 2)
    _need(scale, "scale", torch.uint8, 2)
    N, K = q.shape
    out = torch.empty(N, K, dtype=torch.bfloat16, device=q.device)
    _lib.check("mx_dequantize_bf16_2d", _lib.load().mx_dequantize_bf16_2d(
        _ptr(q), _ptr(scale), N, K, _ptr(out), _stream()))
    return out


def moe_forward_mxfp8_gated_mma_scales(x, gate, w13q, w13s_mma, w2q, w2s_mma, k: int,
                                       renormalize: bool = True, out=None, workspace=None):
    """The MXFP8 layer from the hidden states and the bf16 router gate [E, H]:
    the gate GEMM and softmax top-k run fused in the routing step."""
    w13q, w2q = _u8(w13q), _u8(w2q)
    _need(x, "x", torch.bfloat16, 2)
    _need(gate, "gate", torch.bfloat16, 2)
    for t, n in ((w13q, "w13q"), (w13s_mma, "w13s_mma"), (w2q, "w2q"), (w2s_mma, "w2s_mma")):
        _need(t, n, torch.uint8, 3)
    T, H = x.shape
    E, N2, _ = w13q.shape
    I = N2 // 2
    ws_bytes = moe_forward_mxfp8_workspace_size(T, H, E, k, I)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=x.device)
    _lib.check("moe_forward_mxfp8_gated_mma_scales",
               _lib.load().moe_forward_mxfp8_gated_mma_scales(
                   _ptr(x), _ptr(gate), _ptr(w13q), _ptr(w13s_mma), _ptr(w2q), _ptr(w2s_mma), T,
                   H, E, k, I, int(bool(renormalize)), _ptr(out), _ptr(workspace),
                   workspace.numel(), _stream()))
    return out


def mxfp8_linear_workspace_size(M: int, N: int, K: int) -> int:
    return int(_lib.load().mxfp8_linear_workspace_size(M, N, K))


def _linear(fn, x, wq, ws, out, workspace, packed=False):
    wq = _u8(wq)
    _need(x, "x", torch.bfloat16)
    _need(wq, "wq", torch.uint8, 2)
    _need(ws, "ws", torch.uint8, 2)
    K = x.shape[-1]
    N = wq.shape[0]
    if wq.shape[1] * (2 if packed else 1) != K:
        raise ValueError(f"wq is {tuple(wq.shape)}, x has K = {K}")
    M = x.numel() // K if K else 0
    need = mxfp8_linear_workspace_size(M, N, K)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty(tuple(x.shape[:-1]) + (N,), dtype=torch.bfloat16, device=x.device)
    _need(out, "out", torch.bfloat16)
    _lib.check(fn, getattr(_lib.load(), fn)(
        _ptr(x), _ptr(wq), _ptr(ws), M, N, K, _ptr(out), _ptr(workspace), workspace.numel(),
        _stream()))
    return out


def mxfp8_linear(x, wq, ws, out=None, workspace=None):
    """Dense MXFP8 linear: bf16 x [.., K] -> bf16 [.., N], x MX-quantized per
    token on the device; wq e4m3 [N, K] and ws e8m0 [N, ceil(K/32)] from
    mx_quantize_3d (or an offline checkpoint)."""
    return _linear("mxfp8_linear", x, wq, ws, out, workspace)


def mxfp8_linear_mma_scales(x, wq, ws_mma, out=None, workspace=None):
    """mxfp8_linear with the weight scales already in the tensor-core layout."""
    return _linear("mxfp8_linear_mma_scales", x, wq, ws_mma, out, workspace)


def mxfp4_linear(x, wp, ws, out=None, workspace=None):
    """W4A4 dense linear: bf16 x [.., K] -> bf16 [.., N], x MXFP4-quantized per
    token on the device; wp packed MXFP4 [N, K/2] and ws e8m0 [N, K/32] from
    mx_quantize_fp4_3d (or an offline checkpoint).  K % 128 == 0."""
    return _linear("mxfp4_linear", x, wp, ws, out, workspace, packed=True)


def mxfp4_linear_mma_scales(x, wp, ws_mma, out=None, workspace=None):
    """mxfp4_linear with the weight scales already in the tensor-core layout."""
    return _linear("mxfp4_linear_mma_scales", x, wp, ws_mma, out, workspace, packed=True)


class MXFP4Linear:
    """A W4A4 dense linear layer: packed MXFP4 weights [N, K/2] with e8m0 block
    scales; activations quantized to MXFP4 per token at each call."""

    def __init__(self, wp, ws):
        self.wp, self.ws = _u8(wp), ws
        self.N, k2 = self.wp.shape
        self.K = 2 * k2
        self.ws_mma = mx_scales_to_mma_layout(self.ws, self.K)
        self._ws = None

    @classmethod
    def from_bf16(cls, w):
        return cls(*mx_quantize_fp4_3d(w))

    @classmethod
    def from_quantized(cls, wp, ws):
        return cls(wp, ws)

    def workspace(self, M: int, device):
        need = mxfp8_linear_workspace_size(M, self.N, self.K)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        return self._ws

    def __call__(self, x, out=None):
        M = x.numel() // self.K
        return mxfp4_linear_mma_scales(x, self.wp, self.ws_mma, out=out,
                                       workspace=self.workspace(M, x.device))


class MXFP8Linear:
    """A dense MXFP8 linear layer: e4m3 weights [N, K] with e8m0 block scales.

    ``from_bf16`` quantizes a bf16 weight [N, K] (out_features, in_features)
    on the device at load (the online path); ``from_quantized`` takes an
    offline checkpoint's payload and [N, ceil(K/32)] scales.  The scales are
    re-laid out once into the tensor-core layout; calls quantize the
    activations per token and run the block-scaled GEMM.
    """

    def __init__(self, wq, ws):
        self.wq, self.ws = _u8(wq), ws
        self.N, self.K = self.wq.shape
        self.ws_mma = mx_scales_to_mma_layout(self.ws, self.K)
        self._ws = None

    @classmethod
    def from_bf16(cls, w):
        return cls(*mx_quantize_3d(w))

    @classmethod
    def from_quantized(cls, wq, ws):
        return cls(wq, ws)

    def workspace(self, M: int, device):
        need = mxfp8_linear_workspace_size(M, self.N, self.K)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        return self._ws

    def __call__(self, x, out=None):
        M = x.numel() // self.K
        return mxfp8_linear_mma_scales(x, self.wq, self.ws_mma, out=out,
                                       workspace=self.workspace(M, x.device))


class MXFP8MoELayer:
    """MX-quantized expert weights plus a reusable workspace for one layer shape.

    At construction the weight scales are also re-laid out once into the
    tensor-core layout (``mx_scales_to_mma_layout``); calls go through
    ``moe_forward_mxfp8_mma_scales``.

    ``from_bf16`` quantizes bf16 w13 [E, 2I, H] / w2 [E, H, I] on the device
    (the online, load-time path); ``from_quantized`` takes an offline
    checkpoint's e4m3 payload and e8m0 scales as they are.
    """

    def __init__(self, w13q, w13s, w2q, w2s, k: int, renormalize: bool = True):
        self.w13q, self.w13s, self.w2q, self.w2s = _u8(w13q), w13s, _u8(w2q), w2s
        self.k = k
        self.renormalize = renormalize
        self.E, n2, self.H = self.w13q.shape
        self.I = n2 // 2
        # load time: the scales in the tensor-core layout the layer call reads
        self.w13s_mma = mx_scales_to_mma_layout(self.w13s, self.H)
        self.w2s_mma = mx_scales_to_mma_layout(self.w2s, self.I)
        self._ws = None

    @classmethod
    def from_bf16(cls, w13, w2, k: int, renormalize: bool = True):
        w13q, w13s = mx_quantize_3d(w13)
        w2q, w2s = mx_quantize_3d(w2)
        return cls(w13q, w13s, w2q, w2s, k, renormalize)

    @classmethod
    def from_quantized(cls, w13q, w13s, w2q, w2s, k: int, renormalize: bool = True):
        return cls(w13q, w13s, w2q, w2s, k, renormalize)

    def workspace(self, T: int, device):
        need = moe_forward_mxfp8_workspace_size(T, self.H, self.E, self.k, self.I)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        return self._ws

    def forward_host(self, x_host, logits_host, out_host=None, n_chunks: int = 0, chunks=None):
        """The layer on host tensors (copies overlapped with compute, chunked by tokens)."""
        T = x_host.shape[0]
        if chunks is not None:
            need = moe_forward_mxfp8_host_workspace_size(max(chunks), self.H, self.E, self.k,
                                                         self.I, 1)
        else:
            need = moe_forward_mxfp8_host_workspace_size(T, self.H, self.E, self.k, self.I,
                                                         n_chunks)
        if getattr(self, "_hws", None) is None or self._hws.numel() < need:
            self._hws = torch.empty(max(need, 256), dtype=torch.uint8, device=self.w13q.device)
        return moe_forward_mxfp8_host(x_host, logits_host, self.w13q, self.w13s_mma, self.w2q,
                                      self.w2s_mma, self.k, self.renormalize, out_host=out_host,
                                      n_chunks=n_chunks, workspace=self._hws, chunks=chunks)

    def __call__(self, x, logits, out=None):
        return moe_forward_mxfp8_mma_scales(x, logits, self.w13q, self.w13s_mma, self.w2q,
                                            self.w2s_mma, self.k, self.renormalize, out=out,
                                            workspace=self.workspace(x.shape[0], x.device))

    def forward_gated(self, x, gate, out=None):
        """The layer from the hidden states and the bf16 router gate [E, H] (the
        gate GEMM and top-k fused into the routing step)."""
        return moe_forward_mxfp8_gated_mma_scales(x, gate, self.w13q, self.w13s_mma, self.w2q,
                                                  self.w2s_mma, self.k, self.renormalize,
                                                  out=out,
                                                  workspace=self.workspace(x.shape[0], x.device))


class W4A4MoELayer:
    """MXFP4 (packed e2m1) expert weights with MXFP4 expert inputs (W4A4).

    The routed hidden states and the SwiGLU output are quantized to MXFP4 on
    the device right before the grouped GEMM that reads them.  Weights as for
    ``W4A8MoELayer``.
    """

    def __init__(self, w13p, w13s, w2p, w2s, k: int, renormalize: bool = True):
        self.w13p, self.w13s, self.w2p, self.w2s = _u8(w13p), w13s, _u8(w2p), w2s
        self.k = k
        self.renormalize = renormalize
        self.E, n2, h2 = self.w13p.shape
        self.H, self.I = 2 * h2, n2 // 2
        self.w13s_mma = mx_scales_to_mma_layout(self.w13s, self.H)
        self.w2s_mma = mx_scales_to_mma_layout(self.w2s, self.I)
        self._ws = None

    @classmethod
    def from_bf16(cls, w13, w2, k: int, renormalize: bool = True):
        w13p, w13s = mx_quantize_fp4_3d(w13)
        w2p, w2s = mx_quantize_fp4_3d(w2)
        return cls(w13p, w13s, w2p, w2s, k, renormalize)

    @classmethod
    def from_quantized(cls, w13p, w13s, w2p, w2s, k: int, renormalize: bool = True):
        return cls(w13p, w13s, w2p, w2s, k, renormalize)

    def workspace(self, T: int, device):
        need = moe_forward_mxfp8_workspace_size(T, self.H, self.E, self.k, self.I)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        return self._ws

    def __call__(self, x, logits, out=None):
        return moe_forward_w4a4_mma_scales(x, logits, self.w13p, self.w13s_mma, self.w2p,
                                           self.w2s_mma, self.k, self.renormalize, out=out,
                                           workspace=self.workspace(x.shape[0], x.device))


class W4A8MoELayer:
    """MXFP4 (packed e2m1) expert weights with MXFP8 activations (W4A8).

    ``from_bf16`` quantizes bf16 w13 [E, 2I, H] / w2 [E, H, I] to MXFP4 on the
    device at load (the online path); ``from_quantized`` takes packed FP4
    payloads [E, N, K/2] and e8m0 scales [E, N, K/32] as an offline checkpoint
    ships them.  Scales are re-laid out once into the tensor-core layout.
    """

    def __init__(self, w13p, w13s, w2p, w2s, k: int, renormalize: bool = True):
        self.w13p, self.w13s, self.w2p, self.w2s = _u8(w13p), w13s, _u8(w2p), w2s
        self.k = k
        self.renormalize = renormalize
        self.E, n2, h2 = self.w13p.shape
        self.H, self.I = 2 * h2, n2 // 2
        self.w13s_mma = mx_scales_to_mma_layout(self.w13s, self.H)
        self.w2s_mma = mx_scales_to_mma_layout(self.w2s, self.I)
        self._ws = None

    @classmethod
    def from_bf16(cls, w13, w2, k: int, renormalize: bool = True):
        w13p, w13s = mx_quantize_fp4_3d(w13)
        w2p, w2s = mx_quantize_fp4_3d(w2)
        return cls(w13p, w13s, w2p, w2s, k, renormalize)

    @classmethod
    def from_quantized(cls, w13p, w13s, w2p, w2s, k: int, renormalize: bool = True):
        return cls(w13p, w13s, w2p, w2s, k, renormalize)

    def workspace(self, T: int, device):
        need = moe_forward_mxfp8_workspace_size(T, self.H, self.E, self.k, self.I)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        return self._ws

    def __call__(self, x, logits, out=None):
        return moe_forward_w4a8_mma_scales(x, logits, self.w13p, self.w13s_mma, self.w2p,
                                           self.w2s_mma, self.k, self.renormalize, out=out,
                                           workspace=self.workspace(x.shape[0], x.device))


def moe_route_quant_mxfp8_noalloc(x, logits, k: int, renormalize: bool = True) -> dict:
    """moe_route_quant_mxfp8 through the entry point that takes no workspace.

    For callers that cannot allocate device scratch: the library keeps the
    routing scratch in a fixed 1 MiB device array (ceil(T/64)*E <= 262144).
    The outputs are still allocated here, by torch, like every other binding.
    """
    _need(x, "x", torch.bfloat16, 2)
    _need(logits, "logits", torch.float32, 2)
    T, H = x.shape
    E = logits.shape[1]
    dev = x.device
    M = T * k
    out = dict(
        topk_ids=torch.empty(T, k, dtype=torch.int32, device=dev),
        topk_w=torch.empty(T, k, dtype=torch.float32, device=dev),
        sorted_to_src=torch.empty(M, dtype=torch.int32, device=dev),
        src_to_sorted=torch.empty(M, dtype=torch.int32, device=dev),
        expert_counts=torch.empty(E, dtype=torch.int64, device=dev),
        expert_offsets=torch.empty(E + 1, dtype=torch.int64, device=dev),
        xq=torch.empty(M, H, dtype=torch.uint8, device=dev),
        xs=torch.empty(M, H // 32, dtype=torch.uint8, device=dev),
    )
    _lib.check("moe_route_quant_mxfp8_noalloc", _lib.load().moe_route_quant_mxfp8_noalloc(
        _ptr(x), _ptr(logits), T, H, E, k, int(bool(renormalize)), _ptr(out["xq"]),
        _ptr(out["xs"]), _ptr(out["topk_ids"]), _ptr(out["topk_w"]), _ptr(out["sorted_to_src"]),
        _ptr(out["src_to_sorted"]), _ptr(out["expert_counts"]), _ptr(out["expert_offsets"]),
        _stream()))
    return out
