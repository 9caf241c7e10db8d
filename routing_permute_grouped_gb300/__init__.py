"""GB300 (sm_103a) dropless MoE layer, forward and backward: Python binding.

Every compute step runs in the CUDA library ``_build/libmoe_gb300.so``
(C ABI in ``include/moe.h``); this module only marshals torch tensors into
pointers, sizes and streams.  There is no fallback: if the library is not
built, every call raises.  Build it with ``routing_permute_grouped_gb300.build.build()``
(or ``__graft_entry__.build()``).

Functions carry the names of the C entry points and take the same
arguments, with torch CUDA tensors in place of device pointers and an
optional ``stream`` (default: torch's current stream).  ``MoeLayer`` is the
user-facing object: it packs the weights once, owns a workspace and runs the
whole layer with one call.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

__all__ = [
    "MoeError", "MoeConfig", "MoeWeights", "MoeLayer", "config_of", "load",
    "moe_check_config", "moe_workspace_size", "moe_workspace_layout", "moe_offsets_workspace_size",
    "moe_pack_router", "moe_pack_experts", "moe_pack_weights", "moe_route", "moe_route_splitk",
    "moe_route_splitk_scratch_size", "moe_build_offsets", "moe_build_offsets_noalloc", "moe_permute",
    "moe_grouped_gemm_swiglu", "moe_grouped_gemm_swiglu_gather",
    "moe_grouped_gemm_swiglu_permute", "moe_shared_expert", "moe_shared_expert_up", "moe_shared_expert_down",
    "moe_shared_expert_down_combine", "moe_combine", "moe_layer_fwd",
    "moe_layer_fwd_prerouted", "moe_get_device_status", "moe_status_string", "HostPipeline",
    "MoeWeightsFp8", "moe_pack_experts_fp8", "moe_permute_fp8", "moe_grouped_gemm_swiglu_skinny",
    "moe_grouped_gemm_swiglu_fp8", "moe_layer_fwd_fp8", "moe_layer_fwd_fp8_prerouted",
    "moe_shared_expert_fp8", "moe_workspace_size_fp8", "moe_workspace_layout_fp8",
    "MoeWeightsBwd", "MoeGrads", "moe_pack_experts_bwd", "moe_pack_router_bwd",
    "moe_backward_workspace_size", "moe_layer_bwd", "moe_gate_up_save_size", "moe_layer_fwd_save",
    "moe_widen_e4m3", "moe_grouped_gemm_swiglu_scaled", "moe_shared_expert_scaled",
    "moe_gather_rows", "moe_build_blocks_from_counts", "moe_copy_pieces",
    "moe_build_offsets_unpadded", "moe_grouped_gemm_swiglu_unpadded",
]

MOE_OK = 0
DEVERR_EXPERT_RANGE = 0x1
DEVERR_TIMEOUT = 0x2


class MoeError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"moe status {status}: {detail}")
        self.status = status


class MoeConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("T", "d", "d_e", "E", "k", "n_groups", "topk_groups", "pad_multiple", "d_shared")]


class MoeWeights(ctypes.Structure):
    _fields_ = [("Wg_t", ctypes.c_void_p), ("bias", ctypes.c_void_p), ("W13", ctypes.c_void_p),
                ("W2", ctypes.c_void_p), ("Ws13", ctypes.c_void_p), ("Ws2", ctypes.c_void_p)]


class MoeWeightsFp8(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("Wg_t", "bias", "W13q", "s13", "W2q", "s2", "Ws13q", "ss13", "Ws2q", "ss2")]


class MoeWeightsBwd(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("W13t", "W2", "WgP", "Ws13t", "Ws2")]


_GRAD_FIELDS = ("dx", "dgates", "dWg", "dbias", "dW1", "dW3", "dW2", "dWs1", "dWs3", "dWs2")


class MoeGrads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _GRAD_FIELDS]


_LAYOUT_FIELDS = ("total", "status", "topk_idx", "topk_w", "counts", "padded_offsets",
                  "block_metadata", "num_blocks", "perm_row", "row_src", "row_gate", "x_perm", "h",
                  "y", "hs", "ys", "router_partial", "xs8", "h8", "row_scale", "w16",
                  "visit_ready")


class _Layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in _LAYOUT_FIELDS]


_lib = None


def library_path() -> str:
    return _build.LIB


def load():
    """Load the built CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(f"CUDA library not built: {path} is missing "
                          "(run routing_permute_grouped_gb300.build.build())")
    lib = ctypes.CDLL(path)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    CP = ctypes.POINTER(MoeConfig)
    sigs = {
        "moe_check_config": (ctypes.c_int, [CP]),
        "moe_workspace_size": (SZ, [CP]),
        "moe_workspace_layout": (ctypes.c_int, [CP, ctypes.POINTER(_Layout)]),
        "moe_offsets_workspace_size": (SZ, [CP]),
        "moe_pack_router": (ctypes.c_int, [I32, I32, P, P, P]),
        "moe_pack_experts": (ctypes.c_int, [I32, I32, I32, P, P, P, P, P, P]),
        "moe_pack_weights": (ctypes.c_int, [CP, P, P, P, P]),
        "moe_route": (ctypes.c_int, [CP, P, P, P, P, P, P]),
        "moe_route_splitk_scratch_size": (SZ, [CP]),
        "moe_route_splitk": (ctypes.c_int, [CP, P, P, P, P, P, P, SZ, P]),
        "moe_build_offsets": (ctypes.c_int, [CP, P, P, P, P, P, P, P, P, P, P, SZ, P]),
        "moe_build_offsets_noalloc": (ctypes.c_int, [CP, P, P, P, P, P, P, P, P, P, P, P]),
        "moe_permute": (ctypes.c_int, [CP, P, P, P, P]),
        "moe_grouped_gemm_swiglu": (ctypes.c_int, [CP, P, P, P, P, P, P, P, P, P, P, P]),
        "moe_grouped_gemm_swiglu_gather": (ctypes.c_int, [CP, P, P, P, P, P, P, P, P, P, P, P, P]),
        "moe_grouped_gemm_swiglu_permute": (ctypes.c_int, [CP] + [P] * 14),
        "moe_shared_expert": (ctypes.c_int, [CP, P, P, P, P, P, P, P]),
        "moe_shared_expert_up": (ctypes.c_int, [CP, P, P, P, P, P, P, P]),
        "moe_shared_expert_down": (ctypes.c_int, [CP, P, P, P, P, P]),
        "moe_shared_expert_down_combine": (ctypes.c_int, [CP, P, P, P, P, P, P, P]),
        "moe_combine": (ctypes.c_int, [CP, P, P, P, P, P]),
        "moe_layer_fwd": (ctypes.c_int, [CP, ctypes.POINTER(MoeWeights), P, P, P, SZ, P]),
        "moe_layer_fwd_prerouted": (ctypes.c_int,
                                    [CP, ctypes.POINTER(MoeWeights), P, P, P, P, P, SZ, P]),
        "moe_pack_experts_fp8": (ctypes.c_int, [I32, I32, I32] + [P] * 8),
        "moe_workspace_size_fp8": (SZ, [CP]),
        "moe_workspace_layout_fp8": (ctypes.c_int, [CP, ctypes.POINTER(_Layout)]),
        "moe_permute_fp8": (ctypes.c_int, [CP] + [P] * 7),
        "moe_grouped_gemm_swiglu_skinny": (ctypes.c_int, [CP] + [P] * 10),
        "moe_grouped_gemm_swiglu_fp8": (ctypes.c_int, [CP] + [P] * 15),
        "moe_shared_expert_fp8": (ctypes.c_int, [CP] + [P] * 12),
        "moe_layer_fwd_fp8": (ctypes.c_int, [CP, ctypes.POINTER(MoeWeightsFp8), P, P, P, SZ, P]),
        "moe_layer_fwd_fp8_prerouted": (ctypes.c_int, [CP, ctypes.POINTER(MoeWeightsFp8), P, P, P,
                                                       P, P, SZ, P]),
        "moe_pack_experts_bwd": (ctypes.c_int, [I32, I32, I32, P, P, P, P]),
        "moe_pack_router_bwd": (ctypes.c_int, [I32, I32, P, P, P]),
        "moe_backward_workspace_size": (SZ, [CP]),
        "moe_gate_up_save_size": (SZ, [CP]),
        "moe_widen_e4m3": (ctypes.c_int, [P, P, ctypes.c_int64, P]),
        "moe_gather_rows": (ctypes.c_int, [P, P, P, ctypes.c_int64, I32, P, P, P]),
        "moe_build_blocks_from_counts": (ctypes.c_int, [P, I32, I32, I32, P, P, P, I32, P, P, P]),
        "moe_copy_pieces": (ctypes.c_int, [P, P, I32, P, P, P, I32, I32, P, P, P]),
        "moe_build_offsets_unpadded": (ctypes.c_int, [CP, P, P, P, P, P, P, P, P, SZ, P]),
        "moe_grouped_gemm_swiglu_unpadded": (ctypes.c_int, [CP, P, P, P, P, P, P, P, P, P]),
        "moe_grouped_gemm_swiglu_scaled": (ctypes.c_int, [CP] + [P] * 13),
        "moe_shared_expert_scaled": (ctypes.c_int, [CP] + [P] * 9),
        "moe_layer_fwd_save": (ctypes.c_int, [CP, ctypes.POINTER(MoeWeights), P, P, P, P, P, SZ,
                                              P, SZ, P]),
        "moe_layer_bwd": (ctypes.c_int, [CP, ctypes.POINTER(MoeWeights),
                                         ctypes.POINTER(MoeWeightsBwd), P, P, P, SZ, P, SZ,
                                         ctypes.POINTER(MoeGrads), P, SZ, P]),
        "moe_get_device_status": (ctypes.c_int, [P, ctypes.POINTER(ctypes.c_uint32), P]),
        "moe_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_uint64, P, P]),
        "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "moe_last_error": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int):
    if status != MOE_OK:
        lib = load()
        raise MoeError(status, f"{lib.moe_status_string(status).decode()}: "
                               f"{lib.moe_last_error().decode()}")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def config_of(shape=None, **kw) -> MoeConfig:
    """MoeConfig from a synth.MoeShape (or keyword fields)."""
    if shape is not None:
        kw = dict(T=shape.T, d=shape.d, d_e=shape.d_e, E=shape.E, k=shape.k,
                  n_groups=shape.n_groups, topk_groups=shape.topk_groups,
                  pad_multiple=shape.pad, d_shared=shape.d_shared, **kw)
    kw.setdefault("n_groups", 0)
    kw.setdefault("topk_groups", 0)
    kw.setdefault("pad_multiple", 128)
    kw.setdefault("d_shared", 0)
    return MoeConfig(**kw)


# ------------------------------------------------------------- sizes ------
def moe_check_config(cfg: MoeConfig) -> None:
    _check(load().moe_check_config(ctypes.byref(cfg)))


def moe_workspace_size(cfg: MoeConfig) -> int:
    return int(load().moe_workspace_size(ctypes.byref(cfg)))


def moe_workspace_layout(cfg: MoeConfig) -> dict:
    L = _Layout()
    _check(load().moe_workspace_layout(ctypes.byref(cfg), ctypes.byref(L)))
    return {n: int(getattr(L, n)) for n in _LAYOUT_FIELDS}


def moe_workspace_size_fp8(cfg: MoeConfig) -> int:
    return int(load().moe_workspace_size_fp8(ctypes.byref(cfg)))


def moe_workspace_layout_fp8(cfg: MoeConfig) -> dict:
    L = _Layout()
    _check(load().moe_workspace_layout_fp8(ctypes.byref(cfg), ctypes.byref(L)))
    return {n: int(getattr(L, n)) for n in _LAYOUT_FIELDS}


def moe_offsets_workspace_size(cfg: MoeConfig) -> int:
    return int(load().moe_offsets_workspace_size(ctypes.byref(cfg)))


# ----------------------------------------------------------- packing ------
def moe_pack_router(Wg: torch.Tensor, Wg_t: torch.Tensor, stream=None) -> None:
    d, E = Wg.shape
    _check(load().moe_pack_router(d, E, _ptr(Wg), _ptr(Wg_t), _stream(stream)))


def moe_pack_experts(W1, W3, W2, W13, W2_t, stream=None) -> None:
    E, d, de = W1.shape
    _check(load().moe_pack_experts(E, d, de, _ptr(W1), _ptr(W3), _ptr(W2), _ptr(W13), _ptr(W2_t),
                                   _stream(stream)))


def moe_pack_weights(cfg: MoeConfig, W1, W3, W13_packed, stream=None) -> None:
    _check(load().moe_pack_weights(ctypes.byref(cfg), _ptr(W1), _ptr(W3), _ptr(W13_packed),
                                   _stream(stream)))


def moe_pack_experts_fp8(W1, W3, W2, W13q, s13, W2q, s2, stream=None) -> None:
    E, d, de = W1.shape
    _check(load().moe_pack_experts_fp8(E, d, de, _ptr(W1), _ptr(W3), _ptr(W2), _ptr(W13q),
                                       _ptr(s13), _ptr(W2q), _ptr(s2), _stream(stream)))


# ------------------------------------------------------------ stages ------
def moe_route(cfg, x, Wg_t, bias, topk_idx, topk_w, stream=None) -> None:
    _check(load().moe_route(ctypes.byref(cfg), _ptr(x), _ptr(Wg_t), _ptr(bias), _ptr(topk_idx),
                            _ptr(topk_w), _stream(stream)))


def moe_route_splitk_scratch_size(cfg) -> int:
    return int(load().moe_route_splitk_scratch_size(ctypes.byref(cfg)))


def moe_route_splitk(cfg, x, Wg_t, bias, topk_idx, topk_w, partial, stream=None) -> None:
    nbytes = 0 if partial is None else partial.numel() * partial.element_size()
    _check(load().moe_route_splitk(ctypes.byref(cfg), _ptr(x), _ptr(Wg_t), _ptr(bias),
                                   _ptr(topk_idx), _ptr(topk_w), _ptr(partial), nbytes,
                                   _stream(stream)))


def moe_build_offsets(cfg, topk_idx, topk_w, counts, padded_offsets, block_metadata, num_blocks,
                      perm_row, row_src, row_gate, ws, stream=None) -> None:
    _check(load().moe_build_offsets(
        ctypes.byref(cfg), _ptr(topk_idx), _ptr(topk_w), _ptr(counts), _ptr(padded_offsets),
        _ptr(block_metadata), _ptr(num_blocks), _ptr(perm_row), _ptr(row_src), _ptr(row_gate),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_build_offsets_noalloc(cfg, topk_idx, topk_w, counts, padded_offsets, block_metadata,
                              num_blocks, perm_row, row_src, row_gate, status=None,
                              stream=None) -> None:
    """moe_build_offsets without a caller-provided scratch: for callers that
    cannot allocate device memory here (stream capture, fixed memory pools).
    The scratch is a fixed array inside the library; see include/moe.h for its
    size limit and for why overlapping calls must be ordered."""
    _check(load().moe_build_offsets_noalloc(
        ctypes.byref(cfg), _ptr(topk_idx), _ptr(topk_w), _ptr(counts), _ptr(padded_offsets),
        _ptr(block_metadata), _ptr(num_blocks), _ptr(perm_row), _ptr(row_src), _ptr(row_gate),
        _ptr(status), _stream(stream)))


def moe_permute(cfg, x, perm_row, x_perm, stream=None) -> None:
    _check(load().moe_permute(ctypes.byref(cfg), _ptr(x), _ptr(perm_row), _ptr(x_perm),
                              _stream(stream)))


def moe_grouped_gemm_swiglu(cfg, x_perm, W13, W2_t, block_metadata, num_blocks, padded_offsets,
                            row_gate, h, y, status=None, stream=None) -> None:
    _check(load().moe_grouped_gemm_swiglu(
        ctypes.byref(cfg), _ptr(x_perm), _ptr(W13), _ptr(W2_t), _ptr(block_metadata),
        _ptr(num_blocks), _ptr(padded_offsets), _ptr(row_gate), _ptr(h), _ptr(y), _ptr(status),
        _stream(stream)))


def moe_grouped_gemm_swiglu_permute(cfg, x, row_src, x_perm, visit_ready, W13, W2_t, block_metadata,
                                    num_blocks, padded_offsets, row_gate, h, y, status=None,
                                    stream=None) -> None:
    _check(load().moe_grouped_gemm_swiglu_permute(
        ctypes.byref(cfg), _ptr(x), _ptr(row_src), _ptr(x_perm), _ptr(visit_ready), _ptr(W13),
        _ptr(W2_t), _ptr(block_metadata), _ptr(num_blocks), _ptr(padded_offsets), _ptr(row_gate),
        _ptr(h), _ptr(y), _ptr(status), _stream(stream)))


def moe_grouped_gemm_swiglu_gather(cfg, x, row_src, W13, W2_t, block_metadata, num_blocks,
                                   padded_offsets, row_gate, h, y, status=None,
                                   stream=None) -> None:
    _check(load().moe_grouped_gemm_swiglu_gather(
        ctypes.byref(cfg), _ptr(x), _ptr(row_src), _ptr(W13), _ptr(W2_t), _ptr(block_metadata),
        _ptr(num_blocks), _ptr(padded_offsets), _ptr(row_gate), _ptr(h), _ptr(y), _ptr(status),
        _stream(stream)))


def moe_permute_fp8(cfg, x, perm_row, x8, x_scale, xs8=None, xs_scale=None, stream=None) -> None:
    _check(load().moe_permute_fp8(ctypes.byref(cfg), _ptr(x), _ptr(perm_row), _ptr(x8),
                                  _ptr(x_scale), _ptr(xs8), _ptr(xs_scale), _stream(stream)))


def moe_grouped_gemm_swiglu_skinny(cfg, x_perm, W13, W2_t, block_metadata, num_blocks, row_gate,
                                   h, y, status=None, stream=None) -> None:
    _check(load().moe_grouped_gemm_swiglu_skinny(
        ctypes.byref(cfg), _ptr(x_perm), _ptr(W13), _ptr(W2_t), _ptr(block_metadata),
        _ptr(num_blocks), _ptr(row_gate), _ptr(h), _ptr(y), _ptr(status), _stream(stream)))


def moe_grouped_gemm_swiglu_fp8(cfg, x8, x_scale, W13q, s13, W2q, s2, block_metadata, num_blocks,
                                row_gate, h, h8, h_scale, y, status=None, stream=None) -> None:
    _check(load().moe_grouped_gemm_swiglu_fp8(
        ctypes.byref(cfg), _ptr(x8), _ptr(x_scale), _ptr(W13q), _ptr(s13), _ptr(W2q), _ptr(s2),
        _ptr(block_metadata), _ptr(num_blocks), _ptr(row_gate), _ptr(h), _ptr(h8), _ptr(h_scale),
        _ptr(y), _ptr(status), _stream(stream)))


def moe_shared_expert_fp8(cfg, xs8, xs_scale, Ws13q, ss13, Ws2q, ss2, hs, hs8, hs_scale, ys,
                          status=None, stream=None) -> None:
    _check(load().moe_shared_expert_fp8(ctypes.byref(cfg), _ptr(xs8), _ptr(xs_scale), _ptr(Ws13q),
                                        _ptr(ss13), _ptr(Ws2q), _ptr(ss2), _ptr(hs), _ptr(hs8),
                                        _ptr(hs_scale), _ptr(ys), _ptr(status), _stream(stream)))


def moe_shared_expert(cfg, x, Ws13, Ws2_t, hs, ys, status=None, stream=None) -> None:
    _check(load().moe_shared_expert(ctypes.byref(cfg), _ptr(x), _ptr(Ws13), _ptr(Ws2_t), _ptr(hs),
                                    _ptr(ys), _ptr(status), _stream(stream)))


def moe_shared_expert_up(cfg, x, Ws13, hs, perm_row=None, x_perm=None, status=None,
                         stream=None) -> None:
    _check(load().moe_shared_expert_up(ctypes.byref(cfg), _ptr(x), _ptr(Ws13), _ptr(hs),
                                       _ptr(perm_row), _ptr(x_perm), _ptr(status),
                                       _stream(stream)))


def moe_shared_expert_down(cfg, hs, Ws2_t, ys, status=None, stream=None) -> None:
    _check(load().moe_shared_expert_down(ctypes.byref(cfg), _ptr(hs), _ptr(Ws2_t), _ptr(ys),
                                         _ptr(status), _stream(stream)))


def moe_shared_expert_down_combine(cfg, hs, Ws2_t, y, perm_row, out, status=None,
                                   stream=None) -> None:
    _check(load().moe_shared_expert_down_combine(ctypes.byref(cfg), _ptr(hs), _ptr(Ws2_t),
                                                 _ptr(y), _ptr(perm_row), _ptr(out),
                                                 _ptr(status), _stream(stream)))


def moe_combine(cfg, y, perm_row, shared_out, out, stream=None) -> None:
    _check(load().moe_combine(ctypes.byref(cfg), _ptr(y), _ptr(perm_row), _ptr(shared_out),
                              _ptr(out), _stream(stream)))


def moe_layer_fwd(cfg, weights: MoeWeights, x, out, ws, stream=None) -> None:
    _check(load().moe_layer_fwd(ctypes.byref(cfg), ctypes.byref(weights), _ptr(x), _ptr(out),
                                _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_layer_fwd_prerouted(cfg, weights: MoeWeights, x, topk_idx, topk_w, out, ws,
                            stream=None) -> None:
    _check(load().moe_layer_fwd_prerouted(
        ctypes.byref(cfg), ctypes.byref(weights), _ptr(x), _ptr(topk_idx), _ptr(topk_w), _ptr(out),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_layer_fwd_fp8(cfg, weights: MoeWeightsFp8, x, out, ws, stream=None) -> None:
    _check(load().moe_layer_fwd_fp8(ctypes.byref(cfg), ctypes.byref(weights), _ptr(x), _ptr(out),
                                    _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_layer_fwd_fp8_prerouted(cfg, weights: MoeWeightsFp8, x, topk_idx, topk_w, out, ws,
                                stream=None) -> None:
    _check(load().moe_layer_fwd_fp8_prerouted(
        ctypes.byref(cfg), ctypes.byref(weights), _ptr(x), _ptr(topk_idx), _ptr(topk_w), _ptr(out),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


# ---------------------------------------------------------- backward ------
def moe_pack_experts_bwd(W1, W3, W13t, stream=None) -> None:
    """W13t [E, d, 2*d_e] from W1, W3 [E, d, d_e] (bf16, CUDA)."""
    E, d, de = W1.shape
    _check(load().moe_pack_experts_bwd(E, d, de, _ptr(W1), _ptr(W3), _ptr(W13t), _stream(stream)))


def moe_pack_router_bwd(Wg, WgP, stream=None) -> None:
    """WgP [d, Ep] (Ep = E rounded up to 128, zero past E) from Wg [d, E]."""
    d, E = Wg.shape
    _check(load().moe_pack_router_bwd(d, E, _ptr(Wg), _ptr(WgP), _stream(stream)))


def moe_backward_workspace_size(cfg: MoeConfig) -> int:
    return int(load().moe_backward_workspace_size(ctypes.byref(cfg)))


def moe_gather_rows(src, idx, dst, src_gate=None, dst_gate=None, stream=None) -> None:
    """dst[i] = src[idx[i]] (bf16 rows; gates too when given)."""
    _check(load().moe_gather_rows(_ptr(src), _ptr(idx), _ptr(dst), idx.numel(), src.shape[-1],
                                  _ptr(src_gate), _ptr(dst_gate), _stream(stream)))


def moe_build_blocks_from_counts(counts, P: int, padded_offsets, block_metadata, num_blocks,
                                 piece_row=None, status=None, stream=None) -> None:
    """The expert-major layout of rows that arrive as counts [n_src, E] (int32,
    device): padded offsets, block table, and where each sender's rows land."""
    n_src, E = counts.shape
    _check(load().moe_build_blocks_from_counts(
        _ptr(counts), n_src, E, P, _ptr(padded_offsets), _ptr(block_metadata), _ptr(num_blocks),
        block_metadata.shape[0], _ptr(piece_row), _ptr(status), _stream(stream)))


def moe_copy_pieces(src, dst, src_row, dst_row, rows, max_rows: int, src_gate=None, dst_gate=None,
                    stream=None) -> None:
    """Row pieces src[src_row[i] : + rows[i]] -> dst[dst_row[i] : + rows[i]]
    (device int32 descriptors; gates alongside when given)."""
    _check(load().moe_copy_pieces(_ptr(src), _ptr(dst), src.shape[-1], _ptr(src_row),
                                  _ptr(dst_row), _ptr(rows), rows.numel(), int(max_rows),
                                  _ptr(src_gate), _ptr(dst_gate), _stream(stream)))


def moe_build_offsets_unpadded(cfg, topk_idx, topk_w, counts, group_offsets, perm_row, row_src,
                               row_gate, ws, stream=None) -> None:
    """Counts, group offsets [E + 1] and the permutation of the unpadded
    layout (A rows, no padding, no block table)."""
    _check(load().moe_build_offsets_unpadded(
        ctypes.byref(cfg), _ptr(topk_idx), _ptr(topk_w), _ptr(counts), _ptr(group_offsets),
        _ptr(perm_row), _ptr(row_src), _ptr(row_gate), _ptr(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


def moe_grouped_gemm_swiglu_unpadded(cfg, x_perm, W13, W2_t, group_offsets, row_gate, h, y,
                                     status=None, stream=None) -> None:
    """The grouped GEMMs on the unpadded layout (windows cut by an expert
    boundary run once per expert)."""
    _check(load().moe_grouped_gemm_swiglu_unpadded(
        ctypes.byref(cfg), _ptr(x_perm), _ptr(W13), _ptr(W2_t), _ptr(group_offsets),
        _ptr(row_gate), _ptr(h), _ptr(y), _ptr(status), _stream(stream)))


def moe_widen_e4m3(q, out, stream=None) -> None:
    """bf16 out (same element count) from e4m3 codes q (uint8)."""
    _check(load().moe_widen_e4m3(_ptr(q), _ptr(out), q.numel(), _stream(stream)))


def moe_grouped_gemm_swiglu_scaled(cfg, x_perm, W13, s13, W2_t, s2, block_metadata, num_blocks,
                                   padded_offsets, row_gate, h, y, status=None,
                                   stream=None) -> None:
    _check(load().moe_grouped_gemm_swiglu_scaled(
        ctypes.byref(cfg), _ptr(x_perm), _ptr(W13), _ptr(s13), _ptr(W2_t), _ptr(s2),
        _ptr(block_metadata), _ptr(num_blocks), _ptr(padded_offsets), _ptr(row_gate), _ptr(h),
        _ptr(y), _ptr(status), _stream(stream)))


def moe_shared_expert_scaled(cfg, x, Ws13, ss13, Ws2_t, ss2, hs, ys, status=None,
                             stream=None) -> None:
    _check(load().moe_shared_expert_scaled(ctypes.byref(cfg), _ptr(x), _ptr(Ws13), _ptr(ss13),
                                           _ptr(Ws2_t), _ptr(ss2), _ptr(hs), _ptr(ys), _ptr(status),
                                           _stream(stream)))


def moe_gate_up_save_size(cfg: MoeConfig) -> int:
    return int(load().moe_gate_up_save_size(ctypes.byref(cfg)))


def moe_layer_fwd_save(cfg, weights: MoeWeights, x, out, ws, gu_save, topk_idx=None, topk_w=None,
                       stream=None) -> None:
    """moe_layer_fwd (or the pre-routed form) that also saves the gate/up
    values for moe_layer_bwd in gu_save (moe_gate_up_save_size bytes)."""
    _check(load().moe_layer_fwd_save(
        ctypes.byref(cfg), ctypes.byref(weights), _ptr(x), _ptr(topk_idx), _ptr(topk_w), _ptr(out),
        _ptr(ws), ws.numel() * ws.element_size(), _ptr(gu_save),
        gu_save.numel() * gu_save.element_size(), _stream(stream)))


def moe_layer_bwd(cfg, weights: MoeWeights, wbwd: MoeWeightsBwd, x, dout, ws, grads: dict, bws,
                  gu_saved=None, stream=None) -> None:
    """Backward of moe_layer_fwd(_prerouted / _save); ``grads`` maps the
    moe_grads_t field names to caller-owned CUDA tensors (missing or None =
    NULL); ``gu_saved`` is the gate/up save of moe_layer_fwd_save, or None to
    recompute it."""
    g = MoeGrads(**{n: (None if grads.get(n) is None else _ptr(grads[n]).value)
                    for n in _GRAD_FIELDS})
    gu_bytes = 0 if gu_saved is None else gu_saved.numel() * gu_saved.element_size()
    _check(load().moe_layer_bwd(ctypes.byref(cfg), ctypes.byref(weights), ctypes.byref(wbwd),
                                _ptr(x), _ptr(dout), _ptr(ws), ws.numel() * ws.element_size(),
                                _ptr(gu_saved), gu_bytes, ctypes.byref(g), _ptr(bws),
                                bws.numel() * bws.element_size(), _stream(stream)))


def moe_get_device_status(ws, stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error bits."""
    bits = ctypes.c_uint32(0)
    st = load().moe_get_device_status(_ptr(ws), ctypes.byref(bits), _stream(stream))
    if st not in (MOE_OK, 5):
        _check(st)
    return int(bits.value)


def moe_selftest_wait_timeout(limit_ns: int, status, stream=None) -> None:
    _check(load().moe_selftest_wait_timeout(limit_ns, _ptr(status), _stream(stream)))


def moe_status_string(status: int) -> str:
    return load().moe_status_string(status).decode()


# --------------------------------------------------------- the layer ------
class MoeLayer:
    """One dropless MoE layer on the current CUDA device.

    Packs the weights once (``moe_pack_router`` / ``moe_pack_experts``) and
    owns a workspace sized for ``T`` tokens.  ``forward(x)`` runs
    ``moe_layer_fwd`` (or the pre-routed variant) on the current stream.
    Weights use the pages' orientation: Wg [d, E], W1/W3 [E, d, d_e],
    W2 [E, d_e, d], shared Ws1/Ws3 [d, d_s], Ws2 [d_s, d]; all bf16 CUDA
    tensors; bias fp32 [E] or None.  ``fp8=True`` packs the routed and shared
    expert weights as e4m3 codes with per-output-channel scales
    (``moe_pack_experts_fp8``) and runs ``moe_layer_fwd_fp8``.
    """

    def __init__(self, cfg: MoeConfig, W1, W3, W2, Wg=None, bias=None, Ws1=None, Ws3=None, Ws2=None,
                 stream=None, fp8: bool = False, keep_gate_up: bool = False):
        moe_check_config(cfg)
        self.cfg = cfg
        self.fp8 = fp8
        # keep_gate_up: every forward saves the gate/up values (moe_layer_fwd_save)
        # and the backward reads them instead of recomputing them
        self.keep_gate_up = keep_gate_up and not fp8
        self.gu_save = None
        if self.keep_gate_up:
            self.gu_save = torch.empty(moe_gate_up_save_size(cfg), dtype=torch.uint8,
                                       device=W1.device)
        dev = W1.device
        E, d, de = W1.shape
        if fp8:
            self._init_fp8(cfg, W1, W3, W2, Wg, bias, Ws1, Ws3, Ws2, stream)
            return
        # the caller's weights, kept by reference for the backward packs
        self._user = dict(W1=W1, W3=W3, W2=W2, Wg=Wg, Ws1=Ws1, Ws3=Ws3, Ws2=Ws2)
        self.wbwd = None
        self.W13 = torch.empty((E, 2 * de, d), dtype=torch.bfloat16, device=dev)
        self.W2_t = torch.empty((E, d, de), dtype=torch.bfloat16, device=dev)
        moe_pack_experts(W1, W3, W2, self.W13, self.W2_t, stream)
        self.Wg_t = None
        if Wg is not None:
            self.Wg_t = torch.empty((E, d), dtype=torch.bfloat16, device=dev)
            moe_pack_router(Wg, self.Wg_t, stream)
        self.bias = None if bias is None else bias.to(device=dev, dtype=torch.float32).contiguous()
        self.Ws13 = self.Ws2_t = None
        if cfg.d_shared:
            ds = cfg.d_shared
            self.Ws13 = torch.empty((1, 2 * ds, d), dtype=torch.bfloat16, device=dev)
            self.Ws2_t = torch.empty((1, d, ds), dtype=torch.bfloat16, device=dev)
            moe_pack_experts(Ws1.unsqueeze(0).contiguous(), Ws3.unsqueeze(0).contiguous(),
                             Ws2.unsqueeze(0).contiguous(), self.Ws13, self.Ws2_t, stream)
        self.weights = MoeWeights(
            Wg_t=None if self.Wg_t is None else self.Wg_t.data_ptr(),
            bias=None if self.bias is None else self.bias.data_ptr(),
            W13=self.W13.data_ptr(), W2=self.W2_t.data_ptr(),
            Ws13=None if self.Ws13 is None else self.Ws13.data_ptr(),
            Ws2=None if self.Ws2_t is None else self.Ws2_t.data_ptr())
        self._init_ws(cfg, dev)

    def _init_ws(self, cfg, dev):
        self.layout = moe_workspace_layout_fp8(cfg) if self.fp8 else moe_workspace_layout(cfg)
        self.ws = torch.empty(self.layout["total"], dtype=torch.uint8, device=dev)
        self.ws[:256].zero_()

    def _init_fp8(self, cfg, W1, W3, W2, Wg, bias, Ws1, Ws3, Ws2, stream):
        dev = W1.device
        E, d, de = W1.shape

        def pack(w1, w3, w2, n, width):
            q13 = torch.empty((n, 2 * width, d), dtype=torch.uint8, device=dev)
            s13 = torch.empty((n, 2 * width), dtype=torch.float32, device=dev)
            q2 = torch.empty((n, d, width), dtype=torch.uint8, device=dev)
            s2 = torch.empty((n, d), dtype=torch.float32, device=dev)
            moe_pack_experts_fp8(w1, w3, w2, q13, s13, q2, s2, stream)
            return q13, s13, q2, s2

        self.W13q, self.s13, self.W2q, self.s2 = pack(W1, W3, W2, E, de)
        self.Wg_t = None
        if Wg is not None:
            self.Wg_t = torch.empty((E, d), dtype=torch.bfloat16, device=dev)
            moe_pack_router(Wg, self.Wg_t, stream)
        self.bias = None if bias is None else bias.to(device=dev, dtype=torch.float32).contiguous()
        self.Ws13q = self.ss13 = self.Ws2q = self.ss2 = None
        if cfg.d_shared:
            self.Ws13q, self.ss13, self.Ws2q, self.ss2 = pack(
                Ws1.unsqueeze(0).contiguous(), Ws3.unsqueeze(0).contiguous(),
                Ws2.unsqueeze(0).contiguous(), 1, cfg.d_shared)

        def p(t):
            return None if t is None else t.data_ptr()

        self.weights = MoeWeightsFp8(
            Wg_t=p(self.Wg_t), bias=p(self.bias), W13q=p(self.W13q), s13=p(self.s13),
            W2q=p(self.W2q), s2=p(self.s2), Ws13q=p(self.Ws13q), ss13=p(self.ss13),
            Ws2q=p(self.Ws2q), ss2=p(self.ss2))
        self._init_ws(cfg, dev)

    def forward(self, x, out=None, topk_idx=None, topk_w=None, stream=None):
        if out is None:
            out = torch.empty_like(x)
        if self.fp8:
            if topk_idx is None:
                moe_layer_fwd_fp8(self.cfg, self.weights, x, out, self.ws, stream)
            else:
                moe_layer_fwd_fp8_prerouted(self.cfg, self.weights, x, topk_idx, topk_w, out,
                                            self.ws, stream)
        elif self.keep_gate_up:
            moe_layer_fwd_save(self.cfg, self.weights, x, out, self.ws, self.gu_save,
                               topk_idx=topk_idx, topk_w=topk_w, stream=stream)
        elif topk_idx is None:
            moe_layer_fwd(self.cfg, self.weights, x, out, self.ws, stream)
        else:
            moe_layer_fwd_prerouted(self.cfg, self.weights, x, topk_idx, topk_w, out, self.ws,
                                    stream)
        return out

    __call__ = forward

    def _init_bwd(self, stream=None):
        u = self._user
        dev = u["W1"].device
        E, d, de = u["W1"].shape
        self.W13t = torch.empty((E, d, 2 * de), dtype=torch.bfloat16, device=dev)
        moe_pack_experts_bwd(u["W1"], u["W3"], self.W13t, stream)
        self.WgP = None
        if u["Wg"] is not None:
            self.WgP = torch.empty((d, (E + 127) // 128 * 128), dtype=torch.bfloat16, device=dev)
            moe_pack_router_bwd(u["Wg"], self.WgP, stream)
        self.Ws13t = None
        if self.cfg.d_shared:
            self.Ws13t = torch.empty((1, d, 2 * self.cfg.d_shared), dtype=torch.bfloat16,
                                     device=dev)
            moe_pack_experts_bwd(u["Ws1"].unsqueeze(0).contiguous(),
                                 u["Ws3"].unsqueeze(0).contiguous(), self.Ws13t, stream)

        def p(t):
            return None if t is None else t.data_ptr()

        self.wbwd = MoeWeightsBwd(W13t=p(self.W13t), W2=p(u["W2"]), WgP=p(self.WgP),
                                  Ws13t=p(self.Ws13t), Ws2=p(u["Ws2"]))
        self.bws = torch.empty(moe_backward_workspace_size(self.cfg), dtype=torch.uint8,
                               device=dev)

    def backward(self, x, dout, grads: Optional[dict] = None, prerouted: bool = False,
                 stream=None) -> dict:
        """Gradients of the last ``forward(x)`` (its workspace must be unchanged)
        for the output gradient ``dout`` [T, d] bf16: a dict with dx, dgates,
        dW1, dW3, dW2, the shared dWs1/dWs3/dWs2 and, for a routed forward,
        dWg and dbias (``moe_layer_bwd``).  ``prerouted`` marks a forward that
        was given its routing (no router term)."""
        if self.fp8:
            raise NotImplementedError("the backward runs on bf16 expert weights")
        if self.wbwd is None:
            self._init_bwd(stream)
        cfg, dev = self.cfg, x.device
        T, d, de, E, k = cfg.T, cfg.d, cfg.d_e, cfg.E, cfg.k
        if grads is None:
            bf = dict(dtype=torch.bfloat16, device=dev)
            f32 = dict(dtype=torch.float32, device=dev)
            grads = dict(dx=torch.empty((T, d), **bf), dgates=torch.empty((T, k), **f32),
                         dW1=torch.empty((E, d, de), **bf), dW3=torch.empty((E, d, de), **bf),
                         dW2=torch.empty((E, de, d), **bf))
            routed = self.WgP is not None and not prerouted
            if routed:
                grads["dWg"] = torch.empty((d, E), **f32)
                grads["dbias"] = torch.empty((E,), **f32)
            if cfg.d_shared:
                ds = cfg.d_shared
                grads.update(dWs1=torch.empty((d, ds), **bf), dWs3=torch.empty((d, ds), **bf),
                             dWs2=torch.empty((ds, d), **bf))
        wb = self.wbwd
        if prerouted and wb.WgP is not None:
            wb = MoeWeightsBwd(W13t=wb.W13t, W2=wb.W2, WgP=None, Ws13t=wb.Ws13t, Ws2=wb.Ws2)
        moe_layer_bwd(self.cfg, self.weights, wb, x, dout, self.ws, grads, self.bws,
                      gu_saved=self.gu_save, stream=stream)
        return grads

    def buffer(self, name: str, dtype, shape, offset: int = 0) -> torch.Tensor:
        """A view of one intermediate of the workspace (see moe_workspace_layout),
        starting ``offset`` bytes into its region."""
        off = self.layout[name] + offset
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return self.ws[off:off + nbytes].view(dtype).view(*shape)

    def device_status(self, stream=None) -> int:
        return moe_get_device_status(self.ws, stream)


class HostPipeline:
    """Runs a MoeLayer on token batches held in pinned host memory.

    Each submitted batch is copied to the device, run through the layer and
    copied back; the copies of neighbouring batches overlap the layer's
    compute (three streams: copy-in, compute, copy-out, with ``depth``
    device buffers in rotation).  ``synchronize()`` waits for every submitted
    batch.  The layer's own workspace is reused batch after batch, so layer
    calls stay ordered on the compute stream.
    """

    def __init__(self, layer: MoeLayer, depth: int = 2):
        T, d = layer.cfg.T, layer.cfg.d
        dev = layer.ws.device
        self.layer = layer
        self.depth = depth
        self.s_in = torch.cuda.Stream(device=dev)
        self.s_run = torch.cuda.Stream(device=dev)
        self.s_out = torch.cuda.Stream(device=dev)
        self.x_dev = [torch.empty((T, d), dtype=torch.bfloat16, device=dev) for _ in range(depth)]
        self.o_dev = [torch.empty((T, d), dtype=torch.bfloat16, device=dev) for _ in range(depth)]
        self.ev_in = [torch.cuda.Event() for _ in range(depth)]
        self.ev_run = [torch.cuda.Event() for _ in range(depth)]
        self.ev_out = [torch.cuda.Event() for _ in range(depth)]
        self.used = [False] * depth
        self.i = 0

    def submit(self, x_host: torch.Tensor, out_host: torch.Tensor, topk_idx=None, topk_w=None):
        k = self.i % self.depth
        self.i += 1
        if self.used[k]:
            self.s_in.wait_event(self.ev_run[k])    # x buffer no longer read
            self.s_run.wait_event(self.ev_out[k])   # out buffer copied back
        self.used[k] = True
        with torch.cuda.stream(self.s_in):
            self.x_dev[k].copy_(x_host, non_blocking=True)
            if topk_idx is not None and not topk_idx.is_cuda:
                # pre-routed batches carry their routing from the host too
                if not hasattr(self, "idx_dev"):
                    self.idx_dev = [torch.empty_like(topk_idx, device=self.x_dev[0].device)
                                    for _ in range(self.depth)]
                    self.w_dev = [torch.empty_like(topk_w, device=self.x_dev[0].device)
                                  for _ in range(self.depth)]
                self.idx_dev[k].copy_(topk_idx, non_blocking=True)
                self.w_dev[k].copy_(topk_w, non_blocking=True)
                topk_idx, topk_w = self.idx_dev[k], self.w_dev[k]
            self.ev_in[k].record(self.s_in)
        self.s_run.wait_event(self.ev_in[k])
        self.layer.forward(self.x_dev[k], self.o_dev[k], topk_idx=topk_idx, topk_w=topk_w,
                           stream=self.s_run)
        self.ev_run[k].record(self.s_run)
        self.s_out.wait_event(self.ev_run[k])
        with torch.cuda.stream(self.s_out):
            out_host.copy_(self.o_dev[k], non_blocking=True)
            self.ev_out[k].record(self.s_out)

    def submit_train(self, x_host: torch.Tensor, dout_host: torch.Tensor, dx_host: torch.Tensor,
                     grads: dict, topk_idx=None, topk_w=None):
        """Forward and backward of one batch: x and the output gradient dout
        copied in from pinned host memory, dx copied back; the weight
        gradients (and dgates) land in the device tensors of ``grads``,
        overwritten by every batch.  Copies overlap the compute of the
        neighbouring batches as in ``submit``."""
        k = self.i % self.depth
        self.i += 1
        if not hasattr(self, "dout_dev"):
            self.dout_dev = [torch.empty_like(x) for x in self.x_dev]
            self.dx_dev = [torch.empty_like(x) for x in self.x_dev]
        if self.used[k]:
            self.s_in.wait_event(self.ev_run[k])    # x and dout buffers no longer read
            self.s_run.wait_event(self.ev_out[k])   # dx buffer copied back
        self.used[k] = True
        prerouted = topk_idx is not None
        with torch.cuda.stream(self.s_in):
            self.x_dev[k].copy_(x_host, non_blocking=True)
            self.dout_dev[k].copy_(dout_host, non_blocking=True)
            if prerouted and not topk_idx.is_cuda:
                if not hasattr(self, "idx_dev"):
                    self.idx_dev = [torch.empty_like(topk_idx, device=self.x_dev[0].device)
                                    for _ in range(self.depth)]
                    self.w_dev = [torch.empty_like(topk_w, device=self.x_dev[0].device)
                                  for _ in range(self.depth)]
                self.idx_dev[k].copy_(topk_idx, non_blocking=True)
                self.w_dev[k].copy_(topk_w, non_blocking=True)
                topk_idx, topk_w = self.idx_dev[k], self.w_dev[k]
            self.ev_in[k].record(self.s_in)
        self.s_run.wait_event(self.ev_in[k])
        self.layer.forward(self.x_dev[k], self.o_dev[k], topk_idx=topk_idx, topk_w=topk_w,
                           stream=self.s_run)
        g = dict(grads)
        g["dx"] = self.dx_dev[k]
        self.layer.backward(self.x_dev[k], self.dout_dev[k], grads=g, prerouted=prerouted,
                            stream=self.s_run)
        self.ev_run[k].record(self.s_run)
        self.s_out.wait_event(self.ev_run[k])
        with torch.cuda.stream(self.s_out):
            dx_host.copy_(self.dx_dev[k], non_blocking=True)
            self.ev_out[k].record(self.s_out)

    def synchronize(self):
        for s in (self.s_in, self.s_run, self.s_out):
            s.synchronize()
