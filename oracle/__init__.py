"""Plain fp64 CPU oracle of the dropless MoE layer forward pass.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library: the arithmetic lives in ``moe_oracle.c`` (plain loops,
fp64 on exactly widened bf16 inputs); this module only compiles it with gcc,
marshals numpy arrays and chains the stages in the order the pages give
("MoE & MLA operators", sec. 2.1: router -> permute -> grouped GEMM ->
combine; "Dropless and grouped GEMM", sec. 1: routed + shared).

Array conventions (numpy):
  bf16 tensors are passed as their uint16 bit patterns; x [T, d],
  Wg [d, E], W1/W3 [E, d, de], W2 [E, de, d], Ws1/Ws3 [d, ds], Ws2 [ds, d];
  bias float32 [E]; topk_idx int32 [T, k]; gates float64;
  e4m3 weights as uint8 codes in the layout of the bf16 matrix they stand
  for, with float32 scales per output channel (Q1/Q3 [E, d, de] with S1/S3
  [E, de], Q2 [E, de, d] with S2 [E, d]).

Pinned by ``tests/test_oracle_pins.py`` against the padding worked example
("Dropless and grouped GEMM", sec. 3), the ledger figures, brute-force
routing, a stable library argsort, closed-form softmax identities, the
textbook dense SwiGLU MLP (k = 1, E = 1) and the exact permute/direct
equivalence ("MoE & MLA operators", sec. 2.3).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I, LL, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_double
            sig = {
                "or_bf16_to_double": (D, [ctypes.c_uint16]),
                "or_round_bf16": (D, [D]),
                "or_double_to_bf16_bits": (ctypes.c_uint16, [D]),
                "or_router_logits": (None, [I, I, I, P, P, P, P]),
                "or_route": (I, [I, I, I, I, I, P, P, P, P]),
                "or_rows_capacity": (LL, [LL, I, I]),
                "or_blocks_capacity": (LL, [LL, I, I]),
                "or_build_offsets": (I, [LL, I, I, P, P, P, P, P, P, P, P, P]),
                "or_blocks_from_counts": (I, [I, I, I, P, P, P, P, P]),
                "or_permute": (None, [LL, I, I, P, P, P]),
                "or_grouped_experts": (I, [I, I, I, I, P, P, P, P, P, P, P, P]),
                "or_expert_rows": (I, [I, I, I, I, P, P, P, P, P, P, P, P]),
                "or_shared_expert": (I, [I, I, I, P, P, P, P, P, P]),
                "or_combine": (None, [I, I, I, P, P, P, P]),
                "or_direct_layer": (I, [I, P, I, I, I, I, P, P, P, P, P, P, P, P]),
                "or_round_bf16_array": (None, [LL, P, P]),
                "or_num_threads": (I, []),
                "or_e4m3_to_double": (D, [ctypes.c_uint8]),
                "or_double_to_e4m3": (ctypes.c_uint8, [D]),
                "or_quantize_e4m3_columns": (None, [I, I, P, P, P]),
                "or_quantize_e4m3_batch": (None, [I, I, I, P, P, P]),
                "or_expert_rows_w8": (I, [I, I, I, I] + [P] * 11),
                "or_e4m3_to_double_array": (None, [LL, P, P]),
                "or_double_to_e4m3_array": (None, [LL, P, P]),
                "or_layer_backward": (I, [I] * 6 + [P] * 22),
                "or_weight_grad_columns": (I, [I] * 3 + [P] * 6 + [I] + [P] * 4),
            }
            for name, (res, args) in sig.items():
                f = getattr(lib, name)
                f.restype = res
                f.argtypes = args
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc == 1:
        raise ValueError(f"oracle {what}: invalid argument")
    if rc == 2:
        raise ValueError(f"oracle {what}: expert id out of range")


def num_threads() -> int:
    return int(_L().or_num_threads())


# ---------------------------------------------------------------- bf16 ----
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to fp64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_bf16(v: np.ndarray) -> np.ndarray:
    """fp64 -> nearest bf16 value (ties to even), returned as fp64."""
    a = _c(v, np.float64)
    out = np.empty_like(a)
    _L().or_round_bf16_array(a.size, _p(a), _p(out))
    return out


# --------------------------------------------------------------- stages ----
def rows_capacity(A: int, E: int, P: int) -> int:
    return int(_L().or_rows_capacity(A, E, P))


def blocks_capacity(A: int, E: int, P: int) -> int:
    return int(_L().or_blocks_capacity(A, E, P))


def router_logits(x, Wg, bias=None) -> np.ndarray:
    x = _c(x, np.uint16)
    Wg = _c(Wg, np.uint16)
    T, d = x.shape
    E = Wg.shape[1]
    assert Wg.shape[0] == d
    b = None if bias is None else _c(bias, np.float32)
    out = np.empty((T, E), np.float64)
    _L().or_router_logits(T, d, E, _p(x), _p(Wg), _p(b), _p(out))
    return out


def route(logits, k: int, n_groups: int = 0, topk_groups: int = 0):
    """Top-k (optionally group-limited) routing -> (idx int32 [T,k],
    gates fp64 [T,k], margin fp64 [T])."""
    lg = _c(logits, np.float64)
    T, E = lg.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    m = np.empty((T,), np.float64)
    _check(_L().or_route(T, E, k, n_groups, topk_groups, _p(lg), _p(idx), _p(w), _p(m)), "route")
    return idx, w, m


def build_offsets(topk_idx, topk_w, E: int, P: int) -> dict:
    idx = _c(topk_idx, np.int32).reshape(-1)
    A = idx.size
    w = None if topk_w is None else _c(topk_w, np.float64).reshape(-1)
    R = rows_capacity(A, E, P)
    NB = blocks_capacity(A, E, P)
    counts = np.empty(E, np.int32)
    po = np.empty(E + 1, np.int32)
    meta = np.empty((NB, 3), np.int32)
    nb = np.zeros(1, np.int32)
    perm_row = np.empty(A, np.int32)
    row_src = np.empty(R, np.int32)
    row_gate = np.empty(R, np.float64)
    _check(_L().or_build_offsets(A, E, P, _p(idx), _p(w), _p(counts), _p(po), _p(meta), _p(nb),
                                 _p(perm_row), _p(row_src), _p(row_gate)), "build_offsets")
    n = int(nb[0])
    return dict(counts=counts, padded_offsets=po, block_metadata=meta[:n].copy(), num_blocks=n,
                perm_row=perm_row, row_src=row_src, row_gate=row_gate, rows_capacity=R,
                blocks_capacity=NB)


def blocks_from_counts(counts, P: int) -> dict:
    """The receiver's expert-major layout of an expert-parallel dispatch from
    counts [n_src, E] (rows of sender s for local expert e): padded offsets,
    block table, and piece_row [n_src, E], where sender s's rows for e land."""
    c = _c(counts, np.int32)
    n_src, E = c.shape
    po = np.empty(E + 1, np.int32)
    cap = int(c.sum()) // P + E
    meta = np.empty((max(cap, 1), 3), np.int32)
    nb = np.zeros(1, np.int32)
    piece_row = np.empty((n_src, E), np.int32)
    _check(_L().or_blocks_from_counts(n_src, E, P, _p(c), _p(po), _p(meta), _p(nb),
                                      _p(piece_row)), "blocks_from_counts")
    n = int(nb[0])
    return dict(padded_offsets=po, block_metadata=meta[:n].copy(), num_blocks=n,
                piece_row=piece_row)


def permute(x, row_src, k: int) -> np.ndarray:
    """x_perm [R, d] uint16; pad rows are zero here (the method leaves them
    unspecified and never reads them)."""
    x = _c(x, np.uint16)
    rs = _c(row_src, np.int32)
    R = rs.size
    d = x.shape[1]
    out = np.zeros((R, d), np.uint16)
    _L().or_permute(R, d, k, _p(x), _p(rs), _p(out))
    return out


def grouped_experts(x_perm, W1, W3, W2, block_metadata, row_gate):
    """h [R, de] and y [R, d] in fp64 over the whole padded layout; pad rows
    stay NaN."""
    xp = _c(x_perm, np.uint16)
    W1 = _c(W1, np.uint16)
    W3 = _c(W3, np.uint16)
    W2 = _c(W2, np.uint16)
    E, d, de = W1.shape
    meta = _c(block_metadata, np.int32)
    rg = _c(row_gate, np.float64)
    R = xp.shape[0]
    h = np.full((R, de), np.nan)
    y = np.full((R, d), np.nan)
    _check(_L().or_grouped_experts(d, de, E, meta.shape[0], _p(meta), _p(xp), _p(W1), _p(W3),
                                   _p(W2), _p(rg), _p(h), _p(y)), "grouped_experts")
    return h, y


def expert_rows(xrows, experts, gates, W1, W3, W2):
    """h [n, de], y [n, d] for a compact list of (row, expert, gate)."""
    xr = _c(xrows, np.uint16)
    ex = _c(experts, np.int32)
    g = _c(gates, np.float64)
    W1 = _c(W1, np.uint16)
    W3 = _c(W3, np.uint16)
    W2 = _c(W2, np.uint16)
    E, d, de = W1.shape
    n = ex.size
    h = np.empty((n, de))
    y = np.empty((n, d))
    _check(_L().or_expert_rows(n, d, de, E, _p(xr), _p(ex), _p(g), _p(W1), _p(W3), _p(W2), _p(h),
                               _p(y)), "expert_rows")
    return h, y


def shared_expert(xrows, Ws1, Ws3, Ws2):
    xr = _c(xrows, np.uint16)
    Ws1 = _c(Ws1, np.uint16)
    Ws3 = _c(Ws3, np.uint16)
    Ws2 = _c(Ws2, np.uint16)
    n, d = xr.shape
    ds = Ws1.shape[1]
    hs = np.empty((n, ds))
    ys = np.empty((n, d))
    _check(_L().or_shared_expert(n, d, ds, _p(xr), _p(Ws1), _p(Ws3), _p(Ws2), _p(hs), _p(ys)),
           "shared_expert")
    return hs, ys


def combine(y, perm_row, k: int, ys=None) -> np.ndarray:
    yy = _c(y, np.float64)
    pr = _c(perm_row, np.int32)
    T = pr.size // k
    d = yy.shape[1]
    s = None if ys is None else _c(ys, np.float64)
    out = np.empty((T, d))
    _L().or_combine(T, d, k, _p(yy), _p(pr), _p(s), _p(out))
    return out


def direct_layer(tokens, x, W1, W3, W2, topk_idx, topk_w, ys_rows=None) -> np.ndarray:
    tok = _c(tokens, np.int32)
    x = _c(x, np.uint16)
    W1 = _c(W1, np.uint16)
    W3 = _c(W3, np.uint16)
    W2 = _c(W2, np.uint16)
    idx = _c(topk_idx, np.int32)
    w = _c(topk_w, np.float64)
    E, d, de = W1.shape
    k = idx.shape[1]
    s = None if ys_rows is None else _c(ys_rows, np.float64)
    out = np.empty((tok.size, d))
    _check(_L().or_direct_layer(tok.size, _p(tok), d, de, E, k, _p(x), _p(W1), _p(W3), _p(W2),
                                _p(idx), _p(w), _p(s), _p(out)), "direct_layer")
    return out


# ------------------------------------------------ fp8 (e4m3) weights ----
def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Exact value of e4m3 codes (uint8); NaN for the two NaN codes."""
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    _L().or_e4m3_to_double_array(c.size, _p(c), _p(out))
    return out


def round_e4m3(v: np.ndarray) -> np.ndarray:
    """Nearest e4m3 code (uint8) of each value, ties to even, saturating at
    448."""
    a = _c(v, np.float64)
    out = np.empty(a.shape, np.uint8)
    _L().or_double_to_e4m3_array(a.size, _p(a), _p(out))
    return out


def quantize_e4m3(W) -> tuple:
    """Per-output-channel e4m3 quantization of bf16 matrices W [..., K, N]
    (column n = output channel n) -> (codes uint8 [..., K, N], scales
    float32 [..., N])."""
    W = _c(W, np.uint16)
    K, N = W.shape[-2:]
    batch = int(np.prod(W.shape[:-2], dtype=np.int64)) if W.ndim > 2 else 1
    q = np.empty(W.shape, np.uint8)
    s = np.empty(W.shape[:-2] + (N,), np.float32)
    _L().or_quantize_e4m3_batch(batch, K, N, _p(W), _p(q), _p(s))
    return q, s


def quantize_experts(inp: dict) -> dict:
    """e4m3 codes and scales of the routed expert weights W1, W3, W2."""
    Q1, S1 = quantize_e4m3(inp["W1"])
    Q3, S3 = quantize_e4m3(inp["W3"])
    Q2, S2 = quantize_e4m3(inp["W2"])
    return dict(Q1=Q1, S1=S1, Q3=Q3, S3=S3, Q2=Q2, S2=S2)


def quantize_shared(inp: dict) -> dict:
    """e4m3 codes and scales of the shared expert Ws1, Ws3 [d, ds], Ws2 [ds, d]."""
    Q1, S1 = quantize_e4m3(inp["Ws1"])
    Q3, S3 = quantize_e4m3(inp["Ws3"])
    Q2, S2 = quantize_e4m3(inp["Ws2"])
    return dict(Qs1=Q1, Ss1=S1, Qs3=Q3, Ss3=S3, Qs2=Q2, Ss2=S2)


def shared_expert_w8(xrows, qs: dict):
    """The shared expert with e4m3 weights: the routed evaluation with one
    expert and gate 1 (the arithmetic of shared_expert on the dequantized
    matrices)."""
    n = np.asarray(xrows).shape[0]
    q = dict(Q1=qs["Qs1"][None], S1=qs["Ss1"][None], Q3=qs["Qs3"][None], S3=qs["Ss3"][None],
             Q2=qs["Qs2"][None], S2=qs["Ss2"][None])
    return expert_rows_w8(xrows, np.zeros(n, np.int32), np.ones(n), q)


def expert_rows_w8(xrows, experts, gates, q: dict):
    """expert_rows with e4m3 weights q = quantize_experts(...)."""
    xr = _c(xrows, np.uint16)
    ex = _c(experts, np.int32)
    g = _c(gates, np.float64)
    Q1, Q3, Q2 = (_c(q[n], np.uint8) for n in ("Q1", "Q3", "Q2"))
    S1, S3, S2 = (_c(q[n], np.float32) for n in ("S1", "S3", "S2"))
    E, d, de = Q1.shape
    n = ex.size
    h = np.empty((n, de))
    y = np.empty((n, d))
    _check(_L().or_expert_rows_w8(n, d, de, E, _p(xr), _p(ex), _p(g), _p(Q1), _p(S1), _p(Q3),
                                  _p(S3), _p(Q2), _p(S2), _p(h), _p(y)), "expert_rows_w8")
    return h, y


def grouped_experts_w8(x_perm, q: dict, block_metadata, row_gate):
    """grouped_experts with e4m3 weights: every valid row of the block table
    through its expert; pad rows stay NaN."""
    xp = _c(x_perm, np.uint16)
    meta = _c(block_metadata, np.int32).reshape(-1, 3)
    rows = [np.arange(m0, m0 + vm) for _, m0, vm in meta]
    rows = np.concatenate(rows) if rows else np.zeros(0, np.int64)
    experts = np.concatenate([np.full(vm, e, np.int32) for e, _, vm in meta]) if len(meta) else \
        np.zeros(0, np.int32)
    E, d, de = q["Q1"].shape
    R = xp.shape[0]
    h = np.full((R, de), np.nan)
    y = np.full((R, d), np.nan)
    if rows.size:
        hh, yy = expert_rows_w8(xp[rows], experts, _c(row_gate, np.float64)[rows], q)
        h[rows] = hh
        y[rows] = yy
    return h, y


# ------------------------------------------------------------- backward ----
def weight_grad_columns(x_rows, dout_rows, p, W1, W3, W2, J):
    """Columns J of one expert's weight gradients over the given rows (token
    rows x_rows bf16 bits [n, d], upstream rows dout_rows fp64 [n, d],
    routing weights p [n]; W1/W3 [d, de], W2 [de, d] bf16 bits): returns
    (dW1[:, J], dW3[:, J], dW2[J, :]) in fp64."""
    x = _c(x_rows, np.uint16)
    n, d = x.shape
    de = W1.shape[-1]
    J = _c(J, np.int32)
    dW1c = np.empty((d, J.size))
    dW3c = np.empty((d, J.size))
    dW2r = np.empty((J.size, d))
    _check(_L().or_weight_grad_columns(n, d, de, _p(x), _p(_c(dout_rows, np.float64)),
                                       _p(_c(p, np.float64)), _p(_c(W1, np.uint16)),
                                       _p(_c(W3, np.uint16)), _p(_c(W2, np.uint16)), J.size,
                                       _p(J), _p(dW1c), _p(dW3c), _p(dW2r)),
           "weight_grad_columns")
    return dW1c, dW3c, dW2r


def layer_backward(inp: dict, cfg, fwd: dict, dout) -> dict:
    """Gradients of the layer forward (``layer_forward``'s routing, fixed) for
    an upstream gradient dout [T, d] (fp64): dx, dgates [T, k], dW1, dW3,
    dW2, and with a router dlogits [T, E], dWg [d, E], dbias [E], with a
    shared expert dWs1, dWs3, dWs2 -- all fp64.  The top-k choice is held
    constant and the bf16 rounding of h passes its gradient through."""
    x = _c(inp["x"], np.uint16)
    T, d = x.shape
    W1, W3, W2 = (_c(inp[n], np.uint16) for n in ("W1", "W3", "W2"))
    E, _, de = W1.shape
    k = cfg.k
    ds = cfg.d_shared
    idx = _c(fwd["topk_idx"], np.int32)
    gates = _c(fwd["topk_w"], np.float64)
    routed = inp.get("Wg") is not None and inp.get("topk_idx") is None
    Wg = _c(inp["Wg"], np.uint16) if routed else None
    Ws = [(_c(inp[n], np.uint16) if ds else None) for n in ("Ws1", "Ws3", "Ws2")]
    g = _c(dout, np.float64)
    out = dict(dx=np.empty((T, d)), dgates=np.empty((T, k)), dW1=np.empty((E, d, de)),
               dW3=np.empty((E, d, de)), dW2=np.empty((E, de, d)))
    if routed:
        out.update(dlogits=np.empty((T, E)), dWg=np.empty((d, E)), dbias=np.empty(E))
    if ds:
        out.update(dWs1=np.empty((d, ds)), dWs3=np.empty((d, ds)), dWs2=np.empty((ds, d)))
    gp = lambda n: _p(out.get(n))  # noqa: E731
    _check(_L().or_layer_backward(T, d, de, E, k, ds, _p(x), _p(Wg), _p(idx), _p(gates), _p(W1),
                                  _p(W3), _p(W2), _p(Ws[0]), _p(Ws[1]), _p(Ws[2]), _p(g),
                                  gp("dx"), gp("dgates"), gp("dlogits"), gp("dWg"), gp("dbias"),
                                  gp("dW1"), gp("dW3"), gp("dW2"), gp("dWs1"), gp("dWs3"),
                                  gp("dWs2")), "layer_backward")
    return out


# ---------------------------------------------------------- whole layer ----
def layer_forward(inp: dict, cfg) -> dict:
    """Whole layer through the padded layout (router, offsets, permute,
    grouped experts, shared expert, combine), every intermediate returned.
    ``inp`` holds numpy arrays (see module doc); a pre-routed input carries
    topk_idx / topk_w instead of Wg; an input that also carries the e4m3
    codes and scales of ``quantize_experts`` (``quantize_shared``) runs the
    routed (shared) experts on them."""
    if inp.get("topk_idx") is None:
        logits = router_logits(inp["x"], inp["Wg"], inp.get("bias"))
        idx, w, margin = route(logits, cfg.k, cfg.n_groups, cfg.topk_groups)
    else:
        logits, margin = None, None
        idx = _c(inp["topk_idx"], np.int32)
        w = _c(inp["topk_w"], np.float64)
    off = build_offsets(idx, w, cfg.E, cfg.pad)
    x_perm = permute(inp["x"], off["row_src"], cfg.k)
    if inp.get("Q1") is not None:  # e4m3 routed expert weights
        h, y = grouped_experts_w8(x_perm, inp, off["block_metadata"], off["row_gate"])
    else:
        h, y = grouped_experts(x_perm, inp["W1"], inp["W3"], inp["W2"], off["block_metadata"],
                               off["row_gate"])
    hs = ys = None
    if cfg.d_shared and inp.get("Qs1") is not None:  # e4m3 shared expert weights
        hs, ys = shared_expert_w8(inp["x"], inp)
    elif cfg.d_shared:
        hs, ys = shared_expert(inp["x"], inp["Ws1"], inp["Ws3"], inp["Ws2"])
    out = combine(y, off["perm_row"], cfg.k, ys)
    return dict(logits=logits, topk_idx=idx, topk_w=w, margin=margin, x_perm=x_perm, h=h, y=y,
                hs=hs, ys=ys, out=out, **off)
