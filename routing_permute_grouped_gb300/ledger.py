"""FLOP and byte accounting of the MoE layer forward pass (host logic).

The counting rules restate the pages' ledgers:
  * one token row through one SwiGLU expert costs three d x d_e GEMVs,
    2 * d * d_e * 3 FLOP ("Dropless and grouped GEMM", sec. 4: 88.08 MFLOP
    per row at d=7168, d_e=2048);
  * the router GEMM costs 2 * T * d * E ("MoE & MLA operators", sec. 2.2);
  * the page's permute ledger moves 2 * T * k * d * b bytes (read T*k rows,
    write T*k rows; same page, sec. 2.3) and permute + combine 4 * T * k * d * b
    (sec. 2.6);
  * a single expert fed t tokens reads its 3 * d * d_e weights once plus
    4 * t * d activations (same page, sec. 2.4);
  * the page's grouped-GEMM ledger: b * (3 * A * d + 3 * E * d * d_e) bytes
    (sec. 2.3, 2.89 TFLOP over 2.11 GB at the default shape).
Useful FLOP never counts padding rows.  The algorithmic minimum bytes of this
build's kernels (each token row read once by permute, each routed row written
once) are stated next to the page's figures.
"""
from __future__ import annotations

BF16 = 2


def expert_flops_per_row(d: int, d_e: int) -> int:
    return 2 * d * d_e * 3


def routed_flops(A: int, d: int, d_e: int) -> int:
    return A * expert_flops_per_row(d, d_e)


def shared_flops(T: int, d: int, d_s: int) -> int:
    return T * expert_flops_per_row(d, d_s) if d_s else 0


def router_flops(T: int, d: int, E: int) -> int:
    return 2 * T * d * E


def router_intensity(T: int, d: int, E: int, b: int = BF16) -> float:
    """FLOP per byte of the router GEMM: x [T,d], W_g [d,E] read, logits
    [T,E] written, all b bytes wide."""
    return router_flops(T, d, E) / (b * (T * d + d * E + T * E))


def layer_useful_flops(T: int, k: int, d: int, d_e: int, d_s: int = 0, A: int = None) -> int:
    """Routed (padding excluded) + shared expert FLOP of one layer; the
    router GEMM is excluded (it is < 0.1% of the layer at the default
    shape)."""
    A = T * k if A is None else A
    return routed_flops(A, d, d_e) + shared_flops(T, d, d_s)


def permute_bytes_page(T: int, k: int, d: int, b: int = BF16) -> int:
    return 2 * T * k * d * b


def permute_combine_bytes_page(T: int, k: int, d: int, b: int = BF16) -> int:
    return 4 * T * k * d * b


def permute_bytes_alg(T: int, k: int, d: int, b: int = BF16) -> int:
    """Token-major permute: each token row read once, written k times."""
    return (T + T * k) * d * b


def combine_bytes_alg(T: int, k: int, d: int, shared: bool, b: int = BF16) -> int:
    """k routed rows (+1 shared row) read and one output row written per
    token."""
    return (T * k + T + (T if shared else 0)) * d * b


def single_expert_intensity(t: int, d: int, d_e: int, b: int = BF16) -> float:
    return 2 * t * 3 * d * d_e / (b * (3 * d * d_e + 4 * t * d))


def grouped_gemm_bytes_page(A: int, E: int, d: int, d_e: int, b: int = BF16) -> int:
    return b * (3 * A * d + 3 * E * d * d_e)


def grouped_gemm_bytes_alg(A: int, active_experts: int, d: int, d_e: int, b: int = BF16,
                           fp8_weights: bool = False) -> int:
    """Algorithmic bytes of the two grouped GEMMs (padding excluded): x_perm
    rows read and y rows written (A*d each), h written and read back
    (2*A*d_e), and the weights of every expert that received a row
    (3*d*d_e each, b bytes; with e4m3 weights one byte each plus one fp32
    scale per output channel, 2*d_e + d per expert)."""
    act = b * (2 * A * d + 2 * A * d_e)
    if fp8_weights:
        return act + active_experts * (3 * d * d_e + 4 * (2 * d_e + d))
    return act + b * active_experts * 3 * d * d_e


def gemm1_flops(rows: int, d: int, d_e: int) -> int:
    return 2 * rows * d * 2 * d_e


def gemm2_flops(rows: int, d: int, d_e: int) -> int:
    return 2 * rows * d_e * d


def padded_rows(counts, P: int) -> int:
    return sum(-(-c // P) * P for c in counts)


def padding_waste(counts, P: int) -> float:
    """(sum of padded sizes - assignments) / assignments."""
    A = sum(counts)
    return (padded_rows(counts, P) - A) / A if A else 0.0


def padded_tiles(counts, P: int, tile: int) -> int:
    """Row tiles of height `tile` that the padded layout executes: each
    expert's segment (ceil(c / P) * P rows) split into tiles on its own."""
    return sum(-(-(-(-c // P) * P) // tile) for c in counts if c > 0)


def unpadded_tiles(counts, tile: int) -> int:
    """Row tiles of height `tile` that the unpadded schedule executes
    ("Dropless and grouped GEMM", sec. 11): the experts' rows lie back to
    back without padding, and a tile is executed once for every expert whose
    rows it holds, so a tile that an expert boundary cuts runs twice.
    Between the tile count of the rows and that count + E - 1."""
    n, start = 0, 0
    for c in counts:
        if c > 0:
            n += (start + c - 1) // tile - start // tile + 1
        start += c
    return n


def layer_backward_useful_flops(T: int, k: int, d: int, d_e: int, d_s: int = 0,
                                E: int = 0) -> int:
    """Useful FLOP of the layer backward: every forward GEMM C = A B has a data
    gradient dA = dC B^T and a weight gradient dB = A^T dC of its own cost, so
    twice the forward's routed + shared FLOP, plus twice the router GEMM when
    the router is differentiated (E > 0).  The gate/up recomputation is not
    useful work and is not counted."""
    return 2 * layer_useful_flops(T, k, d, d_e, d_s) + (2 * router_flops(T, d, E) if E else 0)


def layer_backward_gemm_flops(T: int, k: int, d: int, d_e: int, d_s: int = 0, E: int = 0,
                              recompute: bool = True) -> int:
    """FLOP the backward's GEMMs execute on unpadded rows: the useful FLOP plus,
    unless the forward saved them, the recomputed gate/up products
    (2 * d * 2 d_e per routed row, the same for the shared expert)."""
    extra = T * k * 2 * d * 2 * d_e + (T * 2 * d * 2 * d_s if d_s else 0)
    return layer_backward_useful_flops(T, k, d, d_e, d_s, E) + (extra if recompute else 0)


def layer_backward_bytes_alg(T: int, k: int, d: int, d_e: int, d_s: int, E: int, active: int,
                             router: bool, b: int = BF16, recompute: bool = True) -> int:
    """A lower bound of the bytes the layer backward moves: the weights its
    data gradients and the gate/up recomputation read (W2, W13 and W13 in
    the other orientation: 5 * d * d_e per expert that received a row; 3 *
    d * d_e without the recomputation), the weight gradients it writes (3 *
    d * d_e for every expert, zero for the others), the shared expert's
    weights and gradients likewise, the router weight and its fp32 gradient,
    and the token rows x and dout read and dx written once.  The activations
    of the padded layout are not counted."""
    wr = 5 if recompute else 3
    n = b * (active * wr * d * d_e + E * 3 * d * d_e + 3 * T * d)
    if d_s:
        n += b * (wr + 3) * d * d_s
    if router:
        n += b * d * E + 4 * d * E
    return n
