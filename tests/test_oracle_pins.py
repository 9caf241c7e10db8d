"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a worked
example printed on the pages (tests/golden/), brute force over all subsets,
a library routine (numpy stable argsort, numpy matmul, torch's bf16
conversion), a closed form, or the exact permute/direct equivalence that the
TileLang page states.  A plausible mistake in the oracle (a dropped bias, a
wrong sign in silu, a transposed weight, an off-by-one in the padding, an
unstable segment order, a wrong tie-break) fails at least one of them.
"""
import itertools
import os

import numpy as np
import pytest
import torch

import oracle
from routing_permute_grouped_gb300 import ledger
from tests.helpers import bits, rand_bf16

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = [float(v) if "." in v else int(v) for v in rest]
    return vals


# ------------------------------------------------------------- bf16 --------
def test_bf16_widen_matches_torch():
    x = torch.randn(4096) * 10
    b = x.to(torch.bfloat16)
    np.testing.assert_array_equal(oracle.bf16_to_f64(bits(b)), b.to(torch.float64).numpy())


def test_bf16_rounding_matches_torch_rne():
    # every fp32 value converts to bf16 with round-to-nearest-even in torch;
    # the oracle rounds the same (exactly representable) value from fp64
    g = torch.Generator().manual_seed(3)
    f = torch.cat([torch.randn(20000, generator=g) * s for s in (1e-3, 1.0, 1e4)])
    # exact ties: bf16 value + half an ulp
    base = torch.randn(2000, generator=g).to(torch.bfloat16).to(torch.float32)
    ulp_half = torch.ldexp(torch.ones_like(base), torch.frexp(base).exponent - 9)
    f = torch.cat([f, base + ulp_half, base - ulp_half])
    ref = f.to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_bf16(f.to(torch.float64).numpy())
    np.testing.assert_array_equal(got, ref)


def test_bf16_rounding_subnormal_overflow_and_ties_match_torch():
    # the corners of the rounding: bf16 subnormals (quantum 2^-133, below the
    # smallest normal 2^-126), values that overflow to infinity (at and above
    # the midpoint (2 - 2^-8) * 2^127 between the largest finite bf16 and the
    # next power of two), and exact ties in both ranges.  Every input is an
    # fp32 value, which torch converts with round-to-nearest-even.
    g = torch.Generator().manual_seed(4)
    tiny = torch.ldexp(torch.rand(20000, generator=g) * 2 - 1,
                       torch.randint(-149, -120, (20000,), generator=g))
    k = torch.randint(-300, 300, (4000,), generator=g).to(torch.float32)
    q = 2.0 ** -133
    sub_ties = torch.cat([(k + 0.5) * q, (k + 0.25) * q, (k + 0.75) * q])
    fmax = torch.finfo(torch.float32).max
    top = torch.tensor([(2 - 2 ** -8) * 2.0 ** 127, (2 - 2 ** -7) * 2.0 ** 127,
                        (2 - 2 ** -7 - 2 ** -9) * 2.0 ** 127, (2 - 2 ** -8 - 2 ** -20) * 2.0 ** 127,
                        fmax, 2.0 ** 127, (2 - 2 ** -8 + 2 ** -20) * 2.0 ** 127],
                       dtype=torch.float64).to(torch.float32)
    big = torch.ldexp(1 + torch.rand(4000, generator=g), torch.full((4000,), 127))
    f = torch.cat([tiny, sub_ties, top, big, -top, -sub_ties,
                   torch.tensor([2.0 ** -126, 2.0 ** -127, 2.0 ** -133, 2.0 ** -134,
                                 1.5 * 2.0 ** -134, 2.0 ** -135, 2.0 ** -149])])
    ref = f.to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_bf16(f.to(torch.float64).numpy())
    np.testing.assert_array_equal(got, ref)
    assert np.isinf(got).sum() > 0 and (np.abs(got[np.isfinite(got)]) > 0).any()
    assert ((got != 0) & (np.abs(got) < 2.0 ** -126)).sum() > 1000  # subnormal results


# ---------------------------------------------------------- offsets --------
def _prerouted_idx(counts, seed=0):
    labels = np.concatenate([np.full(c, e, np.int32) for e, c in enumerate(counts)])
    rng = np.random.default_rng(seed)
    return labels[rng.permutation(labels.size)]


def test_padding_worked_example():
    gd = _golden("padding_dropless_sec3.txt")
    counts = gd["counts"]
    P = gd["pad"][0]
    off = oracle.build_offsets(_prerouted_idx(counts), None, len(counts), P)
    assert off["counts"].tolist() == counts
    sizes = np.diff(off["padded_offsets"]).tolist()
    assert sizes == gd["padded"]
    assert [s - c for s, c in zip(sizes, counts)] == gd["pad_rows"]
    assert off["padded_offsets"][-1] == gd["total_rows"][0]
    assert off["padded_offsets"][-1] - sum(counts) == gd["total_pad"][0]
    meta = off["block_metadata"]
    per_expert = [int((meta[:, 0] == e).sum()) for e in range(len(counts))]
    assert per_expert == gd["blocks"]
    assert off["num_blocks"] == sum(gd["blocks"])
    last_e0 = meta[meta[:, 0] == 0][-1]
    assert last_e0[2] == gd["last_block_valid_e0"][0]
    assert last_e0[1] == 169 * 128
    # the bound of sec. 3: < P pad rows per expert
    assert max(gd["pad_rows"]) <= P - 1 and sum(gd["pad_rows"]) <= len(counts) * (P - 1)


@pytest.mark.parametrize("P", [64, 128])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_offsets_invariants_and_stable_order(P, seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 40))
    T, k = int(rng.integers(1, 700)), int(rng.integers(1, 5))
    # skewed, some experts empty
    p = rng.dirichlet(np.full(E, 0.3))
    idx = rng.choice(E, size=T * k, p=p).astype(np.int32)
    w = rng.random(T * k)
    off = oracle.build_offsets(idx, w, E, P)
    c, po = off["counts"], off["padded_offsets"]
    assert c.sum() == T * k
    assert np.array_equal(c, np.bincount(idx, minlength=E))
    s = np.diff(po)
    assert (s % P == 0).all() and ((s - c) >= 0).all() and ((s - c) <= P - 1).all()
    assert ((c == 0) == (s == 0)).all()
    # stable order: inside a segment, ascending assignment index == numpy's
    # stable argsort of the expert ids
    order = np.argsort(idx, kind="stable")
    expect_row = np.empty(T * k, np.int64)
    pos = 0
    for e in range(E):
        seg = order[pos:pos + c[e]]
        expect_row[seg] = po[e] + np.arange(c[e])
        pos += c[e]
    assert np.array_equal(off["perm_row"], expect_row)
    rs = off["row_src"]
    assert rs.size == T * k + E * (P - 1)
    valid = rs >= 0
    assert valid.sum() == T * k
    assert np.array_equal(rs[off["perm_row"]], np.arange(T * k))
    assert np.array_equal(off["row_gate"][off["perm_row"]], w)
    assert (off["row_gate"][~valid] == 0).all()
    # block table: ascending expert then m, heights P, valid_m = min(P, rest)
    meta = off["block_metadata"]
    assert off["num_blocks"] == int(np.sum(-(-c // P)))
    assert off["num_blocks"] <= (T * k) // P + E
    exp_meta = [[e, po[e] + m, min(P, c[e] - m)] for e in range(E) for m in range(0, c[e], P)]
    assert meta.tolist() == exp_meta


def test_offsets_decode_block_is_exact():
    # "Dropless and grouped GEMM", sec. 10: 128 rows per expert is exactly one
    # block of 128 with no padding
    off = oracle.build_offsets(_prerouted_idx([128, 128, 0, 128]), None, 4, 128)
    assert np.diff(off["padded_offsets"]).tolist() == [128, 128, 0, 128]
    assert off["block_metadata"].tolist() == [[0, 0, 128], [1, 128, 128], [3, 256, 128]]


def test_offsets_rejects_bad_expert():
    with pytest.raises(ValueError):
        oracle.build_offsets(np.array([0, 5], np.int32), None, 4, 128)


# ------------------------------------------------------------ router -------
def test_router_logits_match_library_matmul():
    x = rand_bf16((37, 96), seed=1)
    Wg = rand_bf16((96, 12), std=0.1, seed=2)
    bias = np.random.default_rng(0).normal(0, 0.5, 12).astype(np.float32)
    ref = oracle.bf16_to_f64(x) @ oracle.bf16_to_f64(Wg) + bias.astype(np.float64)
    np.testing.assert_allclose(oracle.router_logits(x, Wg, bias), ref, rtol=1e-13, atol=1e-13)


def _brute_topk(l, k, n_groups, topk_groups):
    E = l.size
    elig = list(range(E))
    if n_groups:
        gsz = E // n_groups
        gs = [l[g * gsz:(g + 1) * gsz].max() for g in range(n_groups)]
        best = max(itertools.combinations(range(n_groups), topk_groups),
                   key=lambda c: sum(gs[g] for g in c))
        elig = [e for e in range(E) if e // gsz in best]
    best = max(itertools.combinations(elig, k), key=lambda c: sum(l[e] for e in c))
    return sorted(best, key=lambda e: -l[e])


@pytest.mark.parametrize("case", [(8, 2, 0, 0), (8, 3, 4, 2), (6, 1, 0, 0), (8, 4, 2, 1),
                                  (8, 8, 0, 0), (8, 5, 4, 3)])
def test_route_brute_force(case):
    E, k, ng, tg = case
    rng = np.random.default_rng(E * 100 + k * 10 + ng)
    lg = rng.normal(size=(8, E))
    idx, w, m = oracle.route(lg, k, ng, tg)
    for t in range(8):
        assert idx[t].tolist() == _brute_topk(lg[t], k, ng, tg)
    # gates: softmax over the chosen logits == softmax over all E experts,
    # renormalised over the chosen ones
    p = np.exp(lg - lg.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    sel = np.take_along_axis(p, idx.astype(np.int64), 1)
    np.testing.assert_allclose(w, sel / sel.sum(1, keepdims=True), rtol=1e-12)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-14)
    # closed form of the ratio between two gates
    np.testing.assert_allclose(w[:, 0] / w[:, -1],
                               np.exp(np.take_along_axis(lg, idx[:, :1].astype(np.int64), 1)[:, 0] -
                                      np.take_along_axis(lg, idx[:, -1:].astype(np.int64), 1)[:, 0]),
                               rtol=1e-12)
    assert (m > 0).all()


def _brute_margin(l, k, n_groups, topk_groups):
    """The smallest gap between two values whose order decides the routing,
    by enumerating pairs: every kept group against every rejected group
    (group scores), every chosen expert against every eligible rejected one,
    and every pair of chosen experts (their order is part of the output)."""
    E = l.size
    chosen = _brute_topk(l, k, n_groups, topk_groups)
    gaps = []
    elig = set(range(E))
    if n_groups:
        gsz = E // n_groups
        gs = [l[g * gsz:(g + 1) * gsz].max() for g in range(n_groups)]
        kept = max(itertools.combinations(range(n_groups), topk_groups),
                   key=lambda c: sum(gs[g] for g in c))
        gaps += [gs[a] - gs[b] for a in kept for b in range(n_groups) if b not in kept]
        elig = {e for e in range(E) if e // gsz in kept}
    gaps += [l[a] - l[b] for a in chosen for b in elig if b not in chosen]
    gaps += [l[chosen[i]] - l[chosen[j]] for i in range(k) for j in range(i + 1, k)]
    return min(gaps) if gaps else np.inf


@pytest.mark.parametrize("case", [(8, 2, 0, 0), (8, 3, 4, 2), (6, 1, 0, 0), (8, 4, 2, 1),
                                  (8, 8, 0, 0), (8, 5, 4, 3), (12, 3, 6, 2), (9, 2, 3, 1)])
def test_route_margin_brute_force(case):
    # the margin that the tie filter of the parity tests rests on: equal to
    # the pairwise brute force, and no perturbation of the logits smaller
    # than half of it (in every coordinate) changes the routing.  Logits on a
    # coarse grid make near-ties and exact ties (margin 0) frequent.
    E, k, ng, tg = case
    rng = np.random.default_rng(E * 1000 + k * 10 + ng)
    lg = np.concatenate([rng.normal(size=(24, E)), np.round(rng.normal(size=(24, E)) * 4) / 4])
    idx, _, m = oracle.route(lg, k, ng, tg)
    for t in range(lg.shape[0]):
        want = _brute_margin(lg[t], k, ng, tg)
        assert m[t] == want, (t, m[t], want)
        if not np.isfinite(want) or want == 0:
            continue
        for _ in range(20):
            d = rng.uniform(-1, 1, E) * want * 0.49
            assert _brute_topk(lg[t] + d, k, ng, tg) == idx[t].tolist()
    assert (m == 0).any() and (m > 0).any()


def test_route_ties_go_to_lower_index():
    lg = np.array([[1.0, 3.0, 3.0, 0.5, 3.0]])
    idx, w, m = oracle.route(lg, 2)
    assert idx.tolist() == [[1, 2]]
    assert m[0] == 0.0
    lg = np.array([[5.0, 0.0, 0.0, 5.0]])  # two groups with equal score
    idx, _, _ = oracle.route(lg, 1, 2, 1)
    assert idx.tolist() == [[0]]


def test_group_limit_excludes_experts():
    # expert 3 has the second-highest logit but its group (1) loses to group 0
    # (max 9) and group 2 (max 8) when only 2 of 3 groups are kept
    lg = np.array([[9.0, -5, 7.5, 7.6, -1, -1, 8.0, 1.0, 2.0]])
    idx, _, _ = oracle.route(lg, 2, 3, 2)
    assert idx.tolist() == [[0, 6]]
    idx, _, _ = oracle.route(lg, 2)
    assert idx.tolist() == [[0, 6]]
    idx, _, _ = oracle.route(lg, 3, 3, 2)
    assert idx.tolist() == [[0, 6, 2]]


# ------------------------------------------------------ expert / layer -----
class _Cfg:
    def __init__(self, **kw):
        self.__dict__.update(kw)


def _textbook_swiglu(x, W1, W3, W2):
    """Dense SwiGLU MLP with library matmuls; h rounded to bf16."""
    xf = oracle.bf16_to_f64(x)
    g = xf @ oracle.bf16_to_f64(W1)
    u = xf @ oracle.bf16_to_f64(W3)
    h = oracle.round_bf16(g / (1.0 + np.exp(-g)) * u)
    return h, h @ oracle.bf16_to_f64(W2)


def test_moe_with_one_expert_is_dense_swiglu():
    # k = 1, E = 1: every token goes to expert 0 with gate 1, so the layer is
    # the dense SwiGLU MLP of the textbook
    T, d, de = 150, 64, 96
    x = rand_bf16((T, d), seed=5)
    W1 = rand_bf16((1, d, de), std=d ** -0.5, seed=6)
    W3 = rand_bf16((1, d, de), std=d ** -0.5, seed=7)
    W2 = rand_bf16((1, de, d), std=de ** -0.5, seed=8)
    Wg = rand_bf16((d, 1), std=d ** -0.5, seed=9)
    cfg = _Cfg(k=1, E=1, n_groups=0, topk_groups=0, pad=128, d_shared=0)
    res = oracle.layer_forward(dict(x=x, Wg=Wg, bias=None, W1=W1, W3=W3, W2=W2), cfg)
    h_ref, y_ref = _textbook_swiglu(x, W1[0], W3[0], W2[0])
    assert (res["topk_w"] == 1.0).all()
    np.testing.assert_allclose(res["out"], y_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(res["h"][res["perm_row"]], h_ref)


def test_shared_expert_is_dense_swiglu():
    T, d, ds = 40, 64, 32
    x = rand_bf16((T, d), seed=11)
    Ws1 = rand_bf16((d, ds), std=0.125, seed=12)
    Ws3 = rand_bf16((d, ds), std=0.125, seed=13)
    Ws2 = rand_bf16((ds, d), std=0.17, seed=14)
    hs, ys = oracle.shared_expert(x, Ws1, Ws3, Ws2)
    h_ref, y_ref = _textbook_swiglu(x, Ws1, Ws3, Ws2)
    np.testing.assert_array_equal(hs, h_ref)
    np.testing.assert_allclose(ys, y_ref, rtol=1e-12, atol=1e-12)


def test_silu_sign_and_gate_scaling():
    # silu(g) * u with g = u: h = g^2 sigmoid(g) is >= 0; a flipped sign in
    # silu or a swapped gate/up weight gives negative values
    d, de = 32, 16
    x = rand_bf16((20, d), seed=21)
    W = rand_bf16((1, d, de), std=0.2, seed=22)
    W2 = rand_bf16((1, de, d), std=0.2, seed=23)
    h, y = oracle.expert_rows(x, np.zeros(20, np.int32), np.full(20, 0.5), W, W, W2)
    assert (h >= 0).all()
    h1, y1 = oracle.expert_rows(x, np.zeros(20, np.int32), np.full(20, 1.0), W, W, W2)
    np.testing.assert_allclose(y, 0.5 * y1, rtol=1e-15)
    # gate and up are not interchangeable: silu(g) u != silu(u) g
    W3 = rand_bf16((1, d, de), std=0.2, seed=24)
    ha, _ = oracle.expert_rows(x, np.zeros(20, np.int32), np.ones(20), W, W3, W2)
    hb, _ = oracle.expert_rows(x, np.zeros(20, np.int32), np.ones(20), W3, W, W2)
    assert not np.array_equal(ha, hb)
    h_ref, _ = _textbook_swiglu(x, W[0], W3[0], W2[0])
    np.testing.assert_array_equal(ha, h_ref)


@pytest.mark.parametrize("ng,tg,ds,P", [(0, 0, 0, 128), (4, 2, 48, 128), (0, 0, 48, 64)])
def test_permute_combine_equals_direct_evaluation(ng, tg, ds, P):
    # "MoE & MLA operators", sec. 2.3: permute -> per-assignment expert ->
    # scatter-reduce equals evaluating each token's chosen experts directly,
    # with a maximum error of exactly 0
    T, d, de, E, k = 300, 64, 32, 8, 3
    x = rand_bf16((T, d), seed=31)
    inp = dict(x=x, Wg=rand_bf16((d, E), std=d ** -0.5, seed=32),
               bias=np.random.default_rng(1).normal(0, 0.5, E).astype(np.float32),
               W1=rand_bf16((E, d, de), std=d ** -0.5, seed=33),
               W3=rand_bf16((E, d, de), std=d ** -0.5, seed=34),
               W2=rand_bf16((E, de, d), std=de ** -0.5, seed=35))
    if ds:
        inp.update(Ws1=rand_bf16((d, ds), std=d ** -0.5, seed=36),
                   Ws3=rand_bf16((d, ds), std=d ** -0.5, seed=37),
                   Ws2=rand_bf16((ds, d), std=ds ** -0.5, seed=38))
    cfg = _Cfg(k=k, E=E, n_groups=ng, topk_groups=tg, pad=P, d_shared=ds)
    res = oracle.layer_forward(inp, cfg)
    direct = oracle.direct_layer(np.arange(T), x, inp["W1"], inp["W3"], inp["W2"],
                                 res["topk_idx"], res["topk_w"], res["ys"])
    assert np.array_equal(res["out"], direct)
    # the permuted rows really are copies of their token rows
    rs = res["row_src"]
    v = rs >= 0
    assert np.array_equal(res["x_perm"][v], x[rs[v] // k])
    # pad rows of y are never produced, and never needed by combine
    assert np.isnan(res["y"][~v]).all()


def test_direct_evaluation_detects_wrong_layout():
    # plant a layout mistake in the oracle's own tables (swap two rows of
    # perm_row): the equivalence check above must catch it
    T, d, de, E, k = 50, 32, 16, 4, 2
    x = rand_bf16((T, d), seed=41)
    W1 = rand_bf16((E, d, de), std=0.2, seed=42)
    W3 = rand_bf16((E, d, de), std=0.2, seed=43)
    W2 = rand_bf16((E, de, d), std=0.2, seed=44)
    Wg = rand_bf16((d, E), std=0.2, seed=45)
    cfg = _Cfg(k=k, E=E, n_groups=0, topk_groups=0, pad=128, d_shared=0)
    res = oracle.layer_forward(dict(x=x, Wg=Wg, bias=None, W1=W1, W3=W3, W2=W2), cfg)
    pr = res["perm_row"].copy()
    flat = res["topk_idx"].reshape(-1)
    a = 0  # token 0; b: an assignment of another token with another expert
    b = int(np.flatnonzero((flat != flat[0]) & (np.arange(flat.size) // k != 0))[0])
    pr[a], pr[b] = pr[b], pr[a]
    bad = oracle.combine(res["y"], pr, k)
    direct = oracle.direct_layer(np.arange(T), x, W1, W3, W2, res["topk_idx"], res["topk_w"])
    assert not np.array_equal(bad, direct)


# ------------------------------------------------------------ ledgers ------
def test_ledger_figures_of_the_pages():
    g = _golden("ledger_pages.txt")
    d, de = 7168, 2048
    assert round(ledger.expert_flops_per_row(d, de) / 1e6, 2) == g["expert_flops_per_row_mflop"][0]
    assert round(ledger.routed_flops(65536, d, de) / 1e12, 3) == g["routed_tflop_65536_rows"][0]
    assert round(ledger.routed_flops(65792, d, de) / 1e12, 3) == g["routed_tflop_65792_rows"][0]
    assert round(ledger.routed_flops(98304, d, de) / 1e12, 3) == g["routed_tflop_98304_rows"][0]
    assert round(4 * ledger.routed_flops(65792, d, de) / 1e12, 3) == g["ungrouped_tflop_65792x4"][0]
    gib = 2.0 ** 30
    assert round(8192 * d * 2 / gib, 2) == g["mem_x_gib"][0]
    assert round(65792 * d * 2 / gib, 2) == g["mem_recv_x_gib"][0]
    assert round(65792 * 2 * de * 2 / gib, 2) == g["mem_h13_gib"][0]
    assert round(65792 * de * 2 / gib, 2) == g["mem_h_gib"][0]
    assert round(65792 * d * 2 / gib, 2) == g["mem_y_gib"][0]
    T, E, k = 8192, 8, 4
    assert round(ledger.router_flops(T, d, E) / 1e9, 2) == g["router_gflop"][0]
    assert round(ledger.router_intensity(T, d, E), 1) == g["router_ai"][0]
    assert ledger.permute_bytes_page(T, k, d) / 2 ** 20 == g["permute_mib"][0]
    assert round(ledger.routed_flops(T * k, d, de) / 1e12, 2) == g["grouped_tflop"][0]
    gb = ledger.grouped_gemm_bytes_page(T * k, E, d, de)
    assert round(gb / 1e9, 2) == g["grouped_gb"][0]
    assert round(ledger.routed_flops(T * k, d, de) / gb) == g["grouped_ai"][0]
    assert ledger.permute_combine_bytes_page(T, k, d) / gib == g["permute_combine_gib"][0]
    assert round(ledger.single_expert_intensity(16, d, de), 1) == g["single_expert_ai_16"][0]
    assert round(ledger.single_expert_intensity(512, d, de)) == g["single_expert_ai_512"][0]
    gd = _golden("padding_dropless_sec3.txt")
    assert ledger.padded_rows(gd["counts"], 128) == gd["total_rows"][0]
    assert round(100 * ledger.padding_waste(gd["counts"], 128), 2) == 0.39


def test_grouped_gemm_algorithmic_bytes():
    # default shape: 1.913 GB = x_perm + y (2 x 470 MB) + h twice (2 x 134 MB)
    # + the weights of all 8 experts (705 MB)
    b = ledger.grouped_gemm_bytes_alg(8192 * 4, 8, 7168, 2048)
    assert round(b / 1e9, 3) == 1.913
    assert ledger.grouped_gemm_bytes_alg(0, 3, 64, 32) == 2 * 3 * 3 * 64 * 32


def test_grouped_bytes_with_e4m3_weights():
    """e4m3 weights: one byte per weight plus a 4-byte scale per output
    channel; the activation bytes are those of the bf16 ledger."""
    A, act, d, de = 512, 217, 7168, 2048
    b16 = ledger.grouped_gemm_bytes_alg(A, act, d, de)
    b8 = ledger.grouped_gemm_bytes_alg(A, act, d, de, fp8_weights=True)
    acts = 2 * (2 * A * d + 2 * A * de)
    assert b16 - acts == act * 3 * d * de * 2
    assert b8 - acts == act * (3 * d * de + 4 * (2 * de + d))


# ------------------------------------------------------ imbalance sweep ----
def test_zipf_exponents_give_the_stored_loads():
    # the Zipf exponents of the imbalance workloads (constants in synth) are
    # the ones tests/golden/make_zipf_s.py stored, and with them the oracle's
    # routing of the seeded token rows puts the recorded multiple of the mean
    # load on the hottest expert (within 2 % of 1x / 2x / 4x for 2x and 4x)
    import json

    from routing_permute_grouped_gb300 import synth

    with open(os.path.join(GOLDEN, "zipf_s.json")) as f:
        stored = json.load(f)
    shape = synth.WORKLOADS["imbalance_x1_p128"]
    inp = synth.make_inputs(shape, zipf_s=0.0)
    L0 = oracle.router_logits(bits(inp["x"]), bits(inp["Wg"]), None)
    for target in (1, 2, 4):
        for pad in (64, 128):
            name = f"imbalance_x{target}_p{pad}"
            assert synth.ZIPF_S[name] == stored[name]
            assert synth.ZIPF_HOT_OVER_MEAN[name] == stored[name + "_hot_over_mean"]
        name = f"imbalance_x{target}_p128"
        bias = synth.zipf_bias(shape.E, synth.ZIPF_S[name], shape.seed).numpy().astype(np.float64)
        idx, _, _ = oracle.route(L0 + bias[None, :], shape.k)
        counts = np.bincount(idx.reshape(-1), minlength=shape.E)
        ratio = counts.max() / counts.mean()
        assert round(float(ratio), 4) == synth.ZIPF_HOT_OVER_MEAN[name]
        if target > 1:
            assert abs(ratio - target) <= 0.02 * target


def test_tile_counts_of_the_padded_and_unpadded_schedules():
    # "Dropless and grouped GEMM", sec. 11: the pre-routed sizes at tile
    # height 128 execute 515 tiles unpadded (512 tiles of rows, three
    # segment starts inside a tile: +0.59 %) against 514 padded (65,792
    # rows: +0.39 %)
    g = _golden("unpadded_tiles_sec11.txt")
    sizes, tile = g["counts"], g["tile"][0]
    assert np.cumsum([0] + sizes).tolist() == g["group_offsets"]
    assert ledger.unpadded_tiles(sizes, tile) == g["unpadded_tiles"][0]
    assert g["unpadded_tiles"][0] == g["tiles_of_rows"][0] + g["extra_visits"][0]
    assert g["unpadded_tiles"][0] * tile == g["unpadded_rows"][0]
    assert ledger.padded_rows(sizes, tile) == g["padded_rows"][0]
    assert ledger.padded_tiles(sizes, 128, tile) * tile == g["padded_rows"][0]
    A = sum(sizes)
    assert round(100 * (g["unpadded_rows"][0] / A - 1), 2) == g["unpadded_extra_pct"][0]
    assert round(100 * (g["padded_rows"][0] / A - 1), 2) == g["padded_extra_pct"][0]
    # the bounds the page states: rows / tile <= tiles <= rows / tile + E - 1
    rng = np.random.default_rng(8)
    for _ in range(200):
        E = int(rng.integers(1, 40))
        c = rng.integers(0, 700, E)
        c[rng.random(E) < 0.2] = 0
        tile = int(rng.choice([64, 128, 256]))
        A = int(c.sum())
        n = ledger.unpadded_tiles(c.tolist(), tile)
        assert -(-A // tile) <= n <= -(-A // tile) + max(int((c > 0).sum()) - 1, 0)
        # brute force: tiles x experts whose row ranges meet
        starts = np.concatenate([[0], np.cumsum(c)])
        brute = sum(1 for t in range(-(-A // tile)) for e in range(E)
                    if c[e] > 0 and starts[e] < (t + 1) * tile and starts[e + 1] > t * tile)
        assert n == brute
