"""Pins of the oracle's e4m3 (fp8) weight path, CPU only.

The format and the conversion are pinned to a library routine (torch's
float8_e4m3fn casts), the quantizer to its definition (one fp32 scale per
output channel, amax / 448) and to the exact case where every weight is an
e4m3 value times a power of two, and the fp8 expert evaluation to the bf16
one on such weights.  Sources: "MoE & MLA operators", sec. 6.1 (fp8 expert
weights, one byte per element) and "Dropless and grouped GEMM", sec. 12 (the
scale is applied after the matmul when it covers the whole contraction).
"""
import numpy as np
import pytest
import torch

import oracle

E4M3_MAX = 448.0


def _finite_codes():
    c = np.arange(256, dtype=np.uint8)
    return c[(c & 0x7F) != 0x7F]


def _torch_encode(v32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _bf16_bits(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(ours, ref, equal_nan=True)
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF])
    assert ours[0x7E] == E4M3_MAX and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_encode_matches_torch_on_grid_ties_and_random():
    vals = np.sort(np.unique(oracle.e4m3_to_f64(_finite_codes())))
    pos = vals[vals > 0]
    mids = (pos[:-1] + pos[1:]) / 2  # exact in fp32: ties between neighbours
    mids = np.concatenate([[pos[0] / 2], mids])
    m32 = mids.astype(np.float32)
    up = np.nextafter(m32, np.float32(np.inf))
    dn = np.nextafter(m32, np.float32(0))
    rng = np.random.default_rng(7)
    rnd = np.concatenate([rng.uniform(-E4M3_MAX, E4M3_MAX, 20000),
                          rng.standard_normal(20000) * 2.0 ** rng.integers(-14, 6, 20000)])
    allv = np.concatenate([vals, -vals, m32, -m32, up, -up, dn, -dn, rnd, [0.0, -0.0]])
    allv = allv.astype(np.float32)
    allv = allv[np.abs(allv) <= E4M3_MAX]
    ours = oracle.round_e4m3(allv.astype(np.float64))
    ref = _torch_encode(allv)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first value {allv[bad[0]]!r}"


def test_encode_ties_go_to_even_and_saturates():
    # 1 + 1/16 lies halfway between 1 (mantissa 000) and 1.125 (001)
    assert oracle.round_e4m3(np.array([1.0625]))[0] == 0x38
    # 1.1875 halfway between 1.125 (001) and 1.25 (010) -> 010
    assert oracle.round_e4m3(np.array([1.1875]))[0] == 0x3A
    # subnormal tie: 1.5 * 2^-9 between 2^-9 (m 1) and 2^-8 (m 2) -> 2
    assert oracle.round_e4m3(np.array([1.5 * 2.0 ** -9]))[0] == 0x02
    # smallest tie: 2^-10 -> 0 (even)
    assert oracle.round_e4m3(np.array([2.0 ** -10]))[0] == 0x00
    sat = oracle.round_e4m3(np.array([448.0, 470.0, 1e6, -1e30, np.inf, -np.inf]))
    assert list(sat) == [0x7E, 0x7E, 0x7E, 0xFE, 0x7E, 0xFE]
    assert oracle.round_e4m3(np.array([np.nan]))[0] == 0x7F


def test_encode_decode_round_trip():
    codes = _finite_codes()
    assert np.array_equal(oracle.round_e4m3(oracle.e4m3_to_f64(codes)), codes)


def _representable_matrix(rng, K, N):
    """W[i, n] = c * 2^-(8 + n % 5) with c an e4m3 value and one element of
    each column equal to +-448, so the scale of column n is exactly
    2^-(8 + n % 5) and every quotient is exactly its code."""
    vals = oracle.e4m3_to_f64(_finite_codes())
    c = rng.choice(vals, size=(K, N))
    rows = rng.integers(0, K, N)
    c[rows, np.arange(N)] = np.where(rng.random(N) < 0.5, -E4M3_MAX, E4M3_MAX)
    scale = 2.0 ** -(8 + (np.arange(N) % 5))
    W = c * scale[None, :]
    bits = _bf16_bits(W.astype(np.float32))
    assert np.array_equal(oracle.bf16_to_f64(bits), W)  # exact in bf16
    return bits, c, scale


def test_quantize_exact_on_representable_weights():
    rng = np.random.default_rng(11)
    bits, c, scale = _representable_matrix(rng, 96, 40)
    q, s = oracle.quantize_e4m3(bits)
    assert q.shape == bits.shape and s.shape == (40,)
    assert np.array_equal(s.astype(np.float64), scale)
    assert np.array_equal(oracle.e4m3_to_f64(q), c)


def test_quantize_definition_and_error_bound():
    rng = np.random.default_rng(3)
    K, N = 300, 64
    W = rng.standard_normal((2, K, N)) / np.sqrt(K)
    W[1, :, 5] = 0.0  # an all-zero channel
    bits = _bf16_bits(W.astype(np.float32)).reshape(2, K, N)
    w = oracle.bf16_to_f64(bits)
    q, s = oracle.quantize_e4m3(bits)
    amax = np.abs(w).max(axis=1)  # [2, N]
    expect_s = np.where(amax > 0, (amax.astype(np.float32) / np.float32(448.0)), np.float32(1.0))
    assert np.array_equal(s, expect_s.astype(np.float32))
    assert s[1, 5] == 1.0 and not q[1, :, 5].any()
    deq = oracle.e4m3_to_f64(q) * s[:, None, :].astype(np.float64)
    # half an e4m3 quantum: 2^-4 relative for normals, 2^-10 * s absolute for
    # subnormals, with slack for the fp32 quotient
    bound = np.maximum(np.abs(w) * 2.0 ** -4, s[:, None, :] * 2.0 ** -10) * (1 + 2.0 ** -18)
    assert np.all(np.abs(w - deq) <= bound)
    # every non-zero channel reaches the largest code
    mags = np.abs(oracle.e4m3_to_f64(q)).max(axis=1)
    assert np.all(mags[amax > 0] == E4M3_MAX)


def test_fp8_experts_equal_bf16_experts_on_representable_weights():
    """With weights that quantize exactly, the e4m3 expert evaluation is the
    bf16 one operation for operation, so the fp64 results are identical."""
    rng = np.random.default_rng(5)
    E, d, de, n = 3, 64, 48, 7
    W1 = np.stack([_representable_matrix(rng, d, de)[0] for _ in range(E)])
    W3 = np.stack([_representable_matrix(rng, d, de)[0] for _ in range(E)])
    W2 = np.stack([_representable_matrix(rng, de, d)[0] for _ in range(E)])
    x = _bf16_bits(rng.standard_normal((n, d)).astype(np.float32))
    experts = rng.integers(0, E, n).astype(np.int32)
    gates = rng.uniform(0.05, 1.0, n)
    q = oracle.quantize_experts(dict(W1=W1, W3=W3, W2=W2))
    h8, y8 = oracle.expert_rows_w8(x, experts, gates, q)
    h16, y16 = oracle.expert_rows(x, experts, gates, W1, W3, W2)
    assert np.array_equal(h8, h16) and np.array_equal(y8, y16)


def test_fp8_experts_close_to_bf16_experts_on_random_weights():
    """Random weights: the fp8 result differs from the bf16 one by the
    quantisation error only (a few per cent at most), and a wrong scale
    index would not."""
    rng = np.random.default_rng(9)
    E, d, de, n = 2, 128, 64, 6
    W1 = _bf16_bits(rng.standard_normal((E, d, de)) / np.sqrt(d))
    W3 = _bf16_bits(rng.standard_normal((E, d, de)) / np.sqrt(d))
    W2 = _bf16_bits(rng.standard_normal((E, de, d)) / np.sqrt(de))
    x = _bf16_bits(rng.standard_normal((n, d)).astype(np.float32))
    experts = np.array([0, 1, 0, 1, 1, 0], np.int32)
    gates = np.ones(n)
    q = oracle.quantize_experts(dict(W1=W1, W3=W3, W2=W2))
    _, y8 = oracle.expert_rows_w8(x, experts, gates, q)
    _, y16 = oracle.expert_rows(x, experts, gates, W1, W3, W2)
    rel = np.linalg.norm(y8 - y16) / np.linalg.norm(y16)
    assert 1e-4 < rel < 0.05
    # planted mistake: scales of the down projection reversed
    bad = dict(q)
    bad["S2"] = q["S2"][:, ::-1].copy()
    _, yb = oracle.expert_rows_w8(x, experts, gates, bad)
    assert np.linalg.norm(yb - y16) / np.linalg.norm(y16) > 5 * rel


def test_grouped_w8_matches_rows_w8():
    rng = np.random.default_rng(2)
    E, d, de, P = 4, 64, 32, 16
    W1 = _bf16_bits(rng.standard_normal((E, d, de)) / 8)
    W3 = _bf16_bits(rng.standard_normal((E, d, de)) / 8)
    W2 = _bf16_bits(rng.standard_normal((E, de, d)) / 8)
    q = oracle.quantize_experts(dict(W1=W1, W3=W3, W2=W2))
    T, k = 20, 2
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.uniform(0.1, 1, (T, k))
    x = _bf16_bits(rng.standard_normal((T, d)))
    off = oracle.build_offsets(idx, w, E, P)
    xp = oracle.permute(x, off["row_src"], k)
    h, y = oracle.grouped_experts_w8(xp, q, off["block_metadata"], off["row_gate"])
    a = np.arange(T * k)
    hr, yr = oracle.expert_rows_w8(x[a // k], idx.reshape(-1), w.reshape(-1), q)
    assert np.array_equal(y[off["perm_row"]], yr) and np.array_equal(h[off["perm_row"]], hr)
    pad = off["row_src"] < 0
    assert np.all(np.isnan(y[pad]))


def test_shared_w8_equals_one_expert_rows():
    """The e4m3 shared expert is the one-expert routed evaluation with gate 1,
    and with exactly representable weights it equals the bf16 shared expert."""
    rng = np.random.default_rng(4)
    d, ds, n = 64, 48, 5
    Ws1 = _representable_matrix(rng, d, ds)[0]
    Ws3 = _representable_matrix(rng, d, ds)[0]
    Ws2 = _representable_matrix(rng, ds, d)[0]
    x = _bf16_bits(rng.standard_normal((n, d)).astype(np.float32))
    qs = oracle.quantize_shared(dict(Ws1=Ws1, Ws3=Ws3, Ws2=Ws2))
    h8, y8 = oracle.shared_expert_w8(x, qs)
    h16, y16 = oracle.shared_expert(x, Ws1, Ws3, Ws2)
    assert np.array_equal(h8, h16) and np.array_equal(y8, y16)
