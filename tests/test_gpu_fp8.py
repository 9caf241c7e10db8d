"""GPU parity of the small-M (swapped-operand) grouped GEMM and of the e4m3
expert-weight path, against the CPU oracle on the same seeded inputs.

  - moe_pack_experts_fp8: codes and scales bit-exact against the oracle's
    quantizer (the integer codes are decided in fp32 on both sides);
  - moe_permute_fp8 and the split of h: the e4m3 pairs and row scales
    byte-exact against torch's float8 casts under the same row scale;
  - moe_grouped_gemm_swiglu_skinny (bf16 weights) and
    moe_grouped_gemm_swiglu_fp8: h and y of every valid row within the
    tolerances of the bf16 path (relative Frobenius <= 5e-3, max error
    <= 3e-2 * max|ref|), the oracle evaluating the dequantized weights
    exactly;
  - moe_layer_fwd_fp8: routing bit-exact, output within the same tolerances.
Shapes span blocks of 1..128 valid rows, several panels in N, a model width
that is not a multiple of 256 (a half panel), padding 64 and 128, and the
shared expert's tiles in the routed launches.
"""
import numpy as np
import pytest
import torch

import oracle
import routing_permute_grouped_gb300 as moe
from routing_permute_grouped_gb300 import build as moe_build
from routing_permute_grouped_gb300 import synth
from routing_permute_grouped_gb300.synth import MoeShape
from tests.helpers import bits, enforce_margin, oracle_inputs

pytestmark = pytest.mark.gpu

REL_FRO = 5e-3
MAX_REL = 3e-2

SHAPES = {
    "decode_like": MoeShape("decode_like", T=37, d=512, d_e=256, E=64, k=8, n_groups=8,
                            topk_groups=4, d_shared=128, seed=91),
    "full_blocks": MoeShape("full_blocks", T=777, d=1024, d_e=384, E=8, k=4, bias_std=0.5,
                            d_shared=256, seed=92),
    "half_panel_p64": MoeShape("half_panel_p64", T=300, d=384, d_e=128, E=20, k=3, pad=64,
                               bias_std=0.3, seed=93),
    "prerouted": MoeShape("prerouted", T=120, d=512, d_e=256, E=4, k=8,
                          prerouted=(400, 121, 300, 139), seed=94),
    # enough tokens for the warp-per-token form of the e4m3 permute (fewer
    # take a CTA per token)
    "many_tokens": MoeShape("many_tokens", T=3000, d=640, d_e=128, E=8, k=2, d_shared=128,
                            seed=95),
}

_cache = {}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU parity tests need a CUDA device")
    moe_build.build()
    moe.load()


def assert_close(got, ref, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, what
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    mx = np.abs(got - ref).max() if got.size else 0.0
    bound = MAX_REL * (np.abs(ref).max() if ref.size else 0.0)
    assert rel <= REL_FRO, f"{what}: relative Frobenius error {rel:.3e}"
    assert mx <= bound + 1e-30, f"{what}: max error {mx:.3e} > {bound:.3e}"


def cuda(t):
    return None if t is None else t.cuda().contiguous()


def prepared(name, fp8):
    """(shape, CPU inputs after the margin filter, oracle inputs, oracle
    layer result) with e4m3 (fp8=True) or bf16 expert weights."""
    key = (name, fp8)
    if key not in _cache:
        shape = SHAPES[name]
        inp = synth.make_inputs(shape)
        enforce_margin(inp, shape)
        oin = oracle_inputs(inp)
        if fp8:
            oin.update(oracle.quantize_experts(oin))
            if shape.d_shared:
                oin.update(oracle.quantize_shared(oin))
        ref = oracle.layer_forward(oin, shape)
        _cache[key] = (shape, inp, oin, ref)
    return _cache[key]


def _packed_perm(de):
    """Packed W13 row r -> (0 gate / 1 up, output column)."""
    r = np.arange(2 * de)
    blk, within = r // 256, r % 256
    return (within >= 128).astype(np.int64), blk * 128 + within % 128


# ----------------------------------------------------------- packing ----
def test_pack_fp8_matches_oracle():
    g = torch.Generator().manual_seed(5)
    E, d, de = 3, 384, 256
    W1 = (torch.randn(E, d, de, generator=g) / d ** 0.5).to(torch.bfloat16)
    W3 = (torch.randn(E, d, de, generator=g) / d ** 0.5).to(torch.bfloat16)
    W2 = (torch.randn(E, de, d, generator=g) / de ** 0.5).to(torch.bfloat16)
    W1[1, :, 7] = 0  # an all-zero channel
    W2[2, 3, :] *= 64  # a few large weights
    q13 = torch.empty((E, 2 * de, d), dtype=torch.uint8, device="cuda")
    s13 = torch.empty((E, 2 * de), dtype=torch.float32, device="cuda")
    q2 = torch.empty((E, d, de), dtype=torch.uint8, device="cuda")
    s2 = torch.empty((E, d), dtype=torch.float32, device="cuda")
    moe.moe_pack_experts_fp8(cuda(W1), cuda(W3), cuda(W2), q13, s13, q2, s2)
    torch.cuda.synchronize()
    ref = oracle.quantize_experts(dict(W1=bits(W1), W3=bits(W3), W2=bits(W2)))
    which, col = _packed_perm(de)
    Q13 = np.where(which[None, :, None] == 0, ref["Q1"].transpose(0, 2, 1)[:, col, :],
                   ref["Q3"].transpose(0, 2, 1)[:, col, :])
    S13 = np.where(which[None, :] == 0, ref["S1"][:, col], ref["S3"][:, col])
    assert np.array_equal(q13.cpu().numpy(), Q13)
    assert np.array_equal(s13.cpu().numpy(), S13)
    assert np.array_equal(q2.cpu().numpy(), ref["Q2"].transpose(0, 2, 1))
    assert np.array_equal(s2.cpu().numpy(), ref["S2"])


def _pairs_ref(rows_f32: torch.Tensor):
    """Expected e4m3 pairs of float32 rows (CPU): the row scale 2^sig is the
    largest power of two with max|v| * 2^sig <= 448, hi and lo are torch's
    nearest-even float8_e4m3fn casts of v * 2^sig and of the remainder."""
    v = rows_f32.double()
    amax = v.abs().amax(dim=1)
    sig = torch.where(amax > 0, torch.floor(torch.log2(448.0 / amax)), torch.zeros_like(amax))
    # guard the floor of a log against rounding at exact powers of two
    sig = torch.where(amax * 2.0 ** (sig + 1) <= 448.0, sig + 1, sig)
    sig = torch.where(amax * 2.0 ** sig > 448.0, sig - 1, sig)
    a = (v * 2.0 ** sig[:, None]).float()
    hi = a.to(torch.float8_e4m3fn)
    lo = (a - hi.float()).to(torch.float8_e4m3fn)
    return hi.view(torch.uint8), lo.view(torch.uint8), (2.0 ** -sig).float()


@pytest.mark.parametrize("name", ["full_blocks", "many_tokens"])
def test_permute_fp8_pairs_match_float8_casts(name):
    shape, inp, oin, ref = prepared(name, False)
    cfg = moe.config_of(shape)
    x = cuda(inp["x"])
    T, d, R = shape.T, shape.d, shape.rows_capacity
    perm_row = torch.as_tensor(ref["perm_row"], device="cuda")
    x8 = torch.zeros((2 * R, d), dtype=torch.uint8, device="cuda")
    xs = torch.zeros(R, dtype=torch.float32, device="cuda")
    xs8 = torch.zeros((2 * T, d), dtype=torch.uint8, device="cuda")
    xss = torch.zeros(T, dtype=torch.float32, device="cuda")
    moe.moe_permute_fp8(cfg, x, perm_row, x8, xs, xs8, xss)
    torch.cuda.synchronize()
    hi, lo, sc = _pairs_ref(inp["x"].float())
    assert torch.equal(xs8[0::2].cpu(), hi) and torch.equal(xs8[1::2].cpu(), lo)
    assert torch.equal(xss.cpu(), sc)
    rs = ref["row_src"]
    valid = np.flatnonzero(rs >= 0)
    tok = torch.as_tensor(rs[valid] // shape.k)
    vr = torch.as_tensor(valid, device="cuda")
    assert torch.equal(x8[2 * vr].cpu(), hi[tok]) and torch.equal(x8[2 * vr + 1].cpu(), lo[tok])
    assert torch.equal(xs[vr].cpu(), sc[tok])
    # hi + lo carries the bf16 values: exact within 2^10 of the row maximum
    recon = (hi.view(torch.float8_e4m3fn).double() + lo.view(torch.float8_e4m3fn).double()) * \
        sc.double()[:, None]
    xv = inp["x"].double()
    err = (recon - xv).abs()
    assert float((err / xv.abs().amax(dim=1, keepdim=True)).max()) < 2.0 ** -17


# ------------------------------------------------------------- stages ----
def _stage_tables(shape, ref):
    meta = torch.zeros((shape.blocks_capacity, 3), dtype=torch.int32)
    meta[:ref["num_blocks"]] = torch.as_tensor(ref["block_metadata"])
    # stale-looking entries past num_blocks must be ignored
    meta[ref["num_blocks"]:] = torch.tensor([shape.E - 1, 0, 128], dtype=torch.int32)
    nb = torch.tensor([ref["num_blocks"]], dtype=torch.int32)
    row_gate = torch.as_tensor(ref["row_gate"], dtype=torch.float32)
    return cuda(meta), cuda(nb), cuda(row_gate)


def _compare_rows(shape, ref, h, y):
    rs = ref["row_src"]
    valid = np.flatnonzero(rs >= 0)
    vt = torch.as_tensor(valid, device="cuda")
    assert_close(h[vt].double().cpu().numpy(), ref["h"][valid], "h")
    assert_close(y[vt].double().cpu().numpy(), ref["y"][valid], "y")


@pytest.mark.parametrize("name", ["decode_like", "full_blocks", "half_panel_p64"])
def test_skinny_stage_bf16(name):
    shape, inp, oin, ref = prepared(name, False)
    cfg = moe.config_of(shape)
    E, d, de, R = shape.E, shape.d, shape.d_e, shape.rows_capacity
    W13 = torch.empty((E, 2 * de, d), dtype=torch.bfloat16, device="cuda")
    W2t = torch.empty((E, d, de), dtype=torch.bfloat16, device="cuda")
    moe.moe_pack_experts(cuda(inp["W1"]), cuda(inp["W3"]), cuda(inp["W2"]), W13, W2t)
    xp = torch.from_numpy(ref["x_perm"].view(np.int16)).view(torch.bfloat16).cuda()
    meta, nb, row_gate = _stage_tables(shape, ref)
    h = torch.full((R, de), float("nan"), dtype=torch.bfloat16, device="cuda")
    y = torch.full((R, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_grouped_gemm_swiglu_skinny(cfg, xp, W13, W2t, meta, nb, row_gate, h, y, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _compare_rows(shape, ref, h, y)


def _fp8_weights(inp, E, d, de, key=("W1", "W3", "W2")):
    q13 = torch.empty((E, 2 * de, d), dtype=torch.uint8, device="cuda")
    s13 = torch.empty((E, 2 * de), dtype=torch.float32, device="cuda")
    q2 = torch.empty((E, d, de), dtype=torch.uint8, device="cuda")
    s2 = torch.empty((E, d), dtype=torch.float32, device="cuda")
    w = [cuda(inp[k_]) for k_ in key]
    if w[0].dim() == 2:
        w = [t.unsqueeze(0).contiguous() for t in w]
    moe.moe_pack_experts_fp8(w[0], w[1], w[2], q13, s13, q2, s2)
    return q13, s13, q2, s2


@pytest.mark.parametrize("name", ["decode_like", "full_blocks", "half_panel_p64"])
def test_fp8_stage(name):
    shape, inp, oin, ref = prepared(name, True)
    cfg = moe.config_of(shape)
    E, d, de, R = shape.E, shape.d, shape.d_e, shape.rows_capacity
    q13, s13, q2, s2 = _fp8_weights(inp, E, d, de)
    x8 = torch.zeros((2 * R, d), dtype=torch.uint8, device="cuda")
    xs = torch.zeros(R, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_permute_fp8(cfg, cuda(inp["x"]), torch.as_tensor(ref["perm_row"], device="cuda"), x8, xs)
    meta, nb, row_gate = _stage_tables(shape, ref)
    h = torch.full((R, de), float("nan"), dtype=torch.bfloat16, device="cuda")
    h8 = torch.zeros((2 * R, de), dtype=torch.uint8, device="cuda")
    hsc = torch.zeros(R, dtype=torch.float32, device="cuda")
    y = torch.full((R, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_gemm_swiglu_fp8(cfg, x8, xs, q13, s13, q2, s2, meta, nb, row_gate, h, h8, hsc, y,
                                    status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _compare_rows(shape, ref, h, y)
    # the pairs of h that GEMM2 multiplied are those of the GPU's own h
    vt = torch.as_tensor(np.flatnonzero(ref["row_src"] >= 0), device="cuda")
    hi, lo, sc = _pairs_ref(h[vt].float().cpu())
    assert torch.equal(h8[2 * vt].cpu(), hi) and torch.equal(h8[2 * vt + 1].cpu(), lo)
    assert torch.equal(hsc[vt].cpu(), sc)


def test_shared_expert_fp8_stage():
    shape, inp, oin, ref = prepared("full_blocks", True)
    cfg = moe.config_of(shape)
    T, d, ds, R = shape.T, shape.d, shape.d_shared, shape.rows_capacity
    q13, s13, q2, s2 = _fp8_weights(inp, 1, d, ds, key=("Ws1", "Ws3", "Ws2"))
    xs8 = torch.zeros((2 * T, d), dtype=torch.uint8, device="cuda")
    xss = torch.zeros(T, dtype=torch.float32, device="cuda")
    moe.moe_permute_fp8(cfg, cuda(inp["x"]), torch.as_tensor(ref["perm_row"], device="cuda"),
                        torch.zeros((2 * R, d), dtype=torch.uint8, device="cuda"),
                        torch.zeros(R, dtype=torch.float32, device="cuda"), xs8, xss)
    hs = torch.full((T, ds), float("nan"), dtype=torch.bfloat16, device="cuda")
    hs8 = torch.zeros((2 * T, ds), dtype=torch.uint8, device="cuda")
    hss = torch.zeros(T, dtype=torch.float32, device="cuda")
    ys = torch.full((T, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_shared_expert_fp8(cfg, xs8, xss, q13, s13, q2, s2, hs, hs8, hss, ys, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(hs.double().cpu().numpy(), ref["hs"], "hs (e4m3)")
    assert_close(ys.double().cpu().numpy(), ref["ys"], "ys (e4m3)")


# -------------------------------------------------------------- layer ----
def _make_layer(shape, inp, fp8):
    cfg = moe.config_of(shape)
    return cfg, moe.MoeLayer(cfg, cuda(inp["W1"]), cuda(inp["W3"]), cuda(inp["W2"]),
                             Wg=cuda(inp.get("Wg")), bias=cuda(inp.get("bias")),
                             Ws1=cuda(inp.get("Ws1")), Ws3=cuda(inp.get("Ws3")),
                             Ws2=cuda(inp.get("Ws2")), fp8=fp8)


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("fp8", [False, True])
def test_layer_matches_oracle(name, fp8):
    shape, inp, oin, ref = prepared(name, fp8)
    cfg, layer = _make_layer(shape, inp, fp8)
    x = cuda(inp["x"])
    if shape.prerouted:
        out = layer(x, topk_idx=cuda(inp["topk_idx"]), topk_w=cuda(inp["topk_w"]))
    else:
        out = layer(x)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    T, k, E = shape.T, shape.k, shape.E
    i32 = torch.int32
    if not shape.prerouted:
        assert np.array_equal(layer.buffer("topk_idx", i32, (T, k)).cpu().numpy(), ref["topk_idx"])
    nb = int(layer.buffer("num_blocks", i32, (1,)).item())
    assert nb == ref["num_blocks"]
    assert np.array_equal(layer.buffer("perm_row", i32, (shape.A,)).cpu().numpy(), ref["perm_row"])
    assert_close(out.double().cpu().numpy(), ref["out"], f"out ({'e4m3' if fp8 else 'bf16'})")


def test_fp8_layer_is_close_to_bf16_layer():
    """The e4m3 layer differs from the bf16 one by the weight quantisation
    only: a few per cent, far more than the parity tolerance, which is why
    its oracle dequantizes the same codes."""
    shape, inp, _, ref16 = prepared("decode_like", False)
    _, _, _, ref8 = prepared("decode_like", True)
    rel = np.linalg.norm(ref8["out"] - ref16["out"]) / np.linalg.norm(ref16["out"])
    assert 5e-3 < rel < 0.1
    _, layer = _make_layer(shape, inp, True)
    out = layer(cuda(inp["x"]))
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    assert np.linalg.norm(got - ref8["out"]) < 0.2 * np.linalg.norm(got - ref16["out"])


def test_fp8_layer_captures_into_a_cuda_graph():
    shape, inp, oin, ref = prepared("decode_like", True)
    _, layer = _make_layer(shape, inp, True)
    x = cuda(inp["x"])
    out = torch.empty_like(x)
    eager = layer(x).clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer(x, out, stream=s)  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer(x, out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    assert_close(out.double().cpu().numpy(), ref["out"], "out (graph replay)")


@pytest.mark.parametrize("fill", [0x00, 0x7F, 0xFF])
@pytest.mark.parametrize("name,fp8", [("decode_like", False), ("decode_like", True),
                                      ("full_blocks", False), ("full_blocks", True)])
def test_layer_ignores_stale_workspace(name, fp8, fill):
    """Every kernel reads data of the earlier kernels of the launch chain only
    after waiting for them: a workspace holding zeros or stale bytes before
    the call gives the same result, call after call."""
    shape, inp, oin, ref = prepared(name, fp8)
    _, layer = _make_layer(shape, inp, fp8)
    x = cuda(inp["x"])
    for _ in range(3):
        layer.ws.fill_(fill)
        layer.ws[:256].zero_()
        out = layer(x)
        torch.cuda.synchronize()
        assert layer.device_status() == 0
        assert_close(out.double().cpu().numpy(), ref["out"], f"out after a 0x{fill:02x} fill")


def test_widen_e4m3_is_exact():
    """moe_widen_e4m3: every code to the bf16 of its e4m3 value (torch's
    float8_e4m3fn cast), NaN codes to NaN."""
    codes = torch.arange(256, dtype=torch.uint8).repeat(4).cuda()
    out = torch.empty(codes.numel(), dtype=torch.bfloat16, device="cuda")
    moe.moe_widen_e4m3(codes, out)
    torch.cuda.synchronize()
    ref = codes.cpu().view(torch.float8_e4m3fn).to(torch.bfloat16)
    got = out.cpu()
    nan = torch.isnan(ref)
    assert torch.equal(torch.isnan(got), nan)
    assert torch.equal(got[~nan].view(torch.int16), ref[~nan].view(torch.int16))


@pytest.mark.parametrize("name", ["full_blocks", "half_panel_p64"])
def test_widened_scaled_stage(name):
    """The stage calls of the e4m3 layer above the small-M regime:
    moe_widen_e4m3 of the codes, then moe_grouped_gemm_swiglu_scaled (the
    per-channel scales on the accumulators) against the oracle's e4m3
    evaluation; moe_shared_expert_scaled likewise."""
    shape, inp, oin, ref = prepared(name, True)
    cfg = moe.config_of(shape)
    E, d, de, R = shape.E, shape.d, shape.d_e, shape.rows_capacity
    q13, s13, q2, s2 = _fp8_weights(inp, E, d, de)
    w13 = torch.empty(q13.shape, dtype=torch.bfloat16, device="cuda")
    w2 = torch.empty(q2.shape, dtype=torch.bfloat16, device="cuda")
    moe.moe_widen_e4m3(q13, w13)
    moe.moe_widen_e4m3(q2, w2)
    x_perm = torch.zeros((R, d), dtype=torch.bfloat16, device="cuda")
    moe.moe_permute(cfg, cuda(inp["x"]), torch.as_tensor(ref["perm_row"], device="cuda"), x_perm)
    meta, nb, row_gate = _stage_tables(shape, ref)
    po = cuda(torch.as_tensor(ref["padded_offsets"], dtype=torch.int32))
    h = torch.full((R, de), float("nan"), dtype=torch.bfloat16, device="cuda")
    y = torch.full((R, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_grouped_gemm_swiglu_scaled(cfg, x_perm, w13, s13, w2, s2, meta, nb, po, row_gate, h, y,
                                       status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _compare_rows(shape, ref, h, y)
    if shape.d_shared:
        ds, T = shape.d_shared, shape.T
        qs13, ss13, qs2, ss2 = _fp8_weights(inp, 1, d, ds, key=("Ws1", "Ws3", "Ws2"))
        ws13 = torch.empty(qs13.shape, dtype=torch.bfloat16, device="cuda")
        ws2 = torch.empty(qs2.shape, dtype=torch.bfloat16, device="cuda")
        moe.moe_widen_e4m3(qs13, ws13)
        moe.moe_widen_e4m3(qs2, ws2)
        hs = torch.empty((T, ds), dtype=torch.bfloat16, device="cuda")
        ys = torch.empty((T, shape.d), dtype=torch.bfloat16, device="cuda")
        moe.moe_shared_expert_scaled(cfg, cuda(inp["x"]), ws13, ss13, ws2, ss2, hs, ys, status)
        torch.cuda.synchronize()
        assert_close(ys.double().cpu().numpy(), ref["ys"], "shared ys (widened)")
