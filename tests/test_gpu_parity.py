"""GPU parity: every entry point of the C ABI against the CPU oracle on the
same seeded inputs.

Routing indices, counts, offsets, the block table and the permutation must
be bit-exact (the inputs are redrawn until every routing decision has a
fp64 margin >= 1e-3, so fp32 logits decide the same way); permuted rows are
bit-exact copies; floating outputs must have a relative Frobenius error
<= 5e-3 and a max error <= 3e-2 * max|ref|.  Shapes span several tiles in
M, N and K, ragged tails, empty experts, padding 64 and 128, group-limited
routing, a router width that is not a power of two, and a model width that
is not a multiple of 256.
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
    "tiny": synth.WORKLOADS["tiny"],
    "small_default": MoeShape("small_default", T=777, d=1024, d_e=384, E=8, k=4, bias_std=0.5,
                              d_shared=256, seed=77),
    "small_decode": MoeShape("small_decode", T=37, d=512, d_e=256, E=64, k=8, n_groups=8,
                             topk_groups=4, d_shared=128, seed=78),
    "small_prerouted": MoeShape("small_prerouted", T=300, d=512, d_e=256, E=4, k=8,
                                prerouted=(900, 321, 1000, 179), seed=79),
    "small_imbalance_p64": MoeShape("small_imbalance_p64", T=2000, d=512, d_e=256, E=64, k=6,
                                    pad=64, zipf_target=2.0, seed=80),
    "small_e100_d384": MoeShape("small_e100_d384", T=300, d=384, d_e=128, E=100, k=3,
                                bias_std=0.3, seed=81),
}
ZIPF_S = {"small_imbalance_p64": 1.0}

_cache = {}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU parity tests need a CUDA device")
    moe_build.build()
    moe.load()


def prepared(name):
    """(shape, CPU inputs after the margin filter, oracle result)."""
    if name not in _cache:
        shape = SHAPES[name]
        inp = synth.make_inputs(shape, zipf_s=ZIPF_S.get(name))
        enforce_margin(inp, shape)
        ref = oracle.layer_forward(oracle_inputs(inp), shape)
        _cache[name] = (shape, inp, ref)
    return _cache[name]


def cuda(t):
    return None if t is None else t.cuda().contiguous()


def f64(t):
    return t.detach().float().cpu().double().numpy()


def assert_close(got, ref, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, what
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / (nref if nref > 0 else 1.0)
    mx = np.abs(got - ref).max() if got.size else 0.0
    bound = MAX_REL * (np.abs(ref).max() if ref.size else 0.0)
    assert rel <= REL_FRO, f"{what}: relative Frobenius error {rel:.3e}"
    assert mx <= bound + 1e-30, f"{what}: max error {mx:.3e} > {bound:.3e}"


def make_layer(shape, inp):
    cfg = moe.config_of(shape)
    layer = moe.MoeLayer(cfg, cuda(inp["W1"]), cuda(inp["W3"]), cuda(inp["W2"]),
                         Wg=cuda(inp.get("Wg")), bias=cuda(inp.get("bias")),
                         Ws1=cuda(inp.get("Ws1")), Ws3=cuda(inp.get("Ws3")),
                         Ws2=cuda(inp.get("Ws2")))
    return cfg, layer


# ------------------------------------------------------------- packing ----
def test_pack_weights_interleaves_gate_and_up():
    """moe_pack_weights (the config form of the gate/up pack): row 256 j + c
    of expert e's packed matrix is gate column 128 j + c and row
    256 j + 128 + c the matching up column, K (= d) contiguous; the same bytes
    as moe_pack_experts writes."""
    E, d, de = 3, 384, 256
    W1 = torch.randn(E, d, de).to(torch.bfloat16)
    W3 = torch.randn(E, d, de).to(torch.bfloat16)
    W2 = torch.randn(E, de, d).to(torch.bfloat16)
    cfg = moe.config_of(T=1, d=d, d_e=de, E=E, k=1)
    W13 = torch.empty(E, 2 * de, d, dtype=torch.bfloat16, device="cuda")
    moe.moe_pack_weights(cfg, cuda(W1), cuda(W3), W13)
    ref = torch.empty(E, 2 * de, d, dtype=torch.bfloat16)
    for j in range(de // 128):
        ref[:, 256 * j:256 * j + 128] = W1[:, :, 128 * j:128 * j + 128].transpose(1, 2)
        ref[:, 256 * j + 128:256 * j + 256] = W3[:, :, 128 * j:128 * j + 128].transpose(1, 2)
    assert torch.equal(W13.cpu(), ref)
    W13b = torch.empty_like(W13)
    W2t = torch.empty(E, d, de, dtype=torch.bfloat16, device="cuda")
    moe.moe_pack_experts(cuda(W1), cuda(W3), cuda(W2), W13b, W2t)
    assert torch.equal(W13b, W13)
    assert torch.equal(W2t.cpu(), W2.transpose(1, 2))


# ---------------------------------------------------------------- layer ----
@pytest.mark.parametrize("name", list(SHAPES))
def test_layer_matches_oracle(name):
    shape, inp, ref = prepared(name)
    cfg, layer = make_layer(shape, inp)
    x = cuda(inp["x"])
    if shape.prerouted:
        out = layer(x, topk_idx=cuda(inp["topk_idx"]), topk_w=cuda(inp["topk_w"]))
    else:
        out = layer(x)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    T, k, E, d, de = shape.T, shape.k, shape.E, shape.d, shape.d_e
    A, R, NB = shape.A, shape.rows_capacity, shape.blocks_capacity
    i32 = torch.int32
    if not shape.prerouted:
        gidx = layer.buffer("topk_idx", i32, (T, k)).cpu().numpy()
        assert np.array_equal(gidx, ref["topk_idx"])
        gw = layer.buffer("topk_w", torch.float32, (T, k)).cpu().double().numpy()
        np.testing.assert_allclose(gw, ref["topk_w"], rtol=0, atol=2e-5)
    assert np.array_equal(layer.buffer("counts", i32, (E,)).cpu().numpy(), ref["counts"])
    assert np.array_equal(layer.buffer("padded_offsets", i32, (E + 1,)).cpu().numpy(),
                          ref["padded_offsets"])
    nb = int(layer.buffer("num_blocks", i32, (1,)).item())
    assert nb == ref["num_blocks"]
    meta = layer.buffer("block_metadata", i32, (NB, 3)).cpu().numpy()[:nb]
    assert np.array_equal(meta, ref["block_metadata"])
    assert np.array_equal(layer.buffer("perm_row", i32, (A,)).cpu().numpy(), ref["perm_row"])
    assert np.array_equal(layer.buffer("row_src", i32, (R,)).cpu().numpy(), ref["row_src"])
    rg = layer.buffer("row_gate", torch.float32, (R,)).cpu().double().numpy()
    np.testing.assert_allclose(rg, ref["row_gate"], rtol=0, atol=2e-5)
    valid = ref["row_src"] >= 0
    xp = bits(layer.buffer("x_perm", torch.bfloat16, (R, d)).cpu())
    assert np.array_equal(xp[valid], ref["x_perm"][valid])
    h = f64(layer.buffer("h", torch.bfloat16, (R, de)))
    assert_close(h[valid], ref["h"][valid], "h")
    y = f64(layer.buffer("y", torch.bfloat16, (R, d)))
    assert_close(y[valid], ref["y"][valid], "y")
    if shape.d_shared:
        ys = layer.buffer("ys", torch.bfloat16, (T, d))
        assert_close(f64(ys), ref["ys"], "shared ys")
        # the layer's output is the combine of its own buffers, bit for bit
        out2 = torch.empty_like(out)
        moe.moe_combine(cfg, layer.buffer("y", torch.bfloat16, (R, d)),
                        layer.buffer("perm_row", i32, (A,)), ys, out2)
        torch.cuda.synchronize()
        assert torch.equal(out2, out)
    assert_close(f64(out), ref["out"], "out")


@pytest.mark.parametrize("name, permute", [
    ("small_default", "kernel"), ("small_default", "gemm"),
    ("small_prerouted", "kernel"), ("small_prerouted", "gemm"),
    ("small_imbalance_p64", "gemm"),
])
def test_layer_equals_its_stages(name, permute):
    """moe_layer_fwd (on the CTA-pair path: the permute in the shared GEMM1's
    epilogue with a shared expert, its own kernel without) equals the stage
    calls composed by hand, bit for bit: router, offsets, then the permute as
    its own kernel or in GEMM1's copy warps, the grouped GEMMs, the shared
    expert's two halves and the combine.  The arithmetic is the same
    whichever kernel moves the rows."""
    shape, inp, _ = prepared(name)
    cfg, layer = make_layer(shape, inp)
    x = cuda(inp["x"])
    kw = dict(topk_idx=cuda(inp["topk_idx"]), topk_w=cuda(inp["topk_w"])) if shape.prerouted else {}
    out = layer(x, **kw).clone()
    T, k, E, d, de, ds = shape.T, shape.k, shape.E, shape.d, shape.d_e, shape.d_shared
    A, R, NB = shape.A, shape.rows_capacity, shape.blocks_capacity
    dev = dict(device="cuda")
    i32, f32, bf = torch.int32, torch.float32, torch.bfloat16
    if shape.prerouted:
        idx, w = kw["topk_idx"], kw["topk_w"]
    else:
        idx = torch.empty((T, k), dtype=i32, **dev)
        w = torch.empty((T, k), dtype=f32, **dev)
        n = moe.moe_route_splitk_scratch_size(cfg)
        part = torch.empty(max(n // 4, 1), dtype=f32, **dev) if n else None
        moe.moe_route_splitk(cfg, x, layer.Wg_t, layer.bias, idx, w, part)
    counts = torch.empty(E, dtype=i32, **dev)
    po = torch.empty(E + 1, dtype=i32, **dev)
    meta = torch.empty((NB, 3), dtype=i32, **dev)
    nb = torch.empty(1, dtype=i32, **dev)
    perm = torch.empty(A, dtype=i32, **dev)
    row_src = torch.empty(R, dtype=i32, **dev)
    gate = torch.empty(R, dtype=f32, **dev)
    ws = torch.empty(moe.moe_offsets_workspace_size(cfg), dtype=torch.uint8, **dev)
    moe.moe_build_offsets(cfg, idx, w, counts, po, meta, nb, perm, row_src, gate, ws)
    x_perm = torch.zeros((R, d), dtype=bf, **dev)
    h = torch.zeros((R, de), dtype=bf, **dev)
    y = torch.zeros((R, d), dtype=bf, **dev)
    if permute == "kernel":
        moe.moe_permute(cfg, x, perm, x_perm)
        moe.moe_grouped_gemm_swiglu(cfg, x_perm, layer.W13, layer.W2_t, meta, nb, po, gate, h, y)
    else:
        ready = torch.empty(NB, dtype=i32, **dev)
        moe.moe_grouped_gemm_swiglu_permute(cfg, x, row_src, x_perm, ready, layer.W13,
                                            layer.W2_t, meta, nb, po, gate, h, y)
    ys = None
    if ds:
        hs = torch.empty((T, ds), dtype=bf, **dev)
        ys = torch.empty((T, d), dtype=bf, **dev)
        moe.moe_shared_expert_up(cfg, x, layer.Ws13, hs)
        moe.moe_shared_expert_down(cfg, hs, layer.Ws2_t, ys)
    out2 = torch.empty_like(out)
    moe.moe_combine(cfg, y, perm, ys, out2)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    assert torch.equal(out2, out)


def test_layer_is_deterministic():
    shape, inp, _ = prepared("small_default")
    cfg, layer = make_layer(shape, inp)
    x = cuda(inp["x"])
    a = layer(x).clone()
    b = layer(x).clone()
    assert torch.equal(a, b)


def test_layers_on_concurrent_streams():
    """Two layers (different shapes, one on the CTA-pair and one on the
    small-M path) enqueued alternately on two streams, each several times:
    every output equals the same layer's output run alone.  The library
    keeps no per-call state outside the caller's workspaces."""
    runs = []
    for name in ("small_default", "small_decode"):
        shape, inp, _ = prepared(name)
        cfg, layer = make_layer(shape, inp)
        x = cuda(inp["x"])
        alone = layer(x).clone()
        torch.cuda.synchronize()
        runs.append((layer, x, alone))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [[], []]
    for _ in range(4):
        for i, (layer, x, _) in enumerate(runs):
            with torch.cuda.stream(streams[i]):
                out = torch.empty_like(x)
                layer.forward(x, out, stream=streams[i])
                outs[i].append(out)
    torch.cuda.synchronize()
    for i, (layer, _, alone) in enumerate(runs):
        assert layer.device_status() == 0
        for out in outs[i]:
            assert torch.equal(out, alone)


# --------------------------------------------------------------- stages ----
@pytest.mark.parametrize("name", ["tiny", "small_decode", "small_e100_d384", "small_imbalance_p64"])
def test_route_stage(name):
    shape, inp, ref = prepared(name)
    cfg = moe.config_of(shape)
    Wg_t = torch.empty((shape.E, shape.d), dtype=torch.bfloat16, device="cuda")
    moe.moe_pack_router(cuda(inp["Wg"]), Wg_t)
    idx = torch.full((shape.T, shape.k), -7, dtype=torch.int32, device="cuda")
    w = torch.zeros((shape.T, shape.k), dtype=torch.float32, device="cuda")
    moe.moe_route(cfg, cuda(inp["x"]), Wg_t, cuda(inp.get("bias")), idx, w)
    assert np.array_equal(idx.cpu().numpy(), ref["topk_idx"])
    np.testing.assert_allclose(w.cpu().double().numpy(), ref["topk_w"], rtol=0, atol=2e-5)
    # the split-K router (slices over a cluster, or partial logits + a
    # reduce/top-k kernel) decides the same
    nbytes = moe.moe_route_splitk_scratch_size(cfg)
    partial = torch.empty(max(nbytes // 4, 1), dtype=torch.float32, device="cuda")
    idx.fill_(-7)
    w.zero_()
    moe.moe_route_splitk(cfg, cuda(inp["x"]), Wg_t, cuda(inp.get("bias")), idx, w, partial)
    assert np.array_equal(idx.cpu().numpy(), ref["topk_idx"])
    np.testing.assert_allclose(w.cpu().double().numpy(), ref["topk_w"], rtol=0, atol=2e-5)


# Router shapes for the split-K paths: K slices x 128-token tiles.  Up to 4
# slices with E <= 64 run as one clustered kernel (tile width 16, 32 or 64);
# more slices, or more experts, take partial logits and a reduce kernel.
ROUTER_SHAPES = {
    "partial_bn16_s8": MoeShape("partial_bn16_s8", T=2000, d=512, d_e=128, E=8, k=2,
                                bias_std=0.5, seed=90),
    "cluster_bn16_s3": MoeShape("cluster_bn16_s3", T=5000, d=384, d_e=128, E=8, k=2,
                                bias_std=0.5, seed=95),
    "cluster_bn16_s2": MoeShape("cluster_bn16_s2", T=8000, d=1024, d_e=128, E=16, k=4, seed=91),
    "cluster_bn32_s4": MoeShape("cluster_bn32_s4", T=4000, d=1024, d_e=128, E=32, k=3,
                                bias_std=0.3, seed=92),
    "cluster_bn64_s2": MoeShape("cluster_bn64_s2", T=8100, d=768, d_e=128, E=64, k=6,
                                n_groups=8, topk_groups=4, seed=93),
    "partial_bn64_s8": MoeShape("partial_bn64_s8", T=1500, d=1024, d_e=128, E=48, k=5,
                                n_groups=4, topk_groups=2, bias_std=0.2, seed=94),
}


@pytest.mark.parametrize("name", list(ROUTER_SHAPES))
def test_route_splitk_paths(name):
    """moe_route_splitk against the oracle's routing (indices bit-exact after
    the margin filter, gates to 2e-5) on each form of the split-K router, and
    the scratch size that each form asks for."""
    shape = ROUTER_SHAPES[name]
    inp = synth.make_inputs(shape)
    enforce_margin(inp, shape)
    bias = None if inp.get("bias") is None else inp["bias"].numpy()
    lg = oracle.router_logits(bits(inp["x"]), bits(inp["Wg"]), bias)
    ref_idx, ref_w, margin = oracle.route(lg, shape.k, shape.n_groups, shape.topk_groups)
    assert margin.min() >= 1e-3
    cfg = moe.config_of(shape)
    nbytes = moe.moe_route_splitk_scratch_size(cfg)
    assert (nbytes == 0) == name.startswith("cluster"), nbytes
    Wg_t = torch.empty((shape.E, shape.d), dtype=torch.bfloat16, device="cuda")
    moe.moe_pack_router(cuda(inp["Wg"]), Wg_t)
    partial = torch.empty(max(nbytes // 4, 1), dtype=torch.float32, device="cuda")
    idx = torch.full((shape.T, shape.k), -7, dtype=torch.int32, device="cuda")
    w = torch.zeros((shape.T, shape.k), dtype=torch.float32, device="cuda")
    for _ in range(2):  # twice: nothing may depend on what a previous call left
        moe.moe_route_splitk(cfg, cuda(inp["x"]), Wg_t, cuda(inp.get("bias")), idx, w, partial)
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy(), ref_idx)
        np.testing.assert_allclose(w.cpu().double().numpy(), ref_w, rtol=0, atol=2e-5)
        idx.fill_(-7)
        w.zero_()


def _offsets_case(idx, w, E, P):
    T, k = idx.shape
    cfg = moe.config_of(T=T, d=128, d_e=128, E=E, k=k, pad_multiple=P)
    A = T * k
    R = A + E * (P - 1)
    NB = A // P + E
    dev = "cuda"
    out = dict(counts=torch.full((E,), -5, dtype=torch.int32, device=dev),
               padded_offsets=torch.full((E + 1,), -5, dtype=torch.int32, device=dev),
               block_metadata=torch.full((NB, 3), -5, dtype=torch.int32, device=dev),
               num_blocks=torch.full((1,), -5, dtype=torch.int32, device=dev),
               perm_row=torch.full((A,), -5, dtype=torch.int32, device=dev),
               row_src=torch.full((R,), -5, dtype=torch.int32, device=dev),
               row_gate=torch.full((R,), -5.0, dtype=torch.float32, device=dev))
    ws = torch.zeros(moe.moe_offsets_workspace_size(cfg), dtype=torch.uint8, device=dev)
    moe.moe_build_offsets(cfg, cuda(torch.as_tensor(idx)), cuda(torch.as_tensor(w)),
                          out["counts"], out["padded_offsets"], out["block_metadata"],
                          out["num_blocks"], out["perm_row"], out["row_src"], out["row_gate"], ws)
    status = moe.moe_get_device_status(ws)
    return {kk: v.cpu().numpy() for kk, v in out.items()}, status


@pytest.mark.parametrize("P", [64, 128])
@pytest.mark.parametrize("case", ["uniform", "skewed_empty", "one_expert", "worked_example", "exact_blocks",
                                  "large_table"])
def test_build_offsets_stage(P, case):
    # A <= 4096 takes the one-CTA kernel; above it, chunk tables of at most
    # 8192 entries (chunks x experts) the histogram + scan-and-scatter pair,
    # larger ones (large_table: 36 chunks x 256 experts) three launches
    rng = np.random.default_rng(hash(case) % 1000 + P)
    if case == "uniform":
        E, T, k = 8, 4097, 4  # several chunks, ragged tail
        idx = rng.integers(0, E, size=(T, k)).astype(np.int32)
    elif case == "skewed_empty":
        E, T, k = 256, 1111, 8
        p = rng.dirichlet(np.full(E, 0.05))
        idx = rng.choice(E, size=(T, k), p=p).astype(np.int32)
    elif case == "one_expert":
        E, T, k = 5, 3000, 1
        idx = np.full((T, k), 3, np.int32)
    elif case == "worked_example":
        # "Dropless and grouped GEMM", sec. 3 sizes, 8192 tokens x top-8
        sizes = [21733, 15004, 17982, 10817]
        lab = np.concatenate([np.full(c, e, np.int32) for e, c in enumerate(sizes)])
        idx = lab[rng.permutation(lab.size)].reshape(8192, 8)
        E = 4
    elif case == "large_table":
        E, T, k = 256, 9000, 8
        p = rng.dirichlet(np.full(E, 0.1))
        idx = rng.choice(E, size=(T, k), p=p).astype(np.int32)
    else:
        E, T, k = 4, 128, 4  # 128 rows per expert: one exact block each at P=128
        idx = np.repeat(np.arange(4, dtype=np.int32)[None, :], T, 0)
    w = rng.random(idx.shape).astype(np.float32)
    got, status = _offsets_case(idx, w, E, P)
    assert status == 0
    ref = oracle.build_offsets(idx, w.astype(np.float64), E, P)
    for key in ("counts", "padded_offsets", "perm_row", "row_src"):
        assert np.array_equal(got[key], ref[key]), key
    assert int(got["num_blocks"][0]) == ref["num_blocks"]
    assert np.array_equal(got["block_metadata"][:ref["num_blocks"]], ref["block_metadata"])
    assert np.array_equal(got["row_gate"].astype(np.float64), ref["row_gate"])
    if case == "worked_example" and P == 128:
        assert got["padded_offsets"].tolist() == [0, 21760, 36864, 54912, 65792]
        assert int(got["num_blocks"][0]) == 514


def test_build_offsets_flags_bad_expert_ids():
    idx = np.array([[0, 1], [9, 2], [3, -1], [1, 1]], np.int32)
    w = np.ones(idx.shape, np.float32)
    got, status = _offsets_case(idx, w, 4, 128)
    assert status & moe.DEVERR_EXPERT_RANGE
    assert got["perm_row"][2] == -1 and got["perm_row"][5] == -1
    assert got["counts"].tolist() == [1, 3, 1, 1]
    # the valid assignments keep the oracle's layout of the valid ids
    ok = np.array([0, 1, 3, 4, 6, 7])
    assert (got["row_src"][got["perm_row"][ok]] == ok).all()


@pytest.mark.parametrize("name", ["small_default", "small_prerouted"])
def test_permute_stage(name):
    shape, inp, ref = prepared(name)
    cfg = moe.config_of(shape)
    R = shape.rows_capacity
    x_perm = torch.zeros((R, shape.d), dtype=torch.bfloat16, device="cuda")
    moe.moe_permute(cfg, cuda(inp["x"]), cuda(torch.as_tensor(ref["perm_row"])), x_perm)
    got = bits(x_perm.cpu())
    valid = ref["row_src"] >= 0
    assert np.array_equal(got[valid], ref["x_perm"][valid])
    assert (got[~valid] == 0).all()  # pad rows untouched


@pytest.mark.parametrize("name", ["tiny", "small_default", "small_imbalance_p64", "small_e100_d384"])
def test_grouped_gemm_stage(name):
    shape, inp, ref = prepared(name)
    cfg = moe.config_of(shape)
    E, d, de, R, NB = shape.E, shape.d, shape.d_e, shape.rows_capacity, shape.blocks_capacity
    W13 = torch.empty((E, 2 * de, d), dtype=torch.bfloat16, device="cuda")
    W2_t = torch.empty((E, d, de), dtype=torch.bfloat16, device="cuda")
    moe.moe_pack_experts(cuda(inp["W1"]), cuda(inp["W3"]), cuda(inp["W2"]), W13, W2_t)
    # entries past num_blocks are stale: fill them with plausible-looking rows
    # of the real table, which the kernels must never use
    meta = np.resize(ref["block_metadata"], (NB, 3)).astype(np.int32)
    meta[:ref["num_blocks"]] = ref["block_metadata"]
    meta[ref["num_blocks"]:, 1] += 128
    gate32 = ref["row_gate"].astype(np.float32)
    x_perm = torch.from_numpy(ref["x_perm"].view(np.int16)).view(torch.bfloat16).cuda()
    h = torch.zeros((R, de), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((R, d), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_grouped_gemm_swiglu(cfg, x_perm, W13, W2_t, cuda(torch.from_numpy(meta)),
                                cuda(torch.tensor([ref["num_blocks"]], dtype=torch.int32)),
                                cuda(torch.from_numpy(ref["padded_offsets"])),
                                cuda(torch.from_numpy(gate32)), h, y, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    eh, ey = oracle.grouped_experts(ref["x_perm"], bits(inp["W1"]), bits(inp["W3"]),
                                    bits(inp["W2"]), ref["block_metadata"],
                                    gate32.astype(np.float64))
    valid = ref["row_src"] >= 0
    assert_close(f64(h)[valid], eh[valid], "h")
    assert_close(f64(y)[valid], ey[valid], "y")
    # pad rows are never written
    assert (f64(y)[~valid] == 0).all() and (f64(h)[~valid] == 0).all()


@pytest.mark.parametrize("name", ["tiny", "small_default", "small_imbalance_p64", "small_e100_d384",
                                  "small_prerouted"])
def test_grouped_gemm_permute_stage(name):
    """The grouped GEMMs with the permute done by GEMM1's copy warps: x_perm
    equals the oracle's permute on every valid row and keeps its pad rows,
    and h and y equal the stand-alone grouped GEMMs' on that x_perm, bit for
    bit; the call clears a stale visit_ready itself."""
    shape, inp, ref = prepared(name)
    cfg = moe.config_of(shape)
    E, d, de, R, NB = shape.E, shape.d, shape.d_e, shape.rows_capacity, shape.blocks_capacity
    W13 = torch.empty((E, 2 * de, d), dtype=torch.bfloat16, device="cuda")
    W2_t = torch.empty((E, d, de), dtype=torch.bfloat16, device="cuda")
    moe.moe_pack_experts(cuda(inp["W1"]), cuda(inp["W3"]), cuda(inp["W2"]), W13, W2_t)
    meta = cuda(torch.from_numpy(np.resize(ref["block_metadata"], (NB, 3)).astype(np.int32)))
    nb = cuda(torch.tensor([ref["num_blocks"]], dtype=torch.int32))
    po = cuda(torch.from_numpy(ref["padded_offsets"]))
    gate = cuda(torch.from_numpy(ref["row_gate"].astype(np.float32)))
    row_src = cuda(torch.from_numpy(ref["row_src"]))
    g = torch.Generator().manual_seed(11)
    fill = torch.randn((R, d), generator=g).to(torch.bfloat16).cuda()
    x_perm = fill.clone()
    ready = torch.full((NB,), 12345, dtype=torch.int32, device="cuda")
    h = torch.zeros((R, de), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((R, d), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_grouped_gemm_swiglu_permute(cfg, cuda(inp["x"]), row_src, x_perm, ready, W13, W2_t,
                                        meta, nb, po, gate, h, y, status)
    h0 = torch.zeros_like(h)
    y0 = torch.zeros_like(y)
    moe.moe_grouped_gemm_swiglu(cfg, x_perm, W13, W2_t, meta, nb, po, gate, h0, y0, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    valid = ref["row_src"] >= 0
    xp = bits(x_perm.cpu())
    assert np.array_equal(xp[valid], ref["x_perm"][valid])
    assert torch.equal(x_perm[torch.from_numpy(~valid).cuda()], fill[torch.from_numpy(~valid).cuda()])
    assert torch.equal(h, h0) and torch.equal(y, y0)


@pytest.mark.parametrize("name", ["small_default", "small_decode"])
def test_shared_expert_stage(name):
    shape, inp, ref = prepared(name)
    cfg = moe.config_of(shape)
    d, ds, T = shape.d, shape.d_shared, shape.T
    Ws13 = torch.empty((1, 2 * ds, d), dtype=torch.bfloat16, device="cuda")
    Ws2_t = torch.empty((1, d, ds), dtype=torch.bfloat16, device="cuda")
    moe.moe_pack_experts(cuda(inp["Ws1"]).unsqueeze(0).contiguous(),
                         cuda(inp["Ws3"]).unsqueeze(0).contiguous(),
                         cuda(inp["Ws2"]).unsqueeze(0).contiguous(), Ws13, Ws2_t)
    hs = torch.empty((T, ds), dtype=torch.bfloat16, device="cuda")
    ys = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    moe.moe_shared_expert(cfg, cuda(inp["x"]), Ws13, Ws2_t, hs, ys)
    assert_close(f64(hs), ref["hs"], "hs")
    assert_close(f64(ys), ref["ys"], "ys")


def assert_combine_bound(got, expect, y, perm_row, k, ys=None):
    """The combine sums k (+1) bf16 values in fp32 in a fixed order and rounds
    once to bf16.  Against the exact fp64 sum its error is at most half a
    bf16 ulp of the result plus the fp32 additions' error, each at most 2^-24
    of a partial sum, so k (+1) x 2^-24 x the sum of the terms' magnitudes;
    the second term matters only where the terms cancel.  Nearly every
    output is the correctly rounded exact sum."""
    mag = oracle.combine(np.abs(oracle.bf16_to_f64(bits(y))), perm_row, k,
                         None if ys is None else np.abs(oracle.bf16_to_f64(bits(ys))))
    n_terms = k + (0 if ys is None else 1)
    ulp = np.ldexp(1.0, np.frexp(np.abs(expect))[1] - 8)
    bound = ulp + n_terms * 2.0 ** -24 * mag
    assert (np.abs(got - expect) <= bound).all()
    assert np.mean(got == oracle.round_bf16(expect)) > 0.999


@pytest.mark.parametrize("shared", [False, True])
def test_combine_stage(shared):
    shape, inp, ref = prepared("small_default")
    cfg = moe.config_of(shape)
    R, d, T = shape.rows_capacity, shape.d, shape.T
    g = torch.Generator().manual_seed(5)
    y = torch.randn((R, d), generator=g).to(torch.bfloat16)
    ys = torch.randn((T, d), generator=g).to(torch.bfloat16) if shared else None
    out = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(cfg, cuda(y), cuda(torch.as_tensor(ref["perm_row"])), cuda(ys), out)
    expect = oracle.combine(oracle.bf16_to_f64(bits(y)), ref["perm_row"], shape.k,
                            None if ys is None else oracle.bf16_to_f64(bits(ys)))
    got = f64(out)
    assert_combine_bound(got, expect, y, ref["perm_row"], shape.k, ys)


@pytest.mark.parametrize("T, d, k, E", [
    (3000, 1152, 4, 8),   # 375 token CTAs: 3 combine and 2 permute column chunks, the last 16 vectors
    (2500, 2176, 8, 16),  # 313 token CTAs, k = 8: 5 combine and 3 permute chunks, the last 16 vectors
])
def test_permute_combine_column_chunks(T, d, k, E):
    """Grids of a few hundred token CTAs split their rows into column chunks
    (over grid.y) until they span about six waves of resident CTAs; the
    last chunk here is ragged.  The permute copies bit for bit (the
    oracle's rows, pad rows untouched) and the combine stays within the
    fp32 summation bound of the oracle's fp64 sum, with and without a shared
    row."""
    rng = np.random.default_rng(T + d)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    w = rng.random(idx.shape).astype(np.float32)
    off = oracle.build_offsets(idx, w.astype(np.float64), E, 128)
    perm, row_src = off["perm_row"], off["row_src"]
    R = row_src.size
    cfg = moe.config_of(T=T, d=d, d_e=128, E=E, k=k)
    g = torch.Generator().manual_seed(7)
    x = torch.randn((T, d), generator=g).to(torch.bfloat16)
    x_perm = torch.zeros((R, d), dtype=torch.bfloat16, device="cuda")
    moe.moe_permute(cfg, cuda(x), cuda(torch.as_tensor(perm)), x_perm)
    got = bits(x_perm.cpu())
    ref = oracle.permute(bits(x), row_src, k)
    valid = row_src >= 0
    assert np.array_equal(got[valid], ref[valid])
    assert (got[~valid] == 0).all()
    y = torch.randn((R, d), generator=g).to(torch.bfloat16)
    y64 = oracle.bf16_to_f64(bits(y))
    for shared in (False, True):
        ys = torch.randn((T, d), generator=g).to(torch.bfloat16) if shared else None
        out = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
        moe.moe_combine(cfg, cuda(y), cuda(torch.as_tensor(perm)), cuda(ys), out)
        expect = oracle.combine(y64, perm, k, None if ys is None else oracle.bf16_to_f64(bits(ys)))
        assert_combine_bound(f64(out), expect, y, perm, k, ys)


@pytest.mark.parametrize("T, d, ds, k, R", [
    (777, 1024, 384, 4, 3500),   # 3 column slices of 42/43 vectors, ragged last visit
    (300, 384, 128, 3, 1000),    # one slice; d not a multiple of 256 (128-column GEMM2 tiles)
    (40, 7168, 128, 2, 100),     # one slice of 896 vectors (several 64-vector passes)
    (1, 256, 128, 8, 64),        # one token, k = 8
])
def test_shared_expert_halves(T, d, ds, k, R):
    """The shared expert split as the layer runs it, against the stand-alone
    stage calls, bit for bit: moe_shared_expert_up writes the hs of
    moe_shared_expert and, with the permute in its epilogue, the x_perm of
    moe_permute (pad rows untouched); moe_shared_expert_down writes its ys;
    moe_shared_expert_down_combine writes moe_combine's output of those rows.
    Some perm_row entries are negative (rows that take no copy and add
    nothing)."""
    g = torch.Generator().manual_seed(T * 7 + d)
    cfg = moe.config_of(T=T, d=d, d_e=128, E=8, k=k, d_shared=ds)

    def rnd(*shape, std=1.0):
        return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)

    x = cuda(rnd(T, d))
    Ws13 = torch.empty((1, 2 * ds, d), dtype=torch.bfloat16, device="cuda")
    Ws2_t = torch.empty((1, d, ds), dtype=torch.bfloat16, device="cuda")
    moe.moe_pack_experts(cuda(rnd(1, d, ds, std=d ** -0.5)), cuda(rnd(1, d, ds, std=d ** -0.5)),
                         cuda(rnd(1, ds, d, std=ds ** -0.5)), Ws13, Ws2_t)
    perm = torch.randperm(R, generator=g)[:T * k].to(torch.int32)
    perm[::5] = -1
    perm = cuda(perm)
    hs = torch.empty((T, ds), dtype=torch.bfloat16, device="cuda")
    ys = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    moe.moe_shared_expert(cfg, x, Ws13, Ws2_t, hs, ys)
    xp_ref = cuda(rnd(R, d))
    xp = xp_ref.clone()
    moe.moe_permute(cfg, x, perm, xp_ref)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    hs2 = torch.zeros_like(hs)
    moe.moe_shared_expert_up(cfg, x, Ws13, hs2, perm, xp, status)
    ys2 = torch.zeros_like(ys)
    moe.moe_shared_expert_down(cfg, hs2, Ws2_t, ys2, status)
    y = cuda(rnd(R, d))
    expect = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(cfg, y, perm, ys, expect)
    out = torch.zeros_like(expect)
    moe.moe_shared_expert_down_combine(cfg, hs2, Ws2_t, y, perm, out, status)
    hs3 = torch.zeros_like(hs)
    moe.moe_shared_expert_up(cfg, x, Ws13, hs3, None, None, status)  # no permute
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(hs2, hs) and torch.equal(hs3, hs)
    assert torch.equal(xp, xp_ref)
    assert torch.equal(ys2, ys)
    assert torch.equal(out, expect)


def test_host_pipeline_matches_layer():
    # batches in pinned host memory through HostPipeline == the layer on
    # device tensors (same kernels, deterministic order: bit-identical)
    shape, inp, _ = prepared("small_default")
    cfg, layer = make_layer(shape, inp)
    g = torch.Generator().manual_seed(9)
    xs = [inp["x"]] + [torch.randn(inp["x"].shape, generator=g).to(torch.bfloat16)
                       for _ in range(4)]
    xs_host = [x.pin_memory() for x in xs]
    outs = [torch.empty_like(x).pin_memory() for x in xs]
    pipe = moe.HostPipeline(layer)
    for x, o in zip(xs_host, outs):
        pipe.submit(x, o)
    pipe.synchronize()
    for x, o in zip(xs, outs):
        ref = layer(cuda(x)).cpu()
        assert torch.equal(o, ref)


def test_host_pipeline_prerouted():
    shape, inp, ref = prepared("small_prerouted")
    cfg, layer = make_layer(shape, inp)
    x = inp["x"].pin_memory()
    o = torch.empty_like(x).pin_memory()
    pipe = moe.HostPipeline(layer)
    pipe.submit(x, o, topk_idx=inp["topk_idx"].pin_memory(), topk_w=inp["topk_w"].pin_memory())
    pipe.synchronize()
    assert_close(o.double().numpy(), ref["out"], "out")


@pytest.mark.parametrize("name", ["tiny", "small_default", "small_imbalance_p64", "small_e100_d384",
                                  "small_prerouted"])
def test_grouped_gemm_gather_stage(name):
    # the permute fused into GEMM1's A load: token rows gathered through
    # row_src must give the same h and y as the oracle's permuted layout
    shape, inp, ref = prepared(name)
    cfg = moe.config_of(shape)
    E, d, de, R, NB = shape.E, shape.d, shape.d_e, shape.rows_capacity, shape.blocks_capacity
    W13 = torch.empty((E, 2 * de, d), dtype=torch.bfloat16, device="cuda")
    W2_t = torch.empty((E, d, de), dtype=torch.bfloat16, device="cuda")
    moe.moe_pack_experts(cuda(inp["W1"]), cuda(inp["W3"]), cuda(inp["W2"]), W13, W2_t)
    meta = np.resize(ref["block_metadata"], (NB, 3)).astype(np.int32)
    meta[:ref["num_blocks"]] = ref["block_metadata"]
    gate32 = ref["row_gate"].astype(np.float32)
    h = torch.zeros((R, de), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((R, d), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_grouped_gemm_swiglu_gather(
        cfg, cuda(inp["x"]), cuda(torch.from_numpy(ref["row_src"])), W13, W2_t,
        cuda(torch.from_numpy(meta)), cuda(torch.tensor([ref["num_blocks"]], dtype=torch.int32)),
        cuda(torch.from_numpy(ref["padded_offsets"])), cuda(torch.from_numpy(gate32)), h, y, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    eh, ey = oracle.grouped_experts(ref["x_perm"], bits(inp["W1"]), bits(inp["W3"]),
                                    bits(inp["W2"]), ref["block_metadata"],
                                    gate32.astype(np.float64))
    valid = ref["row_src"] >= 0
    assert_close(f64(h)[valid], eh[valid], "h")
    assert_close(f64(y)[valid], ey[valid], "y")
    assert (f64(y)[~valid] == 0).all() and (f64(h)[~valid] == 0).all()


def test_bounded_wait_times_out_and_context_survives():
    # a kernel waits on a barrier that nothing signals: the bounded wait gives
    # up, the timeout bit is set, and the next work on the stream runs normally
    import time
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    moe.moe_selftest_wait_timeout(50_000_000, status)  # 50 ms
    torch.cuda.synchronize()
    assert time.time() - t0 < 5.0
    assert int(status.item()) & moe.DEVERR_TIMEOUT
    shape, inp, ref = prepared("tiny")
    cfg, layer = make_layer(shape, inp)
    out = layer(cuda(inp["x"]))
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    assert_close(f64(out), ref["out"], "out after a timed-out kernel")


def test_layer_captures_into_a_cuda_graph():
    # the whole layer enqueues kernels only (no host sync, no allocation), so
    # it can be recorded once and replayed: the replay equals the eager call
    shape, inp, ref = prepared("small_default")
    cfg, layer = make_layer(shape, inp)
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
    x.copy_(cuda(torch.flip(inp["x"], dims=[0])))  # new tokens, same graph
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, layer(x).clone())


EDGE = {
    "one_token": MoeShape("one_token", T=1, d=256, d_e=128, E=8, k=2, d_shared=128, seed=91),
    "k_equals_E": MoeShape("k_equals_E", T=130, d=256, d_e=128, E=4, k=4, seed=92),
    "single_expert": MoeShape("single_expert", T=300, d=384, d_e=256, E=1, k=1, seed=93),
    "hot_expert": MoeShape("hot_expert", T=700, d=256, d_e=128, E=16, k=2, bias_std=0.0, seed=94),
    "groups_keep_one": MoeShape("groups_keep_one", T=200, d=256, d_e=128, E=32, k=4, n_groups=4,
                                topk_groups=1, seed=95),
}


@pytest.mark.parametrize("name", list(EDGE))
def test_edge_case_layers(name):
    shape = EDGE[name]
    inp = synth.make_inputs(shape)
    if name == "hot_expert":
        # a large bias sends every token's first choice to expert 3
        inp["bias"] = torch.zeros(shape.E)
        inp["bias"][3] = 50.0
    enforce_margin(inp, shape)
    ref = oracle.layer_forward(oracle_inputs(inp), shape)
    cfg, layer = make_layer(shape, inp)
    out = layer(cuda(inp["x"]))
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    T, k, E = shape.T, shape.k, shape.E
    assert np.array_equal(layer.buffer("topk_idx", torch.int32, (T, k)).cpu().numpy(),
                          ref["topk_idx"])
    assert np.array_equal(layer.buffer("counts", torch.int32, (E,)).cpu().numpy(), ref["counts"])
    if name == "hot_expert":
        assert ref["counts"][3] == T
    assert_close(f64(out), ref["out"], "out")
