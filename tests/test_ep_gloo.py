"""Expert parallelism (routing_permute_grouped_gb300/ep.py) on CPU process
groups.

The exchange logic (the counts all-to-all, the receiver's expert-major layout
built from the counts, the piece lists read off it, the two piece-by-piece
exchanges) runs with world size 2 over gloo, with the oracle as the compute
backend on each rank: rank r holds experts
[r*E/2, (r+1)*E/2) and its own half of the tokens.  Every rank's output must
equal, bit for bit, the single-process oracle's output for the same tokens:
dispatch and combine only move rows, and the combine keeps its order.  The
receiver's layout (the oracle's definition, which the device entry point
moe_build_blocks_from_counts is compared with on the GPU) and the piece lists
are checked on hand-worked examples and against the single-GPU offsets of
the same rows.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from routing_permute_grouped_gb300 import ep, synth
from routing_permute_grouped_gb300.synth import MoeShape
from tests.helpers import enforce_margin, oracle_inputs


def test_receiver_layout_worked_example():
    # this rank (0 of W = 2, El = 2, P = 4) keeps experts 0, 1 and receives
    # 5 rows for expert 0 from itself; 4 for expert 0 and 7 for expert 1 from
    # rank 1.  Expert 0's segment: 5 + 4 = 9 rows, padded to 12; expert 1: 7,
    # padded to 8.  Sender 1's rows of expert 0 land right after sender 0's.
    lay = oracle.blocks_from_counts(np.array([[5, 0], [4, 7]]), 4)
    assert lay["padded_offsets"].tolist() == [0, 12, 20]
    assert lay["piece_row"].tolist() == [[0, 12], [5, 12]]
    assert lay["num_blocks"] == 5
    assert lay["block_metadata"].tolist() == [[0, 0, 4], [0, 4, 4], [0, 8, 1], [1, 12, 4],
                                              [1, 16, 3]]


def test_receiver_layout_is_the_single_gpu_layout_of_the_arriving_rows():
    # the expert-major layout built from counts equals the offsets stage's
    # layout of the arriving assignments concatenated in sender order: the
    # same segments and blocks, and sender s's first row of expert e sits
    # where the stable order puts it
    rng = np.random.default_rng(5)
    for W, El, P in ((1, 8, 128), (3, 5, 64), (4, 2, 128)):
        per_src = [rng.choice(El, size=int(rng.integers(0, 400)),
                              p=rng.dirichlet(np.full(El, 0.4))).astype(np.int32)
                   for _ in range(W)]
        counts = np.stack([np.bincount(a, minlength=El) for a in per_src]).astype(np.int32)
        lay = oracle.blocks_from_counts(counts, P)
        cat = np.concatenate(per_src + [np.zeros(0, np.int32)])
        if cat.size == 0:
            continue
        off = oracle.build_offsets(cat, None, El, P)
        assert np.array_equal(lay["padded_offsets"], off["padded_offsets"])
        assert lay["num_blocks"] == off["num_blocks"]
        assert np.array_equal(lay["block_metadata"], off["block_metadata"])
        start = np.cumsum([0] + [a.size for a in per_src])
        for s_ in range(W):
            for e in range(El):
                hit = np.flatnonzero(per_src[s_] == e)
                if hit.size:
                    assert lay["piece_row"][s_, e] == off["perm_row"][start[s_] + hit[0]]
        if W == 1:
            assert np.array_equal(lay["piece_row"][0], off["padded_offsets"][:-1])


def test_plan_pieces_worked_example():
    # rank 0 of W = 2, El = 2: it routes 5, 0, 3, 9 rows to experts 0..3
    # (its own padded segments start at 0, 8, 8, 12); it receives [5, 0] from
    # itself and [4, 7] from rank 1, landing as in the worked layout above
    sends, recvs = ep.plan_pieces(0, 2, [5, 0, 3, 9], [0, 8, 8, 12, 24], [[5, 0], [4, 7]],
                                  [[0, 12], [5, 12]])
    # expert 0 to itself; experts 2, 3 to rank 1, each from its segment start
    assert sends == [(0, 0, 5), (1, 8, 3), (1, 12, 9)]
    # expert-major: expert 0 from ranks 0 and 1, expert 1 from rank 1
    assert recvs == [(0, 0, 5), (1, 5, 4), (1, 12, 7)]


def test_plan_pieces_conserves_rows():
    rng = np.random.default_rng(3)
    W, El, P = 4, 3, 64
    counts = rng.integers(0, 300, W * El)
    recv = rng.integers(0, 300, (W, El))
    own_po = np.concatenate([[0], np.cumsum(-(-counts // P) * P)])
    lay = oracle.blocks_from_counts(recv.astype(np.int32), P)
    sends, recvs = ep.plan_pieces(1, El, counts, own_po, recv, lay["piece_row"])
    assert sum(n for _, _, n in sends) == counts.sum()
    assert sum(n for _, _, n in recvs) == recv.sum()
    # pieces to each peer follow that peer's experts; arrivals fill each
    # segment's valid prefix exactly once
    for peer in range(W):
        assert [n for p, _, n in sends if p == peer] == [c for c in counts[peer * El:(peer + 1) * El]
                                                        if c > 0]
    covered = np.zeros(int(lay["padded_offsets"][-1]), np.int32)
    for _, r, n in recvs:
        covered[r:r + n] += 1
    for e in range(El):
        a, c = lay["padded_offsets"][e], recv[:, e].sum()
        assert (covered[a:a + c] == 1).all() and (covered[a + c:lay["padded_offsets"][e + 1]] == 0).all()


class OracleEp(ep.EpLayerBase):
    """The EP layer with the oracle as compute backend (CPU, fp64)."""

    def __init__(self, shape, inp, group=None):
        super().__init__(shape.E, shape.k, shape.pad, group)
        self.shape = shape
        lo, hi = self.rank * self.El, (self.rank + 1) * self.El
        self.W1, self.W3, self.W2 = (inp[n][lo:hi] for n in ("W1", "W3", "W2"))
        self.inp = inp

    def front(self, x, topk_idx=None, topk_w=None):
        s = self.shape
        xb = x.numpy().view(np.uint16)
        if topk_idx is None:
            lg = oracle.router_logits(xb, self.inp["Wg"], self.inp.get("bias"))
            topk_idx, topk_w, _ = oracle.route(lg, s.k, s.n_groups, s.topk_groups)
        off = oracle.build_offsets(topk_idx, topk_w, s.E, s.pad)
        x_perm = oracle.permute(xb, off["row_src"], s.k)
        # bf16 bits carried as int32 (gloo's all-to-all has no 16-bit type)
        return (torch.as_tensor(off["counts"]), torch.as_tensor(off["padded_offsets"]),
                torch.from_numpy(x_perm.astype(np.int32)),
                torch.from_numpy(off["row_gate"].astype(np.float64)), off)

    def layout(self, recv):
        lay = oracle.blocks_from_counts(recv.numpy().reshape(self.world, self.El), self.P)
        return dict(lay, piece_row=torch.from_numpy(lay["piece_row"]))

    def local_experts(self, xe, ge, lay, valid_rows):
        _, y = oracle.grouped_experts(xe.numpy().astype(np.uint16), self.W1, self.W3, self.W2,
                                      lay["block_metadata"], ge.numpy())
        return torch.from_numpy(y)

    def expert_major_buffers(self, rows, d, like_x, like_g):
        # the oracle reads only the valid rows of each block: any buffer that
        # holds the padded segments will do
        import torch as _t

        n = rows + self.El * self.P
        return (_t.zeros((n, d), dtype=like_x.dtype), _t.zeros((n,), dtype=like_g.dtype))

    def finish(self, x, y, off):
        s = self.shape
        R = off["row_src"].size
        yy = np.full((R, s.d), np.nan)
        yy[:y.shape[0]] = y.numpy()
        ys = None
        if s.d_shared:
            _, ys = oracle.shared_expert(x.numpy().view(np.uint16), self.inp["Ws1"],
                                         self.inp["Ws3"], self.inp["Ws2"])
        return oracle.combine(yy, off["perm_row"], s.k, ys)


CASES = {
    "routed_shared": MoeShape("ep_routed", T=48, d=256, d_e=128, E=8, k=2, pad=64, bias_std=0.5,
                              d_shared=128, seed=401),
    "groups": MoeShape("ep_groups", T=40, d=128, d_e=128, E=8, k=3, n_groups=4, topk_groups=2,
                       pad=128, seed=402),
    "prerouted": MoeShape("ep_pre", T=32, d=128, d_e=128, E=4, k=4, prerouted=(60, 20, 0, 48),
                          seed=403),
}


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _global_inputs(shape):
    inp = synth.make_inputs(shape)
    enforce_margin(inp, shape)
    return oracle_inputs(inp)


def _worker(rank, world, port, name, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    out = None
    try:
        shape = CASES[name]
        inp = _global_inputs(shape)
        T = shape.T // world
        toks = slice(rank * T, (rank + 1) * T)
        layer = OracleEp(shape, inp)
        x = torch.from_numpy(inp["x"][toks].view(np.int16))
        if shape.prerouted:
            out = layer.forward(x, inp["topk_idx"][toks], inp["topk_w"][toks])
        else:
            out = layer.forward(x)
    except Exception:  # report instead of leaving the parent waiting
        import traceback

        out = traceback.format_exc()
    finally:
        q.put((rank, out))
        dist.destroy_process_group()


@pytest.mark.parametrize("name", list(CASES))
def test_ep_forward_matches_the_single_process_layer(name):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    world = 2
    procs = [ctx.Process(target=_worker, args=(r, world, port, name, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    for r in range(world):
        assert not isinstance(res[r], str), res[r]
    for p in procs:
        assert p.exitcode == 0
    shape = CASES[name]
    ref = oracle.layer_forward(_global_inputs(shape), shape)["out"]
    got = np.concatenate([res[r] for r in range(world)])
    assert np.array_equal(got, ref)
