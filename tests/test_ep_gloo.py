"""Expert parallelism (routing_permute_grouped_gb300/ep.py) on CPU process
groups.

The exchange logic (piece sizes, the receiver's expert-major layout and block
table, the two piece-by-piece exchanges) runs with world size 2 over gloo, with the
oracle as the compute backend on each rank: rank r holds experts
[r*E/2, (r+1)*E/2) and its own half of the tokens.  Every rank's output must
equal, bit for bit, the single-process oracle's output for the same tokens:
dispatch and combine only move rows, and the combine keeps its order.  The
plan itself is also checked on a hand-worked example.
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


def test_plan_dispatch_worked_example():
    # this rank (of W = 2, El = 2, P = 4) routes 5, 0, 3, 9 rows to experts
    # 0..3; it receives 2 and 7 rows (experts 0, 1 of its own) from rank 0,
    # 4 and 0 from rank 1
    plan = ep.plan_dispatch(np.array([5, 0, 3, 9]), np.array([[2, 7], [4, 0]]), 4)
    assert plan.send_rows.tolist() == [8, 16]
    assert plan.recv_rows.tolist() == [12, 4]
    assert plan.padded_offsets.tolist() == [0, 8, 16]
    assert plan.rows == 16
    assert plan.block_metadata.tolist() == [[0, 0, 2], [0, 4, 4], [1, 8, 4], [1, 12, 3]]
    # this rank's padded segments (8, 0, 4, 12 rows) go out one per expert:
    # experts 0, 1 to rank 0, experts 2, 3 to rank 1
    assert plan.send_pieces == [(0, 0, 8), (1, 8, 4), (1, 12, 12)]
    # arriving pieces land expert-major, senders in rank order within an expert
    assert plan.recv_pieces == [(0, 0, 4), (1, 4, 4), (0, 8, 8)]


def test_plan_dispatch_conserves_rows():
    rng = np.random.default_rng(3)
    W, El, P = 4, 3, 64
    counts = rng.integers(0, 300, W * El)
    recv = rng.integers(0, 300, (W, El))
    plan = ep.plan_dispatch(counts, recv, P)
    assert plan.send_rows.sum() == ep.padded(counts, P).sum()
    assert plan.rows == plan.recv_rows.sum() == ep.padded(recv, P).sum()
    assert plan.block_metadata[:, 2].sum() == recv.sum()
    # the arriving pieces tile the expert-major layout exactly once, and the
    # sent pieces tile this rank's own padded layout
    for pieces, total in ((plan.recv_pieces, plan.rows), (plan.send_pieces, plan.send_rows.sum())):
        pos = 0
        for _, start, n in sorted(pieces, key=lambda p: p[1]):
            assert start == pos
            pos += n
        assert pos == total
    assert (plan.padded_offsets % P == 0).all()


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
        return (torch.as_tensor(off["counts"]), torch.from_numpy(x_perm.astype(np.int32)),
                torch.from_numpy(off["row_gate"].astype(np.float64)), off)

    def local_experts(self, xe, ge, plan):
        _, y = oracle.grouped_experts(xe.numpy().astype(np.uint16), self.W1, self.W3, self.W2,
                                      plan.block_metadata, ge.numpy())
        return torch.from_numpy(y)

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
