"""Expert parallelism: the layer forward over a torch.distributed group.

Rank r of W holds the routed experts [r * El, (r + 1) * El) (El = E / W) and
a copy of the router and of the shared expert.  One layer forward:

  1. each rank routes its own tokens and permutes them into the padded
     expert-major layout over all E experts (the single-GPU stages);
  2. the per-expert counts are exchanged, then each rank sends rank r' the
     contiguous rows of r''s experts, padded segments included, with their
     routing weights ("Dropless and grouped GEMM", sec. 14: the dispatch
     all-to-all, whose landing write does the permute and the padding);
  3. the receiver lays the W senders' pieces of each local expert out as one
     padded segment per expert (pieces in rank order: every piece is a
     multiple of P rows, so the concatenation is again a padded segment) and
     runs the grouped GEMMs on them with a block table built from the counts;
  4. the rows of y go back into the senders' layout (the combine all-to-all)
     and each rank combines its tokens with its shared expert's rows, as the
     single-GPU layer does.

The summation order of the combine is the single-GPU one, so a token's
output does not depend on W.  NCCL's all-to-all takes its split sizes on the
host: the per-expert counts cross to the host once per layer (a few hundred
bytes).  The plan functions below are plain host logic over those counts;
the compute steps go through a backend object (the CUDA library in
``GpuEp``), so the exchange logic can be exercised on CPU process groups.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def padded(c, P: int):
    """Padded segment size(s): ceil(c / P) * P, 0 for an empty expert."""
    c = np.asarray(c, np.int64)
    return -(-c // P) * P


@dataclass
class DispatchPlan:
    """Split sizes and the receiver's layout for one exchange.

    send_rows[r']   rows this rank sends to rank r' (padded, r''s experts)
    recv_rows[s]    rows this rank receives from rank s
    copies          (src_row, dst_row, rows): the received (source-major)
                    buffer into the expert-major layout, one per non-empty
                    (source, local expert) piece
    padded_offsets  [El + 1] of the expert-major layout
    block_metadata  [num_blocks, 3] = [local expert, m_start, valid_m]
    rows            rows of the expert-major layout (= padded_offsets[-1])
    """
    send_rows: np.ndarray
    recv_rows: np.ndarray
    copies: list
    padded_offsets: np.ndarray
    block_metadata: np.ndarray
    rows: int


def plan_dispatch(counts: np.ndarray, recv_counts: np.ndarray, P: int) -> DispatchPlan:
    """counts [E]: this rank's assignments per global expert; recv_counts
    [W, El]: what every rank s routes to this rank's local experts."""
    recv_counts = np.asarray(recv_counts, np.int64)
    W, El = recv_counts.shape
    counts = np.asarray(counts, np.int64)
    if counts.size != W * El:
        raise ValueError("counts must cover W * El experts")
    send_rows = padded(counts, P).reshape(W, El).sum(axis=1)
    pieces = padded(recv_counts, P)                      # [W, El]
    recv_rows = pieces.sum(axis=1)
    src_start = np.concatenate([[0], np.cumsum(recv_rows)[:-1]])
    seg_rows = pieces.sum(axis=0)                        # per local expert
    po = np.concatenate([[0], np.cumsum(seg_rows)]).astype(np.int32)
    copies, meta = [], []
    for e in range(El):
        dst = int(po[e])
        for s in range(W):
            n = int(pieces[s, e])
            if n == 0:
                continue
            src = int(src_start[s] + pieces[s, :e].sum())
            copies.append((src, dst, n))
            c = int(recv_counts[s, e])
            for m in range(0, c, P):
                meta.append((e, dst + m, min(P, c - m)))
            dst += n
    block_metadata = np.array(meta, np.int32).reshape(-1, 3)
    return DispatchPlan(send_rows, recv_rows, copies, po, block_metadata, int(po[-1]))


class EpLayerBase:
    """The exchange of an expert-parallel layer forward over a process group;
    subclasses supply the compute steps (``front``, ``local_experts``,
    ``finish``) and the tensors' device.  Data moves with
    torch.distributed.all_to_all_single (NCCL between GPUs)."""

    def __init__(self, E: int, k: int, P: int, group=None):
        import torch.distributed as dist

        self.dist = dist
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        if E % self.world:
            raise ValueError(f"E = {E} is not a multiple of the world size {self.world}")
        self.E, self.k, self.P = E, k, P
        self.El = E // self.world

    # -- compute steps (subclasses) ------------------------------------------
    def front(self, x, topk_idx=None, topk_w=None):
        """Route x (or take the given routing) and permute it into the padded
        expert-major layout over all E experts.  Returns (counts [E] device
        int32, x_perm [R, d], row_gate [R], tables for finish)."""
        raise NotImplementedError

    def local_experts(self, xe, ge, plan: DispatchPlan):
        """y rows [plan.rows, d] of the local experts for the expert-major rows
        xe with routing weights ge (the GEMM2 epilogue multiplies by them)."""
        raise NotImplementedError

    def finish(self, x, y, tables):
        """The layer output from this rank's y rows (its own padded layout)
        and its shared expert."""
        raise NotImplementedError

    def expert_major_buffers(self, rows: int, d: int, like_x, like_g):
        """Buffers of at least ``rows`` rows for the expert-major layout (a GPU
        backend hands out buffers of its full capacity: its GEMMs may read
        whole tiles past the last row)."""
        import torch

        return (torch.empty((rows, d), dtype=like_x.dtype, device=like_x.device),
                torch.empty((rows,), dtype=like_g.dtype, device=like_g.device))

    # -- the exchange -------------------------------------------------------
    def _all_to_all(self, inp, send, recv, trailing):
        import torch

        out = torch.empty((int(sum(recv)),) + trailing, dtype=inp.dtype, device=inp.device)
        self.dist.all_to_all_single(out, inp[:int(sum(send))].contiguous(),
                                    [int(v) for v in recv], [int(v) for v in send],
                                    group=self.group)
        return out

    def exchange_counts(self, counts_host: np.ndarray, device) -> np.ndarray:
        """[W, El]: what every rank routes to this rank's experts."""
        import torch

        send = torch.as_tensor(counts_host.astype(np.int64), device=device)
        recv = torch.empty_like(send)
        self.dist.all_to_all_single(recv, send, group=self.group)
        return recv.cpu().numpy().reshape(self.world, self.El)

    def forward(self, x, topk_idx=None, topk_w=None):
        import torch

        counts, x_perm, row_gate, tables = self.front(x, topk_idx, topk_w)
        counts_host = counts.cpu().numpy().astype(np.int64)  # the split sizes
        recv_counts = self.exchange_counts(counts_host, x.device)
        plan = plan_dispatch(counts_host, recv_counts, self.P)
        d = x_perm.shape[1]
        # dispatch: token rows and their routing weights
        xr = self._all_to_all(x_perm, plan.send_rows, plan.recv_rows, (d,))
        gr = self._all_to_all(row_gate, plan.send_rows, plan.recv_rows, ())
        xe, ge = self.expert_major_buffers(plan.rows, d, x_perm, row_gate)
        for src, dst, n in plan.copies:
            xe[dst:dst + n].copy_(xr[src:src + n])
            ge[dst:dst + n].copy_(gr[src:src + n])
        ye = self.local_experts(xe, ge, plan)
        # combine exchange: y rows back to their senders' layout
        yr = torch.empty((int(plan.recv_rows.sum()), d), dtype=ye.dtype, device=x.device)
        for src, dst, n in plan.copies:
            yr[src:src + n].copy_(ye[dst:dst + n])
        ys = self._all_to_all(yr, plan.recv_rows, plan.send_rows, (d,))
        return self.finish(x, ys, tables)
