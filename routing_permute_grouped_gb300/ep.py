"""Expert parallelism: the layer forward over a torch.distributed group.

Rank r of W holds the routed experts [r * El, (r + 1) * El) (El = E / W) and
a copy of the router and of the shared expert.  One layer forward:

  1. each rank routes its own tokens and permutes them into the padded
     expert-major layout over all E experts (the single-GPU stages);
  2. the per-expert counts are exchanged, then each rank sends rank r' the
     padded segment of each of r''s experts, one piece per expert, with
     their routing weights ("Dropless and grouped GEMM", sec. 14: the
     dispatch, whose landing write does the permute and the padding);
  3. the pieces land straight in the receiver's expert-major layout: the W
     senders' pieces of each local expert, in rank order, make one padded
     segment (every piece is a multiple of P rows, so the concatenation is
     again a padded segment), and the grouped GEMMs run on them with a
     block table built from the counts;
  4. the rows of y go back, piece by piece, into the senders' layout (the
     combine exchange) and each rank combines its tokens with its shared
     expert's rows, as the single-GPU layer does.

Pieces between ranks travel as batched point-to-point sends and receives
(NCCL between GPUs); the pieces a rank keeps move in one gather.  The
summation order of the combine is the single-GPU one, so a token's output
does not depend on W.  The piece sizes are needed on the host: the
per-expert counts cross to the host once per layer (a few hundred bytes).  The plan functions below are plain host logic over those counts;
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
    padded_offsets  [El + 1] of the expert-major layout
    block_metadata  [num_blocks, 3] = [local expert, m_start, valid_m]
    rows            rows of the expert-major layout (= padded_offsets[-1])
    send_pieces     (peer, row, rows): this rank's padded segments in its own
                    layout, one per expert with rows, peers in order and each
                    peer's experts in order (the dispatch's sends)
    recv_pieces     (peer, row, rows): where each arriving piece lands in the
                    expert-major layout; for every peer in the order that
                    peer sends them
    """
    send_rows: np.ndarray
    recv_rows: np.ndarray
    padded_offsets: np.ndarray
    block_metadata: np.ndarray
    rows: int
    send_pieces: list
    recv_pieces: list


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
    seg_rows = pieces.sum(axis=0)                        # per local expert
    po = np.concatenate([[0], np.cumsum(seg_rows)]).astype(np.int32)
    # arriving pieces: expert-major, senders in rank order within an expert
    n = pieces.T                                         # [El, W]
    dst = po[:-1, None].astype(np.int64) + np.cumsum(n, axis=1) - n
    ee, ss = np.nonzero(n)                               # row-major: e outer, s inner
    recv_pieces = list(zip(ss.tolist(), dst[ee, ss].tolist(), n[ee, ss].tolist()))
    # the block table: a piece of c rows holds ceil(c / P) blocks of P rows
    c = recv_counts.T[ee, ss]
    nblk = -(-c // P)
    first = np.repeat(np.cumsum(nblk) - nblk, nblk)
    m = (np.arange(int(nblk.sum())) - first) * P
    block_metadata = np.stack([np.repeat(ee, nblk), np.repeat(dst[ee, ss], nblk) + m,
                               np.minimum(P, np.repeat(c, nblk) - m)], axis=1).astype(np.int32)
    own = padded(counts, P)
    own_po = np.concatenate([[0], np.cumsum(own)])
    g = np.flatnonzero(own)
    send_pieces = list(zip((g // El).tolist(), own_po[g].tolist(), own[g].tolist()))
    return DispatchPlan(send_rows, recv_rows, po, block_metadata, int(po[-1]), send_pieces,
                        recv_pieces)


class EpLayerBase:
    """The exchange of an expert-parallel layer forward over a process group;
    subclasses supply the compute steps (``front``, ``local_experts``,
    ``finish``) and the tensors' device.  Row pieces move with
    torch.distributed's batched point-to-point operations (NCCL between
    GPUs), the per-expert counts with one all_to_all_single."""

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

    def gather_rows(self, src, idx: np.ndarray, dst, sgate=None, dgate=None):
        """dst[i] = src[idx[i]] (and the gates) for the i < len(idx) with
        idx[i] >= 0; the other rows are left as they are."""
        import torch

        keep = np.flatnonzero(idx >= 0)
        di = torch.as_tensor(keep, device=src.device)
        si = torch.as_tensor(idx[keep].astype(np.int64), device=src.device)
        dst.index_copy_(0, di, src.index_select(0, si))
        if sgate is not None:
            dgate.index_copy_(0, di, sgate.index_select(0, si))

    # -- the exchange -------------------------------------------------------
    def _exchange(self, src, dst, sends, recvs, sgate=None, dgate=None):
        """Moves row pieces of src to the peers (sends: (peer, row, rows)) and
        lands the peers' pieces in dst (recvs: (peer, row, rows)), the gates
        alongside.  Per pair of ranks the pieces pair up in list order.  The
        pieces between this rank and itself are one gather; the others go
        through batched point-to-point operations."""
        own_s = [(r, n) for p, r, n in sends if p == self.rank]
        own_r = [(r, n) for p, r, n in recvs if p == self.rank]
        if own_s:
            rs, ns = np.array(own_s, np.int64).T
            rd, nd = np.array(own_r, np.int64).T
            if not np.array_equal(ns, nd):
                raise RuntimeError("mismatched local pieces")
            idx = np.full(int((rd + nd).max()), -1, np.int32)
            step = np.arange(int(ns.sum())) - np.repeat(np.cumsum(ns) - ns, ns)
            idx[np.repeat(rd, ns) + step] = np.repeat(rs, ns) + step
            self.gather_rows(src, idx, dst, sgate, dgate)
        ops = []
        P2POp, dist = self.dist.P2POp, self.dist
        for p, r, n in sends:
            if p != self.rank:
                ops.append(P2POp(dist.isend, src[r:r + n], p, self.group))
                if sgate is not None:
                    ops.append(P2POp(dist.isend, sgate[r:r + n], p, self.group))
        for p, r, n in recvs:
            if p != self.rank:
                ops.append(P2POp(dist.irecv, dst[r:r + n], p, self.group))
                if dgate is not None:
                    ops.append(P2POp(dist.irecv, dgate[r:r + n], p, self.group))
        if ops:
            for req in dist.batch_isend_irecv(ops):
                req.wait()

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
        # dispatch: token rows and their routing weights, piece by piece,
        # straight into the expert-major layout
        xe, ge = self.expert_major_buffers(plan.rows, d, x_perm, row_gate)
        self._exchange(x_perm, xe, plan.send_pieces, plan.recv_pieces, row_gate, ge)
        ye = self.local_experts(xe, ge, plan)
        # combine exchange: the y pieces back into their senders' layout
        ys = self.combine_buffer(tables)
        if ys is None:
            ys = torch.empty((int(plan.send_rows.sum()), d), dtype=ye.dtype, device=x.device)
        self._exchange(ye, ys, plan.recv_pieces, plan.send_pieces)
        return self.finish(x, ys, tables)

    def combine_buffer(self, tables):
        """Where the returning y rows land (None: a new tensor)."""
        return None


class GpuEp(EpLayerBase):
    """The expert-parallel layer forward on the CUDA library: this rank's
    slice of the routed experts (W1/W3 [El, d, d_e], W2 [El, d_e, d], bf16,
    CUDA), the router and the shared expert replicated (the pages'
    orientations, as MoeLayer).  ``cfg`` is the global config (E = all
    experts, T = this rank's tokens per call).  Buffers are sized once: the
    expert-major layout holds at most W * T * k rows plus W * El * P of
    padding."""

    def __init__(self, cfg, W1_local, W3_local, W2_local, Wg=None, bias=None, Ws1=None, Ws3=None,
                 Ws2=None, group=None, stream=None):
        import math

        import torch

        from . import (config_of, moe_check_config, moe_pack_experts, moe_pack_router,
                       moe_route_splitk_scratch_size, moe_workspace_layout)

        moe_check_config(cfg)
        super().__init__(cfg.E, cfg.k, cfg.pad_multiple, group)
        El, dev = self.El, W1_local.device
        if W1_local.shape[0] != El:
            raise ValueError(f"this rank holds {El} experts, got {W1_local.shape[0]}")
        self.cfg, self.dev = cfg, dev
        d, de, ds = cfg.d, cfg.d_e, cfg.d_shared
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.W13 = torch.empty((El, 2 * de, d), **bf)
        self.W2_t = torch.empty((El, d, de), **bf)
        moe_pack_experts(W1_local, W3_local, W2_local, self.W13, self.W2_t, stream)
        self.Wg_t = None
        if Wg is not None:
            self.Wg_t = torch.empty((cfg.E, d), **bf)
            moe_pack_router(Wg, self.Wg_t, stream)
        self.bias = None if bias is None else bias.to(device=dev, dtype=torch.float32).contiguous()
        self.Ws13 = self.Ws2_t = None
        if ds:
            self.Ws13 = torch.empty((1, 2 * ds, d), **bf)
            self.Ws2_t = torch.empty((1, d, ds), **bf)
            moe_pack_experts(Ws1.unsqueeze(0).contiguous(), Ws3.unsqueeze(0).contiguous(),
                             Ws2.unsqueeze(0).contiguous(), self.Ws13, self.Ws2_t, stream)
        # this rank's forward workspace over the global experts (routing,
        # offsets, its padded layout, y, the shared expert's rows)
        self.L = moe_workspace_layout(cfg)
        self.ws = torch.empty(self.L["total"], dtype=torch.uint8, device=dev)
        self.ws[:256].zero_()
        n_split = moe_route_splitk_scratch_size(cfg) // 4
        self.partial = self._buf("router_partial", torch.float32, (n_split,)) if n_split else None
        # the expert-major layout of the received rows: capacity R_cap rows
        self.R_cap = self.world * cfg.T * cfg.k + self.world * El * cfg.pad_multiple
        self.cfg_local = config_of(T=math.ceil(self.R_cap / cfg.k), d=d, d_e=de, E=El, k=cfg.k,
                                   pad_multiple=cfg.pad_multiple)
        R_loc = self.cfg_local.T * cfg.k + El * (cfg.pad_multiple - 1)  # the GEMMs' row capacity
        NB_loc = self.cfg_local.T * cfg.k // cfg.pad_multiple + El
        self.xe = torch.zeros((R_loc, d), **bf)
        self.ge = torch.zeros((R_loc,), dtype=torch.float32, device=dev)
        self.he = torch.empty((R_loc, de), **bf)
        self.ye = torch.empty((R_loc, d), **bf)
        self.meta = torch.zeros((NB_loc, 3), dtype=torch.int32, device=dev)
        self.nb = torch.zeros((1,), dtype=torch.int32, device=dev)
        self.po = torch.zeros((El + 1,), dtype=torch.int32, device=dev)
        self.status = torch.zeros((1,), dtype=torch.int32, device=dev)
        self._staging = {}
        # the shared expert needs only x: it runs on a side stream while the
        # routing, the exchange (and its host syncs) and the routed experts run
        self.s_shared = torch.cuda.Stream(device=dev)
        self.ev_shared = torch.cuda.Event()

    def _buf(self, name, dtype, shape):
        import torch

        n = 1
        for v in shape:
            n *= v
        off = self.L[name]
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return self.ws[off:off + nbytes].view(dtype).view(*shape)

    def front(self, x, topk_idx=None, topk_w=None):
        import torch

        from . import moe_build_offsets, moe_permute, moe_route, moe_route_splitk

        from . import moe_shared_expert

        c = self.cfg
        T, k, E, d = c.T, c.k, c.E, c.d
        A, R = T * k, T * k + E * (c.pad_multiple - 1)
        NB = A // c.pad_multiple + E
        i32, f32 = torch.int32, torch.float32
        if c.d_shared:
            self.s_shared.wait_stream(torch.cuda.current_stream(self.dev))
            hs = self._buf("hs", torch.bfloat16, (T, c.d_shared))
            ys = self._buf("ys", torch.bfloat16, (T, d))
            moe_shared_expert(c, x, self.Ws13, self.Ws2_t, hs, ys, self.status, stream=self.s_shared)
            self.ev_shared.record(self.s_shared)
        if topk_idx is None:
            topk_idx = self._buf("topk_idx", i32, (T, k))
            topk_w = self._buf("topk_w", f32, (T, k))
            if self.partial is not None:
                moe_route_splitk(c, x, self.Wg_t, self.bias, topk_idx, topk_w, self.partial)
            else:
                moe_route(c, x, self.Wg_t, self.bias, topk_idx, topk_w)
        t = dict(counts=self._buf("counts", i32, (E,)), po=self._buf("padded_offsets", i32, (E + 1,)),
                 meta=self._buf("block_metadata", i32, (NB, 3)), nb=self._buf("num_blocks", i32, (1,)),
                 perm_row=self._buf("perm_row", i32, (A,)), row_src=self._buf("row_src", i32, (R,)),
                 row_gate=self._buf("row_gate", f32, (R,)))
        moe_build_offsets(c, topk_idx, topk_w, t["counts"], t["po"], t["meta"], t["nb"],
                          t["perm_row"], t["row_src"], t["row_gate"],
                          self.ws[self.L["status"]:self.L["topk_idx"]])
        x_perm = self._buf("x_perm", torch.bfloat16, (R, d))
        moe_permute(c, x, t["perm_row"], x_perm)
        return t["counts"], x_perm, t["row_gate"], t

    def expert_major_buffers(self, rows, d, like_x, like_g):
        if rows > self.xe.shape[0]:
            raise RuntimeError(f"{rows} received rows exceed the capacity {self.xe.shape[0]}")
        return self.xe, self.ge

    def _stage(self, slot: str, a: np.ndarray, out=None):
        """The int32 host array ``a`` on the device (in ``out``, or in the
        slot's own device buffer), through the slot's pinned staging buffer;
        the buffer is reused once its previous copy has finished."""
        import torch

        st = self._staging.get(slot)
        if st is None or st[0].numel() < a.size:
            n = max(2 * a.size, 1024)
            st = (torch.empty(n, dtype=torch.int32).pin_memory(),
                  torch.empty(n, dtype=torch.int32, device=self.dev), torch.cuda.Event())
            self._staging[slot] = st
        else:
            st[2].synchronize()
        host, dev, ev = st
        host[:a.size].numpy()[:] = a.reshape(-1)
        dst = dev[:a.size] if out is None else out.view(-1)[:a.size]
        dst.copy_(host[:a.size], non_blocking=True)
        ev.record()
        return dst

    def gather_rows(self, src, idx, dst, sgate=None, dgate=None):
        from . import moe_gather_rows

        if idx.size == 0:
            return
        slot = "idx_x" if sgate is not None else "idx_y"
        moe_gather_rows(src, self._stage(slot, idx), dst, sgate, dgate)

    def local_experts(self, xe, ge, plan):
        import torch

        from . import moe_grouped_gemm_swiglu, moe_grouped_gemm_swiglu_skinny

        nb = plan.block_metadata.shape[0]
        if nb == 0:
            return self.ye[:0]
        if nb > self.meta.shape[0]:
            raise RuntimeError("block table exceeds its capacity")
        self._stage("meta", plan.block_metadata, self.meta)
        self.nb.fill_(nb)
        self._stage("po", plan.padded_offsets.astype(np.int32), self.po)
        c = self.cfg_local
        valid = int(plan.block_metadata[:, 2].sum())
        if valid <= 32 * self.El:  # few rows per expert: the small-M kernel, as the layer
            moe_grouped_gemm_swiglu_skinny(c, xe, self.W13, self.W2_t, self.meta, self.nb, ge,
                                           self.he, self.ye, self.status)
        else:
            moe_grouped_gemm_swiglu(c, xe, self.W13, self.W2_t, self.meta, self.nb, self.po, ge,
                                    self.he, self.ye, self.status)
        return self.ye[:plan.rows]

    def combine_buffer(self, t):
        import torch

        return self._buf("y", torch.bfloat16, (t["row_src"].shape[0], self.cfg.d))

    def finish(self, x, y, t):
        import torch

        from . import moe_combine

        c = self.cfg
        yy = self.combine_buffer(t)
        if y.shape[0] and y.data_ptr() != yy.data_ptr():
            yy[:y.shape[0]].copy_(y)
        ys = None
        if c.d_shared:  # computed on the side stream since front()
            torch.cuda.current_stream(self.dev).wait_event(self.ev_shared)
            ys = self._buf("ys", torch.bfloat16, (c.T, c.d))
        out = torch.empty_like(x)
        moe_combine(c, yy, t["perm_row"], ys, out)
        return out

    def device_status(self) -> int:
        from . import moe_get_device_status

        return moe_get_device_status(self.status) | moe_get_device_status(self.ws)
