"""Expert parallelism: the layer forward over a torch.distributed group.

Rank r of W holds the routed experts [r * El, (r + 1) * El) (El = E / W) and
a copy of the router and of the shared expert.  One layer forward:

  1. each rank routes its own tokens and permutes them into the padded
     expert-major layout over all E experts (the single-GPU stages);
  2. the per-expert counts are exchanged with one all-to-all on the device,
     and the receiver builds its expert-major layout from them on the device
     (moe_build_blocks_from_counts: the padded offsets, the block table and
     where each sender's rows land);
  3. each rank sends rank r' its rows of each of r''s experts, one piece per
     expert, with their routing weights ("Dropless and grouped GEMM", sec.
     14: the dispatch, whose landing write does the permute and the padding);
     the pieces land back to back, in sender order, in the receiver's segment
     of that expert, so every segment holds its valid rows first, as in the
     single-GPU layout, and the grouped GEMMs run on it as they are;
  4. the rows of y go back, piece by piece, into the senders' layout (the
     combine exchange) and each rank combines its tokens with its shared
     expert's rows, as the single-GPU layer does.

Pieces between ranks travel as batched point-to-point sends and receives
(NCCL between GPUs); the pieces a rank keeps move with one device copy
(moe_copy_pieces) whose descriptors are the device tables.  NCCL takes its
sizes and offsets from the host, so the counts and the landing rows cross to
the host once per layer (one copy of a few hundred bytes); the host only
reads positions out of them (``plan_pieces``), it computes no layout.  The
summation order of the combine is the single-GPU one, so a token's output
does not depend on W.  The compute steps go through a backend object (the
CUDA library in ``GpuEp``), so the exchange logic can be exercised on CPU
process groups.
"""
from __future__ import annotations

import numpy as np


def plan_pieces(rank: int, El: int, counts, own_po, recv, piece_row):
    """The pieces of both exchanges, read from the tables the devices made
    (host copies).

    counts     [E]      this rank's rows per global expert
    own_po     [E + 1]  this rank's padded offsets (its own layout)
    recv       [W, El]  rows every rank sends to this rank's experts
    piece_row  [W, El]  where those rows land in this rank's expert-major
                        layout

    send_pieces (peer, row, rows): this rank's rows of expert g (from its own
        segment start) go to rank g // El; peers in order, each peer's experts
        in order.
    recv_pieces (peer, row, rows): for every local expert (outer) and sender
        (inner), where that sender's rows land.  Between two ranks the pieces
        pair up in list order: both lists follow the receiver's experts."""
    counts = np.asarray(counts, np.int64).reshape(-1)
    own_po = np.asarray(own_po, np.int64).reshape(-1)
    recv = np.asarray(recv, np.int64)
    piece_row = np.asarray(piece_row, np.int64)
    g = np.flatnonzero(counts > 0)
    send_pieces = list(zip((g // El).tolist(), own_po[g].tolist(), counts[g].tolist()))
    ee, ss = np.nonzero(recv.T > 0)  # expert outer, sender inner
    recv_pieces = list(zip(ss.tolist(), piece_row[ss, ee].tolist(), recv[ss, ee].tolist()))
    return send_pieces, recv_pieces


class EpLayerBase:
    """The exchange of an expert-parallel layer forward over a process group;
    subclasses supply the compute steps (``front``, ``layout``,
    ``local_experts``, ``finish``) and the tensors' device.  Row pieces move
    with torch.distributed's batched point-to-point operations (NCCL between
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
        expert-major layout over all E experts.  Returns (counts [E] int32,
        padded offsets [E + 1] int32, x_perm [R, d], row_gate [R], tables for
        finish)."""
        raise NotImplementedError

    def layout(self, recv):
        """The expert-major layout of the arriving rows from recv [W * El]
        (int32, rows of sender s for local expert e at s * El + e): a dict
        with at least ``piece_row`` [W, El]."""
        raise NotImplementedError

    def local_experts(self, xe, ge, lay, valid_rows: int):
        """y rows of the local experts for the expert-major rows xe with routing
        weights ge (the GEMM2 epilogue multiplies by them)."""
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

    def host_tables(self, counts, own_po, recv, piece_row):
        """Host copies of the four tables (numpy)."""
        return tuple(np.asarray(t.cpu() if hasattr(t, "cpu") else t)
                     for t in (counts, own_po, recv, piece_row))

    def move_local(self, src, dst, pieces, sgate=None, dgate=None, combine=False, lay=None):
        """The pieces this rank keeps: pieces = [(src row, dst row, rows)]."""
        import torch

        if not pieces:
            return
        rs, rd, n = (np.array(v, np.int64) for v in zip(*pieces))
        step = np.arange(int(n.sum())) - np.repeat(np.cumsum(n) - n, n)
        si = torch.as_tensor(np.repeat(rs, n) + step, device=src.device)
        di = torch.as_tensor(np.repeat(rd, n) + step, device=src.device)
        dst.index_copy_(0, di, src.index_select(0, si))
        if sgate is not None:
            dgate.index_copy_(0, di, sgate.index_select(0, si))

    # -- the exchange -------------------------------------------------------
    def _exchange(self, src, dst, sends, recvs, sgate=None, dgate=None, combine=False, lay=None):
        """Moves row pieces of src to the peers (sends: (peer, row, rows)) and
        lands the peers' pieces in dst (recvs: (peer, row, rows)), the gates
        alongside.  Per pair of ranks the pieces pair up in list order.  The
        pieces between this rank and itself are one local move; the others
        go through batched point-to-point operations."""
        own_s = [(r, n) for p, r, n in sends if p == self.rank]
        own_r = [(r, n) for p, r, n in recvs if p == self.rank]
        if [n for _, n in own_s] != [n for _, n in own_r]:
            raise RuntimeError("mismatched local pieces")
        self.move_local(src, dst, [(a, b, n) for (a, n), (b, _) in zip(own_s, own_r)], sgate,
                        dgate, combine, lay)
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

    def exchange_counts(self, counts):
        """[W * El] on counts' device: what every rank routes to this rank's
        experts (sender s's counts at s * El + e)."""
        import torch

        recv = torch.empty_like(counts)
        self.dist.all_to_all_single(recv, counts.contiguous(), group=self.group)
        return recv

    def forward(self, x, topk_idx=None, topk_w=None):
        import torch

        counts, own_po, x_perm, row_gate, tables = self.front(x, topk_idx, topk_w)
        recv = self.exchange_counts(counts)
        lay = self.layout(recv)
        h_counts, h_po, h_recv, h_piece = self.host_tables(counts, own_po, recv,
                                                           lay["piece_row"])
        h_recv = h_recv.reshape(self.world, self.El)
        sends, recvs = plan_pieces(self.rank, self.El, h_counts, h_po, h_recv,
                                   h_piece.reshape(self.world, self.El))
        d = x_perm.shape[1]
        rows = int(h_recv.sum())
        # dispatch: token rows and their routing weights, piece by piece,
        # straight into the expert-major layout
        xe, ge = self.expert_major_buffers(max(rows, 1), d, x_perm, row_gate)
        self._exchange(x_perm, xe, sends, recvs, row_gate, ge, lay=lay)
        ye = self.local_experts(xe, ge, lay, rows)
        # combine exchange: the y pieces back into their senders' layout
        ys = self.combine_buffer(tables)
        if ys is None:
            ys = torch.empty((int(h_po[-1]), d), dtype=ye.dtype, device=x.device)
        self._exchange(ye, ys, recvs, sends, combine=True, lay=lay)
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
    expert-major layout holds at most W * T * k rows plus El * P of padding.
    At world size 1 the expert-major layout is the rank's own layout (one
    sender, its rows already back to back per expert), so the layer's own
    buffers serve both sides and no row moves."""

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
        i32 = dict(dtype=torch.int32, device=dev)
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
        self.R_cap = self.world * cfg.T * cfg.k + El * cfg.pad_multiple
        self.cfg_local = config_of(T=math.ceil(self.R_cap / cfg.k), d=d, d_e=de, E=El, k=cfg.k,
                                   pad_multiple=cfg.pad_multiple)
        R_loc = self.cfg_local.T * cfg.k + El * (cfg.pad_multiple - 1)  # the GEMMs' row capacity
        NB_loc = self.cfg_local.T * cfg.k // cfg.pad_multiple + El
        if self.world > 1:
            self.xe = torch.zeros((R_loc, d), **bf)
            self.ge = torch.zeros((R_loc,), dtype=torch.float32, device=dev)
            self.he = torch.empty((R_loc, de), **bf)
            self.ye = torch.empty((R_loc, d), **bf)
        # the receiver's tables, built on the device from the exchanged counts
        self.meta = torch.zeros((NB_loc, 3), **i32)
        self.nb = torch.zeros((1,), **i32)
        self.po = torch.zeros((El + 1,), **i32)
        self.piece_row = torch.zeros((self.world, El), **i32)
        self.status = torch.zeros((1,), **i32)
        self._recv = None
        # the shared expert needs only x: it runs on a side stream while the
        # routing, the exchange (and its host sync) and the routed experts run
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

        from . import moe_build_offsets, moe_permute, moe_route_splitk, moe_shared_expert

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
            # the layer's own router form (fused, clustered split-K, or split-K
            # with partial logits in the scratch), so that the routing weights
            # carry the same bits as MoeLayer's
            moe_route_splitk(c, x, self.Wg_t, self.bias, topk_idx, topk_w, self.partial)
        t = dict(counts=self._buf("counts", i32, (E,)), po=self._buf("padded_offsets", i32, (E + 1,)),
                 meta=self._buf("block_metadata", i32, (NB, 3)), nb=self._buf("num_blocks", i32, (1,)),
                 perm_row=self._buf("perm_row", i32, (A,)), row_src=self._buf("row_src", i32, (R,)),
                 row_gate=self._buf("row_gate", f32, (R,)))
        moe_build_offsets(c, topk_idx, topk_w, t["counts"], t["po"], t["meta"], t["nb"],
                          t["perm_row"], t["row_src"], t["row_gate"],
                          self.ws[self.L["status"]:self.L["topk_idx"]])
        x_perm = self._buf("x_perm", torch.bfloat16, (R, d))
        moe_permute(c, x, t["perm_row"], x_perm)
        return t["counts"], t["po"], x_perm, t["row_gate"], t

    def layout(self, recv):
        from . import moe_build_blocks_from_counts

        self._recv = recv.view(self.world, self.El)
        moe_build_blocks_from_counts(self._recv, self.P, self.po, self.meta, self.nb,
                                     self.piece_row, self.status)
        return dict(po=self.po, meta=self.meta, nb=self.nb, piece_row=self.piece_row)

    def host_tables(self, counts, own_po, recv, piece_row):
        """One device-to-host copy of the four tables (the host sync of the
        layer: NCCL takes its sizes and offsets from the host)."""
        import torch

        parts = (counts, own_po, recv, piece_row)
        packed = torch.cat([t.reshape(-1) for t in parts]).cpu().numpy()
        out, o = [], 0
        for t in parts:
            out.append(packed[o:o + t.numel()])
            o += t.numel()
        return tuple(out)

    def expert_major_buffers(self, rows, d, like_x, like_g):
        if self.world == 1:
            return like_x, like_g  # the rank's own layout is the expert-major one
        if rows > self.xe.shape[0]:
            raise RuntimeError(f"{rows} received rows exceed the capacity {self.xe.shape[0]}")
        return self.xe, self.ge

    def move_local(self, src, dst, pieces, sgate=None, dgate=None, combine=False, lay=None):
        """The pieces this rank keeps, with device descriptors: its own
        segment starts (padded offsets of its experts), the landing rows, the
        counts from the exchange."""
        import torch

        from . import moe_copy_pieces

        if not pieces:
            return
        if src.data_ptr() == dst.data_ptr():
            if any(a != b for a, b, _ in pieces):
                raise RuntimeError("aliased exchange buffers with moving pieces")
            return
        r, El = self.rank, self.El
        own = self._buf("padded_offsets", torch.int32, (self.E + 1,))[r * El:(r + 1) * El]
        land = self.piece_row[r]
        rows = self._recv[r]
        src_row, dst_row = (land, own) if combine else (own, land)
        moe_copy_pieces(src, dst, src_row, dst_row, rows, max(n for _, _, n in pieces), sgate, dgate)

    def local_experts(self, xe, ge, lay, valid_rows):
        import torch

        from . import moe_grouped_gemm_swiglu, moe_grouped_gemm_swiglu_skinny

        if self.world == 1:
            # the layer's own config and buffers: x_perm, h, y of the workspace
            c = self.cfg
            R = c.T * c.k + c.E * (c.pad_multiple - 1)
            he = self._buf("h", torch.bfloat16, (R, c.d_e))
            ye = self._buf("y", torch.bfloat16, (R, c.d))
        else:
            c, he, ye = self.cfg_local, self.he, self.ye
        if valid_rows == 0:
            return ye
        if valid_rows <= 32 * self.El:  # few rows per expert: the small-M kernel, as the layer
            moe_grouped_gemm_swiglu_skinny(c, xe, self.W13, self.W2_t, lay["meta"], lay["nb"], ge,
                                           he, ye, self.status)
        else:
            moe_grouped_gemm_swiglu(c, xe, self.W13, self.W2_t, lay["meta"], lay["nb"], lay["po"],
                                    ge, he, ye, self.status)
        return ye

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
