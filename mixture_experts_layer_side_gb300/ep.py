"""Expert parallelism over G ranks: host orchestration of the exchange (no
arithmetic here; every step on the data runs in libmok.so).

The experts are split over the ranks in contiguous blocks; each rank holds its
own tokens.  One pass moves routed rows once each way, all four directions
driven by the one schedule ("Cursor Open-Sources Mixture-of-Kittens (MoK)",
"Three design decisions that matter", communication-direction paragraph; the
"Results" section runs the layer at EP 64):

  forward   source ranks pack their routed rows in expert-sorted order
            (destination-major), the per-expert counts are exchanged and
            planned (``mok_ep_plan``), the rows move to their experts' ranks,
            each rank runs the ordinary layer calls on what it received with
            k = 1 and score 1 (one output row per received row), the rows come
            back, and the source combines them with its scores in fixed k
            order;
  backward  the sources pack dout rows and their scores along the same plan,
            each rank runs the ordinary backward on its received rows (its
            experts' weight gradients, dX rows, per-row score gradients), the
            dX rows and score gradients come back, and the source sums the dX
            rows in fixed k order and puts the score gradients back in
            [T, k] order.

Rows reach each expert ordered by (source rank, source flat index), i.e. in
ascending global flat index when token t of rank g is global token g*T + t:
every output and gradient is bitwise that of one GPU holding all tokens and
experts.

The exchange is a collective the caller's process group provides
(``DistExchange``: ``torch.distributed.all_to_all_single`` with uneven
splits; NCCL between GPUs).  It needs each pass's row counts on the host: the
per-expert histogram ([E] int32) is read back once per pass.  The pages'
design instead pulls rows over NVLink with device-side signals and no host
step; that data plane needs several GPUs and is not built here.
"""

from __future__ import annotations

import numpy as np
import torch

from . import _lib
from .inputs import Shape
from .layer import PRECISIONS


class ExpertPartition:
    """E experts over G ranks in contiguous blocks whose sizes differ by at most
    one (``mok_ep_first_expert``)."""

    def __init__(self, E, G):
        if not 1 <= G <= E:
            raise ValueError(f"need 1 <= G <= E (G={G}, E={E})")
        self.E, self.G = E, G
        self.bounds = [_lib.mok_ep_first_expert(E, G, g) for g in range(G + 1)]

    def first(self, g):
        return self.bounds[g]

    def count(self, g):
        return self.bounds[g + 1] - self.bounds[g]

    def owner(self, e):
        return int(np.searchsorted(self.bounds, e, side="right") - 1)


class EPPlan:
    """One pass's exchange plan for one rank (host lists and arrays)."""

    def __init__(self, send_rows, recv_rows, recv_expert, n_recv):
        self.send_rows = send_rows        # rows to each rank, from the front of the packed rows
        self.recv_rows = recv_rows        # rows arriving from each rank, in rank order
        self.recv_expert = recv_expert    # local expert of each received row (int32 [n_recv])
        self.n_recv = n_recv
        self.n_send = int(sum(send_rows))


def make_plan(part: ExpertPartition, rank, local_counts, recv_counts, recv_capacity=None) -> EPPlan:
    """``local_counts`` int32 [E] (this rank's schedule histogram),
    ``recv_counts`` int32 [G, E_rank] (each source's counts over this rank's
    experts), both on the host."""
    send, recv, experts, n = _lib.mok_ep_plan(part.E, part.G, rank, local_counts, recv_counts, recv_capacity)
    return EPPlan(send, recv, experts, n)


class DistExchange:
    """The exchange over a ``torch.distributed`` process group: one
    all-to-all with uneven splits per direction (NCCL for device tensors,
    gloo for host tensors)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group

    def counts(self, part: ExpertPartition, rank, local_counts):
        """Send each rank the counts of its experts; returns the [G, E_rank]
        int32 host array of what every source routes to this rank's experts."""
        G, El = part.G, part.count(rank)
        send = local_counts.contiguous()
        out = torch.empty(G * El, dtype=torch.int32, device=send.device)
        self.dist.all_to_all_single(out, send, [El] * G, [part.count(g) for g in range(G)], group=self.group)
        return out.cpu().numpy().reshape(G, El)

    def rows(self, send, send_rows, recv_rows, out):
        """Rows [sum(send_rows), ...] of ``send`` out, rows [sum(recv_rows),
        ...] into the front of ``out``; returns that front."""
        n_send, n_recv = int(sum(send_rows)), int(sum(recv_rows))
        self.dist.all_to_all_single(out[:n_recv], send[:n_send], list(recv_rows), list(send_rows),
                                    group=self.group)
        return out[:n_recv]


class EPMoELayer:
    """One rank's share of an expert-parallel MoE layer on its GPU.

    ``shape`` is this rank's token count T with the GLOBAL expert count E
    (routing ids are global); the rank owns experts
    ``[part.first(rank), part.first(rank + 1))`` and is given only their
    weights ([E_rank, H, I] / [E_rank, I, H]; MXFP8: descriptors from
    ``layer.quantize_weights``).  ``exchange`` moves counts and rows between
    ranks (``DistExchange``).  ``capacity_rows`` bounds the rows one rank can
    receive per pass (default: every routed row of every rank, G*T*k, so no
    row is ever dropped); a pass that would receive more raises
    ``MokError(MOK_ERR_UNSUPPORTED)`` before any row moves.
    """

    def __init__(self, shape: Shape, G, rank, exchange, precision="bf16", capacity_rows=None, minibatch_rows=0,
                 ring_slots=0, device="cuda"):
        self.shape, self.G, self.rank, self.exchange = shape, G, rank, exchange
        self.part = ExpertPartition(shape.E, G)
        self.El = self.part.count(rank)
        self.prec = PRECISIONS[precision]
        self.device = torch.device(device)
        T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
        R = T * k
        self.cap = int(capacity_rows) if capacity_rows else G * R
        self.cfg = _lib.config(minibatch_rows=minibatch_rows, ring_slots=ring_slots)
        self.cshape = _lib.shape_of(T, H, I, E, k)
        d = self.device
        # source side: the schedule of this rank's tokens over all experts
        self.src_ws = torch.empty(_lib.mok_schedule_workspace_size(self.cshape, self.cfg), dtype=torch.uint8,
                                  device=d)
        self.send_rows_buf = torch.empty((R, H), dtype=torch.bfloat16, device=d)
        self.send_s = torch.empty(R, dtype=torch.float32, device=d)
        self.ret_rows = torch.empty((R, H), dtype=torch.bfloat16, device=d)
        self.ret_s = torch.empty(R, dtype=torch.float32, device=d)
        # receiving side: the layer over received rows (k = 1, this rank's experts)
        cap_shape = _lib.shape_of(self.cap, H, I, self.El, 1)
        self.rws = torch.empty(_lib.mok_workspace_size(cap_shape, self.cfg, self.prec), dtype=torch.uint8, device=d)
        self.rws[:256].zero_()  # error word of a pass that received nothing
        self.rctx = torch.empty(_lib.mok_ctx_size(cap_shape, self.cfg, self.prec), dtype=torch.uint8, device=d)
        self.x_recv = torch.empty((self.cap, H), dtype=torch.bfloat16, device=d)
        self.rows_a = torch.empty((self.cap, H), dtype=torch.bfloat16, device=d)
        self.rows_b = torch.empty((self.cap, H), dtype=torch.bfloat16, device=d)
        self.s_recv = torch.empty(self.cap, dtype=torch.float32, device=d)
        self.ds_recv = torch.empty(self.cap, dtype=torch.float32, device=d)
        self.ones = torch.ones(self.cap, dtype=torch.float32, device=d)
        self.idx_recv = torch.empty(self.cap, dtype=torch.int32, device=d)
        self.plan = None

    def _counts_view(self):
        L = _lib.mok_workspace_layout(self.cshape, self.cfg, _lib.MOK_BF16)
        return self.src_ws[L["counts"]:L["counts"] + 4 * self.shape.E].view(torch.int32)

    def _rshape(self):
        return _lib.shape_of(self.plan.n_recv, self.shape.H, self.shape.I, self.El, 1)

    # -- forward ---------------------------------------------------------------
    def forward(self, x, idx, s, W1, W3, W2, out=None):
        """``x`` [T, H] bf16, ``idx`` [T, k] int32 global expert ids, ``s``
        [T, k] f32; W* this rank's experts (forward orientation in MXFP8).
        Returns out [T, H] bf16."""
        sh, cfg = self.shape, self.cfg
        if out is None:
            out = torch.empty((sh.T, sh.H), dtype=torch.bfloat16, device=self.device)
        _lib.mok_build_schedule(self.cshape, cfg, self.src_ws, idx)
        _lib.mok_ep_pack_rows(self.cshape, cfg, self.src_ws, x, None, self.send_rows_buf)
        counts = self._counts_view()
        recv_counts = self.exchange.counts(self.part, self.rank, counts)
        self.plan = plan = make_plan(self.part, self.rank, counts.cpu().numpy(), recv_counts, self.cap)
        if plan.n_recv:
            self.idx_recv[:plan.n_recv].copy_(torch.from_numpy(plan.recv_expert), non_blocking=False)
        self.exchange.rows(self.send_rows_buf, plan.send_rows, plan.recv_rows, self.x_recv)
        if plan.n_recv:
            rs, n = self._rshape(), plan.n_recv
            _lib.mok_build_schedule(rs, cfg, self.rws, self.idx_recv[:n])
            _lib.mok_forward(rs, cfg, self.prec, self.rws, self.x_recv[:n], self.ones[:n], W1, W3, W2,
                             self.rows_a[:n], self.rctx)
        self.exchange.rows(self.rows_a, plan.recv_rows, plan.send_rows, self.ret_rows)
        _lib.mok_ep_combine_rows(self.cshape, cfg, self.src_ws, self.ret_rows, s, out)
        return out

    # -- backward --------------------------------------------------------------
    def backward(self, s, W1, W3, W2, dout, grads=None):
        """After ``forward`` of the same routing: ``s`` the forward's scores,
        W* this rank's experts (backward orientation in MXFP8), ``dout``
        [T, H].  Returns dict(dX [T, H], dW1, dW3 [E_rank, H, I], dW2
        [E_rank, I, H], ds [T, k])."""
        sh, cfg, plan = self.shape, self.cfg, self.plan
        if plan is None:
            raise RuntimeError("backward before forward")
        d = self.device
        if grads is None:
            grads = dict(dX=torch.empty((sh.T, sh.H), dtype=torch.bfloat16, device=d),
                         dW1=torch.empty((self.El, sh.H, sh.I), dtype=torch.bfloat16, device=d),
                         dW3=torch.empty((self.El, sh.H, sh.I), dtype=torch.bfloat16, device=d),
                         dW2=torch.empty((self.El, sh.I, sh.H), dtype=torch.bfloat16, device=d),
                         ds=torch.empty((sh.T, sh.k), dtype=torch.float32, device=d))
        _lib.mok_ep_pack_rows(self.cshape, cfg, self.src_ws, dout, s, self.send_rows_buf, self.send_s)
        self.exchange.rows(self.send_rows_buf, plan.send_rows, plan.recv_rows, self.rows_a)
        self.exchange.rows(self.send_s, plan.send_rows, plan.recv_rows, self.s_recv)
        n = plan.n_recv
        if n:
            _lib.mok_backward(self._rshape(), cfg, self.prec, self.rws, self.rctx, self.x_recv[:n],
                              self.s_recv[:n], W1, W3, W2, self.rows_a[:n], self.rows_b[:n], grads["dW1"],
                              grads["dW3"], grads["dW2"], self.ds_recv[:n])
        else:
            # no routed row reached this rank's experts: their gradients are zero
            for name in ("dW1", "dW3", "dW2"):
                grads[name].zero_()
        self.exchange.rows(self.rows_b, plan.recv_rows, plan.send_rows, self.ret_rows)
        self.exchange.rows(self.ds_recv, plan.recv_rows, plan.send_rows, self.ret_s)
        _lib.mok_ep_combine_rows(self.cshape, cfg, self.src_ws, self.ret_rows, None, grads["dX"])
        _lib.mok_ep_unsort_scores(self.cshape, cfg, self.src_ws, self.ret_s, grads["ds"])
        return grads

    def check(self):
        """Synchronise and raise if either side recorded a device error."""
        for ws in (self.src_ws, self.rws):
            st = _lib.mok_check(ws)
            if st != 0:
                raise _lib.MokError(st, "device")
