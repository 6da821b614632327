"""Host-side convenience wrapper around the C ABI (no compute here).

``MoKLayer`` owns the caller-side buffers the C ABI asks for (workspace and
forward context, allocated once and reused, as the pages' workspace is:
"Mixture-of-Kittens (MoK)", "Core concepts", Workspace row) and forwards the
calls of the pages' functional API -- build_schedule, forward, backward --
to libmok.so.
"""

from __future__ import annotations

import torch

from . import _lib
from .inputs import Shape

PRECISIONS = {"bf16": _lib.MOK_BF16, "mxfp8": _lib.MOK_MXFP8}


def quantize_weights(W1, W3, W2, stream=None):
    """Pre-quantise bf16 weights for MXFP8 mode (the pages' ops.mxfp8_quantize
    step), in both orientations: the forward contracts W1/W3 over H and W2
    over I (blocks along the rows of each matrix, block_axis 0), the
    backward contracts W1/W3 over I and W2 over H (block_axis 1).
    Returns {"fwd": (mx1, mx3, mx2), "bwd": (...), "bwd_replay": (...)} of
    descriptors; "bwd_replay" is what the bounded-memory backward (replay)
    takes: W1 and W3 as two descriptors each, the backward orientation then
    the forward one (its replayed GEMM1 contracts over H).  The code and
    scale tensors are kept alive on the returned object."""
    out = {"tensors": []}
    for orient, axis in (("fwd", 0), ("bwd", 1)):
        descs = []
        for W in (W1, W3, W2):
            E, r, c = W.shape
            q = torch.empty((E, r, c), dtype=torch.uint8, device=W.device)
            sf_shape = (E, r // 32, c) if axis == 0 else (E, r, c // 32)
            sf = torch.empty(sf_shape, dtype=torch.uint8, device=W.device)
            _lib.mok_mxfp8_quantize(W, axis, q, sf, stream)
            out["tensors"] += [q, sf]
            descs.append(_lib.mx(q, sf))
        out[orient] = tuple(descs)
    pair = _lib.MokMx * 2
    out["bwd_replay"] = (pair(out["bwd"][0], out["fwd"][0]), pair(out["bwd"][1], out["fwd"][1]), out["bwd"][2])
    return out


class MoKLayer:
    def __init__(self, shape: Shape, precision="bf16", minibatch_rows=0, ring_slots=0, debug_flags=0,
                 replay=False, overlap_sms=0, device="cuda"):
        self.shape = shape
        self.cshape = _lib.shape_of(shape.T, shape.H, shape.I, shape.E, shape.k)
        self.cfg = _lib.config(minibatch_rows=minibatch_rows, ring_slots=ring_slots, debug_flags=debug_flags,
                               replay=int(bool(replay)), overlap_sms=overlap_sms)
        self.prec = PRECISIONS[precision]
        self.device = torch.device(device)
        ws_bytes = _lib.mok_workspace_size(self.cshape, self.cfg, self.prec)
        ctx_bytes = _lib.mok_ctx_size(self.cshape, self.cfg, self.prec)
        if ws_bytes == 0 or ctx_bytes == 0:
            raise _lib.MokError(2, "unsupported shape or config")
        self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device=self.device)
        self.ctx = torch.empty(ctx_bytes, dtype=torch.uint8, device=self.device)
        self.layout = _lib.mok_workspace_layout(self.cshape, self.cfg, self.prec)

    # -- the functional API -------------------------------------------------
    def build_schedule(self, topk_idx, stream=None):
        _lib.mok_build_schedule(self.cshape, self.cfg, self.ws, topk_idx, stream)

    def forward(self, x, scores, W1, W3, W2, out=None, stream=None):
        if out is None:
            out = torch.empty((self.shape.T, self.shape.H), dtype=torch.bfloat16, device=self.device)
        _lib.mok_forward(self.cshape, self.cfg, self.prec, self.ws, x, scores, W1, W3, W2, out, self.ctx, stream)
        return out

    def forward_fused(self, topk_idx, x, scores, W1, W3, W2, out=None, stream=None):
        """Schedule and forward in one launch (MXFP8: the routing-independent
        quantisation and scale tiling ahead of it); backward may follow."""
        if out is None:
            out = torch.empty((self.shape.T, self.shape.H), dtype=torch.bfloat16, device=self.device)
        _lib.mok_forward_fused(self.cshape, self.cfg, self.prec, self.ws, topk_idx, x, scores, W1, W3, W2, out,
                               self.ctx, stream)
        return out

    def backward(self, x, scores, W1, W3, W2, dout, grads=None, stream=None):
        s = self.shape
        if grads is None:
            grads = self.alloc_grads()
        _lib.mok_backward(self.cshape, self.cfg, self.prec, self.ws, self.ctx, x, scores, W1, W3, W2, dout,
                          grads["dX"], grads["dW1"], grads["dW3"], grads["dW2"], grads["ds"], stream)
        return grads

    def alloc_grads(self):
        s, d = self.shape, self.device
        return dict(dX=torch.empty((s.T, s.H), dtype=torch.bfloat16, device=d),
                    dW1=torch.empty((s.E, s.H, s.I), dtype=torch.bfloat16, device=d),
                    dW3=torch.empty((s.E, s.H, s.I), dtype=torch.bfloat16, device=d),
                    dW2=torch.empty((s.E, s.I, s.H), dtype=torch.bfloat16, device=d),
                    ds=torch.empty((s.T, s.k), dtype=torch.float32, device=d))

    # -- MXFP8 weights ------------------------------------------------------
    def quantize_weights(self, W1, W3, W2, stream=None):
        return quantize_weights(W1, W3, W2, stream)

    def check(self, stream=None):
        """Synchronise and raise if the device recorded an error."""
        st = _lib.mok_check(self.ws, stream)
        if st != 0:
            raise _lib.MokError(st, "device")

    # -- inspection ---------------------------------------------------------
    def schedule_arrays(self):
        """Views of the schedule arrays inside the workspace (int32)."""
        s, L = self.shape, self.layout
        R, E = s.T * s.k, s.E

        def view(off, n):
            return self.ws[off:off + 4 * n].view(torch.int32)

        hdr = view(L["header"], 16)
        return dict(header=hdr, counts=view(L["counts"], E), offsets=view(L["offsets"], E + 1),
                    padded_offsets=view(L["padded_offsets"], E + 1), perm=view(L["perm"], R),
                    inv_perm=view(L["inv_perm"], R), pad_perm=view(L["pad_perm"], L["pad_capacity"]),
                    pad_inv=view(L["pad_inv"], R), tile_expert=view(L["tile_expert"], L["tile_capacity"]))


class MoKRouter:
    """Owns the router workspace; forward gives the layer its routing
    (top-k ids, softmax scores), backward turns the layer's score gradient
    into router-weight and input gradients (mok_router_forward / _backward)."""

    def __init__(self, shape: Shape, device="cuda"):
        self.shape = shape
        self.device = torch.device(device)
        self.cshape = _lib.shape_of(shape.T, shape.H, shape.I, shape.E, shape.k)
        n = _lib.mok_router_workspace_size(self.cshape)
        if n == 0:
            raise _lib.MokError(1, "mok_router_workspace_size")
        self.ws = torch.empty(n, dtype=torch.uint8, device=self.device)

    def forward(self, x, Wr, bias=None, with_logits=False, stream=None):
        s = self.shape
        idx = torch.empty((s.T, s.k), dtype=torch.int32, device=self.device)
        scores = torch.empty((s.T, s.k), dtype=torch.float32, device=self.device)
        logits = torch.empty((s.T, s.E), dtype=torch.float32, device=self.device) if with_logits else None
        _lib.mok_router_forward(self.cshape, self.ws, x, Wr, bias, idx, scores, logits, stream)
        return (idx, scores, logits) if with_logits else (idx, scores)

    def backward(self, x, Wr, idx, scores, dscores, stream=None):
        s = self.shape
        dWr = torch.empty((s.H, s.E), dtype=torch.float32, device=self.device)
        dx = torch.empty((s.T, s.H), dtype=torch.bfloat16, device=self.device)
        _lib.mok_router_backward(self.cshape, self.ws, x, Wr, idx, scores, dscores, dWr, dx, stream)
        return dWr, dx

    def check(self):
        st = _lib.mok_check(self.ws)
        if st != 0:
            raise _lib.MokError(st, "router device status")
