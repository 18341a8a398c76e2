"""Neuron-sharded decode over torch.distributed ranks, one GPU per rank.

Rank g of G holds the neurons g, g + G, g + 2G, ... of a layer (its rows of
A, b1, W1, W2; a full copy of Bm; b2 on rank 0 only), decodes them with the
library's ordinary calls into a partial output, exchanges the partial
outputs with one all-gather, and sums them in rank order with
pi_shard_reduce (deterministic).  The neuron partition and the sum follow
include/pi.h (pi_shard_desc / pi_shard_layer / pi_shard_reduce).

Marshalling and the collective only: every arithmetic step runs in libpi's
kernels.  Peer data moves only through the torch.distributed collective.
"""
from __future__ import annotations

from . import (check, make_weights, pi_ffn_desc, pi_layer_decode, pi_shard_desc,
               pi_shard_layer, pi_shard_reduce, workspace)


def shard_desc(desc, G: int, g: int) -> pi_ffn_desc:
    """The descriptor of rank g's shard (host only)."""
    out = pi_ffn_desc()
    check(pi_shard_desc(desc, G, g, out), "pi_shard_desc")
    return out


def exchange(part, world: int, group=None):
    """All ranks' partial outputs, [world][batch][d], in rank order (one
    all-gather; the identity on one rank)."""
    import torch
    if world == 1:
        return part.unsqueeze(0)
    import torch.distributed as dist
    p = part.contiguous()
    out = torch.empty((world * p.shape[0],) + tuple(p.shape[1:]), dtype=p.dtype, device=p.device)
    dist.all_gather_into_tensor(out, p, group=group)  # rank g's rows at [g * batch, ...)
    return out.view((world,) + tuple(p.shape))


class ShardedLayer:
    """Rank g's shard of one layer, resident on `device`.

    A, Bm, b1, W1, W2, b2: the whole layer's device tensors (W2 None for a
    packed layout), read once here to build the shard."""

    def __init__(self, desc, A, Bm, b1, W1, W2, b2, G: int, g: int, device, stream=None):
        import torch
        self.G, self.g, self.d = G, g, desc.d
        self.desc = shard_desc(desc, G, g)
        n = self.desc.n
        self.A = torch.empty((n, desc.r), dtype=torch.int16, device=device)
        self.b1 = torch.empty((n,), dtype=torch.float32, device=device)
        self.W1 = torch.empty((n,) + tuple(W1.shape[1:]), dtype=W1.dtype, device=device)
        self.W2 = (torch.empty((n, desc.d), dtype=W2.dtype, device=device)
                   if W2 is not None else None)
        self.Bm = Bm
        self.b2 = b2 if g == 0 else None
        src = make_weights(A, Bm, b1, W1, W2, b2)
        dst = make_weights(self.A, Bm, self.b1, self.W1, self.W2, self.b2)
        check(pi_shard_layer(desc, src, G, g, dst, stream=stream), "pi_shard_layer")
        self.w = dst
        self.ws = None

    def partial(self, x, batch: int, part, idx_out, cnt_out, dev_status, stream=None):
        """This rank's partial output over its own neurons (no residual)."""
        if self.ws is None:
            self.ws = workspace(self.desc, 32, x.device)
        check(pi_layer_decode(self.desc, self.w, x, batch, part, None, idx_out, cnt_out,
                              dev_status, self.ws, stream=stream), "pi_layer_decode")


def decode(shard: ShardedLayer, x, batch: int, y, residual, dev_status, world: int, group=None,
           idx_out=None, cnt_out=None, stream=None):
    """One decode step of a sharded layer on every rank: partial output,
    all-gather, rank-ordered sum (+ residual) into y [batch][d] (the same y
    on every rank).  idx_out / cnt_out receive the rank's own active list in
    local rows (local row k is neuron g + k G)."""
    import torch
    part = torch.empty((batch, shard.d), dtype=torch.float32, device=x.device)
    shard.partial(x, batch, part, idx_out, cnt_out, dev_status, stream=stream)
    parts = exchange(part, world, group)
    check(pi_shard_reduce(parts, world, batch, shard.d, residual, y, stream=stream),
          "pi_shard_reduce")
    return y
