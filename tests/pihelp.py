"""Shared helpers of the GPU tests: upload a generated layer, run the C ABI
through the binding, and compare with the oracle under the parity rules.

Parity rules (the tolerances the tests enforce):
  * active set: bit-exact, except neurons whose oracle logit satisfies
    |logit| < 1e-4 * rms(logits); those near-ties are excluded and counted;
  * y: the oracle is re-run on the GPU's own active list and
    max|y_gpu - y_oracle| / max|y_dense| <= 2e-3 (absolute 1e-6 if the dense
    output is identically 0);
  * integer outputs (lists, counts, masks) computed from the same logits are
    compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

import activation_sparse_decode_rank_gb300 as pi
import oracle

Y_TOL = 2e-3
TIE_REL = 1e-4


def up(a, dev):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).to(dev)


class DevLayer:
    """A generated layer resident on the GPU, with its descriptor.  packed:
    the weights are held as per-neuron records built by pi_pack_weights."""

    def __init__(self, L, dev, hot_prefix: int = 0, with_b2: bool = True, packed: bool = False):
        self.L = L
        self.dev = dev
        self.A = up(L.A, dev)
        self.Bm = up(L.Bm, dev)
        self.b1 = up(L.b1, dev)
        self.W1 = up(L.W1, dev)
        self.W2 = up(L.W2, dev)
        self.b2 = up(L.b2, dev) if (with_b2 and L.b2 is not None) else None
        self.desc = pi.make_desc(L.d, L.n, L.r, L.dtype, L.gated, hot_prefix)
        self.w = pi.make_weights(self.A, self.Bm, self.b1, self.W1, self.W2, self.b2)
        self.packed = None
        if packed:
            self.set_packed(True)

    def set_packed(self, on: bool):
        """Switches the descriptor and weights between the two layouts."""
        if on and self.packed is None:
            m = 3 if self.L.gated else 2
            self.packed = torch.empty((self.L.n, m * self.L.d), dtype=torch.int16, device=self.dev)
            pi.check(pi.pi_pack_weights(self.desc, self.W1, self.W2, self.packed),
                     "pi_pack_weights")
        self.desc.layout = pi.PI_LAYOUT_PACKED if on else pi.PI_LAYOUT_SPLIT
        if on:
            self.w = pi.make_weights(self.A, self.Bm, self.b1, self.packed, None, self.b2)
        else:
            self.w = pi.make_weights(self.A, self.Bm, self.b1, self.W1, self.W2, self.b2)

    def workspace(self, batch=1):
        return pi.workspace(self.desc, batch, self.dev)


def near_ties(lg):
    lg = np.asarray(lg, np.float64)
    rms = float(np.sqrt(np.mean(lg * lg))) if lg.size else 0.0
    return np.abs(lg) < TIE_REL * rms


def check_active_set(gpu_idx, oracle_logits):
    """Returns the number of near-ties; raises if the sets differ elsewhere."""
    gpu_idx = np.asarray(gpu_idx)
    assert np.all(np.diff(gpu_idx) > 0), "active list not strictly ascending"
    tie = near_ties(oracle_logits)
    want = oracle_logits > 0
    got = np.zeros_like(want)
    got[gpu_idx] = True
    bad = np.nonzero((want != got) & ~tie)[0]
    assert bad.size == 0, f"active set differs at {bad[:10]} (logits {oracle_logits[bad[:10]]})"
    return int(tie.sum())


def y_rel_err(L, x, gpu_idx, y_gpu, y_dense=None):
    yo = oracle.sparse_ffn(L, x, np.asarray(gpu_idx, np.int32))
    yd = oracle.dense_ffn(L, x) if y_dense is None else y_dense
    den = float(np.abs(yd).max())
    diff = float(np.abs(np.asarray(y_gpu, np.float64) - yo).max())
    if den > 0:
        return diff / den
    return 0.0 if diff <= 1e-6 else float("inf")


def zeros_i32(n, dev):
    return torch.zeros(max(n, 4), dtype=torch.int32, device=dev)
