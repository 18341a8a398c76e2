"""Offline profiling and neuron placement on the GPU (pi_profile_counts,
pi_hot_order, pi_permute_neurons) against the oracle.

Integer outputs are compared bit for bit: counts from the same fp32 logits,
the hot-first order from the same counts, every permuted tensor byte for
byte.  End to end: a layer stored in a shuffled order is profiled over
sample tokens with the GPU predictor, placed hot first, and decoded; the
placed layer gives the oracle's y for the shuffled layer, and its active
list maps back through the neuron table.
"""
import numpy as np
import pytest
import torch

import activation_sparse_decode_rank_gb300 as pi
import oracle
import synth
from pihelp import DevLayer, Y_TOL, check_active_set, up, zeros_i32

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def gpu_counts(lg_host, counts=None):
    batch, n = lg_host.shape
    c = torch.zeros(max(n, 4), dtype=torch.int32, device=DEV)
    if counts is not None:
        c[:n] = up(np.asarray(counts, np.uint32), DEV)
    pi.check(pi.pi_profile_counts(up(lg_host.astype(np.float32), DEV), n, batch, c))
    torch.cuda.synchronize()
    return c.cpu().numpy()[:n].view(np.uint32)


@pytest.mark.parametrize("n,batch", [(1, 1), (777, 3), (28672, 32), (100003, 7)])
def test_profile_counts_bit_exact(n, batch):
    rng = np.random.default_rng(n + batch)
    lg = rng.standard_normal((batch, n)).astype(np.float32)
    lg[0, : min(n, 3)] = [0.0, -0.0, 1e-38][: min(n, 3)]
    c = gpu_counts(lg)
    np.testing.assert_array_equal(c, oracle.profile_counts(lg.astype(np.float64)))
    c2 = gpu_counts(lg, c)  # accumulates
    np.testing.assert_array_equal(c2, 2 * c)


@pytest.mark.parametrize("n,top", [(1, 3), (1000, 2), (28672, 50), (100003, 400)])
def test_hot_order_bit_exact(n, top):
    rng = np.random.default_rng(n)
    counts = rng.integers(0, top, n).astype(np.uint32)  # many ties
    c = up(counts, DEV)
    perm = torch.full((max(n, 4),), -1, dtype=torch.int32, device=DEV)
    pi.check(pi.pi_hot_order(c, n, perm))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(perm.cpu().numpy()[:n], oracle.hot_order(counts))


def _alloc_like(D):
    L = D.L
    A = torch.empty_like(D.A)
    b1 = torch.empty_like(D.b1)
    if D.packed is not None and D.desc.layout == pi.PI_LAYOUT_PACKED:
        W1 = torch.empty_like(D.packed)
        W2 = None
    else:
        W1 = torch.empty_like(D.W1)
        W2 = torch.empty_like(D.W2)
    return A, b1, W1, W2


@pytest.mark.parametrize("shape", [(1024, 4096, 64, "f16", False), (256, 1001, 24, "bf16", True),
                                   (4096, 16384, 128, "f16", False)])
@pytest.mark.parametrize("packed", [False, True])
def test_permute_neurons_bit_exact(shape, packed):
    d, n, r, dt, g = shape
    L = synth.make_layer(d, n, r, dt, gated=g, alpha=0.9, density=0.1, seed=31)
    D = DevLayer(L, DEV, packed=packed)
    perm_h = np.random.default_rng(31).permutation(n).astype(np.int32)
    A, b1, W1, W2 = _alloc_like(D)
    dst = pi.make_weights(A, D.Bm, b1, W1, W2, D.b2)
    st = zeros_i32(1, DEV)
    pi.check(pi.pi_permute_neurons(D.desc, D.w, up(perm_h, DEV), dst, st))
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    np.testing.assert_array_equal(A.cpu().numpy().view(np.uint16), oracle.permute_rows(L.A, perm_h))
    np.testing.assert_array_equal(b1.cpu().numpy(), oracle.permute_rows(L.b1, perm_h))
    if packed:
        rec = D.packed.cpu().numpy()
        np.testing.assert_array_equal(W1.cpu().numpy(), oracle.permute_rows(rec, perm_h))
    else:
        np.testing.assert_array_equal(W1.cpu().numpy().view(np.uint16),
                                      oracle.permute_rows(L.W1, perm_h))
        np.testing.assert_array_equal(W2.cpu().numpy().view(np.uint16),
                                      oracle.permute_rows(L.W2, perm_h))


def test_permute_rejects_out_of_range_entries():
    L = synth.make_layer(256, 512, 16, "f16", alpha=0.9, density=0.1, seed=32)
    D = DevLayer(L, DEV)
    perm_h = np.arange(512, dtype=np.int32)[::-1].copy()
    perm_h[7] = 512
    perm_h[9] = -3
    A, b1, W1, W2 = _alloc_like(D)
    A.fill_(0)
    dst = pi.make_weights(A, D.Bm, b1, W1, W2, D.b2)
    st = zeros_i32(1, DEV)
    pi.check(pi.pi_permute_neurons(D.desc, D.w, up(perm_h, DEV), dst, st))
    torch.cuda.synchronize()
    assert int(st[0]) == pi.PI_ERR_INDEX
    Ah = A.cpu().numpy().view(np.uint16)
    assert not Ah[7].any() and not Ah[9].any()  # not followed
    np.testing.assert_array_equal(Ah[8], L.A[perm_h[8]])


def test_profile_place_decode_end_to_end():
    # a hot-first layer stored shuffled; the GPU predictor over 320 sample
    # tokens profiles it, the GPU ranks and permutes it
    d, n, r = 1024, 4096, 64
    L = synth.make_layer(d, n, r, "f16", alpha=0.8, density=0.08, seed=33)
    shuf = np.random.default_rng(33).permutation(n).astype(np.int32)
    Ls = synth.permute_layer(L, shuf)
    D = DevLayer(Ls, DEV)
    ws = D.workspace(32)
    counts = torch.zeros(n, dtype=torch.int32, device=DEV)
    lg = torch.empty((32, n), dtype=torch.float32, device=DEV)
    host_counts = np.zeros(n, np.uint32)
    for s in range(10):
        x = synth.gen_x(34, s, 32, d)
        pi.check(pi.pi_predict(D.desc, D.A, D.Bm, D.b1, up(x, DEV), 32, lg, ws))
        pi.check(pi.pi_profile_counts(lg, n, 32, counts))
        torch.cuda.synchronize()
        host_counts = oracle.profile_counts(lg.cpu().numpy().astype(np.float64), host_counts)
    ch = counts.cpu().numpy().view(np.uint32)
    np.testing.assert_array_equal(ch, host_counts)  # from the GPU's own logits
    perm = torch.empty(n, dtype=torch.int32, device=DEV)
    pi.check(pi.pi_hot_order(counts, n, perm))
    A, b1, W1, W2 = _alloc_like(D)
    dst = pi.make_weights(A, D.Bm, b1, W1, W2, D.b2)
    st = zeros_i32(1, DEV)
    pi.check(pi.pi_permute_neurons(D.desc, D.w, perm, dst, st))
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    ph = perm.cpu().numpy()
    np.testing.assert_array_equal(ph, oracle.hot_order(ch))
    # the placed order is hot first: mostly the generator's own hot prefix
    orig = shuf[ph]
    assert np.mean(orig[:200]) < 0.25 * np.mean(orig[-2000:])
    # decode the placed layer
    desc_p = pi.make_desc(d, n, r, "f16", False, hot_prefix=90)
    y = torch.empty((1, d), device=DEV)
    idx = torch.full((1, n), -1, dtype=torch.int32, device=DEV)
    cnt = zeros_i32(1, DEV)
    for t in range(3):
        x = synth.gen_x(35, t, 1, d)
        pi.check(pi.pi_layer_decode(desc_p, dst, up(x, DEV), 1, y, None, idx, cnt, st,
                                    pi.workspace(desc_p, 1, DEV)))
        torch.cuda.synchronize()
        assert int(st[0]) == 0
        gi = idx[0, : int(cnt[0])].cpu().numpy()
        orig_idx = np.sort(ph[gi])          # through the neuron table
        _, lo = oracle.predict(Ls, x)
        check_active_set(orig_idx, lo[0])
        yo = oracle.sparse_ffn(Ls, x[0], orig_idx)
        yd = oracle.dense_ffn(Ls, x[0])
        assert float(np.abs(y.cpu().numpy()[0] - yo).max()) <= Y_TOL * float(np.abs(yd).max())
