"""Neuron-sharded decode, its G ranks emulated one after another on one GPU
(each shard's launches are independent; only the exchange joins them): the
shards' active sets are the oracle's restricted to each rank's neurons, and
the rank-ordered sum of the partial outputs equals the oracle on the union
of the shards' lists."""
import numpy as np
import pytest
import torch

import activation_sparse_decode_rank_gb300 as pi
from activation_sparse_decode_rank_gb300 import sharded
import oracle
import synth
from pihelp import Y_TOL, check_active_set, up, y_rel_err, zeros_i32

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")

SHAPES = [(1024, 4096, 64, "f16", False, 0.8, 0.08, 51, 90),
          (200, 1001, 24, "bf16", False, 0.9, 0.10, 52, 37),
          (136, 777, 16, "f16", True, 1.0, 0.12, 53, 20)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    pi.build()
    yield


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("G", [2, 3])
@pytest.mark.parametrize("packed", [False, True])
def test_sharded_layer_matches_the_oracle(shape, G, packed):
    d, n, r, dt, gated, a, rho, seed, hot = shape
    L = synth.make_layer(d, n, r, dt, gated=gated, alpha=a, density=rho, seed=seed)
    desc = pi.make_desc(d, n, r, dt, gated, hot, packed=packed)
    A, Bm, b1, W1, W2, b2 = (up(L.A, DEV), up(L.Bm, DEV), up(L.b1, DEV), up(L.W1, DEV),
                             up(L.W2, DEV), up(L.b2, DEV))
    if packed:
        m = 3 if gated else 2
        rec = torch.empty((n, m * d), dtype=torch.int16, device=DEV)
        sdesc = pi.make_desc(d, n, r, dt, gated, hot)
        pi.check(pi.pi_pack_weights(sdesc, W1, W2, rec))
        W1, W2 = rec, None
    batch = 3
    xs = synth.gen_x(seed + 5, 0, batch, d)
    res = synth.gen_x(seed + 6, 0, batch, d)
    shards = [sharded.ShardedLayer(desc, A, Bm, b1, W1, W2, b2, G, g, DEV) for g in range(G)]
    assert sum(s.desc.n for s in shards) == n
    for g, s in enumerate(shards):
        assert s.desc.n == len(range(g, n, G))
        assert s.desc.hot_prefix == len(range(g, hot, G))
    x = up(xs, DEV)
    outs = []
    for rep in range(2):
        parts = torch.empty((G, batch, d), device=DEV)
        lists = []
        st = zeros_i32(1, DEV)
        for g, s in enumerate(shards):
            idx = torch.full((batch, s.desc.n), -1, dtype=torch.int32, device=DEV)
            cnt = zeros_i32(batch, DEV)
            s.partial(x, batch, parts[g], idx, cnt, st)
            torch.cuda.synchronize()
            lists.append((idx.cpu().numpy(), cnt.cpu().numpy()))
        y = torch.empty((batch, d), device=DEV)
        pi.check(pi.pi_shard_reduce(parts, G, batch, d, up(res, DEV), y))
        torch.cuda.synchronize()
        assert int(st[0]) == 0
        outs.append(y.cpu().numpy())
    np.testing.assert_array_equal(outs[1], outs[0])  # deterministic
    for t in range(batch):
        _, lg = oracle.predict(L, xs[t])
        glob = []
        for g, (idx, cnt) in enumerate(lists):
            local = idx[t, :cnt[t]]
            check_active_set(local, lg[0][g::G])      # the oracle's mask on rank g's rows
            glob.extend((g + G * local).tolist())     # local row k is neuron g + k G
        gidx = np.array(sorted(glob), dtype=np.int32)
        assert y_rel_err(L, xs[t], gidx, outs[0][t] - res[t]) <= Y_TOL


def test_shard_calls_check_their_arguments():
    desc = pi.make_desc(1024, 4096, 64, "f16")
    out = pi.pi_ffn_desc()
    assert pi.pi_shard_desc(desc, 0, 0, out) == pi.PI_ERR_SHAPE
    assert pi.pi_shard_desc(desc, 4, 4, out) == pi.PI_ERR_SHAPE
    assert pi.pi_shard_desc(desc, 4, -1, out) == pi.PI_ERR_SHAPE
    y = torch.empty((1, 1024), device=DEV)
    assert pi.pi_shard_reduce(y, 1, 0, 1024, None, y) == pi.PI_ERR_SHAPE
    assert pi.pi_shard_reduce(y, 1, 1, 1020, None, y) == pi.PI_ERR_SHAPE
