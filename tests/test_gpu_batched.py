"""Batched decode (2 <= batch <= 32): per-token masks, the union of the
tokens' active neurons read once, the contraction on tensor cores.

Parity: every token's active set under the near-tie rule, and every token's
y against the oracle run on that token's own GPU list (the batched result
must equal the batch-1 definition for each token).  Workloads: the
OPT-13B-shaped layer of the density sweep at full size, the gated
Llama-2-7B-shaped layer, a small layer with ragged union tiles.
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
_cache = {}


def dev_layer(key, maker):
    if key not in _cache:
        _cache.clear()
        torch.cuda.empty_cache()
        _cache[key] = DevLayer(maker(), DEV)
    return _cache[key]


def opt13b(density):
    return dev_layer(("opt13b", density), lambda: synth.make_layer(
        5120, 20480, 192, "f16", alpha=0.9, density=density, seed=5))


def decode_batch(D, x, packed=False):
    L = D.L
    B = x.shape[0]
    D.set_packed(packed)
    try:
        y = torch.full((B, L.d), float("nan"), device=DEV)
        idx = torch.full((B, L.n), -1, dtype=torch.int32, device=DEV)
        cnt = zeros_i32(B, DEV)
        st = zeros_i32(1, DEV)
        pi.check(pi.pi_layer_decode(D.desc, D.w, up(x, DEV), B, y, None, idx, cnt, st,
                                    D.workspace(B)), "pi_layer_decode")
        torch.cuda.synchronize()
    finally:
        D.set_packed(False)
    c = cnt.cpu().numpy()[:B]
    return y.cpu().numpy(), [idx[t, : c[t]].cpu().numpy() for t in range(B)], int(st[0])


def check_tokens(L, x, y, idxs, tokens=None):
    for t in (range(x.shape[0]) if tokens is None else tokens):
        _, lo = oracle.predict(L, x[t])
        check_active_set(idxs[t], lo[0])
        yo = oracle.sparse_ffn(L, x[t], idxs[t])
        yd = oracle.dense_ffn(L, x[t])
        err = float(np.abs(y[t].astype(np.float64) - yo).max()) / float(np.abs(yd).max())
        assert err <= Y_TOL, (t, err)


@pytest.mark.parametrize("batch", [2, 4, 16, 32])
@pytest.mark.parametrize("density", [0.02, 0.10, 0.50])
def test_batched_decode_opt13b(batch, density):
    D = opt13b(density)
    x = synth.gen_x(50 + batch, 0, batch, D.L.d)
    y, idxs, st = decode_batch(D, x, packed=(batch % 2 == 0 and density == 0.10))
    assert st == 0
    check_tokens(D.L, x, y, idxs, tokens=sorted({0, batch // 2, batch - 1}))


def test_batched_decode_gated_bf16_packed():
    D = dev_layer("llama", lambda: synth.make_layer(4096, 11008, 256, "bf16", gated=True,
                                                     alpha=1.0, density=0.10, seed=3))
    x = synth.gen_x(60, 0, 8, D.L.d)
    for packed in (False, True):
        y, idxs, st = decode_batch(D, x, packed=packed)
        assert st == 0
        check_tokens(D.L, x, y, idxs, tokens=[0, 3, 7])


def test_batched_ragged_tiles_and_residual():
    # d = 256 (two 128-column chunks), n = 1001: union tiles end mid-tile
    D = dev_layer("ragged", lambda: synth.make_layer(256, 1001, 24, "f16", alpha=0.9,
                                                      density=0.15, seed=61))
    L = D.L
    for batch in (3, 17, 32):
        x = synth.gen_x(61, batch, batch, L.d)
        y, idxs, st = decode_batch(D, x)
        assert st == 0
        check_tokens(L, x, y, idxs)
        # residual: y + x
        yr = torch.empty((batch, L.d), device=DEV)
        st2 = zeros_i32(1, DEV)
        xd = up(x, DEV)
        pi.check(pi.pi_layer_decode(D.desc, D.w, xd, batch, yr, xd, None, None, st2,
                                    D.workspace(batch)))
        torch.cuda.synchronize()
        np.testing.assert_allclose(yr.cpu().numpy(), y + x, rtol=0, atol=1e-5)


def test_batched_sparse_ffn_on_oracle_union():
    D = opt13b(0.10)
    L = D.L
    batch = 8
    x = synth.gen_x(62, 0, batch, L.d)
    _, lo = oracle.predict(L, x)
    uidx, tmask = oracle.union(lo)
    ui = up(np.ascontiguousarray(uidx, np.int32), DEV)
    uc = torch.tensor([len(uidx), 0, 0, 0], dtype=torch.int32, device=DEV)
    tm = up(np.ascontiguousarray(tmask, np.uint32), DEV)
    y = torch.empty((batch, L.d), device=DEV)
    st = zeros_i32(1, DEV)
    pi.check(pi.pi_sparse_ffn(D.desc, D.w, up(x, DEV), batch, None, None, 0, ui, uc, tm, y, st,
                              D.workspace(batch)))
    torch.cuda.synchronize()
    yh = y.cpu().numpy()
    for t in range(batch):
        S = oracle.compact(lo[t])
        yo = oracle.sparse_ffn(L, x[t], S)
        yd = oracle.dense_ffn(L, x[t])
        assert float(np.abs(yh[t] - yo).max()) / float(np.abs(yd).max()) <= Y_TOL


def test_batched_empty_union():
    L = synth.make_layer(256, 512, 16, "f16", alpha=0.9, density=0.1, seed=63)
    L.b1[:] = -1e4
    D = DevLayer(L, DEV)
    x = synth.gen_x(63, 0, 5, 256)
    y, idxs, st = decode_batch(D, x)
    assert st == 0 and all(len(i) == 0 for i in idxs)
    np.testing.assert_array_equal(y, np.broadcast_to(L.b2, y.shape))


@pytest.mark.parametrize("batch", [2, 16, 32])
def test_dense_batched(batch):
    D = dev_layer("ragged", lambda: synth.make_layer(256, 1001, 24, "f16", alpha=0.9,
                                                      density=0.15, seed=61))
    L = D.L
    x = synth.gen_x(64, batch, batch, L.d)
    y = torch.empty((batch, L.d), device=DEV)
    pi.check(pi.pi_dense_ffn(D.desc, D.w, up(x, DEV), batch, y, D.workspace(batch)))
    torch.cuda.synchronize()
    yh = y.cpu().numpy()
    for t in range(batch):
        yd = oracle.dense_ffn(L, x[t])
        assert float(np.abs(yh[t] - yd).max()) / float(np.abs(yd).max()) <= Y_TOL


def test_dense_batched_gated_full_size():
    D = dev_layer("llama", lambda: synth.make_layer(4096, 11008, 256, "bf16", gated=True,
                                                     alpha=1.0, density=0.10, seed=3))
    x = synth.gen_x(65, 0, 4, D.L.d)
    for packed in (False, True):
        D.set_packed(packed)
        try:
            y = torch.empty((4, D.L.d), device=DEV)
            pi.check(pi.pi_dense_ffn(D.desc, D.w, up(x, DEV), 4, y, D.workspace(4)))
            torch.cuda.synchronize()
        finally:
            D.set_packed(False)
        yh = y.cpu().numpy()
        for t in (0, 3):
            yd = oracle.dense_ffn(D.L, x[t])
            assert float(np.abs(yh[t] - yd).max()) / float(np.abs(yd).max()) <= Y_TOL


@pytest.mark.parametrize("gated", [False, True])
def test_tcgen05_up_projection(gated, monkeypatch):
    """The tcgen05 up projection (PI_BATCH_TC=1) under the same rules."""
    monkeypatch.setenv("PI_BATCH_TC", "1")
    if gated:
        D = dev_layer("llama", lambda: synth.make_layer(4096, 11008, 256, "bf16", gated=True,
                                                         alpha=1.0, density=0.10, seed=3))
        x = synth.gen_x(70, 0, 5, 4096)
        tokens = [0, 4]
    else:
        D = opt13b(0.10)
        x = synth.gen_x(71, 0, 32, 5120)
        tokens = [0, 17, 31]
    for packed in (False, True):
        y, idxs, st = decode_batch(D, x, packed=packed)
        assert st == 0
        check_tokens(D.L, x, y, idxs, tokens=tokens)
    yd = torch.empty((x.shape[0], D.L.d), device=DEV)
    pi.check(pi.pi_dense_ffn(D.desc, D.w, up(x, DEV), x.shape[0], yd, D.workspace(x.shape[0])))
    torch.cuda.synchronize()
    for t in tokens:
        want = oracle.dense_ffn(D.L, x[t])
        assert float(np.abs(yd.cpu().numpy()[t] - want).max()) <= Y_TOL * float(np.abs(want).max())


def dense_batch(D, x, packed):
    B = x.shape[0]
    D.set_packed(packed)
    try:
        y = torch.full((B, D.L.d), float("nan"), device=DEV)
        pi.check(pi.pi_dense_ffn(D.desc, D.w, up(x, DEV), B, y, D.workspace(B)), "pi_dense_ffn")
        torch.cuda.synchronize()
    finally:
        D.set_packed(False)
    return y.cpu().numpy()


@pytest.mark.parametrize("batch,packed", [(2, False), (16, True), (32, False), (32, True)])
def test_dense_batched_tensor_memory_opt13b(batch, packed):
    """The dense batched FFN on the tcgen05 / TMA phases, OPT-13B shape:
    128 or 136 weight rows per block as the MMA's N in phase 1 (x's high and
    low parts as its M), phase 2's (column tile, neuron block) items split
    over every block, the blocks' partials summed in block order."""
    D = opt13b(0.10)
    x = synth.gen_x(72, batch, batch, 5120)
    y = dense_batch(D, x, packed)
    for t in sorted({0, batch // 2, batch - 1}):
        want = oracle.dense_ffn(D.L, x[t])
        assert float(np.abs(y[t] - want).max()) <= Y_TOL * float(np.abs(want).max()), t


def test_dense_batched_wide_layer():
    """n = 65536: 432 rows per block, more than one accumulator tile of the
    tensor-memory phases holds, so the dense FFN takes the mma.sync phases;
    bit-identical on a second call."""
    D = dev_layer("wide", lambda: synth.make_layer(1024, 65536, 64, "f16", alpha=0.9,
                                                    density=0.1, seed=73))
    x = synth.gen_x(74, 0, 3, 1024)
    y = dense_batch(D, x, False)
    for t in range(3):
        want = oracle.dense_ffn(D.L, x[t])
        assert float(np.abs(y[t] - want).max()) <= Y_TOL * float(np.abs(want).max()), t
    np.testing.assert_array_equal(dense_batch(D, x, False), y)


@pytest.mark.parametrize("batch", [8, 24])
def test_dense_batched_tensor_memory_128_column_tiles(batch):
    """d = 1152 (a multiple of 128, not of 256): phase 2 takes 128-column
    tiles; 16 and 32 padded tokens (the one-warp and the two-warp
    epilogue); n = 4096: 32 rows per block in phase 1."""
    D = dev_layer("d1152", lambda: synth.make_layer(1152, 4096, 64, "f16", alpha=0.9,
                                                     density=0.1, seed=75))
    x = synth.gen_x(76, batch, batch, 1152)
    for packed in (False, True):
        y = dense_batch(D, x, packed)
        for t in sorted({0, batch - 1}):
            want = oracle.dense_ffn(D.L, x[t])
            assert float(np.abs(y[t] - want).max()) <= Y_TOL * float(np.abs(want).max()), (packed, t)


def test_dense_batched_tensor_memory_gated_batch32():
    """Gated bf16 Llama-2-7B shape at batch 32: two weight tiles (gate, up)
    per stage in phase 1, 256-column tiles and the two-warp epilogue in
    phase 2."""
    D = dev_layer("llama", lambda: synth.make_layer(4096, 11008, 256, "bf16", gated=True,
                                                     alpha=1.0, density=0.10, seed=3))
    x = synth.gen_x(77, 0, 32, 4096)
    y = dense_batch(D, x, True)
    for t in (0, 13, 31):
        want = oracle.dense_ffn(D.L, x[t])
        assert float(np.abs(y[t] - want).max()) <= Y_TOL * float(np.abs(want).max()), t


def test_dense_batched_legacy_phases_subprocess():
    """PI_BATCH_LEGACY=1 (read once per process, so in a child process)
    keeps the dense batched FFN on the mma.sync phases: the same layer and
    tokens against the oracle, at 16 and 32 padded tokens."""
    import os
    import subprocess
    import sys
    code = r'''
import sys, numpy as np, torch
import activation_sparse_decode_rank_gb300 as pi, oracle, synth
sys.path.insert(0, "tests")
from pihelp import DevLayer, Y_TOL, up
dev = torch.device("cuda:0")
D = DevLayer(synth.make_layer(1152, 4096, 64, "f16", alpha=0.9, density=0.1, seed=75), dev)
for B in (8, 24):
    x = synth.gen_x(78, B, B, 1152)
    y = torch.full((B, 1152), float("nan"), device=dev)
    pi.check(pi.pi_dense_ffn(D.desc, D.w, up(x, dev), B, y, D.workspace(B)))
    torch.cuda.synchronize()
    yh = y.cpu().numpy()
    for t in (0, B - 1):
        want = oracle.dense_ffn(D.L, x[t])
        err = float(np.abs(yh[t] - want).max()) / float(np.abs(want).max())
        assert err <= Y_TOL, (B, t, err)
print("ok")
'''
    env = dict(os.environ, PI_BATCH_LEGACY="1")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]
