"""pi_decode_layers: J batch-1 decode steps over a table of layers in one
persistent launch (residual stack, or independent steps).

Parity per step against the oracle on the GPU's own input of that step
(teacher forcing for the stack), under the near-tie rule for the mask
(mask_out) and the y tolerance on the GPU's own active set; the step counts
(cnt_out) equal the masks' popcounts; and the steps agree with one
pi_layer_decode call per step (same masks outside near-ties, y within the
tolerance: the two kernels sum the predictor in different orders).
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


def run_seq(layers, J, x, chain):
    """layers: list of DevLayer; returns y [J][d], masks [J][n], counts [J]."""
    d, n = layers[0].desc.d, layers[0].desc.n
    y = torch.full((J, d), float("nan"), device=DEV)
    cnt = torch.full((max(J, 4),), -1, dtype=torch.int32, device=DEV)
    mask = torch.full((J, n), 7, dtype=torch.uint8, device=DEV)
    st = zeros_i32(1, DEV)
    ws = pi.workspace(layers[0].desc, 1, DEV)
    pi.check(pi.pi_decode_layers([D.desc for D in layers], [D.w for D in layers], J, up(x, DEV),
                                 int(chain), y, cnt, mask, st, ws), "pi_decode_layers")
    torch.cuda.synchronize()
    assert int(st[0]) == 0, pi.status_string(int(st[0]))
    return y.cpu().numpy(), mask.cpu().numpy(), cnt.cpu().numpy()[:J]


def check_steps(layers, J, x, chain, y, mask, cnt, steps=None):
    R = len(layers)
    ties = 0
    for j in (range(J) if steps is None else steps):
        L = layers[j % R].L
        xj = (x[0] if j == 0 else y[j - 1]) if chain else x[j]
        assert np.all((mask[j] == 0) | (mask[j] == 1))
        gi = np.nonzero(mask[j])[0].astype(np.int32)
        assert cnt[j] == gi.size
        _, lo = oracle.predict(L, xj)
        ties += check_active_set(gi, lo[0])
        yo = oracle.sparse_ffn(L, xj, gi)
        if chain:
            yo = xj.astype(np.float64) + yo
        yd = oracle.dense_ffn(L, xj)
        err = float(np.abs(y[j].astype(np.float64) - yo).max()) / float(np.abs(yd).max())
        assert err <= Y_TOL, (j, err)
    return ties


def tiny_layers(R, seed=21, dtype="f16", gated=False, hot=90, packed=False):
    out = []
    for l in range(R):
        L = synth.make_layer(1024, 4096, 64, dtype, gated=gated, alpha=0.8, density=0.08,
                             seed=seed, layer=l)
        out.append(DevLayer(L, DEV, hot_prefix=hot, packed=packed))
    return out


@pytest.mark.parametrize("packed,balance", [(False, "0"), (True, "0"), (False, "1"), (True, "1")])
def test_stack_chain_tiny(packed, balance, monkeypatch):
    # balance = 1: the cold active neurons are spread over the blocks by
    # global rank (one more grid-wide wait); the results obey the same rules
    monkeypatch.setenv("PI_SEQ_BALANCE", balance)
    layers = tiny_layers(4, packed=packed)
    x = synth.gen_x(21, 0, 1, 1024)
    y, mask, cnt = run_seq(layers, 4, x, chain=True)
    assert check_steps(layers, 4, x, True, y, mask, cnt) <= 8


@pytest.mark.parametrize("J", [1, 2, 3])
@pytest.mark.parametrize("chain", [True, False])
def test_short_launches(J, chain):
    # independent steps reduce step j - 1 beside step j's stage 1, and the
    # last step after the loop; the shortest launches cover both ends
    layers = tiny_layers(2, seed=28)
    x = synth.gen_x(28, 0, 1 if chain else J, 1024)
    y, mask, cnt = run_seq(layers, J, x, chain=chain)
    check_steps(layers, J, x, chain, y, mask, cnt)


@pytest.mark.parametrize("chain", [True, False])
def test_rank_per_layer(chain):
    # each layer its own predictor rank (64, 16, 48, 32): the launch sizes
    # its buffers for the largest, every step uses its layer's own
    ranks = (64, 16, 48, 32)
    layers = []
    for l, r in enumerate(ranks):
        L = synth.make_layer(1024, 4096, r, "f16", alpha=0.8, density=0.08, seed=27, layer=l)
        layers.append(DevLayer(L, DEV, hot_prefix=90, packed=True))
    J = 6
    x = synth.gen_x(27, 0, 1 if chain else J, 1024)
    d, n = 1024, 4096
    y = torch.full((J, d), float("nan"), device=DEV)
    cnt = torch.full((max(J, 4),), -1, dtype=torch.int32, device=DEV)
    mask = torch.full((J, n), 7, dtype=torch.uint8, device=DEV)
    st = zeros_i32(1, DEV)
    big = max(layers, key=lambda D: D.desc.r).desc
    ws = pi.workspace(big, 1, DEV)
    pi.check(pi.pi_decode_layers([D.desc for D in layers], [D.w for D in layers], J, up(x, DEV),
                                 int(chain), y, cnt, mask, st, ws), "pi_decode_layers")
    torch.cuda.synchronize()
    assert int(st[0]) == 0, pi.status_string(int(st[0]))
    check_steps(layers, J, x, chain, y.cpu().numpy(), mask.cpu().numpy(), cnt.cpu().numpy()[:J])


@pytest.mark.parametrize("balance", ["0", "1"])
def test_independent_steps_wrap_the_table(balance, monkeypatch):
    monkeypatch.setenv("PI_SEQ_BALANCE", balance)
    layers = tiny_layers(3, seed=22, hot=0)
    J = 7
    x = synth.gen_x(22, 0, J, 1024)
    y, mask, cnt = run_seq(layers, J, x, chain=False)
    check_steps(layers, J, x, False, y, mask, cnt)


@pytest.mark.parametrize("balance", ["0", "1"])
def test_many_steps_one_launch(balance, monkeypatch):
    monkeypatch.setenv("PI_SEQ_BALANCE", balance)
    layers = tiny_layers(2, seed=23)
    J = 301
    x = synth.gen_x(23, 0, J, 1024)
    y, mask, cnt = run_seq(layers, J, x, chain=False)
    check_steps(layers, J, x, False, y, mask, cnt, steps=[0, 1, 150, 299, 300])
    assert np.isfinite(y).all()


def test_gated_bf16_llama_shape():
    L = synth.make_layer(4096, 11008, 256, "bf16", gated=True, alpha=1.0, density=0.10, seed=3)
    for packed in (False, True):
        D = DevLayer(L, DEV, hot_prefix=463, packed=packed)
        x = synth.gen_x(24, 0, 3, 4096)
        y, mask, cnt = run_seq([D], 3, x, chain=False)
        check_steps([D], 3, x, False, y, mask, cnt)
        del D
        torch.cuda.empty_cache()


@pytest.mark.parametrize("balance", ["0", "1"])
def test_opt67_shape_is_reproducible(balance, monkeypatch):
    # every sum has a fixed order (with balancing too: the split of the cold
    # work depends only on the lists), so two launches give the same bits;
    # and the steps obey the oracle's rules
    monkeypatch.setenv("PI_SEQ_BALANCE", balance)
    L = synth.make_layer(4096, 16384, 128, "f16", alpha=0.9, density=0.06, seed=2)
    D = DevLayer(L, DEV, hot_prefix=304, packed=True)
    J = 6
    x = synth.gen_x(26, 0, J, 4096)
    y, mask, cnt = run_seq([D], J, x, chain=False)
    y2, mask2, cnt2 = run_seq([D], J, x, chain=False)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))
    assert np.array_equal(mask, mask2) and np.array_equal(cnt, cnt2)
    check_steps([D], J, x, False, y, mask, cnt)


def test_opt67_shape_matches_layer_decode():
    L = synth.make_layer(4096, 16384, 128, "f16", alpha=0.9, density=0.06, seed=2)
    D = DevLayer(L, DEV, hot_prefix=304, packed=True)
    J = 5
    x = synth.gen_x(25, 0, J, 4096)
    y, mask, cnt = run_seq([D], J, x, chain=False)
    check_steps([D], J, x, False, y, mask, cnt)
    ws = D.workspace(1)
    st = zeros_i32(1, DEV)
    for j in range(J):
        y1 = torch.empty((1, 4096), device=DEV)
        idx = torch.full((1, 16384), -1, dtype=torch.int32, device=DEV)
        c1 = zeros_i32(1, DEV)
        pi.check(pi.pi_layer_decode(D.desc, D.w, up(x[j:j + 1], DEV), 1, y1, None, idx, c1, st,
                                    ws))
        torch.cuda.synchronize()
        g1 = idx[0, : int(c1[0])].cpu().numpy()
        gs = np.nonzero(mask[j])[0]
        _, lo = oracle.predict(L, x[j])
        from pihelp import near_ties
        tie = near_ties(lo[0])
        diff = np.setxor1d(g1, gs)
        assert all(tie[i] for i in diff)
        yd = oracle.dense_ffn(L, x[j])
        assert float(np.abs(y1.cpu().numpy()[0] - y[j]).max()) <= 2 * Y_TOL * float(np.abs(yd).max())


@pytest.mark.parametrize("balance", ["0", "1"])
def test_opt30_shape_stack_three_layers(balance, monkeypatch):
    monkeypatch.setenv("PI_SEQ_BALANCE", balance)
    d, n, r = 7168, 28672, 256
    seed = 4
    alpha, rho, cz, scale = synth.stack_plan(seed, 48, n)
    gls, layers = [], []
    for l in range(3):
        g = synth.make_layer_gpu(d, n, r, "f16", alpha=float(alpha[l]), zipf_c=float(cz[l]),
                                 seed=seed, layer=l, bias_scale=float(scale[l]), device=DEV)
        desc = pi.make_desc(d, n, r, "f16", False, hot_prefix=n // 36)
        gls.append(g)

        class G:  # minimal DevLayer stand-in over GPU-made tensors
            pass
        D = G()
        D.desc = desc
        D.w = pi.make_weights(g["A"], g["Bm"], g["b1"], g["W1"], g["W2"], g["b2"])
        layers.append(D)
    torch.cuda.synchronize()
    x = synth.gen_x(seed, 0, 1, d)
    y, mask, cnt = run_seq(layers, 3, x, chain=True)
    for l in range(3):
        layers[l].L = synth.to_host_layer(gls[l])
    check_steps(layers, 3, x, True, y, mask, cnt)
    # per-layer densities near the plan's targets
    for l in range(3):
        assert 0.5 * rho[l] < cnt[l] / n < 1.6 * rho[l] + 0.01


def test_layer_decode_still_runs_after_sequences():
    layers = tiny_layers(1, seed=26)
    D = layers[0]
    x = synth.gen_x(26, 0, 2, 1024)
    run_seq(layers, 2, x, chain=False)
    y1 = torch.empty((1, 1024), device=DEV)
    st = zeros_i32(1, DEV)
    pi.check(pi.pi_layer_decode(D.desc, D.w, up(x[:1], DEV), 1, y1, None, None, None, st,
                                D.workspace(1)))
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    yd = oracle.dense_ffn(D.L, x[0])
    _, lo = oracle.predict(D.L, x[0])
    yo = oracle.sparse_ffn(D.L, x[0], oracle.compact(lo[0]))
    assert float(np.abs(y1.cpu().numpy()[0] - yo).max()) <= Y_TOL * float(np.abs(yd).max())
