"""The GPU build of the input generator, and the 48-layer OPT-30B-shaped FFN
stack with residual adds (d=7168, n=28672, r=256, fp16, ~39 GB resident).

Generator: the GPU build must write the host generator's bytes (possible
last-bit differences of log / sin / cos may flip a 16-bit rounding very
rarely; the test bounds that).

Stack: one decode step through all 48 layers with pi_layer_decode and the
residual stream x_{l+1} = x_l + FFN_l(x_l) kept in fp32.  Parity per layer
with teacher forcing (the oracle gets the GPU's x_l) under the near-tie rule,
an end-to-end check of the final residual stream against the oracle's own
chain, and the per-layer density against the plan's target.
"""
import numpy as np
import pytest
import torch

import activation_sparse_decode_rank_gb300 as pi
import oracle
import synth
from pihelp import Y_TOL, check_active_set, near_ties, up, zeros_i32

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.mark.parametrize("shape", [(256, 640, 32, "f16", False), (136, 777, 16, "bf16", True),
                                   (4096, 2048, 128, "f16", False)])
def test_gpu_generator_writes_the_host_bytes(shape):
    d, n, r, dt, g = shape
    h = synth.make_layer(d, n, r, dt, gated=g, alpha=0.9, density=0.1, seed=41, layer=3)
    gg = synth.make_layer_gpu(d, n, r, dt, gated=g, alpha=0.9, density=0.1, seed=41, layer=3,
                              device=DEV)
    torch.cuda.synchronize()
    gh = synth.to_host_layer(gg)
    np.testing.assert_array_equal(gh.b1, h.b1)
    for name in ("A", "Bm", "W1", "W2"):
        a, b = getattr(gh, name), getattr(h, name)
        diff = a != b
        # any difference must be one unit in the last place, and very rare
        assert diff.mean() <= 1e-6, f"{name}: {diff.sum()} of {diff.size} differ"
        if diff.any():
            assert np.all(np.abs(a[diff].astype(np.int32) - b[diff].astype(np.int32)) == 1)


def test_opt30b_stack_48_layers():
    d, n, r, L = 7168, 28672, 256, 48
    seed = 4
    alpha, rho, c, scale = synth.stack_plan(seed, L, n)
    layers, descs, wts = [], [], []
    for l in range(L):
        g = synth.make_layer_gpu(d, n, r, "f16", alpha=float(alpha[l]), zipf_c=float(c[l]),
                                 seed=seed, layer=l, bias_scale=float(scale[l]), device=DEV)
        layers.append(g)
        descs.append(pi.make_desc(d, n, r, "f16", False, hot_prefix=n // 36))
        wts.append(pi.make_weights(g["A"], g["Bm"], g["b1"], g["W1"], g["W2"], g["b2"]))
    ws = pi.workspace(descs[0], 1, DEV)
    st = zeros_i32(1, DEV)
    x0 = synth.gen_x(seed, 0, 1, d)
    xs = [up(x0, DEV)]
    idx = torch.full((L, n), -1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros((L, 4), dtype=torch.int32, device=DEV)
    for l in range(L):
        y = torch.empty((1, d), dtype=torch.float32, device=DEV)
        pi.check(pi.pi_layer_decode(descs[l], wts[l], xs[l], 1, y, xs[l], idx[l], cnt[l], st, ws),
                 f"layer {l}")
        xs.append(y)
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    xh = [t.cpu().numpy()[0] for t in xs]
    cnts = cnt[:, 0].cpu().numpy()
    ties = 0
    x_or = x0[0].copy()
    for l in range(L):
        Lh = synth.to_host_layer(layers[l])
        # teacher forcing: the oracle runs on the GPU's own input of layer l
        _, lo = oracle.predict(Lh, xh[l])
        gi = idx[l, : cnts[l]].cpu().numpy()
        ties += check_active_set(gi, lo[0])
        yo = oracle.sparse_ffn(Lh, xh[l], gi)
        yd = oracle.dense_ffn(Lh, xh[l])
        want = (xh[l].astype(np.float64) + yo).astype(np.float32)
        err = float(np.abs(xh[l + 1].astype(np.float64) - want).max()) / float(np.abs(yd).max())
        assert err <= Y_TOL, f"layer {l}: {err}"
        # the per-layer density stays near the plan's target (bias scaling)
        assert 0.5 * rho[l] < cnts[l] / n < 1.6 * rho[l] + 0.01, (l, cnts[l] / n, rho[l])
        # the oracle's own chain, end to end
        _, _, _, x_or = oracle.layer_decode(Lh, x_or, residual=True)
        del Lh
    assert ties <= 4 * L
    end = float(np.abs(xh[L].astype(np.float64) - x_or).max()) / float(np.abs(x_or).max())
    assert end <= 1e-2, end
