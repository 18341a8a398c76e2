"""Execution of the dispatch plan: pi_decode_planned runs each path the plan
can name, and a pi_decoder replays one captured graph per batch size.

Every path is checked against the oracle under the usual parity rules: the
sparse paths (fused, per token, union) on each token's own predicted set,
the dense path against the plain dense FFN (it has no predictor).
"""
import numpy as np
import pytest
import torch

import activation_sparse_decode_rank_gb300 as pi
import oracle
import synth
from pihelp import Y_TOL, check_active_set, up, y_rel_err, zeros_i32

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
D_, N_, R_ = 1024, 4096, 64


@pytest.fixture(scope="module")
def layer():
    pi.build()
    L = synth.make_layer(D_, N_, R_, "f16", alpha=0.9, density=0.05, seed=41)
    t = [up(L.A, DEV), up(L.Bm, DEV), up(L.b1, DEV), up(L.W1, DEV), up(L.W2, DEV), up(L.b2, DEV)]
    desc = pi.make_desc(D_, N_, R_, "f16", False, 64)
    return L, desc, pi.make_weights(*t), t


def _check_tokens(L, xs, y, idx, cnt, path, residual=None):
    for t in range(xs.shape[0]):
        x = xs[t]
        res = residual[t] if residual is not None else 0.0
        if path == pi.PI_PATH_DENSE:
            want = oracle.dense_ffn(L, x) + res
            den = float(np.abs(oracle.dense_ffn(L, x)).max())
            assert float(np.abs(y[t] - want).max()) / den <= Y_TOL
            continue
        c = int(cnt[t])
        gi = idx[t, :c]
        _, lg = oracle.predict(L, x)
        check_active_set(gi, lg[0])
        assert y_rel_err(L, x, gi, y[t] - res) <= Y_TOL


@pytest.mark.parametrize("path,batch", [(pi.PI_PATH_FUSED, 1), (pi.PI_PATH_PER_TOKEN, 3),
                                        (pi.PI_PATH_UNION, 4), (pi.PI_PATH_DENSE, 4),
                                        (pi.PI_PATH_DENSE, 1)])
@pytest.mark.parametrize("with_residual", [False, True])
def test_every_path_matches_the_oracle(layer, path, batch, with_residual):
    L, desc, w, _ = layer
    xs = synth.gen_x(42, batch, batch, D_)
    res = synth.gen_x(43, batch, batch, D_) if with_residual else None
    y = torch.empty((batch, D_), device=DEV)
    idx = torch.full((batch, N_), -1, dtype=torch.int32, device=DEV)
    cnt = zeros_i32(batch, DEV)
    st = zeros_i32(1, DEV)
    ws = pi.workspace(desc, batch, DEV)
    rc = pi.pi_decode_planned(desc, w, path, up(xs, DEV), batch, y,
                              up(res, DEV) if res is not None else None, idx, cnt, st, ws)
    pi.check(rc, "pi_decode_planned")
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    _check_tokens(L, xs, y.cpu().numpy(), idx.cpu().numpy(), cnt.cpu().numpy(), path, res)


def test_paths_the_batch_does_not_allow_are_refused(layer):
    L, desc, w, _ = layer
    x = torch.zeros((4, D_), device=DEV)
    y = torch.empty((4, D_), device=DEV)
    st = zeros_i32(1, DEV)
    ws = pi.workspace(desc, 4, DEV)
    assert pi.pi_decode_planned(desc, w, pi.PI_PATH_FUSED, x, 4, y, None, None, None, st,
                                ws) == pi.PI_ERR_SHAPE
    assert pi.pi_decode_planned(desc, w, pi.PI_PATH_UNION, x, 1, y, None, None, None, st,
                                ws) == pi.PI_ERR_SHAPE
    assert pi.pi_decode_planned(desc, w, 7, x, 1, y, None, None, None, st, ws) == pi.PI_ERR_SHAPE


@pytest.mark.parametrize("density,allow_dense", [(0.05, 0), (0.05, 1), (0.6, 1)])
def test_decoder_runs_its_plan_and_replays_the_graph(layer, density, allow_dense):
    L, desc, w, _ = layer
    xs_h = synth.gen_x(44, 0, 32, D_)
    res_h = synth.gen_x(45, 0, 32, D_)
    x = up(xs_h, DEV)
    res = up(res_h, DEV)
    y = torch.empty((32, D_), device=DEV)
    st = zeros_i32(1, DEV)
    ws = pi.workspace(desc, 32, DEV)
    rc, dec = pi.pi_decoder_create(desc, w, None, density, allow_dense, None, x, y, res, st, ws)
    pi.check(rc, "pi_decoder_create")
    try:
        for batch in (1, 4, 16):
            plan = pi.pi_plan()
            pi.check(pi.pi_decoder_plan(dec, batch, plan))
            if not allow_dense:
                assert plan.path != pi.PI_PATH_DENSE
            outs = []
            for rep in range(3):  # direct + capture, then two graph replays
                y.fill_(float("nan"))
                pi.check(pi.pi_decoder_run(dec, batch), "pi_decoder_run")
                torch.cuda.synchronize()
                assert int(st[0]) == 0
                outs.append(y[:batch].cpu().numpy().copy())
            np.testing.assert_array_equal(outs[1], outs[0])
            np.testing.assert_array_equal(outs[2], outs[0])
            # the same path called directly gives the same bits
            yd = torch.empty((batch, D_), device=DEV)
            idx = torch.full((batch, N_), -1, dtype=torch.int32, device=DEV)
            cnt = zeros_i32(batch, DEV)
            ws2 = pi.workspace(desc, batch, DEV)
            pi.check(pi.pi_decode_planned(desc, w, plan.path, x, batch, yd, res, idx, cnt, st,
                                          ws2))
            torch.cuda.synchronize()
            np.testing.assert_array_equal(yd.cpu().numpy(), outs[0])
            _check_tokens(L, xs_h[:batch], outs[0], idx.cpu().numpy(), cnt.cpu().numpy(),
                          plan.path, res_h[:batch])
    finally:
        pi.pi_decoder_destroy(dec)


def test_decoder_creation_checks_its_arguments(layer):
    L, desc, w, _ = layer
    x = torch.zeros((32, D_), device=DEV)
    st = zeros_i32(1, DEV)
    small = pi.workspace(desc, 4, DEV)
    rc, dec = pi.pi_decoder_create(desc, w, None, 0.05, 0, None, x, x, None, st, small)
    assert rc == pi.PI_ERR_WORKSPACE and dec == 0
    ws = pi.workspace(desc, 32, DEV)
    rc, dec = pi.pi_decoder_create(desc, w, None, 1.5, 0, None, x, x, None, st, ws)
    assert rc == pi.PI_ERR_SHAPE and dec == 0
