"""pi_layer_decode_static: the one-token decode for callers that cannot
allocate device memory (a plugin inside a framework that owns all device
memory, or a loop that must not call cudaMalloc).  It uses the library's
fixed scratch array instead of a caller workspace; its results must match
pi_layer_decode's, call after call, since every call reuses the same array.

Collected last on purpose (test_zz_*): if it fails, a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import activation_sparse_decode_rank_gb300 as pi
import synth
from pihelp import DevLayer, Y_TOL, up, y_rel_err, zeros_i32

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    pi.build()
    yield


def _run(D, x, static):
    L = D.L
    xd = up(x, DEV)
    y = torch.full((1, L.d), float("nan"), device=DEV)
    idx = torch.full((1, L.n), -1, dtype=torch.int32, device=DEV)
    cnt = zeros_i32(1, DEV)
    st = zeros_i32(1, DEV)
    if static:
        rc = pi.pi_layer_decode_static(D.desc, D.w, xd, y, None, idx, cnt, st)
    else:
        rc = pi.pi_layer_decode(D.desc, D.w, xd, 1, y, None, idx, cnt, st, D.workspace(1))
    pi.check(rc, "decode")
    torch.cuda.synchronize()
    c = int(cnt[0])
    return y[0].cpu().numpy(), idx[0, :c].cpu().numpy(), int(st[0])


@pytest.mark.parametrize("shape", [(1024, 4096, 64, "f16", False, 0.8, 0.08, 1),
                                   (4096, 16384, 128, "f16", False, 0.9, 0.06, 2),
                                   (4096, 11008, 256, "bf16", True, 1.0, 0.10, 3)])
def test_static_scratch_matches_workspace_call(shape):
    d, n, r, dt, g, a, rho, seed = shape
    L = synth.make_layer(d, n, r, dt, gated=g, alpha=a, density=rho, seed=seed)
    D = DevLayer(L, DEV, hot_prefix=n // 40, packed=True)
    for step in range(2):  # two calls in a row share the fixed array
        x = synth.gen_x(seed + 77, step, 1, d)
        y0, i0, s0 = _run(D, x, static=False)
        y1, i1, s1 = _run(D, x, static=True)
        assert s0 == 0 and s1 == 0
        # the same kernel, grid and summation order on both calls: identical
        # bits (a stale or aliased region of the shared array would show here)
        np.testing.assert_array_equal(i1, i0)
        np.testing.assert_array_equal(y1, y0)
        # and the result itself within the oracle tolerance on the GPU's list
        assert y_rel_err(L, x[0], i0, y0) <= Y_TOL


def test_static_scratch_rejects_too_large_a_shape_on_the_gpu():
    # the rejection happens on the host; every pointer is a real buffer of
    # this test (small: the shape is refused before anything is launched)
    d, n, r = 8192, pi.PI_STATIC_SCRATCH_BYTES, 64
    desc = pi.make_desc(d, n, r, "f16")
    buf = torch.zeros(4096, dtype=torch.float32, device=DEV)
    w = pi.make_weights(buf, buf, buf, buf, buf, None)
    st = zeros_i32(1, DEV)
    rc = pi.pi_layer_decode_static(desc, w, buf, buf, None, None, None, st)
    assert rc == pi.PI_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert int(st[0]) == 0
