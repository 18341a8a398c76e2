"""GPU parity of every C-ABI entry point against the fp64 oracle.

Workloads: the tiny ReLU layer and the OPT-6.7B-, Llama-2-7B- (gated) and
OPT-30B-shaped layers at full size, a ragged layer whose sizes are not
multiples of the tiles, and batched predictor cases of the OPT-13B shape.
"""
import math

import numpy as np
import pytest
import torch

import activation_sparse_decode_rank_gb300 as pi
import oracle
import synth
from pihelp import DevLayer, Y_TOL, check_active_set, near_ties, up, y_rel_err, zeros_i32

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")

# (name, d, n, r, dtype, gated, alpha, density, seed, hot_prefix)
WL = {
    "tiny_d1024_n4096": (1024, 4096, 64, "f16", False, 0.8, 0.08, 1, 90),
    "ragged_d200_n1001_r24": (200, 1001, 24, "bf16", False, 0.9, 0.10, 11, 37),
    "ragged_gated_d136_n777_r16": (136, 777, 16, "f16", True, 1.0, 0.12, 12, 0),
    "opt6.7b_d4096_n16384": (4096, 16384, 128, "f16", False, 0.9, 0.06, 2, 304),
    "llama2_7b_gated_d4096_n11008": (4096, 11008, 256, "bf16", True, 1.0, 0.10, 3, 463),
    "opt30b_layer_d7168_n28672": (7168, 28672, 256, "f16", False, 0.9, 0.09, 4, 800),
}
_host = {}
_dev = {}


def layer(name):
    """The named layer on the GPU (host copies are kept; one device copy)."""
    if name not in _dev:
        d, n, r, dt, g, a, rho, seed, hot = WL[name]
        if name not in _host:
            _host[name] = synth.make_layer(d, n, r, dt, gated=g, alpha=a, density=rho, seed=seed)
        _dev.clear()
        torch.cuda.empty_cache()
        _dev[name] = DevLayer(_host[name], DEV, hot_prefix=hot)
    return _dev[name]


def logits_bound(L, x, u_ref, split=False):
    """fp32 error bound of the GPU logits: stage-1 dot products of length d,
    stage-2 of length r (+ bias), gamma_K = K u / (1 - K u), u = 2^-24.
    split: stage 2 ran on the tensor cores with u as a high + low 16-bit
    pair (batch > 1), which leaves |u - hi - lo| <= 2^-22 |u| (+ 2^-25 for
    the f16 subnormal range of lo) for f16 and 2^-16 |u| for bf16."""
    uu = 2.0**-24
    g = lambda k: k * uu / (1 - k * uu)
    dec = (lambda b: b.view(np.float16).astype(np.float64)) if L.dtype == "f16" else \
        (lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64))
    A = np.abs(dec(L.A))
    B = np.abs(dec(L.Bm))
    du = g(L.d) * (B @ np.abs(x.astype(np.float64)))
    au = np.abs(u_ref)
    if split:
        du = du + (2.0**-22 * au + 2.0**-25 if L.dtype == "f16" else 2.0**-16 * au)
    return 2.0 * (A @ du + g(L.r + 1) * (A @ au + np.abs(L.b1))) + 1e-30


# ---------------------------------------------------------------- predictor
@pytest.mark.parametrize("name", ["tiny_d1024_n4096", "ragged_d200_n1001_r24",
                                  "opt6.7b_d4096_n16384", "llama2_7b_gated_d4096_n11008"])
@pytest.mark.parametrize("batch", [1, 5])
def test_predict_parity(name, batch):
    D = layer(name)
    L = D.L
    x = synth.gen_x(100 + batch, 0, batch, L.d)
    lg = torch.empty((batch, L.n), dtype=torch.float32, device=DEV)
    ws = D.workspace(batch)
    pi.check(pi.pi_predict(D.desc, D.A, D.Bm, D.b1, up(x, DEV), batch, lg, ws), "pi_predict")
    torch.cuda.synchronize()
    g = lg.cpu().numpy().astype(np.float64)
    u, lo = oracle.predict(L, x)
    split = batch > 1 and L.r % 16 == 0  # the batched predictor's tensor-core stage 2
    for t in range(batch):
        bound = logits_bound(L, x[t], u[t], split)
        assert np.all(np.abs(g[t] - lo[t]) <= bound)
        tie = near_ties(lo[t])
        np.testing.assert_array_equal((g[t] > 0)[~tie], (lo[t] > 0)[~tie])


def test_predict_batch32_opt13b_shape():
    L = synth.make_layer(5120, 20480, 192, "f16", alpha=0.9, density=0.05, seed=5)
    D = DevLayer(L, DEV)
    x = synth.gen_x(5, 0, 32, 5120)
    lg = torch.empty((32, L.n), dtype=torch.float32, device=DEV)
    pi.check(pi.pi_predict(D.desc, D.A, D.Bm, D.b1, up(x, DEV), 32, lg, D.workspace(32)))
    torch.cuda.synchronize()
    g = lg.cpu().numpy().astype(np.float64)
    u, lo = oracle.predict(L, x)
    for t in (0, 13, 31):
        assert np.all(np.abs(g[t] - lo[t]) <= logits_bound(L, x[t], u[t], split=True))
        tie = near_ties(lo[t])
        np.testing.assert_array_equal((g[t] > 0)[~tie], (lo[t] > 0)[~tie])


# ---------------------------------------------------------------- compaction
def _compact(lg_host, cap, union=False, dev_status=True, grid=False):
    """grid: pass a workspace, so that the grid-wide compaction runs (else
    the one-block-per-token kernels)."""
    batch, n = lg_host.shape
    lg = up(lg_host.astype(np.float32), DEV)
    idx = torch.full((batch, max(cap, 1)), -7, dtype=torch.int32, device=DEV)
    cnt = zeros_i32(batch, DEV)
    st = zeros_i32(1, DEV)
    ui = torch.full((n,), -7, dtype=torch.int32, device=DEV) if union else None
    uc = zeros_i32(1, DEV) if union else None
    tm = torch.zeros(n, dtype=torch.int32, device=DEV) if union else None
    ws = pi.workspace(pi.make_desc(8, n, 8), batch, DEV) if grid else None
    pi.check(pi.pi_compact(lg, n, batch, idx, cnt, cap, ui, uc, tm, st if dev_status else None,
                           ws, ws.numel() if grid else 0))
    torch.cuda.synchronize()
    out = dict(idx=idx.cpu().numpy(), cnt=cnt.cpu().numpy()[:batch], status=int(st[0]))
    if union:
        c = int(uc[0])
        out.update(uidx=ui.cpu().numpy()[:c], tmask=tm.cpu().numpy().view(np.uint32)[:c])
    return out


@pytest.mark.parametrize("grid", [False, True])
@pytest.mark.parametrize("n", [1, 31, 255, 256, 257, 1023, 1024, 1025, 4096, 28672, 100003])
def test_compact_bit_exact(n, grid):
    rng = np.random.default_rng(n)
    for density in (0.0, 0.07, 0.5, 1.0):
        lg = np.where(rng.random((3, n)) < density, rng.random((3, n)) + 1e-3,
                      -rng.random((3, n))).astype(np.float32)
        lg[:, : min(n, 3)] = [0.0, -0.0, 1e-38][: min(n, 3)]  # zeros are inactive
        o = _compact(lg, n, grid=grid)
        assert o["status"] == 0
        for t in range(3):
            want = oracle.compact(lg[t].astype(np.float64))
            assert o["cnt"][t] == len(want)
            np.testing.assert_array_equal(o["idx"][t][: len(want)], want)


@pytest.mark.parametrize("grid", [False, True])
def test_compact_capacity_overflow_reported(grid):
    lg = np.ones((2, 5000), np.float32)
    lg[1, ::2] = -1.0
    o = _compact(lg, 1000, grid=grid)
    assert o["status"] == pi.PI_ERR_CAPACITY
    assert list(o["cnt"]) == [5000, 2500]
    np.testing.assert_array_equal(o["idx"][0], np.arange(1000))
    np.testing.assert_array_equal(o["idx"][1], np.arange(1, 2001, 2))


@pytest.mark.parametrize("grid", [False, True])
@pytest.mark.parametrize("batch", [1, 4, 16, 32])
def test_union_bit_exact(batch, grid):
    rng = np.random.default_rng(batch)
    for n in (20480, 777):
        lg = (rng.standard_normal((batch, n)) - 1.8).astype(np.float32)
        o = _compact(lg, n, union=True, grid=grid)
        want_i, want_m = oracle.union(lg.astype(np.float64))
        np.testing.assert_array_equal(o["uidx"], want_i)
        np.testing.assert_array_equal(o["tmask"], want_m)
        for t in range(batch):  # and every token's own list
            want = oracle.compact(lg[t].astype(np.float64))
            assert o["cnt"][t] == len(want)
            np.testing.assert_array_equal(o["idx"][t][: len(want)], want)


# ---------------------------------------------------------------- sparse / dense FFN
def _sparse(D, x, idx_list, cap=None):
    L = D.L
    cap = L.n if cap is None else cap
    idx = torch.zeros(max(cap, 1), dtype=torch.int32, device=DEV)
    k = min(len(idx_list), cap)
    if k:
        idx[:k] = torch.from_numpy(np.asarray(idx_list[:k], np.int32)).to(DEV)
    cnt = torch.tensor([len(idx_list), 0, 0, 0], dtype=torch.int32, device=DEV)
    y = torch.full((1, L.d), float("nan"), device=DEV)
    st = zeros_i32(1, DEV)
    pi.check(pi.pi_sparse_ffn(D.desc, D.w, up(x, DEV), 1, idx, cnt, cap, None, None, None, y, st,
                              D.workspace()))
    torch.cuda.synchronize()
    return y[0].cpu().numpy(), int(st[0])


@pytest.mark.parametrize("name", list(WL))
def test_sparse_ffn_parity(name):
    D = layer(name)
    L = D.L
    x = synth.gen_x(7, 0, 1, L.d)
    _, lo = oracle.predict(L, x)
    idx = oracle.compact(lo[0])
    y, st = _sparse(D, x, idx)
    assert st == 0
    assert y_rel_err(L, x, idx, y) <= Y_TOL


def test_sparse_ffn_edge_lists():
    D = layer("ragged_d200_n1001_r24")
    L = D.L
    x = synth.gen_x(8, 0, 1, L.d)
    # empty list: y = b2
    y, st = _sparse(D, x, [])
    assert st == 0
    np.testing.assert_array_equal(y, L.b2)
    # every neuron (dense through the sparse operator)
    y, st = _sparse(D, x, np.arange(L.n))
    assert st == 0 and y_rel_err(L, x, np.arange(L.n), y) <= Y_TOL
    # one neuron, the last one
    y, st = _sparse(D, x, [L.n - 1])
    assert st == 0 and y_rel_err(L, x, [L.n - 1], y) <= Y_TOL
    # more active than the list holds: reported, nothing computed
    y, st = _sparse(D, x, np.arange(50), cap=20)
    assert st == pi.PI_ERR_CAPACITY
    # an entry outside [0, n) is reported and skipped, never read
    y, st = _sparse(D, x, [3, L.n, 7])
    assert st == pi.PI_ERR_INDEX
    y2, _ = _sparse(D, x, [3, 7])
    np.testing.assert_array_equal(y, y2)


@pytest.mark.parametrize("name", ["tiny_d1024_n4096", "ragged_gated_d136_n777_r16",
                                  "opt6.7b_d4096_n16384", "llama2_7b_gated_d4096_n11008"])
def test_dense_ffn_parity(name):
    D = layer(name)
    L = D.L
    batch = 2
    x = synth.gen_x(9, 0, batch, L.d)
    y = torch.empty((batch, L.d), device=DEV)
    pi.check(pi.pi_dense_ffn(D.desc, D.w, up(x, DEV), batch, y, D.workspace(batch)))
    torch.cuda.synchronize()
    for t in range(batch):
        yd = oracle.dense_ffn(L, x[t])
        err = float(np.abs(y[t].cpu().numpy() - yd).max()) / float(np.abs(yd).max())
        assert err <= Y_TOL


# ---------------------------------------------------------------- fused decode
def _decode(D, x, batch=1, residual=None, want_idx=True):
    L = D.L
    xd = up(x, DEV)
    y = torch.full((batch, L.d), float("nan"), device=DEV)
    idx = torch.full((batch, L.n), -1, dtype=torch.int32, device=DEV) if want_idx else None
    cnt = zeros_i32(batch, DEV) if want_idx else None
    st = zeros_i32(1, DEV)
    res = xd if residual else None
    pi.check(pi.pi_layer_decode(D.desc, D.w, xd, batch, y, res, idx, cnt, st,
                                D.workspace(batch)), "pi_layer_decode")
    torch.cuda.synchronize()
    out = dict(y=y.cpu().numpy(), status=int(st[0]))
    if want_idx:
        out["cnt"] = cnt.cpu().numpy()[:batch]
        out["idx"] = [idx[t, : out["cnt"][t]].cpu().numpy() for t in range(batch)]
    return out


@pytest.mark.parametrize("name", list(WL))
def test_layer_decode_parity(name):
    D = layer(name)
    L = D.L
    steps = 3 if L.d >= 4096 else 6
    ties = 0
    for s in range(steps):
        x = synth.gen_x(20 + s, s, 1, L.d)
        o = _decode(D, x)
        assert o["status"] == 0
        _, lo = oracle.predict(L, x)
        ties += check_active_set(o["idx"][0], lo[0])
        assert y_rel_err(L, x, o["idx"][0], o["y"][0]) <= Y_TOL
        if not np.any(near_ties(lo[0])):
            # no near-ties: the end-to-end result must match too
            np.testing.assert_array_equal(o["idx"][0], oracle.compact(lo[0]))
    assert ties <= steps * 2


def test_layer_decode_residual_and_hot_prefix_variants():
    D = layer("ragged_d200_n1001_r24")
    L = D.L
    x = synth.gen_x(30, 0, 1, L.d)
    base = _decode(D, x)
    for hot in (0, 1, 500, L.n):
        D.desc.hot_prefix = hot
        o = _decode(D, x, residual=True)
        # the hot prefix only changes what is fetched early, never the result
        np.testing.assert_array_equal(o["idx"][0], base["idx"][0])
        np.testing.assert_allclose(o["y"][0], base["y"][0] + x[0], rtol=0, atol=1e-6)
    D.desc.hot_prefix = WL["ragged_d200_n1001_r24"][-1]
    # without the optional outputs
    o = _decode(D, x, want_idx=False)
    np.testing.assert_array_equal(o["y"][0], base["y"][0])


def test_layer_decode_deterministic():
    D = layer("opt6.7b_d4096_n16384")
    x = synth.gen_x(31, 0, 1, D.L.d)
    a = _decode(D, x)
    b = _decode(D, x)
    np.testing.assert_array_equal(a["y"], b["y"])
    np.testing.assert_array_equal(a["idx"][0], b["idx"][0])


def test_layer_decode_batch_equals_per_token():
    """A batched step gives every token its own mask and the batch-1 result
    (within the tolerance: the batched contraction runs on tensor cores)."""
    D = layer("tiny_d1024_n4096")
    L = D.L
    x = synth.gen_x(32, 0, 4, L.d)
    ob = _decode(D, x, batch=4)
    assert ob["status"] == 0
    for t in range(4):
        o1 = _decode(D, x[t:t + 1])
        _, lo = oracle.predict(L, x[t])
        check_active_set(ob["idx"][t], lo[0])
        yd = oracle.dense_ffn(L, x[t])
        assert float(np.abs(ob["y"][t] - o1["y"][0]).max()) <= Y_TOL * float(np.abs(yd).max())


def test_layer_decode_no_active_neuron():
    L = synth.make_layer(256, 512, 16, "f16", alpha=0.9, density=0.1, seed=33)
    L.b1[:] = -1e4  # every logit is negative
    D = DevLayer(L, DEV)
    x = synth.gen_x(33, 0, 1, 256)
    o = _decode(D, x)
    assert o["status"] == 0 and o["cnt"][0] == 0
    np.testing.assert_array_equal(o["y"][0], L.b2)


def test_layer_decode_in_cuda_graph():
    D = layer("tiny_d1024_n4096")
    L = D.L
    x = up(synth.gen_x(34, 0, 1, L.d), DEV)
    y = torch.empty((1, L.d), device=DEV)
    st = zeros_i32(1, DEV)
    ws = D.workspace()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pi.check(pi.pi_layer_decode(D.desc, D.w, x, 1, y, None, None, None, st, ws, stream=s))
        s.synchronize()
        ref = y.clone()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            pi.check(pi.pi_layer_decode(D.desc, D.w, x, 1, y, None, None, None, st, ws,
                                        stream=s))
        y.zero_()
        for _ in range(3):
            g.replay()
        s.synchronize()
    assert int(st[0]) == 0
    torch.testing.assert_close(y, ref, rtol=0, atol=0)


# ---------------------------------------------------------------- packed layout
@pytest.mark.parametrize("name", ["ragged_d200_n1001_r24", "ragged_gated_d136_n777_r16",
                                  "opt6.7b_d4096_n16384", "llama2_7b_gated_d4096_n11008"])
def test_pack_weights_bit_exact(name):
    D = layer(name)
    L = D.L
    D.set_packed(True)
    try:
        got = D.packed.cpu().numpy().view(np.uint16)
        m1 = 2 if L.gated else 1
        want = np.concatenate([L.W1.reshape(L.n, m1 * L.d), L.W2], axis=1)
        np.testing.assert_array_equal(got, want)
    finally:
        D.set_packed(False)


@pytest.mark.parametrize("name", list(WL))
def test_packed_layout_same_results(name):
    """The packed records hold the same bytes: every entry point gives
    bit-identical outputs on both layouts."""
    D = layer(name)
    L = D.L
    x = synth.gen_x(40, 0, 1, L.d)
    a = _decode(D, x)
    _, lo = oracle.predict(L, x)
    idx = oracle.compact(lo[0])
    ys, _ = _sparse(D, x, idx)
    D.set_packed(True)
    try:
        b = _decode(D, x)
        yp, st = _sparse(D, x, idx)
        assert b["status"] == 0 and st == 0
        np.testing.assert_array_equal(a["y"], b["y"])
        np.testing.assert_array_equal(a["idx"][0], b["idx"][0])
        np.testing.assert_array_equal(ys, yp)
        if L.d <= 4096:
            y = torch.empty((1, L.d), device=DEV)
            pi.check(pi.pi_dense_ffn(D.desc, D.w, up(x, DEV), 1, y, D.workspace()))
            torch.cuda.synchronize()
            yd = oracle.dense_ffn(L, x[0])
            assert float(np.abs(y[0].cpu().numpy() - yd).max()) / float(np.abs(yd).max()) <= Y_TOL
    finally:
        D.set_packed(False)


# ---------------------------------------------------------------- failure path
def test_bounded_wait_times_out_and_reports():
    D = layer("tiny_d1024_n4096")
    ws = D.workspace()
    st = zeros_i32(1, DEV)
    pi.check(pi.pi_selftest_wait_timeout(st, ws, 2_000_000))  # 2 ms
    torch.cuda.synchronize()
    assert int(st[0]) == pi.PI_ERR_TIMEOUT
    # the context is still usable: a fresh workspace decodes normally
    x = synth.gen_x(35, 0, 1, D.L.d)
    o = _decode(D, x)
    assert o["status"] == 0


@pytest.mark.parametrize("packed", [False, True])
def test_ring_wait_times_out_and_returns(packed):
    # every block's first listed neuron is never copied: its ring wait runs
    # out after 2 ms, the block abandons its ring (issuing nothing more and
    # letting what it issued land) and the launch ends within about one bound
    import time
    D = layer("tiny_d1024_n4096")
    D.set_packed(packed)
    L = D.L
    n = L.n
    idx = torch.arange(n, dtype=torch.int32, device=DEV)  # 26+ neurons per block
    cnt = torch.tensor([n, 0, 0, 0], dtype=torch.int32, device=DEV)
    x = up(synth.gen_x(36, 0, 1, L.d), DEV)
    y = torch.empty((1, L.d), device=DEV)
    ws = D.workspace()
    st = zeros_i32(1, DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    pi.check(pi.pi_selftest_ring_timeout(D.desc, D.w, x, idx, cnt, n, y, st, ws, 2_000_000))
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st[0]) == pi.PI_ERR_TIMEOUT
    assert dt < 0.5, f"a timed-out ring took {dt:.3f} s to return"
    # the context is still usable: the same list decodes normally
    ws2 = D.workspace()
    st2 = zeros_i32(1, DEV)
    pi.check(pi.pi_sparse_ffn(D.desc, D.w, x, 1, idx, cnt, n, None, None, None, y, st2, ws2))
    torch.cuda.synchronize()
    assert int(st2[0]) == 0
    xh = synth.gen_x(36, 0, 1, L.d)[0]
    assert y_rel_err(L, xh, np.arange(n, dtype=np.int32), y[0].cpu().numpy()) <= Y_TOL
    D.set_packed(False)
