"""Pins of the fp64 oracle to things other than itself (no GPU).

Each oracle function is checked against at least one of: a hand-worked
example (tests/golden), an exhaustive or brute-force enumeration, a library
routine computing the same quantity another way, or a closed-form identity
of the seeded construction.  The choices are meant to catch a dropped term,
a wrong sign or index, or a transposed operand anywhere in the oracle.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _to_bits(vals, dtype):
    v = np.asarray(vals, np.float64)
    if dtype == "f16":
        out = v.astype(np.float16)
        assert np.array_equal(out.astype(np.float64), v), "fixture value not exact in fp16"
        return out.view(np.uint16)
    f = v.astype(np.float32)
    b = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((b.astype(np.uint32) << 16).view(np.float32).astype(np.float64), v)
    return b


def _golden_layer(g, dtype, gated):
    n, d = g["n"], g["d"]
    W1 = _to_bits(g["W1"], dtype).reshape(n, d)
    if gated:
        W1 = np.ascontiguousarray(np.stack([W1, _to_bits(g["Wup"], dtype).reshape(n, d)], axis=1))
    return synth.Layer(d, n, g["r"], dtype, gated,
                       _to_bits(g["A"], dtype).reshape(n, g["r"]),
                       _to_bits(g["Bm"], dtype).reshape(g["r"], d),
                       np.asarray(g["b1"], np.float32), W1,
                       _to_bits(g["W2"], dtype).reshape(n, d),
                       np.asarray(g["b2"], np.float32))


def _f64(bits, dtype):
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ----------------------------------------------------------- decode
def test_decode_f16_exhaustive_vs_numpy():
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode_half(b, "f16")
    want = b.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    np.testing.assert_array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], want[~nan])
    np.testing.assert_array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_decode_bf16_exhaustive_vs_fp32_bits():
    b = np.arange(65536, dtype=np.uint32)
    got = oracle.decode_half(b.astype(np.uint16), "bf16")
    with np.errstate(invalid="ignore"):  # the NaN patterns widen as NaN
        want = (b << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(want)
    np.testing.assert_array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], want[~nan])


# ----------------------------------------------------------- golden
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_hand_worked_example(dtype):
    g = json.load(open(os.path.join(GOLD, "tiny_ffn_d4_n8_r2.json")))
    e = g["expect"]
    x = np.asarray(g["x"], np.float32)
    L = _golden_layer(g, dtype, gated=False)
    u, lg = oracle.predict(L, x)
    np.testing.assert_array_equal(u[0], e["u"])
    np.testing.assert_array_equal(lg[0], e["logits"])
    idx = oracle.compact(lg[0])
    np.testing.assert_array_equal(idx, e["idx"])
    np.testing.assert_array_equal(oracle.hidden(L, x, idx), e["h_plain"])
    np.testing.assert_array_equal(oracle.sparse_ffn(L, x, idx), e["y_plain"])
    np.testing.assert_array_equal(oracle.dense_ffn(L, x), e["y_dense_plain"])
    lg2, idx2, y2, xn = oracle.layer_decode(L, x, residual=True)
    np.testing.assert_array_equal(idx2, e["idx"])
    np.testing.assert_array_equal(y2, e["y_plain"])
    np.testing.assert_array_equal(xn, np.asarray(e["x_next_plain"], np.float32))
    G = _golden_layer(g, dtype, gated=True)
    np.testing.assert_array_equal(oracle.hidden(G, x, idx), e["h_gated"])
    np.testing.assert_array_equal(oracle.sparse_ffn(G, x, idx), e["y_gated"])
    np.testing.assert_array_equal(oracle.dense_ffn(G, x), e["y_dense_gated"])
    # no b2: the same sums without the bias
    L.b2 = None
    np.testing.assert_array_equal(oracle.sparse_ffn(L, x, idx),
                                  np.asarray(e["y_plain"]) - np.asarray(g["b2"]))


# ----------------------------------------------------------- compaction
def test_compact_exhaustive_n12():
    n = 12
    for m in range(1 << n):
        bits = [(m >> i) & 1 for i in range(n)]
        lg = np.array([1.0 if b else -1.0 for b in bits])
        idx = oracle.compact(lg)
        assert list(idx) == [i for i in range(n) if bits[i]]
        assert len(idx) == bin(m).count("1")


def test_compact_strict_threshold_and_specials():
    lg = np.array([0.0, -0.0, 1e-300, -1e-300, np.nan, np.inf, -np.inf, 5e-324])
    assert list(oracle.compact(lg)) == [2, 5, 7]
    assert len(oracle.compact(np.zeros(0))) == 0


def test_union_matches_set_union():
    rng = np.random.default_rng(4)
    for batch in (1, 3, 32):
        lg = rng.standard_normal((batch, 300)) - 1.2
        uidx, mask = oracle.union(lg)
        sets = [set(np.nonzero(lg[t] > 0)[0].tolist()) for t in range(batch)]
        assert list(uidx) == sorted(set().union(*sets))
        for k, i in enumerate(uidx):
            assert int(mask[k]) == sum(1 << t for t in range(batch) if i in sets[t])


# ----------------------------------------------------------- FFN vs BLAS
@pytest.mark.parametrize("dtype,gated", [("f16", False), ("bf16", False), ("bf16", True)])
def test_dense_ffn_equals_textbook_gemv_pair(dtype, gated):
    """Full density reduces to the dense FFN, computed here by numpy's
    matrix-vector products from the decoded weights."""
    L = synth.make_layer(192, 384, 24, dtype, gated=gated, alpha=0.9, density=0.2, seed=21)
    x = synth.gen_x(21, 0, 1, 192)[0]
    W1 = _f64(L.W1, dtype)
    W2 = _f64(L.W2, dtype)
    xd = x.astype(np.float64)
    if gated:
        g = W1[:, 0, :] @ xd + L.b1
        up = W1[:, 1, :] @ xd
        h = np.maximum(g, 0.0) * up
    else:
        h = np.maximum(W1 @ xd + L.b1, 0.0)
    want = W2.T @ h + L.b2
    got = oracle.dense_ffn(L, x)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12 * max(1.0, np.abs(want).max()))
    # and the hidden vector itself, on an arbitrary neuron list
    idx = np.array([0, 5, 17, 383, 100], np.int32)
    np.testing.assert_allclose(oracle.hidden(L, x, idx), h[idx], rtol=0, atol=1e-12)
    np.testing.assert_allclose(oracle.down(L, idx, h[idx]), W2[idx].T @ h[idx] + L.b2,
                               rtol=0, atol=1e-12)


def test_predict_equals_blas_low_rank_product():
    L = synth.make_layer(160, 320, 24, "f16", alpha=0.9, density=0.1, seed=22)
    x = synth.gen_x(22, 3, 2, 160)
    u, lg = oracle.predict(L, x)
    A = _f64(L.A, "f16")
    B = _f64(L.Bm, "f16")
    U = x.astype(np.float64) @ B.T
    np.testing.assert_allclose(u, U, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lg, U @ A.T + L.b1, rtol=0, atol=1e-12)


# ----------------------------------------------------------- identities
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_predictor_equals_preactivation_without_noise(dtype):
    """With zero noise W1 = round(A Bm), so the predictor logit A(Bm x) + b1
    and the up-projection pre-activation W1 x + b1 differ only by the
    rounding of A, Bm and W1 to 16 bits:
      |logit_i - pre_i| <= sum_j |x_j| ((2u + u^2)/(1-u)^2 sum_k |A_ik||Bm_kj|
                                        + u/(1-u) |W1_ij|)
    with u the unit roundoff (2^-11 fp16, 2^-8 bf16); outside that band the
    two masks must agree exactly."""
    d, n, r = 256, 1024, 32
    L = synth.make_layer(d, n, r, dtype, alpha=0.9, density=0.1, seed=23, noise=0.0)
    u = 2.0**-11 if dtype == "f16" else 2.0**-8
    A = np.abs(_f64(L.A, dtype))
    B = np.abs(_f64(L.Bm, dtype))
    W1 = _f64(L.W1, dtype)
    agree = 0
    for step in range(4):
        x = synth.gen_x(23, step, 1, d)[0]
        _, lg = oracle.predict(L, x)
        pre = W1 @ x.astype(np.float64) + L.b1
        ax = np.abs(x.astype(np.float64))
        band = ((2 * u + u * u) / (1 - u) ** 2) * (A @ (B @ ax)) + (u / (1 - u)) * (np.abs(W1) @ ax)
        band = band * (1 + 1e-9) + 1e-12
        assert np.all(np.abs(lg[0] - pre) <= band)
        clear = np.abs(pre) > band
        np.testing.assert_array_equal(lg[0][clear] > 0, pre[clear] > 0)
        agree += int(clear.sum())
    assert agree > 0.5 * 4 * n


def test_sparse_over_true_relu_set_equals_dense():
    """Over the true ReLU-active set {i : W1_i x + b1_i > 0} the sparse FFN is
    the dense FFN: the neurons left out have h = 0 and contribute nothing."""
    L = synth.make_layer(128, 512, 16, "f16", alpha=0.9, density=0.15, seed=24)
    for step in range(3):
        x = synth.gen_x(24, step, 1, 128)[0]
        pre = _f64(L.W1, "f16") @ x.astype(np.float64) + L.b1
        S = np.nonzero(pre > 0)[0].astype(np.int32)
        assert 0 < len(S) < 512
        np.testing.assert_array_equal(oracle.sparse_ffn(L, x, S), oracle.dense_ffn(L, x))


def test_skipped_neuron_contributes_exactly_zero():
    L = synth.make_layer(128, 512, 16, "bf16", gated=True, alpha=0.9, density=0.15, seed=25)
    x = synth.gen_x(25, 0, 1, 128)[0]
    Wg = _f64(L.W1[:, 0, :], "bf16")
    pre = Wg @ x.astype(np.float64) + L.b1
    S = np.nonzero(pre > 0)[0]
    off = np.nonzero(pre <= 0)[0]
    base = oracle.sparse_ffn(L, x, S.astype(np.int32))
    rng = np.random.default_rng(0)
    for extra in rng.choice(off, size=5, replace=False):
        S2 = np.sort(np.append(S, extra)).astype(np.int32)
        np.testing.assert_array_equal(oracle.sparse_ffn(L, x, S2), base)


def test_neuron_permutation_invariance():
    """Storing the neurons in another order (rows of A, b1, W1, W2 moved
    together, the neuron-table view of placement) maps the active set by the
    permutation and leaves y unchanged up to fp64 summation order."""
    L = synth.make_layer(128, 600, 16, "f16", alpha=0.9, density=0.12, seed=26)
    perm = np.random.default_rng(1).permutation(600)
    P = synth.permute_layer(L, perm)
    for step in range(3):
        x = synth.gen_x(26, step, 1, 128)[0]
        lg, idx, y, _ = oracle.layer_decode(L, x)
        lgp, idxp, yp, _ = oracle.layer_decode(P, x)
        np.testing.assert_array_equal(np.sort(perm[idxp]), idx)
        np.testing.assert_allclose(yp, y, rtol=0, atol=1e-12)
        np.testing.assert_array_equal(lgp, lg[perm])


def test_brute_force_tiny_all_masks():
    """n = 8, d = 4: for every one of the 256 neuron subsets the sparse FFN
    equals a direct sum over the subset computed from decoded weights."""
    L = synth.make_layer(4, 8, 2, "f16", alpha=0.5, density=0.4, seed=27)
    x = synth.gen_x(27, 0, 1, 4)[0].astype(np.float64)
    W1 = _f64(L.W1, "f16")
    W2 = _f64(L.W2, "f16")
    for m in range(256):
        S = [i for i in range(8) if (m >> i) & 1]
        want = np.array(L.b2, np.float64)
        for i in S:
            h = max(0.0, float(W1[i] @ x) + float(L.b1[i]))
            want = want + h * W2[i]
        got = oracle.sparse_ffn(L, x.astype(np.float32), np.array(S, np.int32))
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-14)


def test_expected_active_count_matches_closed_form():
    """For x ~ N(0, I) the logit of neuron i is N(b1_i, ||A_i Bm||^2) given
    the weights, so E[cnt] = sum_i Phi(b1_i / ||A_i Bm||).  The oracle's mean
    count over many fresh steps must sit within 5 standard errors."""
    from scipy.stats import norm
    d, n, r = 256, 2048, 32
    L = synth.make_layer(d, n, r, "f16", alpha=0.9, density=0.08, seed=28)
    AB = _f64(L.A, "f16") @ _f64(L.Bm, "f16")
    s = np.sqrt((AB * AB).sum(axis=1))
    p = norm.cdf(L.b1.astype(np.float64) / s)
    steps = 400
    X = synth.gen_x(28, 0, steps, d)
    _, lg = oracle.predict(L, X)
    cnt = (lg > 0).sum(axis=1)
    sd = math.sqrt(float((p * (1 - p)).sum()) / steps)
    assert abs(cnt.mean() - p.sum()) < 5 * sd
    # per-neuron frequency follows the hot-first profile
    freq = (lg > 0).mean(axis=0)
    assert freq[:16].mean() > 0.6 and freq[-512:].mean() < 0.05


def test_layer_decode_composes_predict_compact_sparse():
    L = synth.make_layer(256, 1024, 32, "bf16", gated=True, alpha=1.0, density=0.1, seed=29)
    x = synth.gen_x(29, 0, 1, 256)[0]
    lg, idx, y, xn = oracle.layer_decode(L, x, residual=True)
    _, lg2 = oracle.predict(L, x)
    np.testing.assert_array_equal(lg, lg2[0])
    np.testing.assert_array_equal(idx, oracle.compact(lg))
    np.testing.assert_array_equal(y, oracle.sparse_ffn(L, x, idx))
    np.testing.assert_array_equal(xn, (x.astype(np.float64) + y).astype(np.float32))


def test_thread_count_does_not_change_results():
    L = synth.make_layer(256, 1024, 32, "f16", alpha=0.9, density=0.1, seed=30)
    x = synth.gen_x(30, 0, 1, 256)[0]
    prev = oracle.get_threads()
    try:
        oracle.set_threads(1)
        a = oracle.layer_decode(L, x)
        b1 = oracle.dense_ffn(L, x)
        oracle.set_threads(max(2, prev))
        b = oracle.layer_decode(L, x)
        b2 = oracle.dense_ffn(L, x)
    finally:
        oracle.set_threads(prev)
    for u, v in zip(a[:3], b[:3]):
        np.testing.assert_array_equal(u, v)
    np.testing.assert_array_equal(b1, b2)


# ---------------------------------------------------------------- offline placement
def test_profile_counts_brute_force():
    rng = np.random.default_rng(7)
    lg = rng.standard_normal((5, 37))
    lg[0, :4] = [0.0, -0.0, 1e-300, -1e-300]  # only the positive one counts
    c = oracle.profile_counts(lg)
    want = [sum(1 for t in range(5) if lg[t, i] > 0) for i in range(37)]
    assert c.tolist() == want
    assert c[0] == sum(1 for t in range(1, 5) if lg[t, 0] > 0)
    # counts accumulate over calls
    c2 = oracle.profile_counts(lg, c)
    assert c2.tolist() == [2 * v for v in want]


def test_hot_order_hand_worked():
    # counts 3 5 5 0 3 7 -> 7 (neuron 5), then the two 5s by index (1, 2),
    # the two 3s (0, 4), then 0 (3)
    assert oracle.hot_order(np.array([3, 5, 5, 0, 3, 7])).tolist() == [5, 1, 2, 0, 4, 3]
    assert oracle.hot_order(np.zeros(6)).tolist() == list(range(6))
    assert oracle.hot_order(np.array([9])).tolist() == [0]


def test_hot_order_properties_with_many_ties():
    rng = np.random.default_rng(8)
    c = rng.integers(0, 6, 2000).astype(np.uint32)
    p = oracle.hot_order(c)
    assert sorted(p.tolist()) == list(range(2000))          # a permutation
    cp = c[p]
    assert np.all(np.diff(cp.astype(np.int64)) <= 0)        # hot first
    same = np.diff(cp.astype(np.int64)) == 0
    assert np.all(np.diff(p)[same] > 0)                     # ties keep index order
    want = [i for _, i in sorted((-int(v), i) for i, v in enumerate(c))]
    assert p.tolist() == want


def test_permute_rows_and_inverse():
    rng = np.random.default_rng(9)
    rows = rng.integers(0, 2**16, (50, 24)).astype(np.uint16)
    perm = rng.permutation(50).astype(np.int32)
    out = oracle.permute_rows(rows, perm)
    for k in range(50):
        assert np.array_equal(out[k], rows[perm[k]])
    inv = np.empty_like(perm)
    inv[perm] = np.arange(50, dtype=np.int32)
    assert np.array_equal(oracle.permute_rows(out, inv), rows)
    b = rng.standard_normal(50).astype(np.float32)
    assert np.array_equal(oracle.permute_rows(b, perm), b[perm])


def _oracle_permuted(L, perm):
    return synth.Layer(L.d, L.n, L.r, L.dtype, L.gated, oracle.permute_rows(L.A, perm), L.Bm,
                       oracle.permute_rows(L.b1, perm), oracle.permute_rows(L.W1, perm),
                       oracle.permute_rows(L.W2, perm), L.b2, dict(L.meta))


def test_placement_keeps_the_decode_and_maps_the_table():
    # A layer stored in a random order, profiled and placed hot first,
    # decodes to the same y; its active list maps back through the table.
    L = synth.make_layer(64, 300, 8, "f16", alpha=0.9, density=0.2, seed=10)
    rng = np.random.default_rng(10)
    shuf = rng.permutation(300).astype(np.int32)
    Ls = _oracle_permuted(L, shuf)
    xs = synth.gen_x(10, 0, 40, 64)
    _, lg = oracle.predict(Ls, xs)
    perm = oracle.hot_order(oracle.profile_counts(lg))
    Lp = _oracle_permuted(Ls, perm)
    for t in range(3):
        x = synth.gen_x(11, t, 1, 64)[0]
        _, _, ys, _ = oracle.layer_decode(Ls, x)
        lgp, idxp, yp, _ = oracle.layer_decode(Lp, x)
        np.testing.assert_allclose(yp, ys, rtol=0, atol=1e-12 * max(1.0, np.abs(ys).max()))
        _, ids, _, _ = oracle.layer_decode(Ls, x)
        assert sorted(perm[idxp].tolist()) == sorted(ids.tolist())


def test_placement_recovers_hot_first_order():
    # the generated layer is hot first; shuffled, then profiled over 400
    # tokens and placed, the activation rate falls along the new order
    L = synth.make_layer(64, 512, 8, "f16", alpha=0.9, density=0.1, seed=12)
    shuf = np.random.default_rng(12).permutation(512).astype(np.int32)
    Ls = _oracle_permuted(L, shuf)
    c = np.zeros(512, np.uint32)
    for s in range(10):
        _, lg = oracle.predict(Ls, synth.gen_x(12, s, 40, 64))
        c = oracle.profile_counts(lg, c)
    perm = oracle.hot_order(c)
    orig = shuf[perm]              # original (hot-first) index at each placed position
    assert np.mean(orig[:50]) < 0.25 * np.mean(orig[-200:])
    assert np.all(np.diff(c[perm].astype(np.int64)) <= 0)
