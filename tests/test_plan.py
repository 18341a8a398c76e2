"""Density / batch-aware dispatch plan (pi_plan_dispatch): host logic, no GPU.

The expected rows are pinned by exact enumeration over every activation
outcome of a tiny layer and against the union of the oracle's own
predicted masks; the rest checks the byte counts, the availability of each
path, the choice of the cheapest estimate and the error channel.
"""
import itertools

import numpy as np
import pytest

import activation_sparse_decode_rank_gb300 as pi


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pi.build()
    pi.lib()


def plan(desc, batch, p=None, density=0.0, allow_dense=1, model=None):
    out = pi.pi_plan()
    st = pi.pi_plan_dispatch(desc, batch, p, density, allow_dense, model, out)
    return st, out


def test_expected_rows_match_exact_enumeration():
    # every outcome of n neurons x B tokens, each neuron active with its own
    # probability, independently: the mean of |union| and of a token's count
    p = np.array([0.25, 0.5, 0.125, 0.75], dtype=np.float32)
    n, B = p.size, 3
    desc = pi.make_desc(128, n, 8)
    eu = ea = 0.0
    for bits in itertools.product((0, 1), repeat=n * B):
        m = np.array(bits).reshape(B, n)
        pr = np.prod(np.where(m == 1, p, 1 - p).astype(np.float64))
        eu += pr * m.any(axis=0).sum()
        ea += pr * m[0].sum()
    st, out = plan(desc, B, p)
    assert st == pi.PI_OK
    assert out.union_rows == pytest.approx(eu, rel=1e-12)
    assert out.active_rows == pytest.approx(ea, rel=1e-12)


def test_uniform_density_equals_a_flat_profile():
    desc = pi.make_desc(5120, 20480, 192)
    for B in (1, 2, 7, 32):
        for rho in (0.0, 0.02, 0.3, 1.0):
            _, a = plan(desc, B, None, rho)
            _, b = plan(desc, B, np.full(20480, rho, np.float32))
            assert a.union_rows == pytest.approx(b.union_rows, rel=1e-9, abs=1e-6)
            assert a.active_rows == pytest.approx(b.active_rows, rel=1e-9, abs=1e-6)
    _, z = plan(desc, 4, None, 0.0)
    assert z.union_rows == 0.0 and z.active_rows == 0.0
    _, f = plan(desc, 4, None, 1.0)
    assert f.union_rows == 20480 and f.active_rows == 20480


def test_union_grows_with_batch_and_stays_bounded():
    rng = np.random.default_rng(0)
    p = (rng.random(4096) ** 4).astype(np.float32)
    desc = pi.make_desc(1024, 4096, 64)
    prev = 0.0
    for B in range(1, 33):
        _, o = plan(desc, B, p)
        assert o.union_rows >= prev - 1e-9
        assert o.union_rows <= min(4096.0, B * o.active_rows) + 1e-6
        assert o.union_rows >= o.active_rows - 1e-6
        prev = o.union_rows


def test_bytes_and_availability():
    d, n, r = 5120, 20480, 192
    desc = pi.make_desc(d, n, r)
    pred = n * r * 2 + r * d * 2 + 4 * n
    row = 2 * d * 2
    _, o1 = plan(desc, 1, None, 0.1, allow_dense=0)
    assert o1.path == pi.PI_PATH_FUSED
    assert list(o1.est_us)[1:] == [-1.0, -1.0, -1.0]
    assert o1.bytes[pi.PI_PATH_FUSED] == pytest.approx(pred + 0.1 * n * row)
    _, o4 = plan(desc, 4, None, 0.1, allow_dense=1)
    assert o4.est_us[pi.PI_PATH_FUSED] == -1.0
    assert o4.bytes[pi.PI_PATH_PER_TOKEN] == pytest.approx(4 * (pred + 0.1 * n * row))
    assert o4.bytes[pi.PI_PATH_UNION] == pytest.approx(pred + o4.union_rows * row)
    assert o4.bytes[pi.PI_PATH_DENSE] == pytest.approx(n * row)
    gated = pi.make_desc(d, n, r, gated=True)
    _, og = plan(gated, 4, None, 0.1)
    assert og.bytes[pi.PI_PATH_DENSE] == pytest.approx(n * 3 * d * 2)
    odd = pi.make_desc(1000, n, r)  # d % 128 != 0: no union path
    _, oo = plan(odd, 4, None, 0.1)
    assert oo.est_us[pi.PI_PATH_UNION] == -1.0 and oo.path != pi.PI_PATH_UNION


def test_choice_is_the_least_estimate():
    desc = pi.make_desc(5120, 20480, 192)
    for B in (1, 2, 4, 9, 16, 32):
        for rho in (0.01, 0.05, 0.2, 0.6):
            for allow in (0, 1):
                _, o = plan(desc, B, None, rho, allow)
                ok = [(o.est_us[k], k) for k in range(pi.PI_PATHS) if o.est_us[k] >= 0]
                assert o.path == min(ok)[1]
                if not allow:
                    assert o.est_us[pi.PI_PATH_DENSE] == -1.0


def test_estimates_follow_the_model():
    desc = pi.make_desc(4096, 16384, 128)
    m = pi.pi_cost_model()
    pi.pi_default_cost_model(m)
    for t in range(pi.PI_COST_TIERS):
        for k in range(pi.PI_PATHS):
            m.fixed_us[k][t] = 10.0 * (k + 1)
            m.gbs[k][t] = 1000.0 * (t + 1)
    _, o = plan(desc, 5, None, 0.05, 1, m)  # batch 5: tier of batch <= 16 (index 2)
    for k in (pi.PI_PATH_UNION, pi.PI_PATH_DENSE):
        assert o.est_us[k] == pytest.approx(10.0 * (k + 1) + o.bytes[k] / (3000.0 * 1e3))
    # per token: batch x the fused tier-0 estimate of one token
    one = o.bytes[pi.PI_PATH_PER_TOKEN] / 5
    assert o.est_us[pi.PI_PATH_PER_TOKEN] == pytest.approx(5 * (20.0 + one / 1e6))


def test_errors():
    desc = pi.make_desc(4096, 16384, 128)
    out = pi.pi_plan()
    assert pi.pi_plan_dispatch(desc, 0, None, 0.1, 1, None, out) == pi.PI_ERR_SHAPE
    assert pi.pi_plan_dispatch(desc, 33, None, 0.1, 1, None, out) == pi.PI_ERR_SHAPE
    assert pi.pi_plan_dispatch(desc, 4, None, 1.5, 1, None, out) == pi.PI_ERR_SHAPE
    assert pi.pi_plan_dispatch(desc, 4, None, float("nan"), 1, None, out) == pi.PI_ERR_SHAPE
    bad = pi.make_desc(4096, 16384, 7)
    assert pi.pi_plan_dispatch(bad, 4, None, 0.1, 1, None, out) == pi.PI_ERR_SHAPE
    m = pi.pi_cost_model()
    pi.pi_default_cost_model(m)
    m.gbs[pi.PI_PATH_UNION][1] = 0.0
    assert pi.pi_plan_dispatch(desc, 4, None, 0.1, 1, m, out) == pi.PI_ERR_SHAPE
    pi.pi_default_cost_model(m)
    m.tier_max_batch[2] = 2
    assert pi.pi_plan_dispatch(desc, 4, None, 0.1, 1, m, out) == pi.PI_ERR_SHAPE
    L = pi.lib()
    assert L.pi_plan_dispatch(None, 4, None, 0.1, 1, None, out) == pi.PI_ERR_NULL
    assert L.pi_plan_dispatch(desc, 4, None, 0.1, 1, None, None) == pi.PI_ERR_NULL


def test_expected_union_matches_the_oracles_masks():
    # p_i profiled from the oracle's own predicted masks over many tokens;
    # the plan's expected union of B tokens against the mean union measured
    # on other tokens of the same layer (tokens are independent, so the
    # formula holds in expectation; the tolerance covers both samples)
    import oracle
    import synth
    d, n, r = 64, 512, 16
    L = synth.make_layer(d, n, r, "f16", alpha=0.8, density=0.1, seed=31)
    prof = np.concatenate([oracle.predict(L, synth.gen_x(31, s, 64, d))[1] > 0
                           for s in range(64)])
    p = prof.mean(axis=0).astype(np.float32)  # 4096 tokens
    desc = pi.make_desc(d, n, r)
    masks = np.concatenate([oracle.predict(L, synth.gen_x(32, s, 64, d))[1] > 0
                            for s in range(32)])  # 2048 other tokens
    for B in (2, 4, 16):
        groups = masks[: (len(masks) // B) * B].reshape(-1, B, n)
        unions = groups.any(axis=1).sum(axis=1)
        _, o = plan(desc, B, p)
        assert o.union_rows == pytest.approx(unions.mean(), rel=0.03)
        assert o.active_rows == pytest.approx(masks.sum(axis=1).mean(), rel=0.03)


# Measured on a GB300 (bench.py --sweep, OPT-13B-shaped layer d 5120,
# n 20480, r 192, fp16, packed records, Zipf exponent 0.9, seed 5): the
# sparse path's and the dense path's µs per step of B tokens at each
# density.  Batch 1's sparse path is the fused layer kernel, larger
# batches' the union path.
SWEEP_US = {
    # density: {B: (sparse, dense)}
    0.02: {1: (19.4, 72.6), 4: (47.5, 75.9), 16: (75.8, 77.4), 32: (123.0, 83.7)},
    0.05: {1: (22.9, 72.6), 4: (61.7, 76.1), 16: (104.9, 77.4), 32: (181.9, 83.6)},
    0.10: {1: (27.1, 72.9), 4: (81.2, 76.1), 16: (148.2, 77.3), 32: (225.2, 83.4)},
    0.25: {1: (40.8, 72.9), 4: (132.0, 76.4), 16: (192.9, 77.5), 32: (275.4, 83.7)},
    0.50: {1: (66.9, 73.4), 4: (175.1, 76.6), 16: (219.2, 77.6), 32: (276.5, 84.0)},
}


@pytest.mark.parametrize("rho", sorted(SWEEP_US))
def test_default_model_picks_the_measured_faster_path(rho):
    # the built-in constants against the sweep they were fitted to: at every
    # measured point the plan names the path that ran faster, and its
    # estimate of that path lies within 10 % of the measurement
    import synth

    d, n, r, alpha = 5120, 20480, 192, 0.9
    pz = synth.zipf_probs(n, alpha, synth.zipf_calibrate(n, alpha, rho))
    desc = pi.make_desc(d, n, r, "f16", False, int((pz >= 0.5).sum()), packed=True)
    for B, (sparse_us, dense_us) in SWEEP_US[rho].items():
        st, o = plan(desc, B, pz.astype(np.float32), 0.0, 1)
        assert st == pi.PI_OK
        sp = pi.PI_PATH_FUSED if B == 1 else pi.PI_PATH_UNION
        want = pi.PI_PATH_DENSE if dense_us < sparse_us else sp
        assert o.path == want, (rho, B, [o.est_us[k] for k in range(pi.PI_PATHS)])
        meas = min(sparse_us, dense_us)
        assert o.est_us[want] == pytest.approx(meas, rel=0.10), (rho, B)
