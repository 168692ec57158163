"""Pins for the oracle: checks against what the paper and mathematics fix.

Nothing here re-types the oracle's own formulas to compare them with
themselves.  The pins are: a library implementation of Philox (cuRAND's host
generator), closed forms of Definition 2, exhaustive enumeration of all 2^|L|
Poisson outcomes on tiny inputs (Theorem 1's MSE, Lemma 1 and Theorem 2
coverage), library softmax / SDPA, identities such as sum r = eta n, values
the paper prints (tests/golden/paper_values.json) and brute force vs closed
form agreement.  Paper: "Verify Before You Fetch: Reliable KV Cache
Compression for LLM Inference".
"""
import ctypes
import ctypes.util
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "paper_values.json")


def golden(key):
    with open(GOLDEN) as f:
        for v in json.load(f)["values"]:
            if v["id"] == key:
                return v
    raise KeyError(key)


# ----------------------------------------------------------------------------- Philox
def _curand():
    for name in ("libcurand.so", "libcurand.so.10"):
        for base in (os.environ.get("CUDA_HOME", "/usr/local/cuda"), "/usr/local/cuda"):
            p = os.path.join(base, "lib64", name)
            if os.path.exists(p):
                return ctypes.CDLL(p)
    p = ctypes.util.find_library("curand")
    if p:
        return ctypes.CDLL(p)
    pytest.skip("libcurand not available")


def _curand_host_stream(cr, seed, offset, count):
    CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161
    g = ctypes.c_void_p()
    assert cr.curandCreateGeneratorHost(ctypes.byref(g), CURAND_RNG_PSEUDO_PHILOX4_32_10) == 0
    try:
        assert cr.curandSetPseudoRandomGeneratorSeed(g, ctypes.c_ulonglong(seed)) == 0
        assert cr.curandSetGeneratorOffset(g, ctypes.c_ulonglong(offset)) == 0
        out = np.zeros(count, np.uint32)
        assert cr.curandGenerate(g, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(count)) == 0
    finally:
        cr.curandDestroyGenerator(g)
    return out


@pytest.mark.parametrize("seed", [0, 0x123456789ABCDEF, 0xFFFFFFFFFFFFFFFF, 42])
@pytest.mark.parametrize("offset", [0, 4 * 5, 4 * ((1 << 20) + 7), 4 * ((1 << 48) + (3 << 16) + 9)])
def test_philox_matches_curand_host_generator(seed, offset):
    """cuRAND's host Philox4x32-10 stream: output block b of the stream is the
    Philox block at key (seed_lo, seed_hi) and counter
    (b >> 16 low word, b >> 48, b & 0xffff, 0)."""
    cr = _curand()
    got = _curand_host_stream(cr, seed, offset, 16)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for i in range(4):
        blk = offset // 4 + i
        ctr = [(blk >> 16) & 0xFFFFFFFF, (blk >> 48) & 0xFFFFFFFF, blk & 0xFFFF, 0]
        assert list(oracle.philox4x32_10(ctr, key)) == list(got[4 * i:4 * i + 4])


def test_uniform_is_top_24_bits():
    for tok in range(50):
        x = oracle.philox4x32_10([tok, 3, 5, 7], [11, 13])[0]
        u = oracle.uniform(11 | (13 << 32), tok, 3, 5, 7)
        assert u == (int(x) >> 8) * 2.0 ** -24
        assert 0.0 <= u < 1.0


# ----------------------------------------------------------------------------- water-filling
def _random_tau(rng, n, kind):
    if kind == "uniform":
        t = rng.random(n)
    elif kind == "heavy":   # a few dominant tokens, as with needles
        t = rng.random(n) ** 8
        t[rng.choice(n, 30, replace=False)] = 1.0
    elif kind == "lognormal":
        t = np.exp(rng.standard_normal(n) * 3)
        t /= t.max()
    else:
        raise ValueError(kind)
    return np.maximum(t, 2.0 ** -38).astype(np.float32)


@pytest.mark.parametrize("kind", ["uniform", "heavy", "lognormal"])
@pytest.mark.parametrize("n,eta", [(1024, 1 / 8), (4099, 1 / 16), (20000, 1 / 32), (777, 0.5)])
def test_waterfill_inclusion_identity_and_bisection(kind, n, eta):
    """Algorithm 1, water-filling step: sum_i min(1, c tau_i) = eta n (to 1e-12), and c agrees
    with an independent plain bisection on c."""
    rng = np.random.default_rng(n)
    tau = _random_tau(rng, n, kind)
    n_sink, n_local = 4, 64
    budget = eta * n
    c, tstar, r64, r32 = oracle.waterfill(tau, n_sink, n_local, budget)
    assert abs(r64.sum() - budget) <= 1e-12 * budget
    forced = np.zeros(n, bool)
    forced[:n_sink] = True
    forced[n - n_local:] = True
    assert np.all(r64[forced] == 1.0)
    assert np.all((r64 > 0) & (r64 <= 1))
    # independent bisection on c in double
    tu = tau[~forced].astype(np.float64)
    target = budget - forced.sum()
    lo, hi = 0.0, 1.0
    while np.minimum(1.0, hi * tu).sum() < target:
        hi *= 2
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if np.minimum(1.0, mid * tu).sum() < target:
            lo = mid
        else:
            hi = mid
    assert abs(c - hi) <= 1e-12 * c
    # the capped tokens are the top t* scores, and they satisfy c tau >= 1
    capped = (~forced) & (r64 == 1.0)
    assert capped.sum() == tstar
    if tstar:
        assert tau[capped].min() >= tau[(~forced) & ~capped].max()


def test_waterfill_equal_scores_closed_form():
    """All scores equal on U: r_i = B'/|U| for every non-forced token."""
    n, n_sink, n_local = 8192, 4, 128
    tau = np.full(n, 0.3, np.float32)
    budget = n / 16
    c, tstar, r64, r32 = oracle.waterfill(tau, n_sink, n_local, budget)
    expect = (budget - n_sink - n_local) / (n - n_sink - n_local)
    u = r64[n_sink:n - n_local]
    assert tstar == 0
    assert np.allclose(u, expect, rtol=1e-15, atol=0)


def test_waterfill_degenerate_budgets():
    n = 512
    tau = np.linspace(0.01, 1, n).astype(np.float32)
    c, t, r64, r32 = oracle.waterfill(tau, 4, 64, n)  # budget covers everything
    assert math.isinf(c) and np.all(r32 == 1.0)
    with pytest.raises(ValueError):
        oracle.waterfill(tau, 4, 64, 68.0)  # budget == forced set


def test_resident_fraction_printed_value():
    """Paper: 16x compression keeps 6.25% of the cache resident (expected size)."""
    g = golden("resident_fraction_percent_16x")
    rng = np.random.default_rng(5)
    n = 32768
    tau = _random_tau(rng, n, "heavy")
    c, t, r64, r32 = oracle.waterfill(tau, 4, 128, n / 16)
    assert abs(100 * r64.sum() / n - g["value"]) <= g["rounding"]


def test_u128_to_double_is_correctly_rounded():
    rng = np.random.default_rng(0)
    for _ in range(2000):
        bits = int(rng.integers(1, 127))
        v = int(rng.integers(0, 2 ** 63)) << 64 | int(rng.integers(0, 2 ** 63))
        v &= (1 << bits) - 1
        assert oracle.u128_to_double(v) == float(v)


# ----------------------------------------------------------------------------- Poisson sample
def test_poisson_sample_frequencies_match_r():
    """Z_i ~ Bernoulli(r_i) independently (Algorithm 1, sampling step): over many seeds
    the empirical inclusion frequency of each token matches r_i."""
    rng = np.random.default_rng(1)
    n = 200
    r = rng.uniform(0.02, 0.98, n).astype(np.float32)
    seeds = 3000
    hits = np.zeros(n)
    for s in range(seeds):
        hits += oracle.poisson_sample(r, seed=s * 7919 + 1, kv_head=0, layer=0, seq=0) == 1
    p = r.astype(np.float64)
    z = (hits - seeds * p) / np.sqrt(seeds * p * (1 - p))
    assert np.abs(z).max() < 4.5          # Bonferroni over 200 tokens
    chi2 = (z ** 2).sum()                 # ~ chi^2_200
    assert chi2 < 200 + 6 * math.sqrt(400)


def test_poisson_sample_counter_fields_are_independent_streams():
    r = np.full(4096, 0.5, np.float32)
    a = oracle.poisson_sample(r, 9, 0, 0, 0)
    for other in [(1, 0, 0), (0, 1, 0), (0, 0, 1)]:
        b = oracle.poisson_sample(r, 9, *other)
        agree = (a == b).mean()
        assert 0.45 < agree < 0.55
    assert np.array_equal(a, oracle.poisson_sample(r, 9, 0, 0, 0))
    r2 = r.copy()
    r2[:10] = 1.0
    f = oracle.poisson_sample(r2, 9, 0, 0, 0)
    assert np.all(f[:10] == 2) and np.all(f[10:] != 2)


# ----------------------------------------------------------------------------- sketches
def test_int8_sketch_hand_example_and_bound():
    K = np.array([[127.0, -64.0, 63.5, 0.5], [0.0, 0.0, 0.0, 0.0]], np.float32)
    codes, scale = oracle.sketch_int8(K)
    assert scale[0] == 1.0 and scale[1] == 0.0
    assert list(codes[0]) == [127, -64, 64, 0]     # round half to even
    assert list(codes[1]) == [0, 0, 0, 0]
    rng = np.random.default_rng(2)
    K = rng.standard_normal((500, 128)).astype(np.float32) * rng.uniform(0.1, 10, (500, 1)).astype(np.float32)
    codes, scale = oracle.sketch_int8(K)
    rec = codes.astype(np.float64) * scale[:, None]
    assert np.all(np.abs(K - rec) <= scale[:, None] * 0.5 * (1 + 1e-6))
    assert np.all(np.abs(codes).max(axis=1) == 127)


def test_2bit_sketch_hand_example_and_bound():
    d, n = 16, 8
    K = np.zeros((n, d), np.float32)
    K[:, 0] = [0, 1, 2, 3, 3, 2, 1, 0]            # pair (0, 8) has the largest energy
    K[:, 8] = [3, 3, 3, 3, 0, 0, 0, 0]
    K[:, 3] = 0.1
    pairs, codes, zero, scale = oracle.sketch_2bit(K, group=8)
    assert list(pairs) == [0, 3]                  # d/8 = 2 pairs
    kept = oracle.kept_channels(pairs, d)
    assert list(kept) == [0, 3, 8, 11]
    assert list(codes[:, 0]) == [0, 1, 2, 3, 3, 2, 1, 0]
    assert list(codes[:, 2]) == [3, 3, 3, 3, 0, 0, 0, 0]
    assert oracle.f16_to_f32(zero[0, 0]) == 0.0 and oracle.f16_to_f32(scale[0, 0]) == 1.0
    rng = np.random.default_rng(3)
    d, n = 128, 1000
    K = (rng.standard_normal((n, d)) * np.linspace(0.2, 3, d)).astype(np.float32)
    pairs, codes, zero, scale = oracle.sketch_2bit(K, group=128)
    energy = (K.astype(np.float64) ** 2)[:, :d // 2] + (K.astype(np.float64) ** 2)[:, d // 2:]
    top = np.sort(np.argsort(-energy.sum(0), kind="stable")[:d // 8])
    assert list(pairs) == list(top)
    kept = oracle.kept_channels(pairs, d)
    zf, sf = oracle.f16_to_f32(zero), oracle.f16_to_f32(scale)
    for g in range((n + 127) // 128):
        blk = K[g * 128:(g + 1) * 128][:, kept].astype(np.float64)
        rec = zf[g].astype(np.float64) + sf[g].astype(np.float64) * codes[g * 128:(g + 1) * 128]
        mn = blk.min(0)
        slack = sf[g] / 2 + 3 * 2.0 ** -11 * sf[g] + 2.0 ** -11 * np.abs(mn) + 1e-6
        assert np.all(np.abs(blk - rec) <= slack)


def test_2bit_sketch_size_matches_printed_fraction():
    """Appendix A.1: the sketch costs 1.76% of the cache (d = 128, bf16 K+V)."""
    g = golden("sketch_fraction_percent")
    d, n, group = 128, 4096, 128
    K = np.random.default_rng(4).standard_normal((n, d)).astype(np.float32)
    pairs, codes, zero, scale = oracle.sketch_2bit(K, group=group)
    assert codes.shape[1] == golden("kept_channels_d128")["value"]
    code_bits = codes.size * 2
    param_bits = (zero.size + scale.size) * 16
    sketch_bytes_per_token = (code_bits + param_bits) / 8 / n
    full_bytes_per_token = 2 * d * 2
    frac = 100 * sketch_bytes_per_token / full_bytes_per_token
    assert abs(frac - g["value"]) <= g["rounding"]
    K256 = np.random.default_rng(4).standard_normal((256, 256)).astype(np.float32)
    assert oracle.sketch_2bit(K256)[1].shape[1] == golden("kept_channels_d256")["value"]


def test_sketch_logits_reduce_to_exact_on_grid_keys():
    """A key that lies on the sketch's grid is reproduced exactly, so its
    sketch logit equals the exact logit (computed with numpy's matmul)."""
    rng = np.random.default_rng(6)
    d, n = 128, 300
    q = rng.standard_normal(d)
    codes = rng.integers(-127, 128, (n, d)).astype(np.int8)
    codes[:, 0] = 127
    scale = rng.uniform(0.01, 0.1, n).astype(np.float32)
    K = codes.astype(np.float64) * scale[:, None].astype(np.float64)
    c2, s2 = oracle.sketch_int8(K.astype(np.float32))
    assert np.array_equal(c2, codes)
    ref = K @ q / math.sqrt(d)
    assert np.allclose(oracle.logits_int8(q, codes, scale), ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(oracle.logits_exact(q, K), ref, rtol=1e-12, atol=1e-12)
    # 2-bit: kept channels on the {0,1,2,3} grid, dropped channels zero
    K2 = np.zeros((256, d), np.float32)
    kept_pairs = np.arange(0, 64, 4)
    ch = np.concatenate([kept_pairs, kept_pairs + 64])
    K2[:, ch] = rng.integers(0, 4, (256, ch.size)) * 2.0 + 1.0
    K2[0, ch] = 1.0
    K2[1, ch] = 7.0
    K2[2:, ch] *= 1.0 + 0 * K2[2:, ch]
    pairs, codes2, zero, sc = oracle.sketch_2bit(K2)
    assert list(pairs) == list(kept_pairs)
    lg = oracle.logits_2bit(q, pairs, codes2, zero, sc)
    assert np.allclose(lg, K2.astype(np.float64) @ q / math.sqrt(d), rtol=1e-12, atol=1e-12)


def test_tau_matches_library_softmax():
    from scipy.special import softmax
    rng = np.random.default_rng(7)
    n, d, rows = 700, 128, 8
    K = rng.standard_normal((n, d)).astype(np.float32)
    Q = rng.standard_normal((rows, d)).astype(np.float32)
    t = oracle.tau(K, Q, 4, 64)
    p = softmax(Q.astype(np.float64) @ K.astype(np.float64).T / math.sqrt(d), axis=1).max(0)
    ref = (p / p.max()).astype(np.float32)
    ref = np.maximum(ref, np.float32(2.0 ** -38))
    ref[:4] = 1
    ref[-64:] = 1
    assert np.allclose(t, ref, rtol=2e-7, atol=0)
    assert t.max() == 1.0


# ----------------------------------------------------------------------------- estimator (Def. 2, Thm. 1)
def _lam(beta, w, r):
    return np.clip(beta * r / (w * (1 - r)), r, 1.0)


def test_beta_closed_forms():
    """|L| = 1: lambda = r, beta = w (1 - r).  m identical tokens:
    lambda = m r / (1 - r + m r)."""
    for w, r in [(1.0, 0.3), (5.0, 0.01), (1e-3, 0.9)]:
        beta = oracle.beta_breakpoints([w], [r])
        assert math.isclose(beta, w * (1 - r), rel_tol=1e-12)
    for m in [2, 3, 10, 1000]:
        for r in [0.05, 0.5, 0.9]:
            w = np.full(m, 2.5)
            rr = np.full(m, r)
            beta = oracle.beta_breakpoints(w, rr)
            lam = _lam(beta, w, rr)
            assert np.allclose(lam, m * r / (1 - r + m * r), rtol=1e-12)


def _mse_enumerated(w, r, lam):
    """E[(D^ - D)^2] over all 2^|L| Poisson outcomes (exact sketch)."""
    L = len(w)
    tot = 0.0
    for z in itertools.product([0, 1], repeat=L):
        z = np.array(z)
        p = np.prod(np.where(z == 1, r, 1 - r))
        err = (z * lam * w / r).sum() - w.sum()
        tot += p * err * err
    return tot


def test_theorem1_minimality_by_enumeration():
    """Theorem 1: the clipped fixed point minimises the exact MSE over
    lambda in [r, 1]^L; random feasible perturbations never lower it, and the
    enumerated MSE equals eq. (6)."""
    rng = np.random.default_rng(8)
    for trial in range(12):
        L = int(rng.integers(1, 9))
        w = np.exp(rng.standard_normal(L) * 2)
        r = rng.uniform(0.02, 0.95, L)
        beta = oracle.beta_breakpoints(w, r)
        lam = _lam(beta, w, r)
        best = _mse_enumerated(w, r, lam)
        eq6 = (w * (1 - lam)).sum() ** 2 + (lam ** 2 * w ** 2 * (1 - r) / r).sum()
        assert math.isclose(best, eq6, rel_tol=1e-10)
        for _ in range(30):
            pert = np.clip(lam + rng.normal(0, 0.05, L), r, 1.0)
            assert _mse_enumerated(w, r, pert) >= best * (1 - 1e-12)
        # KKT: interior coordinates have zero gradient, boundary ones the right sign
        grad = -2 * (w * (1 - lam)).sum() * w + 2 * lam * w ** 2 * (1 - r) / r
        interior = (lam > r + 1e-12) & (lam < 1 - 1e-12)
        assert np.allclose(grad[interior], 0, atol=1e-9 * max(1.0, np.abs(grad).max()))
        assert np.all(grad[lam <= r + 1e-12] >= -1e-9 * max(1.0, np.abs(grad).max()))
        assert np.all(grad[lam >= 1 - 1e-12] <= 1e-9 * max(1.0, np.abs(grad).max()))


def test_beta_breakpoints_vs_plain_bisection():
    rng = np.random.default_rng(9)
    for L in [1, 5, 100, 5000]:
        w = np.exp(rng.standard_normal(L) * 3)
        r = rng.uniform(0.001, 0.999, L)
        beta = oracle.beta_breakpoints(w, r)
        lo, hi = 0.0, (w * (1 - r)).sum()
        for _ in range(300):
            mid = 0.5 * (lo + hi)
            if mid - (w * (1 - _lam(mid, w, r))).sum() < 0:
                lo = mid
            else:
                hi = mid
        assert math.isclose(beta, hi, rel_tol=1e-12)


# ----------------------------------------------------------------------------- binary shrinkage (App. A.2)
def _gamma_order(w, r):
    """L by decreasing w (1 - r) / r, ties by lower index (the visiting order of App. A.2)."""
    g = w * (1 - r) / r
    return np.lexsort((np.arange(len(w)), -g))


def test_binary_shrinkage_closed_forms():
    """|L| = 1: the only token is shrunk (gamma > 0 = 2 beta), lambda = r, beta = w (1 - r),
    the same as Definition 2.  m identical tokens: token k (0-based) is shrunk while
    w (1 - r) / r > 2 k w (1 - r), i.e. 2 k r < 1, so min(m, ceil(1 / (2 r))) are shrunk."""
    for w, r in [(1.0, 0.3), (5.0, 0.01), (1e-3, 0.9)]:
        lam, beta, ns = oracle.binary_shrinkage([w], [r])
        assert ns == 1 and lam[0] == r and math.isclose(beta, w * (1 - r), rel_tol=1e-15)
    for m in [1, 2, 3, 10, 1000]:
        for r in [0.03, 0.3, 0.7, 0.9]:
            lam, beta, ns = oracle.binary_shrinkage(np.full(m, 2.5), np.full(m, r))
            k0 = min(m, math.ceil(1 / (2 * r)))
            assert ns == k0
            assert np.array_equal(lam, np.where(np.arange(m) < k0, r, 1.0))   # ties: lower index first
            assert math.isclose(beta, k0 * 2.5 * (1 - r), rel_tol=1e-12)
    # a zero weight has gamma = 0, never above 2 beta >= 0
    lam, beta, ns = oracle.binary_shrinkage([0.0, 0.0], [0.5, 0.2])
    assert ns == 0 and beta == 0.0 and np.all(lam == 1.0)


def test_binary_shrinkage_is_prefix_minimum_by_enumeration():
    """App. A.2: switching token i from lambda = 1 to lambda = r_i changes the MSE by
    w_i (1 - r_i) (2 beta - w_i (1 - r_i) / r_i), and the stop is the MSE minimum over all
    prefixes of the order -- both checked against the MSE of every prefix computed by
    enumerating all 2^|L| Poisson outcomes.  Theorem 1 places the continuous minimiser below it."""
    rng = np.random.default_rng(81)
    for trial in range(25):
        L = int(rng.integers(1, 9))
        w = np.exp(rng.standard_normal(L) * 2)
        r = rng.uniform(0.02, 0.95, L)
        if trial % 3 == 0:
            r = rng.uniform(0.005, 0.06, L)   # small r: long prefixes
        lam, beta, ns = oracle.binary_shrinkage(w, r)
        order = _gamma_order(w, r)
        mse = []
        for k in range(L + 1):
            lk = np.ones(L)
            lk[order[:k]] = r[order[:k]]
            mse.append(_mse_enumerated(w, r, lk))
        for k in range(L):
            i = order[k]
            bk = (w[order[:k]] * (1 - r[order[:k]])).sum()
            ai = w[i] * (1 - r[i])
            assert math.isclose(mse[k + 1] - mse[k], ai * (2 * bk - ai / r[i]),
                                rel_tol=1e-8, abs_tol=1e-10 * max(mse))
        expect = np.ones(L)
        expect[order[:ns]] = r[order[:ns]]
        assert np.array_equal(lam, expect)
        assert math.isclose(beta, (w * (1 - lam)).sum(), rel_tol=1e-12)
        assert mse[ns] <= min(mse) * (1 + 1e-10)
        cont = _lam(oracle.beta_breakpoints(w, r), w, r)
        assert _mse_enumerated(w, r, cont) <= mse[ns] * (1 + 1e-10) <= mse[0] * (1 + 1e-10)


def test_binary_shrinkage_certificate_coverage_and_fetch():
    """Lemma 1 and Theorem 2 hold for any fixed lambda in [r, 1]: with the binary
    coefficients, Pr(|D^ - D|/D > eps^(L)) <= delta and, after fetching L_g[:k*], the
    (eps, delta) guarantee -- both exactly over all outcomes; brute-force and closed-form
    gains and k* agree."""
    rng = np.random.default_rng(82)
    for trial in range(30):
        L = int(rng.integers(1, 10))
        flags, r32, t = _tiny_row(rng, L)
        eps = float(rng.choice([0.01, 0.05, 0.2]))
        delta = float(rng.choice([0.05, 0.1, 0.3]))
        brute = oracle.kvfetch_row(flags, r32, t, t, eps, delta, mode=0, shrinkage=1)
        fast = oracle.kvfetch_row(flags, r32, t, t, eps, delta, mode=1, shrinkage=1)
        assert brute["kstar"] == fast["kstar"]
        assert np.array_equal(brute["exact_mask"], fast["exact_mask"])
        Lm = flags != 2
        w = np.exp(t - fast["m"])
        D = w.sum()
        r = r32[Lm].astype(np.float64)
        lam, beta, _ = oracle.binary_shrinkage(w[Lm], r)
        assert np.array_equal(fast["lam"][Lm], lam)
        assert math.isclose(fast["beta"], beta, rel_tol=1e-12, abs_tol=1e-300)
        E = fast["exact_mask"]
        idx = np.nonzero(Lm)[0]
        fail_all = fail_fetch = 0.0
        for z, p in _outcomes(r):
            Z = np.zeros(len(flags))
            Z[idx] = z
            full = w[~Lm].sum() + (Z * fast["lam"] * w / r32)[Lm].sum()
            if abs(full - D) / D > fast["eps_hat"]:
                fail_all += p
            keep = ~Lm | E
            dhat = w[keep].sum() + (Z * fast["lam"] * w / r32)[Lm & ~E].sum()
            if abs(dhat - D) / D > eps:
                fail_fetch += p
        assert fail_all <= delta + 1e-12
        assert fail_fetch <= delta + 1e-12


# ----------------------------------------------------------------------------- shortlist (App. A.1)
def test_shortlist_is_top_k_of_the_largest_sketch_logit():
    """The shortlist of a KV head: among tokens of L outside the sample (flags 0), the k with the
    largest sketch logit over the head's query rows, ties by lower index -- against a plain sort."""
    rng = np.random.default_rng(91)
    for trial in range(20):
        n, G, k = int(rng.integers(5, 400)), int(rng.choice([1, 2, 4, 8])), int(rng.integers(0, 150))
        flags = rng.choice([0, 1, 2], size=n, p=[0.6, 0.2, 0.2]).astype(np.uint8)
        ts = np.round(rng.standard_normal((G, n)) * 3, 1)   # coarse values: ties occur
        got = oracle.shortlist(flags, ts, k)
        score = ts.max(axis=0)
        cand = np.nonzero(flags == 0)[0]
        order = cand[np.lexsort((cand, -score[cand]))]
        want = np.zeros(n, bool)
        want[order[:k]] = True
        assert np.array_equal(got, want)


def test_exact_weight_mask_reductions():
    """App. A.1's certificate weights: exact logits where the mask is set, sketch logits elsewhere.
    With an exact sketch the mask changes nothing; a mask over all of L equals the exact sketch; and D
    is sum_H w + sum_L of the chosen weights."""
    rng = np.random.default_rng(92)
    for trial in range(12):
        L = int(rng.integers(2, 60))
        flags, r32, t = _tiny_row(rng, L, H=3)
        ts = t + rng.standard_normal(len(t)) * 0.4
        mask = (rng.random(len(t)) < 0.4) & (flags != 2)
        eps, delta = float(rng.choice([0.01, 0.05])), 0.1
        a = oracle.kvfetch_row(flags, r32, t, t, eps, delta)
        b = oracle.kvfetch_row(flags, r32, t, t, eps, delta, use_exact=mask)
        for key in ["D", "beta", "eps_hat", "kstar"]:
            assert a[key] == b[key]
        assert np.array_equal(a["exact_mask"], b["exact_mask"])
        c = oracle.kvfetch_row(flags, r32, t, ts, eps, delta, use_exact=flags != 2)
        for key in ["D", "beta", "eps_hat", "kstar"]:
            assert c[key] == a[key]
        d = oracle.kvfetch_row(flags, r32, t, ts, eps, delta, use_exact=mask)
        Lm = flags != 2
        used = np.where(mask, t, ts)
        m = max(t[~Lm].max(), used[Lm].max())
        D = np.exp(t[~Lm] - m).sum() + np.exp(used[Lm] - m).sum()
        assert math.isclose(d["D"], D, rel_tol=1e-12)


# ----------------------------------------------------------------------------- certificate / fetch (Lemma 1, Thm. 2)
def _tiny_row(rng, L, H=2):
    n = L + H
    flags = np.zeros(n, np.uint8)
    flags[:H] = 2
    r32 = np.ones(n, np.float32)
    r32[H:] = rng.uniform(0.05, 0.9, L).astype(np.float32)
    t = rng.standard_normal(n) * 1.5
    return flags, r32, t


def _outcomes(r):
    for z in itertools.product([0, 1], repeat=len(r)):
        z = np.array(z)
        yield z, float(np.prod(np.where(z == 1, r, 1 - r)))


def _outcome_flags(flags, z):
    """The row's flags with the sample set to the Poisson outcome z over L (1 = sampled)."""
    f = flags.copy()
    f[flags != 2] = z.astype(np.uint8)
    return f


def test_lemma1_coverage_exact_enumeration():
    """Lemma 1: Pr(|D^ - D|/D > eps^(L)) <= delta, computed exactly over all Poisson outcomes (exact
    sketch: sketch logits = exact logits), with D^ read from the oracle's estimator for every outcome."""
    rng = np.random.default_rng(10)
    for trial in range(40):
        L = int(rng.integers(1, 11))
        flags, r32, t = _tiny_row(rng, L)
        delta = float(rng.choice([0.05, 0.1, 0.3]))
        res = oracle.kvfetch_row(flags, r32, t, t, eps=1e9, delta=delta)
        w = np.exp(t - res["m"])
        assert math.isclose(res["D"], w.sum(), rel_tol=1e-12)
        assert not res["exact_mask"].any()
        Lm = flags != 2
        fail = 0.0
        for z, p in _outcomes(r32[Lm].astype(np.float64)):
            dhat, _ = oracle.estimate_row(_outcome_flags(flags, z), r32, t, res["lam"], res["exact_mask"], res["m"])
            if abs(dhat - res["D"]) / res["D"] > res["eps_hat"]:
                fail += p
        assert fail <= delta + 1e-12
    empty = oracle.kvfetch_row(np.full(5, 2, np.uint8), np.ones(5, np.float32), np.zeros(5), np.zeros(5), 0.1, 0.1)
    assert empty["eps_hat"] == 0.0 and empty["no_fetch"] == 1


def test_theorem2_coverage_and_monotone_residual_certificate():
    """Theorem 2: after fetching L_g[:k*] the estimator meets (eps, delta),
    checked exactly over all outcomes; eps^(L_g[k:]) is nonincreasing in k;
    g_i >= 0; brute-force and closed-form gains and k* agree."""
    rng = np.random.default_rng(11)
    for trial in range(40):
        L = int(rng.integers(2, 11))
        flags, r32, t = _tiny_row(rng, L)
        eps = float(rng.choice([0.01, 0.05, 0.2]))
        delta = float(rng.choice([0.05, 0.1]))
        brute = oracle.kvfetch_row(flags, r32, t, t, eps, delta, mode=0)
        fast = oracle.kvfetch_row(flags, r32, t, t, eps, delta, mode=1)
        assert brute["kstar"] == fast["kstar"]
        assert np.array_equal(brute["exact_mask"], fast["exact_mask"])
        Lm = flags != 2
        if not fast["no_fetch"]:
            gb, gf = brute["gain"][Lm], fast["gain"][Lm]
            assert np.all(gf >= 0)
            big = gf > 1e-9 * fast["eps_hat"]
            assert np.allclose(gb[big], gf[big], rtol=1e-8)
        w = np.exp(t - fast["m"])
        D = w.sum()
        lam = fast["lam"]
        # residual certificate along the order, recomputed from Lemma 1's sums
        order = fast["order"]
        ld = math.log(2 / delta)
        a = w * (1 - lam)
        v = lam ** 2 * w ** 2 * (1 - r32) / r32
        b = lam * w / r32 * np.maximum(r32, 1 - r32)
        prev = math.inf
        for k in range(len(order) + 1):
            rest = order[k:]
            bb = b[rest].max() if len(rest) else 0.0
            e = (a[rest].sum() + bb * ld / 3 + math.sqrt((bb * ld / 3) ** 2 + 2 * v[rest].sum() * ld)) / D
            assert e <= prev * (1 + 1e-12)
            prev = e
        # exact coverage of the returned estimator, D^ read from the oracle for every outcome
        E = fast["exact_mask"]
        fail = 0.0
        for z, p in _outcomes(r32[Lm].astype(np.float64)):
            dhat, _ = oracle.estimate_row(_outcome_flags(flags, z), r32, t, lam, E, fast["m"])
            if abs(dhat - D) / D > eps:
                fail += p
        assert fail <= delta + 1e-12


def test_certificate_invariant_to_logit_shift():
    rng = np.random.default_rng(12)
    n = 3000
    flags = (rng.random(n) < 0.05).astype(np.uint8) * 2
    r32 = np.where(flags == 2, 1.0, rng.uniform(0.01, 0.3, n)).astype(np.float32)
    t = rng.standard_normal(n) * 2
    ts = t + rng.standard_normal(n) * 0.1
    a = oracle.kvfetch_row(flags, r32, t, ts, 0.02, 0.05)
    b = oracle.kvfetch_row(flags, r32, t + 37.5, ts + 37.5, 0.02, 0.05)
    assert math.isclose(a["eps_hat"], b["eps_hat"], rel_tol=1e-12)
    assert a["kstar"] == b["kstar"] and np.array_equal(a["exact_mask"], b["exact_mask"])
    assert math.isclose(a["beta"] / a["D"], b["beta"] / b["D"], rel_tol=1e-12)


def test_eps_zero_fetches_everything_and_equals_dense_attention():
    """eps = 0 forces the full fetch (k* = |L|), and the output is plain softmax
    attention (numpy double loop and torch float64 SDPA)."""
    import torch
    rng = np.random.default_rng(13)
    n, d = 600, 64
    K = rng.standard_normal((n, d))
    V = rng.standard_normal((n, d))
    q = rng.standard_normal(d)
    t = K @ q / math.sqrt(d)
    flags = (rng.random(n) < 0.1).astype(np.uint8)
    flags[:8] = 2
    r32 = np.where(flags == 2, 1.0, 0.1).astype(np.float32)
    res = oracle.kvfetch_row(flags, r32, t, t + rng.standard_normal(n) * 0.3, 0.0, 0.05)
    assert res["kstar"] == (flags != 2).sum() and res["exact_mask"][flags != 2].all()
    out = oracle.attention_row(flags, r32, t, V, res["lam"], res["exact_mask"])
    p = np.exp(t - t.max())
    dense = (p[:, None] * V).sum(0) / p.sum()
    sdpa = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q)[None, None, None], torch.tensor(K)[None, None], torch.tensor(V)[None, None])[0, 0, 0].numpy()
    assert np.allclose(out, dense, rtol=1e-12, atol=1e-13)
    assert np.allclose(out, sdpa, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("sketch", ["int8", "2bit"])
def test_appended_tokens_at_eps_zero_equal_dense_attention(sketch):
    """Decode-time growth (App. A.3.1): tokens appended after compress are H.  At eps = 0 every token of
    L is fetched, so the decision over the compressed prefix plus the appended tokens must return plain
    softmax attention over all of them (closed form), whatever the prefix's sample; and the certificate
    denominator must count the appended tokens (D = sum of every exact weight when the sketch is exact
    on H, checked here through the output).  Pins the test harness's extension of a compressed slot."""
    import dataclasses

    from vkcase import oracle_compress, oracle_decode, oracle_tau
    from verified_kv_cache_gb300 import workloads
    n0, t = 700, 40
    full = workloads.qwen_layer_case(seed=5, n=n0 + t, n_kv=1, n_q=2, n_needles=2, W=4, steps=2, sketch=sketch,
                                     eta=0.25, eps=0.0, delta=0.05, n_sink=4, n_local=64)
    w0 = dataclasses.replace(full, n=n0, K=full.K[:, :, :n0], V=full.V[:, :, :n0])
    osl = oracle_compress(w0, 0, oracle_tau(w0, 0))
    for s in range(2):
        rows, unions = oracle_decode(full, 0, osl, full.queries[s, 0], 0.0, 0.05)
        assert len(unions[0]) == int((osl.flags[0] == 0).sum())   # all of L minus S, nothing appended
        for hq in range(full.n_q):
            q = full.queries[s, 0, hq].astype(np.float64)
            K, V = full.K[0, 0].astype(np.float64), full.V[0, 0].astype(np.float64)
            lg = K @ q / math.sqrt(full.d)
            p = np.exp(lg - lg.max())
            dense = (p[:, None] * V).sum(0) / p.sum()
            assert np.allclose(rows[hq]["out"], dense, rtol=1e-10, atol=1e-12), (s, hq)
            if s == 1:   # a random query spreads its weight: the appended tokens carry a visible share
                p0 = p[:n0]
                prefix_only = (p0[:, None] * V[:n0]).sum(0) / p0.sum()
                assert not np.allclose(prefix_only, dense, rtol=1e-6, atol=1e-8)


@pytest.mark.parametrize("sketch_noise", [0.0, 0.4])
@pytest.mark.parametrize("eps", [1e9, 0.02])
def test_attention_weights_follow_eq5_by_one_hot_values(sketch_noise, eps):
    """The oracle's output weights, pinned by enumeration: with one-hot value rows (V_i = e_i, d = n)
    the attention returns each token's share of the estimator itself, o_i = omega_i w_i / D^.  Eq. (5)
    after the fetch gives omega_i = 1 on H and on L_g[:k*], lambda_i / r_i on the rest of the sample
    and 0 on unsampled, unfetched tokens, with the EXACT weight w_i (the keys of S are resident and
    those of L_g[:k*] fetched), while lambda and the order come from the sketch weights.  Checked for
    every Poisson outcome of tiny rows, with no fetch (eps huge) and with part of L made exact."""
    rng = np.random.default_rng(15)
    checked_exact = 0
    for trial in range(12):
        L = int(rng.integers(2, 9))
        flags, r32, t = _tiny_row(rng, L)
        ts = t + sketch_noise * rng.standard_normal(len(t))
        res = oracle.kvfetch_row(flags, r32, t, ts, eps, 0.1)
        lam, E = res["lam"], res["exact_mask"]
        checked_exact += int(E.sum())
        n = len(flags)
        V = np.eye(n)
        w = np.exp(t - t.max())
        for z, _ in _outcomes(r32[flags != 2].astype(np.float64)):
            f = _outcome_flags(flags, z)
            out = oracle.attention_row(f, r32, t, V, lam, E)
            term = np.where((f == 2) | E, w, np.where(f == 1, lam * w / r32.astype(np.float64), 0.0))
            assert np.allclose(out, term / term.sum(), rtol=1e-12, atol=1e-15), (trial, z)
            # lambda_i / r_i, not lambda_i: a sampled, unfetched token of L is weighted above its lambda
            s_only = (f == 1) & ~E
            if s_only.any():
                i = int(np.nonzero(s_only)[0][0])
                assert out[i] / out[f == 2][0] == pytest.approx(lam[i] / r32[i] * w[i] / w[f == 2][0], rel=1e-12)
    if eps < 1:
        assert checked_exact > 0, "no row made part of L exact"


def test_estimator_moments_match_bias_and_eq6():
    """Theorem 1's objects, read from two different oracle functions: over all Poisson outcomes the
    oracle's D^ (no fetch) has mean D - beta(L) (the bias sum_L w_i (1 - lambda_i), i.e. sum_a of the
    certificate) and mean squared error beta(L)^2 + V(L) (eq. (6) at the returned lambda), both from
    kvfetch_row.  A weight lambda_i instead of lambda_i / r_i, or a nonzero weight on unsampled tokens,
    moves both moments."""
    rng = np.random.default_rng(16)
    for trial in range(30):
        L = int(rng.integers(1, 11))
        flags, r32, t = _tiny_row(rng, L)
        res = oracle.kvfetch_row(flags, r32, t, t, 1e9, 0.1)
        D = res["D"]
        m1 = m2 = 0.0
        for z, p in _outcomes(r32[flags != 2].astype(np.float64)):
            dhat, _ = oracle.estimate_row(_outcome_flags(flags, z), r32, t, res["lam"], res["exact_mask"], res["m"])
            m1 += p * dhat
            m2 += p * (dhat - D) ** 2
        assert math.isclose(m1, D - res["sum_a"], rel_tol=1e-12), (m1, D, res["sum_a"])
        assert math.isclose(m2, res["sum_a"] ** 2 + res["V"], rel_tol=1e-10), (m2, res["sum_a"], res["V"])
    # lambda forced to one: the Horvitz-Thompson estimator, read from the oracle, is unbiased
    flags, r32, t = _tiny_row(rng, 8)
    ones = np.where(flags != 2, 1.0, 0.0)
    m1 = sum(p * oracle.estimate_row(_outcome_flags(flags, z), r32, t, ones, np.zeros(len(flags), bool), 0.0)[0]
             for z, p in _outcomes(r32[flags != 2].astype(np.float64)))
    assert math.isclose(m1, np.exp(t).sum(), rel_tol=1e-12)


@pytest.mark.slow
def test_empirical_coverage_over_philox_seeds_tiny_case():
    """Coverage over many independent Poisson samples (Philox seeds) on the
    tiny exact-sketch workload: the fraction of decisions whose denominator
    misses eps exceeds delta rarely (paper, Sec. 5.5: under 0.7% with a
    perfect sketch at delta = 0.1)."""
    from verified_kv_cache_gb300 import workloads
    w = workloads.tiny_oracle_case()
    K, V = w.K[0, 0].astype(np.float64), w.V[0, 0]
    tau = oracle.tau(w.K[0, 0], w.obs_q[0, 0], w.n_sink, w.n_local)
    c, t, r64, r32 = oracle.waterfill(tau, w.n_sink, w.n_local, w.eta * w.n)
    seeds = 1500
    fails = 0
    total = 0
    for s in range(w.queries.shape[0]):
        q = w.queries[s, 0, 0].astype(np.float64)
        tl = K @ q / math.sqrt(w.d)
        base = oracle.poisson_sample(r32, 0, 0, 0, 0)
        res = oracle.kvfetch_row(base, r32, tl, tl, w.eps, w.delta)
        ww = np.exp(tl - res["m"])
        D = ww.sum()
        Lm = base != 2
        E = res["exact_mask"]
        lam = res["lam"]
        for seed in range(seeds):
            f = oracle.poisson_sample(r32, seed, 0, 0, 0)
            dhat, _ = oracle.estimate_row(f, r32, tl, lam, E, res["m"])
            fails += abs(dhat - D) / D > w.eps
            total += 1
    assert fails / total <= w.delta
