"""Pins for oracle.pages: metadata, bounds, Gaussian model, τ̂ and selection."""

import json
import math
import os

import numpy as np
import pytest

from oracle import entmax as em
from oracle import pages as pg

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_metadata_twopass_welford_chan_agree():
    rng = np.random.default_rng(10)
    keys = rng.normal(size=(77, 9)) * 3.0 + 1.5
    P = 16
    meta = pg.page_metadata(keys, P)
    assert list(meta["n"]) == [16, 16, 16, 16, 13]
    for p in range(5):
        blk = keys[p * P: (p + 1) * P]
        # token-by-token (append of one token at a time)
        n, mean, m2 = 0, np.zeros(9), np.zeros(9)
        for x in blk:
            n, mean, m2 = pg.welford_append(n, mean, m2, x)
        np.testing.assert_allclose(mean, meta["mean"][p], rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(m2 / n, meta["var"][p], rtol=1e-12, atol=1e-13)
        # two halves merged (append of a block to a partly filled page)
        h = len(blk) // 3
        a, b = blk[:h], blk[h:]
        ma, mb = a.mean(0), b.mean(0)
        n2, mean2, m22 = pg.chan_merge(len(a), ma, ((a - ma) ** 2).sum(0),
                                       len(b), mb, ((b - mb) ** 2).sum(0))
        np.testing.assert_allclose(mean2, meta["mean"][p], rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(m22 / n2, meta["var"][p], rtol=1e-12, atol=1e-13)
        # bounding box: every key inside, and each face attained by some key
        assert np.all(blk >= meta["kmin"][p]) and np.all(blk <= meta["kmax"][p])
        assert np.all((blk == meta["kmin"][p]).any(0)) and np.all((blk == meta["kmax"][p]).any(0))


def test_bbox_is_an_upper_bound_and_tight():
    rng = np.random.default_rng(11)
    d, P = 16, 8
    keys = rng.normal(size=(8 * P + 3, d))
    meta = pg.page_metadata(keys, P)
    for _ in range(20):
        q = rng.normal(size=d)
        U = pg.bbox_bound(q, meta["kmin"], meta["kmax"])
        s = keys @ q / math.sqrt(d)
        for p in range(U.size):
            assert U[p] >= s[p * P:(p + 1) * P].max() - 1e-12
        # equivalent split form: positive part of q meets kmax, negative kmin
        U2 = (meta["kmax"] @ np.maximum(q, 0) + meta["kmin"] @ np.minimum(q, 0)) / math.sqrt(d)
        np.testing.assert_allclose(U, U2, atol=1e-12)
    # tight for one-token pages and for pages of identical tokens
    one = pg.page_metadata(keys[:5], 1)
    q = rng.normal(size=d)
    np.testing.assert_allclose(pg.bbox_bound(q, one["kmin"], one["kmax"]),
                               keys[:5] @ q / math.sqrt(d), atol=1e-12)
    same = pg.page_metadata(np.repeat(keys[:1], 4, axis=0), 4)
    np.testing.assert_allclose(pg.bbox_bound(q, same["kmin"], same["kmax"]),
                               keys[:1] @ q / math.sqrt(d), atol=1e-12)


def test_hand_decode_case_bbox_and_topk():
    c = json.load(open(os.path.join(GOLD, "decode_hand_case.json")))
    meta = pg.page_metadata(np.array(c["k"]), c["page_size"])
    U = pg.bbox_bound(np.array(c["q"][0]), meta["kmin"], meta["kmax"])
    assert abs(U[0] - eval(c["bbox_U_page0"])) < 1e-15
    assert abs(U[1] - eval(c["bbox_U_page1"])) < 1e-15
    k = c["topk_budget_tokens"] // c["page_size"]
    assert list(pg.select_topk(U, k)) == c["topk_page_ids"]


def test_topk_matches_stable_sort_with_ties():
    rng = np.random.default_rng(12)
    for n in (1, 5, 64, 300):
        u = np.round(rng.normal(size=n), 1)  # many exact ties
        for k in (1, 3, n // 2 + 1, n, n + 5):
            got = pg.select_topk(u, k)
            order = np.lexsort((np.arange(n), -u))  # by -u, then index
            want = np.sort(order[:k])
            assert list(got) == list(want)


def _hadamard(n):
    H = np.array([[1.0]])
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]])
    return H


def test_gauss_model_is_exact_for_uncorrelated_page():
    # Columns 1..d of a Hadamard matrix are centred and mutually orthogonal,
    # so the page's empirical covariance is diagonal; then the model's μ_p and
    # σ_p² equal the empirical mean and variance of the page's token scores.
    d, n = 12, 32
    H = _hadamard(n)[:, 1:d + 1]
    rng = np.random.default_rng(13)
    scale = rng.uniform(0.5, 2.0, size=d)
    keys = rng.normal(size=d) + H * scale
    meta = pg.page_metadata(keys, n)
    q = rng.normal(size=d)
    mu, sig = pg.gauss_page_scores(q, meta["mean"], meta["var"])
    s = keys @ q / math.sqrt(d)
    assert abs(mu[0] - s.mean()) < 1e-12
    assert abs(sig[0] ** 2 - s.var()) < 1e-12


def test_partial_moments_match_quadrature():
    rng = np.random.default_rng(14)
    for beta in (1.0, 2.0):
        for _ in range(25):
            a = rng.normal() * 3.0
            if a + 12 * 3.0 <= 0.0:
                continue
            sg = rng.uniform(0.05, 3.0)
            # the integrand vanishes below 0 and is smooth above it, so integrate
            # from the kink at 0 (or a − 12σ if that is larger)
            x = np.linspace(max(0.0, a - 12 * sg), a + 12 * sg, 100001)
            dens = np.exp(-0.5 * ((x - a) / sg) ** 2) / (sg * math.sqrt(2 * math.pi))
            f = np.clip(x, 0, None) ** beta * dens
            h = x[1] - x[0]  # composite Simpson on an even number of intervals
            quad = float(h / 3.0 * (f[0] + f[-1] + 4.0 * f[1:-1:2].sum() + 2.0 * f[2:-1:2].sum()))
            got = float(pg.partial_moment(a, sg, beta))
            assert abs(got - quad) < 1e-9 * max(1.0, abs(quad)), (beta, a, sg, got, quad)
        # σ = 0 reduces to the plain power of the positive part
        assert float(pg.partial_moment(0.7, 0.0, beta)) == 0.7 ** beta
        assert float(pg.partial_moment(-0.7, 0.0, beta)) == 0.0


def test_tauhat_degenerate_equals_exact_entmax_of_means():
    # With σ_p = 0 every page is a point mass, so F(τ) = Σ_p n_p (m_p − τ)_+^β
    # is the exact entmax normaliser of the page means repeated n_p times.
    rng = np.random.default_rng(15)
    for alpha in (1.5, 2.0):
        m = rng.normal(size=40)
        n = rng.integers(1, 33, size=40)
        th = pg.tauhat(m, np.zeros(40), n, alpha)
        ref = em.threshold(np.repeat(m, n), alpha)
        assert abs(th - ref) < 1e-10


def test_tauhat_solves_normaliser_and_F_decreasing():
    rng = np.random.default_rng(16)
    for alpha in (1.5, 2.0):
        beta = 1.0 / (alpha - 1.0)
        m = rng.normal(size=200) * 0.4
        sg = rng.uniform(0.1, 0.8, size=200)
        n = np.full(200, 32)
        th = pg.tauhat(m, sg, n, alpha)
        assert abs(pg.normaliser(th, m, sg, n, beta) - 1.0) < 1e-10
        ts = np.linspace(m.max() - 1.0, th + 2.0, 50)
        F = [pg.normaliser(t, m, sg, n, beta) for t in ts]
        assert all(F[i] > F[i + 1] for i in range(len(F) - 1))
        assert th >= m.max() - 1.0


def test_gaussian_selection_monotone_in_margin():
    rng = np.random.default_rng(17)
    mh = rng.normal(size=(4, 500))
    thr = rng.normal(size=4) + 1.0
    prev = None
    for delta in (0.0, 0.25, 0.5, 1.0, 2.0):
        sel = set(pg.select_gaussian(mh, thr - delta))
        if prev is not None:
            assert prev <= sel
        prev = sel
    # equality selects
    assert list(pg.select_gaussian(np.array([[1.0, 0.5]]), np.array([0.5]))) == [0, 1]


def test_est_max_one_token_page_is_mean():
    assert pg.est_max(np.array([0.3]), np.array([5.0]), np.array([1]))[0] == 0.3


# --------------------------------------------------------------------------
# General entmax order in the Gaussian selector: J_ν(t) = E[(t + Z)_+^ν]
# --------------------------------------------------------------------------

def test_jfun_reduces_to_the_integer_closed_forms():
    # ν = 0: Φ(t); ν = 1: tΦ + φ; ν = 2: (1+t²)Φ + tφ; ν = 3: (t³+3t)Φ + (t²+2)φ
    # (integrate (t + z)^n φ(z) over z > −t term by term); both routes of jfun.
    from scipy.special import ndtr
    t = np.concatenate([np.linspace(-10.0, 19.5, 60), np.linspace(20.0, 40.0, 9)])
    ph, Ph = np.exp(-0.5 * t * t) / math.sqrt(2 * math.pi), ndtr(t)
    forms = {0: Ph, 1: t * Ph + ph, 2: (1 + t * t) * Ph + t * ph, 3: (t ** 3 + 3 * t) * Ph + (t * t + 2) * ph}
    for nu, ref in forms.items():
        # for ν ≥ 1 the closed forms cancel in the far left tail (tΦ against φ),
        # so they are compared where they keep their digits
        keep = t >= (-10.0 if nu == 0 else -4.0)
        got = pg.jfun(t[keep], float(nu))
        np.testing.assert_allclose(got, ref[keep], rtol=1e-11, atol=1e-300)


def test_jfun_matches_quadrature_of_its_definition():
    from scipy.integrate import quad
    for nu in (-0.5, 0.5, 1.5, 3.3, 6.0):
        for t in (-6.0, -2.5, 0.0, 1.0, 4.0, 12.0, 19.0, 21.0, 25.0):
            f = lambda y: y ** nu * math.exp(-0.5 * (y - t) ** 2) / math.sqrt(2 * math.pi)
            ref = quad(f, 0.0, max(1.0, t) + 40.0, points=[max(t, 1e-3)], limit=400,
                       epsabs=0.0, epsrel=1e-13)[0]
            got = float(pg.jfun(np.array([t]), nu)[0])
            # quad's own accuracy next to the y^ν end point (ν < 0) is about 1e-9
            assert abs(got - ref) <= 5e-9 * abs(ref), (nu, t, got, ref)


def test_jfun_derivative_is_nu_times_the_next_lower_order():
    # d/dt ∫_0^∞ y^ν φ(y − t) dy = ν·J_{ν−1}(t) (integrate by parts), so the
    # Halley step's D1 and D2 come from the orders β − 1 and β − 2.
    h = 1e-5
    for nu in (1.7, 2.5, 4.0):
        for t in (-3.0, 0.0, 2.0, 25.0):
            fd = (pg.jfun(np.array([t + h]), nu)[0] - pg.jfun(np.array([t - h]), nu)[0]) / (2 * h)
            ref = nu * pg.jfun(np.array([t]), nu - 1.0)[0]
            assert abs(fd - ref) <= 1e-6 * max(1.0, abs(ref)), (nu, t, fd, ref)


def test_jfun_is_continuous_across_the_series_switch():
    for nu in (0.5, 3.3, 7.0):
        a = pg.jfun(np.array([pg.J_SERIES_FROM * (1 - 1e-12)]), nu)[0]
        b = pg.jfun(np.array([pg.J_SERIES_FROM]), nu)[0]
        assert abs(a - b) <= 1e-11 * abs(b)


def test_partial_moment_general_beta_matches_quadrature():
    from scipy.integrate import quad
    rng = np.random.default_rng(17)
    for beta in (0.5, 1.5, 3.3):
        for _ in range(15):
            a, sg = rng.normal() * 2.0, rng.uniform(0.05, 2.0)
            f = lambda x: max(x, 0.0) ** beta * math.exp(-0.5 * ((x - a) / sg) ** 2) / (sg * math.sqrt(2 * math.pi))
            lo = max(0.0, a - 14 * sg)
            if lo >= a + 14 * sg:
                continue
            ref = quad(f, lo, a + 14 * sg, points=[max(a, lo + 1e-12)], limit=400, epsabs=0.0, epsrel=1e-12)[0]
            got = float(pg.partial_moment(a, sg, beta))
            assert abs(got - ref) <= 1e-9 * max(abs(ref), 1e-300), (beta, a, sg, got, ref)
        assert float(pg.partial_moment(0.7, 0.0, beta)) == 0.7 ** beta


@pytest.mark.parametrize("alpha", [1.25, 1.75, 3.0])
def test_tauhat_general_alpha(alpha):
    beta = 1.0 / (alpha - 1.0)
    rng = np.random.default_rng(18)
    # point masses: the exact entmax threshold of the repeated means
    m = rng.normal(size=30)
    n = rng.integers(1, 33, size=30)
    assert abs(pg.tauhat(m, np.zeros(30), n, alpha) - em.threshold(np.repeat(m, n), alpha)) < 1e-10
    # Gaussian pages: F(τ̂) = 1, F decreasing, τ̂ ≥ max m − 1
    m = rng.normal(size=150) * 0.4
    sg = rng.uniform(0.1, 0.8, size=150)
    n = np.full(150, 32)
    th = pg.tauhat(m, sg, n, alpha)
    assert abs(pg.normaliser(th, m, sg, n, beta) - 1.0) < 1e-10
    F = [pg.normaliser(t, m, sg, n, beta) for t in np.linspace(m.max() - 1.0, th + 2.0, 30)]
    assert all(F[i] > F[i + 1] for i in range(len(F) - 1))
    assert th >= m.max() - 1.0


def test_jfun_matches_high_precision_quadrature():
    # 40-digit tanh-sinh quadrature of the defining integral (mpmath), across
    # all three routes of jfun and both sides of each switch
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    for nu in (-0.5, 0.5, 1.5, 3.3, 6.0):
        for t in (-14.0, -6.0, -2.0, -1.999, 0.0, 3.0, 12.0, 19.99, 20.0, 30.0):
            if t < 0:  # φ(y − t) = φ(t)·e^{−y²/2 − |t|y}: integrate the factor, split at its scale
                x = mp.mpf(-t)
                ref = mp.npdf(x) * mp.quad(lambda y: y ** nu * mp.exp(-y * y / 2 - x * y),
                                           [0, 1 / x, 10 / x, mp.inf])
            else:
                ref = mp.quad(lambda y: y ** nu * mp.npdf(y - t), [0, max(t, 1.0), mp.inf])
            got = pg.jfun(np.array([t]), nu)[0]
            assert abs(got - float(ref)) <= 1e-12 * abs(float(ref)), (nu, t, got, float(ref))


# --------------------------------------------------------------------------
# Estimated maximum with n_p > 1, the Gaussian cap, bf16 statistics
# --------------------------------------------------------------------------

def test_est_max_golden_pages():
    """μ_p, σ_p and M̂_p = μ_p + σ_p·sqrt(2 ln n_p) of hand-built pages (a full
    page and a partly filled one), through page_metadata, gauss_page_scores
    and est_max: a missing factor 2 in the log, or the page size in place of
    the valid count, fails here."""
    c = json.load(open(os.path.join(GOLD, "est_max_cases.json")))
    q = np.array(c["q"])
    for pg_case in c["pages"]:
        cols = [eval(pg_case["k%d" % i]) for i in range(c["d"])]
        keys = np.array(cols, dtype=np.float64).T
        assert keys.shape[0] == pg_case["n"]
        meta = pg.page_metadata(keys, c["page_size"])
        assert list(meta["n"]) == [pg_case["n"]]
        mu, sig = pg.gauss_page_scores(q, meta["mean"], meta["var"])
        assert abs(mu[0] - eval(pg_case["mu"])) < 1e-14
        assert abs(sig[0] - eval(pg_case["sigma"])) < 1e-14
        mh = pg.est_max(mu, sig, meta["n"])
        assert abs(mh[0] - eval(pg_case["mhat"])) < 1e-13, (mh[0], pg_case["mhat"])


def test_gaussian_cap_golden_case():
    """The Gaussian selector's cap on hand-built point-mass pages: τ̂, the
    uncapped selection, and which pages survive each cap (ties to the lower
    page index), with the capacity flag."""
    from oracle import decode as odec
    c = json.load(open(os.path.join(GOLD, "gaussian_cap_case.json")))
    P, other = c["page_size"], c["other_dims"]
    keys = np.array([[s] + other for s in c["page_scores"] for _ in range(P)])
    vals = np.arange(keys.shape[0] * 4, dtype=np.float64).reshape(-1, 4)
    Q = np.array(c["q"])
    r = odec.decode_group(keys, vals, Q, c["alpha"], "gaussian", P, 0, c["margin"])
    assert abs(r["tauhat"][0] - eval(c["tauhat"])) < 1e-10
    assert list(r["page_ids"]) == c["uncapped_page_ids"] and not r["capacity_flag"]
    for case in c["capped"]:
        r = odec.decode_group(keys, vals, Q, c["alpha"], "gaussian", P, case["budget_tokens"],
                              c["margin"])
        assert list(r["page_ids"]) == case["page_ids"], (case, r["page_ids"])
        assert r["capacity_flag"] == case["capacity_flag"]


def test_bf16_round_hand_cases_and_library_conversion():
    """Round-to-nearest-even to bfloat16 (8 significant bits): halfway cases
    go to the even neighbour, and on float32-representable inputs the result
    equals torch's float32 → bfloat16 conversion (a library routine)."""
    r = pg.bf16_round
    assert r(1.0 + 2.0 ** -8) == 1.0                      # tie between 1 and 1 + 2^-7: even is 1
    assert r(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6      # tie: 1 + 2^-6 has the even last bit
    assert r(1.0 + 2.0 ** -8 + 2.0 ** -30) == 1.0 + 2.0 ** -7  # just above the tie
    assert r(-(1.0 + 3 * 2.0 ** -8)) == -(1.0 + 2.0 ** -6)
    assert r(0.0) == 0.0 and r(2.0 ** -130) == 2.0 ** -130 and r(3.0) == 3.0
    assert r(255.5) == 256.0 and r(254.5) == 254.0       # spacing 1 in [128, 256): ties to even
    import torch
    rng = np.random.default_rng(21)
    x = np.concatenate([rng.normal(size=20000) * 10.0 ** rng.integers(-6, 6, size=20000),
                        rng.uniform(-3, 3, size=5000)]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(r(x.astype(np.float64)), want)


def test_bf16_metadata_rounds_mean_and_m2():
    rng = np.random.default_rng(22)
    keys = rng.normal(size=(70, 8)) * 2.0 + 0.3
    meta = pg.page_metadata(keys, 16)
    b = pg.bf16_metadata(meta)
    n = meta["n"][:, None].astype(np.float64)
    assert np.array_equal(b["mean"], pg.bf16_round(meta["mean"]))
    assert np.array_equal(b["var"] * n, pg.bf16_round(meta["var"] * n))
    assert np.array_equal(b["kmin"], meta["kmin"]) and np.array_equal(b["kmax"], meta["kmax"])
    # within half a bfloat16 spacing (at most 2^-8 of the value) of the exact statistics
    assert np.all(np.abs(b["mean"] - meta["mean"]) <= 2.0 ** -8 * np.abs(meta["mean"]))
