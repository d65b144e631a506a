"""Pins for the oracle's rejection-sampling acceptance (CPU only).

"Decoding Speculative Decoding from First Principles", section "How does this
drafter maintain the same distribution of the target?": a drafted token x is
kept with probability min(1, p(x)/q(x)); at the first rejection a token is
drawn from max(p - q, 0) renormalised; the emitted token then follows p
exactly.  The oracle is pinned to the page's worked example, to that
distribution identity (chi-square over many independent draws), to the
all-accept case (bonus drawn from p), to the generator's published
known-answer outputs and to the Gumbel law's closed-form moments.  Each pin
was checked to catch a planted slip: q/p instead of p/q, the residual
max(q - p, 0), a flipped Gumbel sign, dropping the temperature.
"""
from __future__ import annotations

import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                key, *vals = line.split()
                rows[key] = vals
    return rows


def chi2_ok(counts, probs, n, z=5.0):
    """Every cell within z standard deviations of its binomial expectation."""
    probs = np.asarray(probs, np.float64)
    exp = n * probs
    sd = np.sqrt(n * probs * (1 - probs)) + 1e-12
    return np.all(np.abs(counts - exp) <= z * sd + 1e-9)


def test_splitmix64_known_answers(oracle_mod):
    g = read_golden("splitmix64_seed0.txt")
    for n, hexval in g.items():
        assert oracle_mod.splitmix64(0, int(n)) == int(hexval[0], 16)


def test_uniform_and_gumbel_moments(oracle_mod):
    # u in [0, 1) with mean 1/2; Gumbel noise with mean = Euler-Mascheroni
    # constant and variance pi^2 / 6
    u = np.array([oracle_mod.accept_uniform(7, b, i) for b in range(200) for i in range(50)])
    assert u.min() >= 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 0.02
    g = np.array([oracle_mod.gumbel(7, b, x) for b in range(100) for x in range(200)])
    assert abs(g.mean() - 0.5772156649) < 0.05
    assert abs(g.var() - np.pi ** 2 / 6) < 0.1


def worked_inputs(B, T=1.0):
    g = read_golden("rejection_worked_example.txt")
    p = np.array(g["p"], np.float64)
    q = np.array(g["q"], np.float64)
    draft = int(g["draft"][0])
    tl = np.tile((np.log(np.stack([p, p])) * T)[None], (B, 1, 1)).astype(np.float32)
    dl = np.tile((np.log(q) * T)[None, None], (B, 1, 1)).astype(np.float32)
    dr = np.full((B, 1), draft, np.int32)
    return g, tl, dl, dr


def test_worked_example(oracle_mod):
    B = 40000
    g, tl, dl, dr = worked_inputs(B)
    acc, nxt, ratio, unif, gap = oracle_mod.accept_rejection(tl, dl, "f32", dr, 1.0, 12345)
    pa = float(g["accept_prob"][0])
    assert np.allclose(ratio[:, 0], pa, rtol=1e-6)
    assert chi2_ok(np.array([np.sum(acc == 1)]), [pa], B)
    # rejected -> a residual draw
    rej = nxt[acc == 0]
    counts = np.bincount(rej, minlength=3)
    assert counts[1] == 0  # the residual has no mass on the rejected token
    assert chi2_ok(counts, np.array(g["residual"], np.float64), len(rej))


def test_temperature_scales_logits(oracle_mod):
    # softmax(logits / T): logits multiplied by T at temperature T give the
    # same distributions, hence the same draws
    B = 3000
    _, tl, dl, dr = worked_inputs(B)
    _, tl2, dl2, _ = worked_inputs(B, T=2.0)
    a1 = oracle_mod.accept_rejection(tl, dl, "f32", dr, 1.0, 99)
    a2 = oracle_mod.accept_rejection(tl2, dl2, "f32", dr, 2.0, 99)
    assert np.array_equal(a1[0], a2[0]) and np.array_equal(a1[1], a2[1])


@pytest.mark.parametrize("seed", [1, 2])
def test_emitted_token_follows_target(oracle_mod, seed):
    # k = 1, drafts drawn from q: the first emitted token (the draft if kept,
    # else the residual draw) must follow p
    rng = np.random.default_rng(seed)
    V, B = 6, 60000
    lp = rng.standard_normal(V) * 1.5
    lq = rng.standard_normal(V) * 1.5
    p = np.exp(lp - lp.max()); p /= p.sum()
    q = np.exp(lq - lq.max()); q /= q.sum()
    dr = rng.choice(V, size=(B, 1), p=q).astype(np.int32)
    tl = np.tile(np.stack([lp, lp])[None], (B, 1, 1)).astype(np.float64).astype(np.float32)
    dl = np.tile(lq[None, None], (B, 1, 1)).astype(np.float32)
    acc, nxt, *_ = oracle_mod.accept_rejection(tl, dl, "f32", dr, 1.0, 1000 + seed)
    first = np.where(acc == 1, dr[:, 0], nxt)
    # the float32-rounded logits define p exactly as the oracle sees them
    lp32 = tl[0, 0].astype(np.float64)
    p32 = np.exp(lp32 - lp32.max()); p32 /= p32.sum()
    assert chi2_ok(np.bincount(first, minlength=V), p32, B)


def test_all_accept_draws_bonus_from_target(oracle_mod):
    # p == q: every draft is kept (p/q = 1 > u) and the bonus follows p_k
    rng = np.random.default_rng(5)
    V, k, B = 5, 3, 40000
    lg = rng.standard_normal((k + 1, V)).astype(np.float32)
    tl = np.tile(lg[None], (B, 1, 1))
    dl = np.ascontiguousarray(tl[:, :k])
    dr = rng.integers(0, V, size=(B, k)).astype(np.int32)
    acc, nxt, ratio, *_ = oracle_mod.accept_rejection(tl, dl, "f32", dr, 1.0, 7)
    assert np.all(acc == k)
    assert np.allclose(ratio, 1.0, atol=1e-12)
    pk = np.exp(lg[k].astype(np.float64) - lg[k].max()); pk /= pk.sum()
    assert chi2_ok(np.bincount(nxt, minlength=V), pk, B)


def test_invariants_and_errors(oracle_mod):
    rng = np.random.default_rng(9)
    B, k, V = 64, 4, 50
    tl = rng.standard_normal((B, k + 1, V)).astype(np.float32) * 2
    dl = rng.standard_normal((B, k, V)).astype(np.float32) * 2
    dr = rng.integers(0, V, size=(B, k)).astype(np.int32)
    acc, nxt, ratio, unif, gap = oracle_mod.accept_rejection(tl, dl, "f32", dr, 0.7, 3)
    assert np.all((acc >= 0) & (acc <= k)) and np.all((nxt >= 0) & (nxt < V))
    for b in range(B):
        n = acc[b]
        # kept while u < p/q, rejected at the first u >= p/q
        assert np.all(unif[b, :n] < ratio[b, :n])
        if n < k:
            assert unif[b, n] >= ratio[b, n]
            assert np.all(np.isnan(ratio[b, n + 1:]))
            # the residual excludes tokens where q >= p, the rejected one included
            assert nxt[b] != dr[b, n]
    bad = dr.copy()
    bad[0, 0] = V
    with pytest.raises(ValueError):
        oracle_mod.accept_rejection(tl, dl, "f32", bad, 1.0, 3)
