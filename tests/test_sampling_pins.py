"""Pins of the oracle's exact speculative sampling verify (no GPU).

What they fix, beyond the oracle's own arithmetic:
  * closed forms of the sampling chain on hand-sized logits (top-k, top-p,
    min-p, temperature, each in llama.cpp's order);
  * with every filter off, the distribution is the softmax of the 32 best
    logits (scipy's softmax);
  * temperature 0 reduces to the greedy verify;
  * the pages' correctness claim itself: with drafts, the emitted token is
    distributed exactly as without them (Monte Carlo over the uniforms, as
    the engine's 2000-sample test per position), and the accept rate of a
    draft is p(draft).  A planted mistake (resampling without removing the
    rejected draft) must fail the same test.
"""
import math

import numpy as np
import pytest

scipy_special = pytest.importorskip("scipy.special")
scipy_stats = pytest.importorskip("scipy.stats")


def probs(d):
    return (d.w / d.W).astype(np.float64)


def test_top_p_closed_forms(oracle):
    v = np.array([2.0, 1.0, 0.0, -1.0], np.float32)
    ids = np.arange(4, dtype=np.int32)
    e = [math.exp(-j) for j in range(4)]
    S = sum(e)
    # cumulative softmax: 0.644, 0.881, 0.968, 1.0
    for top_p, keep in [(0.5, 1), (0.8, 2), (0.95, 3), (0.99, 4)]:
        d = oracle.sampling_dist(v, ids, 1.0, top_p=top_p)
        assert d.ids.tolist() == list(range(keep))
        want = np.array(e[:keep]) / sum(e[:keep])
        assert np.allclose(probs(d), want, rtol=0, atol=1e-6)
    assert abs(sum(e[:2]) / S - 0.8807970779778823) < 1e-12


def test_min_p_closed_forms(oracle):
    v = np.array([2.0, 1.0, 0.0, -1.0], np.float32)
    ids = np.array([7, 3, 9, 1], np.int32)
    # exp(l - max) = 1, 0.368, 0.135, 0.0498
    for min_p, keep in [(0.5, 1), (0.2, 2), (0.1, 3), (0.04, 4)]:
        d = oracle.sampling_dist(v, ids, 1.0, min_p=min_p)
        assert d.ids.tolist() == [7, 3, 9, 1][:keep]


def test_top_k_then_temperature_closed_form(oracle):
    v = np.array([2.0, 1.0, 0.0, -1.0], np.float32)
    d = oracle.sampling_dist(v, np.arange(4, dtype=np.int32), 0.5, top_k=3)
    want = np.array([1.0, math.exp(-2.0), math.exp(-4.0)])
    assert np.allclose(probs(d), want / want.sum(), rtol=0, atol=1e-6)


def test_order_top_p_before_temperature(oracle):
    """top-p sees the temperature-1 distribution: at temperature 0.25 the
    same two candidates survive top_p = 0.8 as at temperature 1."""
    v = np.array([2.0, 1.0, 0.0, -1.0], np.float32)
    d = oracle.sampling_dist(v, np.arange(4, dtype=np.int32), 0.25, top_p=0.8)
    assert d.ids.tolist() == [0, 1]
    want = np.array([1.0, math.exp(-4.0)])
    assert np.allclose(probs(d), want / want.sum(), rtol=0, atol=1e-6)


def test_filters_off_is_softmax_of_the_32_best(oracle):
    rng = np.random.default_rng(5)
    logits = (rng.standard_normal((1, 1000)) * 3).astype(np.float32)
    order = np.argsort(-logits[0], kind="stable")[:32]
    r = oracle.verify_sampled_from_logits(logits, [], [0.5, 0.5], 1.0)
    d = r.dists[0]
    assert d.ids.tolist() == order.tolist()
    want = scipy_special.softmax(logits[0][order].astype(np.float64))
    assert np.allclose(probs(d), want, rtol=0, atol=1e-6)


def test_temperature_zero_is_the_greedy_verify(oracle):
    rng = np.random.default_rng(6)
    T = 5
    logits = (rng.standard_normal((T, 300)) * 2).astype(np.float32)
    a = np.argmax(logits, axis=1).astype(np.int32)
    for p in range(T):
        drafts = a[:T - 1].copy()
        if p < T - 1:
            drafts[p] = (drafts[p] + 1) % 300
        u = rng.random(2 * T).astype(np.float32)
        r = oracle.verify_sampled_from_logits(logits, drafts, u, 0.0)
        acc, nxt = oracle.verify(a, drafts)
        assert (r.accept_len, r.next_token) == (acc, nxt) == (p, int(a[p]))


def test_top_k_one_ignores_the_uniforms(oracle):
    rng = np.random.default_rng(7)
    logits = (rng.standard_normal((3, 200)) * 2).astype(np.float32)
    a = np.argmax(logits, axis=1)
    for _ in range(20):
        u = rng.random(6).astype(np.float32)
        r = oracle.verify_sampled_from_logits(logits, [int(a[0]), 5], u, 0.8, top_k=1)
        want_acc = 2 if int(a[1]) == 5 else 1
        assert r.accept_len == want_acc
        assert r.next_token == int(a[want_acc])


def test_draft_outside_the_kept_set_is_never_accepted(oracle):
    rng = np.random.default_rng(8)
    logits = (rng.standard_normal((2, 500)) * 2).astype(np.float32)
    worst = int(np.argmin(logits[0]))
    for _ in range(50):
        r = oracle.verify_sampled_from_logits(logits, [worst], rng.random(4).astype(np.float32), 1.0)
        assert r.accept_len == 0 and r.next_token != worst


def _monte_carlo(oracle, logits, draft, n, seed, **chain):
    rng = np.random.default_rng(seed)
    first = {}
    second = {}
    accepted = 0
    for _ in range(n):
        u = rng.random(4).astype(np.float32)
        r = oracle.verify_sampled_from_logits(logits, [draft], u, **chain)
        tok0 = draft if r.accept_len >= 1 else r.next_token
        first[tok0] = first.get(tok0, 0) + 1
        if r.accept_len >= 1:
            accepted += 1
            second[r.next_token] = second.get(r.next_token, 0) + 1
    return first, second, accepted


def _chi2(counts, dist, n):
    p = probs(dist)
    ids = dist.ids.tolist()
    assert set(counts) <= set(ids), "a token outside the sampling distribution was emitted"
    obs = np.array([counts.get(t, 0) for t in ids], np.float64)
    exp = p * n
    stat = float(((obs - exp) ** 2 / exp).sum())
    return stat, scipy_stats.chi2.ppf(0.999, df=max(1, len(ids) - 1))


CHAIN = dict(temperature=0.7, top_k=20, top_p=0.95)   # one of the settings measured on the pages


@pytest.mark.parametrize("rank", [0, 3, 60])
def test_emitted_token_is_distributed_as_without_drafts(oracle, rank):
    """The first emitted token follows p_0 whatever the draft (the top
    candidate, a mid-ranked one, one outside the kept set); the draft is
    accepted at rate p_0(draft); given acceptance the bonus token follows p_1."""
    rng = np.random.default_rng(40 + rank)
    logits = (rng.standard_normal((2, 80)) * 1.5).astype(np.float32)
    draft = int(np.argsort(-logits[0], kind="stable")[rank])
    n = 6000
    first, second, accepted = _monte_carlo(oracle, logits, draft, n, seed=rank, **CHAIN)
    r0 = oracle.verify_sampled_from_logits(logits, [draft], [0.5] * 4, **CHAIN)
    d0, d1 = r0.dists
    stat, bound = _chi2(first, d0, n)
    assert stat < bound, (stat, bound)
    pd = float(probs(d0)[d0.ids.tolist().index(draft)]) if draft in d0.ids.tolist() else 0.0
    assert abs(accepted - n * pd) <= 4.5 * math.sqrt(n * pd * (1 - pd)) + 1
    if accepted > 500:
        stat1, bound1 = _chi2(second, d1, accepted)
        assert stat1 < bound1, (stat1, bound1)


def test_planted_residual_mistake_is_caught(oracle, monkeypatch):
    """Drawing the replacement from p itself (not from p without the
    rejected draft) over-weights the draft; the same test must reject it."""
    real = oracle.sample_from
    monkeypatch.setattr(oracle, "sample_from", lambda dist, u, exclude=None: real(dist, u, None))
    rng = np.random.default_rng(40)
    logits = (rng.standard_normal((2, 80)) * 1.5).astype(np.float32)
    draft = int(np.argsort(-logits[0], kind="stable")[0])
    n = 6000
    first, _, _ = _monte_carlo(oracle, logits, draft, n, seed=0, **CHAIN)
    r0 = oracle.verify_sampled_from_logits(logits, [draft], [0.5] * 4, **CHAIN)
    stat, bound = _chi2(first, r0.dists[0], n)
    assert stat > bound
