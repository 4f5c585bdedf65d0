"""GPU parity of the exact speculative sampling verify
(lmhead_verify_sampled / lmhead_sampling_dist) against the oracle.

The kernel and the oracle take every decision in fp32 in the same order;
they can still differ where the GPU's fp32 logits (another summation order)
or its expf move a decision across its threshold.  So ids and outcomes are
compared exactly where the oracle reports every decision on the path clear
of rounding (relative margin >= 1e-4, candidate orders >= 1e-3 apart), and
probabilities within 1e-4 everywhere the kept set is the same."""
import numpy as np
import pytest

import gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CHAINS = [dict(temperature=1.0), dict(temperature=0.7, top_k=20, top_p=0.95),
          dict(temperature=1.3, top_p=0.9, min_p=0.05), dict(temperature=0.5, top_k=5),
          dict(temperature=1.0, min_p=0.3), dict(temperature=0.0)]


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_verify_gb300 as m
    from speculative_verify_gb300 import build
    build.build()
    m.load()
    return m


def dev16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def dev32(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).cuda()


def devf(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def head(seed, V, K, T, spread=1.0):
    rng = np.random.default_rng(seed)
    Wq, sc = gen.weights(rng, V, K)
    if spread != 1.0:
        f = (sc.astype(np.uint32) << 16).view(np.float32) * np.float32(spread)
        sc = gen.f32_to_bf16_bits(f)
    x = gen.activations(rng, T, K)
    return rng, Wq, sc, x


def chain_args(c):
    return (c.get("temperature", 1.0), c.get("top_k", 0), c.get("top_p", 1.0), c.get("min_p", 0.0))


@pytest.mark.parametrize("V,K,T,seed", [(3000, 256, 3, 1), (20000, 1024, 8, 2), (20, 128, 2, 3),
                                        (7001, 640, 1, 4), (300000, 128, 2, 5)])
@pytest.mark.parametrize("ci", range(len(CHAINS)))
def test_sampling_distribution_matches_oracle(sv, oracle, V, K, T, seed, ci):
    chain = CHAINS[ci]
    _, Wq, sc, x = head(seed, V, K, T)
    logits = oracle.lmhead_logits(x, Wq, sc, K, T, V)
    ref = oracle.verify_sampled_from_logits(logits, np.zeros(T - 1, np.int32), np.zeros(2 * T), **chain)
    ids, probs = sv.lmhead_sampling_dist(dev16(x), dev32(Wq), dev16(sc), *chain_args(chain))
    torch.cuda.synchronize()
    ids, probs = ids.cpu().numpy(), probs.cpu().numpy()
    checked = 0
    for t in range(T):
        d = ref.dists[t]
        if not d.cut_clear(1e-4, 1e-3):
            continue
        n = d.ids.size
        assert (ids[t, n:] == -1).all() and (probs[t, n:] == 0).all()
        got = dict(zip(ids[t, :n].tolist(), probs[t, :n].tolist()))
        want = dict(zip(d.ids.tolist(), (d.w / d.W).tolist()))
        assert set(got) == set(want), t
        for k, v in want.items():
            assert abs(got[k] - v) <= 1e-4, (t, k, got[k], v)
        assert abs(sum(got.values()) - 1.0) <= 1e-5
        checked += 1
    assert checked >= T // 2


def drafts_for(rng, ref_dists, n_draft, V):
    """Per row: the best candidate, a random kept one, or a token outside."""
    out = np.empty(n_draft, np.int32)
    for i in range(n_draft):
        d = ref_dists[i]
        r = rng.random()
        if r < 0.5:
            out[i] = d.ids[0]
        elif r < 0.85:
            out[i] = d.ids[rng.integers(0, d.ids.size)]
        else:
            out[i] = (int(d.ids.max()) + 1 + rng.integers(0, 50)) % V
    return out


@pytest.mark.parametrize("V,K,n_draft,seed", [(5000, 512, 3, 11), (30000, 768, 7, 12), (600, 128, 1, 13),
                                              (4000, 256, 0, 14)])
@pytest.mark.parametrize("ci", [0, 1, 2, 5])
def test_sampled_verify_matches_oracle(sv, oracle, V, K, n_draft, seed, ci):
    chain = CHAINS[ci]
    T = n_draft + 1
    rng, Wq, sc, x = head(seed, V, K, T, spread=0.5)
    logits = oracle.lmhead_logits(x, Wq, sc, K, T, V)
    base = oracle.verify_sampled_from_logits(logits, np.zeros(n_draft, np.int32), np.zeros(2 * T), **chain)
    dx, dW, ds = dev16(x), dev32(Wq), dev16(sc)
    clear = 0
    trials = 24
    for _ in range(trials):
        drafts = drafts_for(rng, base.dists, n_draft, V)
        u = rng.random(2 * T).astype(np.float32)
        ref = oracle.verify_sampled_from_logits(logits, drafts, u, **chain)
        acc, nxt = sv.lmhead_verify_sampled(dx, dW, ds, dev32(drafts), devf(u), *chain_args(chain))
        torch.cuda.synchronize()
        if ref.clear:
            clear += 1
            assert (int(acc.item()), int(nxt.item())) == (ref.accept_len, ref.next_token)
        else:
            assert 0 <= int(acc.item()) <= n_draft
    assert clear >= trials // 2


def test_temperature_zero_is_the_greedy_verify(sv, oracle):
    V, K, n_draft = 9000, 640, 4
    rng, Wq, sc, x = head(21, V, K, n_draft + 1)
    ref = oracle.lmhead_verify(x, Wq, sc, K, V, np.zeros(n_draft, np.int32))
    dx, dW, ds = dev16(x), dev32(Wq), dev16(sc)
    for p in range(n_draft + 1):
        drafts = gen.drafts_with_mismatch(rng, ref.a, p, V)
        u = devf(rng.random(2 * (n_draft + 1)))
        acc, nxt = sv.lmhead_verify_sampled(dx, dW, ds, dev32(drafts), u, temperature=0.0)
        acc_g, nxt_g = sv.lmhead_verify(dx, dW, ds, dev32(drafts))
        torch.cuda.synchronize()
        assert (int(acc.item()), int(nxt.item())) == (int(acc_g.item()), int(nxt_g.item()))
        if all(ref.margin[: p + 1] > 1e-3):
            assert int(acc.item()) == p and int(nxt.item()) == int(ref.a[p])


def test_gpu_emitted_token_is_distributed_as_without_drafts(sv, oracle):
    """The engine's own check: 2000 draws per position, with a draft on the
    row, follow the drafts-free distribution (chi-square at 99.9%)."""
    stats = pytest.importorskip("scipy.stats")
    V, K = 3000, 256
    rng, Wq, sc, x = head(31, V, K, 2, spread=0.25)
    chain = dict(temperature=1.0, top_k=20, top_p=0.95)
    ids, probs = sv.lmhead_sampling_dist(dev16(x), dev32(Wq), dev16(sc), *chain_args(chain))
    ids, probs = ids.cpu().numpy()[0], probs.cpu().numpy()[0].astype(np.float64)
    n = int((ids >= 0).sum())
    assert n >= 3
    draft = int(ids[1])                  # a kept candidate, not the best
    N = 2000
    us = devf(rng.random((N, 4)))
    dx, dW, ds, dd = dev16(x), dev32(Wq), dev16(sc), dev32(np.array([draft], np.int32))
    acc_all = torch.empty(N, dtype=torch.int32, device="cuda")
    nxt_all = torch.empty(N, dtype=torch.int32, device="cuda")
    for i in range(N):
        sv.lmhead_verify_sampled(dx, dW, ds, dd, us[i], *chain_args(chain), accept_len=acc_all[i:i + 1],
                                 next_token=nxt_all[i:i + 1])
    torch.cuda.synchronize()
    acc, nxt = acc_all.cpu().numpy(), nxt_all.cpu().numpy()
    tok0 = np.where(acc >= 1, draft, nxt)
    pos = {int(t): j for j, t in enumerate(ids[:n])}
    assert all(int(t) in pos for t in tok0)
    obs = np.bincount([pos[int(t)] for t in tok0], minlength=n).astype(np.float64)
    exp = probs[:n] * N
    stat = float(((obs - exp) ** 2 / exp).sum())
    assert stat < stats.chi2.ppf(0.999, df=n - 1), (stat, n)
    pd = probs[1]
    assert abs(int((acc >= 1).sum()) - N * pd) <= 4.5 * np.sqrt(N * pd * (1 - pd)) + 1


def test_sampled_verify_full_size_head(sv, oracle):
    """The lm_head at full size (V = 248,320, K = 5120), four rows."""
    V, K, n_draft = gen.VOCAB, gen.HIDDEN, 3
    rng, Wq, sc, x = head(41, V, K, n_draft + 1)
    logits = oracle.lmhead_logits(x, Wq, sc, K, n_draft + 1, V)
    chain = CHAINS[1]
    base = oracle.verify_sampled_from_logits(logits, np.zeros(n_draft, np.int32), np.zeros(8), **chain)
    dx, dW, ds = dev16(x), dev32(Wq), dev16(sc)
    clear = 0
    for _ in range(8):
        drafts = drafts_for(rng, base.dists, n_draft, V)
        u = rng.random(8).astype(np.float32)
        ref = oracle.verify_sampled_from_logits(logits, drafts, u, **chain)
        acc, nxt = sv.lmhead_verify_sampled(dx, dW, ds, dev32(drafts), devf(u), *chain_args(chain))
        torch.cuda.synchronize()
        if ref.clear:
            clear += 1
            assert (int(acc.item()), int(nxt.item())) == (ref.accept_len, ref.next_token)
    assert clear >= 4


def test_sampling_distribution_with_maxima_clustered_in_one_chunk(sv, oracle):
    """Rows 0..16383 get 8x the scales, so the row's 32 best logits all sit
    in the first chunk of slice maxima: the exact threshold takes over."""
    V, K, T = 248320, 256, 2
    rng = np.random.default_rng(51)
    Wq, sc = gen.weights(rng, V, K)
    f = (sc.astype(np.uint32) << 16).view(np.float32).copy()
    f[:16384] *= 8.0
    sc = gen.f32_to_bf16_bits(f)
    x = gen.activations(rng, T, K)
    logits = oracle.lmhead_logits(x, Wq, sc, K, T, V)
    ref = oracle.verify_sampled_from_logits(logits, np.zeros(T - 1, np.int32), np.zeros(2 * T), temperature=1.0)
    ids, probs = sv.lmhead_sampling_dist(dev16(x), dev32(Wq), dev16(sc), 1.0, 0, 1.0, 0.0)
    torch.cuda.synchronize()
    ids, probs = ids.cpu().numpy(), probs.cpu().numpy()
    checked = 0
    for t in range(T):
        d = ref.dists[t]
        assert all(c < 16384 for c in d.ids.tolist())
        if not d.cut_clear(1e-4, 1e-3):
            continue
        got = dict(zip(ids[t].tolist(), probs[t].tolist()))
        want = dict(zip(d.ids.tolist(), (d.w / d.W).tolist()))
        assert set(got) == set(want)
        for k, v in want.items():
            assert abs(got[k] - v) <= 1e-4
        checked += 1
    assert checked >= 1
