"""GPU parity of the rescored verify (lmhead_verify_rescored /
lmhead_argmax_rescored) against the oracle: the int4 head's top-k candidates
of every row, rescored with the bf16 head.

Bit-exact ids are required where both decisions are clear of fp32
reordering: the gap between the k-th and (k+1)-th int4 logit (which fixes the
candidate set) and the margin between the two best bf16 logits among the
candidates both exceed 1e-3.  Otherwise the GPU's id must be one of the
candidates within 1e-3 of the best."""
import numpy as np
import pytest

import gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MARGIN = 1e-3


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


def bf16_head(rng, V, K, scale=0.02):
    return gen.f32_to_bf16_bits((rng.standard_normal((V, K)) * scale).astype(np.float32))


def check_rows(ids, vals, ref):
    for t in range(ids.size):
        cand = ref.cand[t].tolist()
        assert int(ids[t]) in cand
        j = cand.index(int(ids[t]))
        best = float(ref.bf16[t].max())
        assert float(ref.bf16[t, j]) >= best - MARGIN
        assert abs(float(vals[t]) - float(ref.bf16[t, j])) <= 1e-4 * max(1.0, np.abs(ref.bf16[t]).max())
        if ref.cand_gap[t] > MARGIN and ref.margin[t] > MARGIN:
            assert int(ids[t]) == int(ref.a[t]), t


@pytest.mark.parametrize("V,K,T,k,seed", [(3000, 768, 4, 16, 1), (20000, 1024, 8, 64, 2), (500, 256, 1, 1, 3),
                                          (7000, 5120, 4, 32, 4), (64, 128, 2, 64, 5)])
def test_rescored_argmax_matches_oracle(sv, oracle, V, K, T, k, seed):
    rng = np.random.default_rng(800 + seed)
    Wq, sc = gen.weights(rng, V, K)
    Wbf = bf16_head(rng, V, K)
    x = gen.activations(rng, T, K)
    ref = oracle.lmhead_verify_rescored(x, Wq, sc, Wbf, K, V, np.zeros(T - 1, np.int32), k)
    ids, vals = sv.lmhead_argmax_rescored(dev16(x), dev32(Wq), dev16(sc), dev16(Wbf), top_k=k)
    torch.cuda.synchronize()
    check_rows(ids.cpu().numpy(), vals.cpu().numpy(), ref)


def test_rescored_verify_accept_len_and_next_token(sv, oracle):
    rng = np.random.default_rng(870)
    V, K, n_draft, k = 4096, 512, 3, 16
    Wq, sc = gen.weights(rng, V, K)
    Wbf = bf16_head(rng, V, K)
    x = gen.activations(rng, n_draft + 1, K)
    ref0 = oracle.lmhead_verify_rescored(x, Wq, sc, Wbf, K, V, np.zeros(n_draft, np.int32), k)
    for p in range(n_draft + 1):
        drafts = gen.drafts_with_mismatch(rng, ref0.a, p, V)
        ref = oracle.lmhead_verify_rescored(x, Wq, sc, Wbf, K, V, drafts, k)
        acc, nxt = sv.lmhead_verify_rescored(dev16(x), dev32(Wq), dev16(sc), dev16(Wbf), dev32(drafts), top_k=k)
        torch.cuda.synchronize()
        clear = all(ref.cand_gap[t] > MARGIN and ref.margin[t] > MARGIN for t in range(int(ref.accept_len[0]) + 1))
        if clear:
            assert int(acc.item()) == int(ref.accept_len[0]) == p
            assert int(nxt.item()) == int(ref.next_token[0])


def test_rescored_planted_flip(sv):
    """The int4 head ranks row 5 first and row 9 second; the bf16 head
    prefers row 9: one candidate gives 5, two or more give 9."""
    V, K = 16, 128
    Wq = np.full((V, K // 8), 0x88888888, np.uint32)
    Wq[5] = 0xFFFFFFFF
    Wq[9] = 0xEEEEEEEE
    sc = np.full((V, 1), gen.f32_to_bf16_bits(np.float32(1.0)), np.uint16)
    Wbf = np.zeros((V, K), np.uint16)
    Wbf[5] = gen.f32_to_bf16_bits(np.float32(1.0))
    Wbf[9] = gen.f32_to_bf16_bits(np.float32(2.0))
    x = np.full((1, K), gen.f32_to_bf16_bits(np.float32(1.0)), np.uint16)
    got = {}
    for k in (1, 2, 16):
        ids, vals = sv.lmhead_argmax_rescored(dev16(x), dev32(Wq), dev16(sc), dev16(Wbf), top_k=k)
        torch.cuda.synchronize()
        got[k] = (int(ids.item()), float(vals.item()))
    assert got[1] == (5, 128.0)
    assert got[2] == (9, 256.0)
    assert got[16] == (9, 256.0)


def test_rescored_with_one_candidate_is_the_int4_argmax(sv, oracle):
    rng = np.random.default_rng(880)
    V, K, T = 5000, 640, 4
    Wq, sc = gen.weights(rng, V, K)
    Wbf = bf16_head(rng, V, K)
    x = gen.activations(rng, T, K)
    ids1, _ = sv.lmhead_argmax_rescored(dev16(x), dev32(Wq), dev16(sc), dev16(Wbf), top_k=1)
    ids4, _ = sv.lmhead_argmax(dev16(x), dev32(Wq), dev16(sc))
    torch.cuda.synchronize()
    assert torch.equal(ids1, ids4)


def test_rescored_candidates_clustered_in_one_slice(sv, oracle):
    """Rows 1000..1127 (one 128-row slice) get 8x the scales, so most of the
    k best int4 logits sit in that slice: the threshold from the slices'
    maxima must still keep all of them."""
    rng = np.random.default_rng(890)
    V, K, T, k = 5000, 256, 3, 64
    Wq, sc = gen.weights(rng, V, K)
    f = (sc.astype(np.uint32) << 16).view(np.float32).copy()
    f[1000:1128] *= 8.0
    sc = gen.f32_to_bf16_bits(f)
    Wbf = bf16_head(rng, V, K)
    x = gen.activations(rng, T, K)
    ref = oracle.lmhead_verify_rescored(x, Wq, sc, Wbf, K, V, np.zeros(T - 1, np.int32), k)
    assert sum(1000 <= c < 1128 for c in ref.cand[0].tolist()) > 32
    ids, vals = sv.lmhead_argmax_rescored(dev16(x), dev32(Wq), dev16(sc), dev16(Wbf), top_k=k)
    torch.cuda.synchronize()
    check_rows(ids.cpu().numpy(), vals.cpu().numpy(), ref)


@pytest.mark.parametrize("k", [16, 64])
def test_rescored_maxima_clustered_in_one_chunk(sv, oracle, k):
    """Rows 0..16383 (the slices of the first chunk of 128 slice maxima) get
    8x the scales: the first threshold (the k-th best of every chunk's 8
    best maxima) is then reached by far more than 64 slices and the exact
    threshold must take over."""
    rng = np.random.default_rng(900 + k)
    V, K, T = 248320, 256, 2
    Wq, sc = gen.weights(rng, V, K)
    f = (sc.astype(np.uint32) << 16).view(np.float32).copy()
    f[:16384] *= 8.0
    sc = gen.f32_to_bf16_bits(f)
    Wbf = bf16_head(rng, V, K)
    x = gen.activations(rng, T, K)
    ref = oracle.lmhead_verify_rescored(x, Wq, sc, Wbf, K, V, np.zeros(T - 1, np.int32), k)
    assert all(c < 16384 for c in ref.cand[0].tolist())
    ids, vals = sv.lmhead_argmax_rescored(dev16(x), dev32(Wq), dev16(sc), dev16(Wbf), top_k=k)
    torch.cuda.synchronize()
    check_rows(ids.cpu().numpy(), vals.cpu().numpy(), ref)
