"""GPU parity of the dynamic draft list (draft_list_* in the C ABI) against
the oracle: the id array and the count must be identical after every call;
the greedy draft step over the list (lmhead_argmax, T = 1) must return the
oracle's restricted argmax where the top-1 margin exceeds 1e-3."""
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


def dev_i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def check_same(dl_gpu, dl_ref):
    torch.cuda.synchronize()
    assert dl_gpu.count() == dl_ref.count
    assert np.array_equal(dl_gpu.ids.cpu().numpy(), dl_ref.ids())


@pytest.mark.parametrize("V,n_static,cap,seed", [(500, 37, 64, 1), (248320, 32768, 4096, 2), (97, 1, 5, 3),
                                                 (4096, 300, 0, 4)])
def test_draft_list_matches_oracle_over_calls(sv, oracle, V, n_static, cap, seed):
    rng = np.random.default_rng(seed)
    static = rng.choice(V, size=n_static, replace=False).astype(np.int32)
    dl = sv.DraftList(dev_i32(static), V, cap)
    ref = oracle.draft_list_init(static, V, cap)
    check_same(dl, ref)
    for call in range(12):
        n = int(rng.integers(0, 80)) if call else 0
        # mostly fresh tokens, some repeats, some static ids, some out of range
        toks = rng.integers(-3, V + 3, size=n).astype(np.int32)
        if n > 4:
            toks[: n // 4] = rng.choice(static, size=n // 4)
            toks[n // 4: n // 3] = toks[0]
        dl.add(dev_i32(toks))
        oracle.draft_list_add(ref, toks)
        check_same(dl, ref)


def test_draft_list_prompt_sized_call_and_overflow(sv, oracle):
    """One call with a 6,000-token prompt against cap 4,096: the first 4,096
    new tokens in order, later ones dropped."""
    rng = np.random.default_rng(9)
    V = 248320
    static = rng.choice(V, size=32768, replace=False).astype(np.int32)
    toks = rng.integers(0, V, size=6000).astype(np.int32)
    dl = sv.DraftList(dev_i32(static), V, 4096)
    ref = oracle.draft_list_init(static, V, 4096)
    dl.add(dev_i32(toks))
    oracle.draft_list_add(ref, toks)
    check_same(dl, ref)
    assert ref.count == 4096
    more = rng.integers(0, V, size=100).astype(np.int32)
    dl.add(dev_i32(more))
    oracle.draft_list_add(ref, more)
    check_same(dl, ref)


def test_greedy_draft_step_over_the_list(sv, oracle):
    """lmhead_argmax with the list as vocab_map (n_static + cap entries,
    unused slots repeating the first static id) equals the oracle's argmax
    over the distinct ids of the list."""
    rng = np.random.default_rng(12)
    V, K = 6000, 768
    Wq, sc = gen.weights(rng, V, K)
    static = rng.choice(V, size=700, replace=False).astype(np.int32)
    dl = sv.DraftList(dev_i32(static), V, 256)
    ref = oracle.draft_list_init(static, V, 256)
    toks = rng.integers(0, V, size=150).astype(np.int32)
    dl.add(dev_i32(toks))
    oracle.draft_list_add(ref, toks)
    x = gen.activations(rng, 1, K)
    dx = torch.from_numpy(x.view(np.int16)).cuda()
    dW = torch.from_numpy(Wq.view(np.int32)).cuda()
    ds = torch.from_numpy(sc.view(np.int16)).cuda()
    ids, vals = sv.lmhead_argmax(dx, dW, ds, vocab_map=dl.ids)
    torch.cuda.synchronize()
    assert sv.last_device_error() == 0
    cand = np.unique(ref.ids())
    lg = oracle.lmhead_logits(x, Wq, sc, K, 1, V, rows=cand)
    a, best, second = oracle.argmax(lg, ids=cand)
    got = int(ids.cpu().item())
    assert got in set(cand.tolist())
    if best[0] - second[0] > MARGIN:
        assert got == int(a[0])
    j = int(np.where(cand == got)[0][0])
    assert abs(float(vals.cpu().item()) - float(lg[0, j])) <= 1e-4 * np.abs(lg).max()
