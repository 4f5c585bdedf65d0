"""lmhead_verify_noalloc: the verify for callers that cannot allocate GPU
memory when they call -- serving runtimes that hand out every device byte
from their own arena, latency-critical paths that cannot take cudaMalloc's
implicit synchronisation.  Its scratch is a fixed array inside the library,
so the call itself never allocates.

The test drives it through the C ABI, twice in a row on the same inputs and
once more on other drafts, and requires exactly the results of the regular
lmhead_verify (same kernel, same launch shape), and the CPU oracle's outcome
(bit-exact where the deciding rows' top-1 margin exceeds 1e-3, else one of
the correct outcomes).  Across its calls after the first, the device's free
memory must not change.  The file is named so that pytest collects it last;
it needs no state left by other tests.
"""
import ctypes

import numpy as np
import pytest

import gen
from verify_check import check_verify

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_verify_gb300 as sv
    from speculative_verify_gb300 import build
    build.build()
    return sv.load()


def _dev(a, dt):
    return torch.from_numpy(np.ascontiguousarray(a).view(dt)).cuda()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def resident_vocab(K):
    """A vocabulary large enough that the call takes the resident-activation
    path (at least 80 units of 64 rows x 128 columns per thread block)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return (80 * sms + K // 128 - 1) // (K // 128) * 64 + 37


@pytest.mark.parametrize("V,K,n_draft,n_map", [(30011, 1024, 3, 0), (20000, 512, 7, 5000),
                                                 (9000, 1280, 15, 0), (7000, 768, 31, 3000),
                                                 ("resident", 1024, 3, 0)])
def test_noalloc_matches_regular_entry_point(lib, oracle, V, K, n_draft, n_map):
    if V == "resident":
        V = resident_vocab(K)
    rng = np.random.default_rng(4242 + V + n_map)
    Wq, sc = gen.weights(rng, V, K)
    T = n_draft + 1
    x = gen.activations(rng, T, K)
    vm = gen.vocab_map(rng, V, n_map) if n_map else None
    a, _, _ = oracle.argmax(oracle.lmhead_logits(x, Wq, sc, K, T, V, rows=vm), ids=vm)
    dx, dW, ds = _dev(x, np.int16), _dev(Wq, np.int32), _dev(sc, np.int16)
    dvm = None if vm is None else _dev(vm, np.int32)
    n_map_arg = 0 if vm is None else vm.size
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    draft_sets = [gen.drafts_with_mismatch(rng, a, 1, V, pool=vm),
                  gen.drafts_with_mismatch(rng, a, n_draft, V, pool=vm)]
    acc_r = torch.empty(1, dtype=torch.int32, device="cuda")
    nxt_r = torch.empty(1, dtype=torch.int32, device="cuda")
    acc_n = torch.empty(1, dtype=torch.int32, device="cuda")
    nxt_n = torch.empty(1, dtype=torch.int32, device="cuda")
    ids = torch.empty(T, dtype=torch.int32, device="cuda")
    # the GPU's per-row argmax ids (regular entry point), for the near-tie check
    rc = lib.lmhead_argmax(_p(dx), _p(dW), _p(ds), K, T, None if dvm is None else _p(dvm), n_map_arg, V,
                           _p(ids), None, stream)
    assert rc == 0
    dds = [_dev(d.astype(np.int32), np.int32) for d in draft_sets]
    torch.cuda.synchronize()
    free_after_first = None
    for call, di in enumerate([0, 0, 1]):
        d, dd = draft_sets[di], dds[di]
        acc_r.fill_(-7)
        acc_n.fill_(-7)
        rc = lib.lmhead_verify(_p(dx), _p(dW), _p(ds), K, _p(dd), n_draft,
                               None if dvm is None else _p(dvm), n_map_arg, V, _p(acc_r), _p(nxt_r),
                               stream)
        assert rc == 0
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        rc = lib.lmhead_verify_noalloc(_p(dx), _p(dW), _p(ds), K, _p(dd), n_draft,
                                       None if dvm is None else _p(dvm), n_map_arg, V, _p(acc_n),
                                       _p(nxt_n), stream)
        assert rc == 0, "lmhead_verify_noalloc returned %d on call %d" % (rc, call)
        torch.cuda.synchronize()
        free_now = torch.cuda.mem_get_info()[0]
        if call == 0:
            free_after_first = free_now
        else:
            # no device memory taken by the calls after the first
            assert free_now == free_before == free_after_first, (call, free_before, free_now)
        assert int(acc_n.item()) == int(acc_r.item()), call
        assert int(nxt_n.item()) == int(nxt_r.item()), call
        ref = oracle.lmhead_verify(x, Wq, sc, K, V, d, vocab_map=vm)
        check_verify(ref, d, acc_n.cpu().numpy(), nxt_n.cpu().numpy(), ids.cpu().numpy(), n_draft, 1, vm)


def test_noalloc_rejects_too_many_drafts(lib):
    buf = torch.zeros(64, dtype=torch.int32, device="cuda")
    rc = lib.lmhead_verify_noalloc(_p(buf), _p(buf), _p(buf), 128, _p(buf), 32, None, 0, 16,
                                   _p(buf), _p(buf), None)
    assert rc == -2


def test_noalloc_rejects_long_rows_with_more_than_7_drafts(lib):
    """With more than 7 drafts the activations go through the library's
    fixed conversion buffer, sized for K <= 16384: a longer row is refused
    before anything is enqueued."""
    buf = torch.zeros(64, dtype=torch.int32, device="cuda")
    out = torch.full((2,), -7, dtype=torch.int32, device="cuda")
    rc = lib.lmhead_verify_noalloc(_p(buf), _p(buf), _p(buf), 16384 + 128, _p(buf), 15, None, 0, 16,
                                   _p(out), _p(out[1:]), None)
    assert rc == -2
    torch.cuda.synchronize()
    assert out.tolist() == [-7, -7]
