"""sv_verify_cycle: one verify cycle's weight reads (a layer's GEMMs, then the
lm_head verify) in one C-ABI call, captured in a CUDA graph and replayed on
new inputs, checked against the oracle -- every y element-wise within the
GEMM tolerance, accept_len and next_token as in the greedy verify tests.
Also: a bad descriptor anywhere in the cycle is refused before anything is
enqueued."""
import numpy as np
import pytest

import gen
from verify_check import check_verify

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SHAPES = (("qkv", 1024, 1280), ("gate_up", 1024, 4352), ("down", 2176, 1024))


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_verify_gb300 as m
    from speculative_verify_gb300 import build
    build.build()
    m.load()
    assert m.last_device_error() == 0
    return m


def _d16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def _d32(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).cuda()


def _check_gemm(yg, y32):
    yg = gen.bf16_bits_to_f32(yg.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
    rowmax = np.abs(y32).max(axis=1, keepdims=True)
    err = np.abs(yg - y32.astype(np.float64))
    assert np.all(err <= 1e-2 * rowmax), "tolerance 1e-2 of the row maximum violated"


@pytest.mark.parametrize("T,n_streams", [(4, 1), (8, 1), (32, 4)])
def test_captured_cycle_matches_oracle(sv, oracle, T, n_streams):
    rng = np.random.default_rng(5100 + T)
    V, Kh = 6000, 1024
    n_draft = T // n_streams - 1
    weights = [gen.weights(rng, N, K) for _, K, N in SHAPES]
    Wh, sh = gen.weights(rng, V, Kh)
    dW = [(_d32(W), _d16(s)) for W, s in weights]
    dWh, dsh = _d32(Wh), _d16(sh)
    # device input buffers the graph reads; refilled before each replay
    xs = [torch.zeros((T, K), dtype=torch.int16, device="cuda") for _, K, _ in SHAPES]
    ys = [torch.empty((T, N), dtype=torch.bfloat16, device="cuda") for _, _, N in SHAPES]
    xh = torch.zeros((T, Kh), dtype=torch.int16, device="cuda")
    dr = torch.zeros((n_streams, n_draft), dtype=torch.int32, device="cuda")
    acc = torch.full((n_streams,), -7, dtype=torch.int32, device="cuda")
    nxt = torch.full((n_streams,), -7, dtype=torch.int32, device="cuda")
    gemms = [(xs[i], dW[i][0], dW[i][1], ys[i]) for i in range(len(SHAPES))]
    verify = dict(x=xh, Wq=dWh, scales=dsh, drafts=dr, accept_len=acc, next_token=nxt)
    sv.verify_cycle(gemms, verify)          # first call outside capture
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            sv.verify_cycle(gemms, verify, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for replay in range(2):
        xh_np = gen.activations(rng, T, Kh)
        x_np = [gen.activations(rng, T, K) for _, K, _ in SHAPES]
        lg = oracle.lmhead_logits(xh_np, Wh, sh, Kh, T, V)
        a, _, _ = oracle.argmax(lg)
        drafts = np.stack([gen.drafts_with_mismatch(rng, a[s * (n_draft + 1):(s + 1) * (n_draft + 1)],
                                                    int(rng.integers(0, n_draft + 1)), V)
                           for s in range(n_streams)]).astype(np.int32)
        for i in range(len(SHAPES)):
            xs[i].copy_(_d16(x_np[i]))
        xh.copy_(_d16(xh_np))
        dr.copy_(torch.from_numpy(drafts).cuda())
        acc.fill_(-7)
        nxt.fill_(-7)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        for i, (_, K, N) in enumerate(SHAPES):
            y32, _ = oracle.w4a16_gemm(x_np[i], weights[i][0], weights[i][1], T, K, N)
            _check_gemm(ys[i], y32)
        ids, _ = sv.lmhead_argmax(xh, dWh, dsh)
        torch.cuda.synchronize()
        res = oracle.lmhead_verify(xh_np, Wh, sh, Kh, V, drafts, n_streams=n_streams)
        check_verify(res, drafts, acc.cpu().numpy(), nxt.cpu().numpy(), ids.cpu().numpy(), n_draft, n_streams)
    assert sv.last_device_error() == 0


def raw_cycle(sv, gemms):
    """sv_verify_cycle through the C ABI with raw descriptors (the binding's
    own checks would reject a bad entry before the library sees it)."""
    import ctypes
    arr = (sv.GemmCall * len(gemms))()
    for i, (x, Wq, sc, y) in enumerate(gemms):
        arr[i] = sv.GemmCall(x.data_ptr(), Wq.data_ptr(), sc.data_ptr(), x.shape[0], x.shape[1], Wq.shape[0],
                             y.data_ptr())
    return sv.load().sv_verify_cycle(arr, len(gemms), None,
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_cycle_refuses_a_bad_entry_before_enqueuing(sv):
    """The second GEMM's output is misaligned: the call returns SV_ERR_ALIGN
    and the first GEMM, though valid, was not enqueued (its output keeps
    the value written before)."""
    rng = np.random.default_rng(5200)
    T, K, N = 4, 1024, 640
    W, s = gen.weights(rng, N, K)
    x = _d16(gen.activations(rng, T, K))
    dW, ds = _d32(W), _d16(s)
    y1 = torch.full((T, N), 7.0, dtype=torch.bfloat16, device="cuda")
    y2 = torch.full((T * N + 8,), 7.0, dtype=torch.bfloat16, device="cuda")
    bad_y = y2[1:1 + T * N].view(T, N)          # 2-byte offset: not 16-byte aligned
    torch.cuda.synchronize()
    assert raw_cycle(sv, [(x, dW, ds, y1), (x, dW, ds, bad_y)]) == -3
    torch.cuda.synchronize()
    assert bool((y1.float() == 7.0).all()), "a refused cycle enqueued work"
    assert raw_cycle(sv, [(x, dW, ds, y1)]) == 0
    torch.cuda.synchronize()
    assert not bool((y1.float() == 7.0).all())
