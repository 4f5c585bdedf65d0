"""Calls with 17 <= T <= 32 and K a multiple of 1024 on both of their
kernels -- the tcgen05 kernel (5th-generation tensor cores, accumulators in
tensor memory; the default) and the mma.sync kernel (sv_debug_set_tcgen05(0))
-- against the CPU oracle: the
one-hot pin of the levels' order in tensor memory against the activations'
K-major layout, wide-range activations, GEMM shapes with split tiles, and the
greedy verify up to the full four-stream lm_head."""
import numpy as np
import pytest

import gen
from test_parity_gpu import (assert_gemm_close, dev_bits16, dev_words, run_head_case, to_f32,
                             wide_range_activations)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=["tcgen05", "mma_sync"])
def sv(request):
    """The library with calls of 17 <= T <= 32 on the tcgen05 kernel (the
    default) and, for the second pass, on the mma.sync kernel."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_verify_gb300 as m
    from speculative_verify_gb300 import build
    build.build()
    m.load()
    assert m.last_device_error() == 0
    m.debug_set_tcgen05(request.param == "tcgen05")
    yield m
    m.debug_set_tcgen05(True)


def test_one_hot_pins_tensor_memory_layout(sv, oracle):
    """The same one-hot pin through the tcgen05 kernel (32 token rows, K a
    multiple of 1024): x = e_k gives y[n] = (nibble - 8) * s exactly for
    every k, which pins the levels' order in tensor memory against the
    activations' K-major layout, the swizzled weight rows and the scale
    ring."""
    K, N = 1024, 300
    W = K // 8
    rng = np.random.default_rng(61)
    Wq = rng.integers(0, 2**32, size=(N, W), dtype=np.uint32)
    Wq[:16, :] = np.array([int(("%x" % n) * 8, 16) for n in range(16)], np.uint32)[:, None]
    lv = ((Wq[:, :, None] >> (4 * np.arange(8, dtype=np.uint32))) & 0xF).reshape(N, K).astype(np.int64) - 8
    s = gen.f32_to_bf16_bits((2.0 ** rng.integers(-4, 3, size=(N, K // 128))).astype(np.float32))
    sval = gen.bf16_bits_to_f32(s).astype(np.float64)
    one = gen.f32_to_bf16_bits(np.float32(1.0))
    for k0 in range(0, K, 32):
        x = np.zeros((32, K), np.uint16)
        x[np.arange(32), k0 + np.arange(32)] = one
        y = sv.w4a16_gemm(dev_bits16(x), dev_words(Wq), dev_bits16(s))
        torch.cuda.synchronize()
        got = to_f32(y).astype(np.float64)
        ks = k0 + np.arange(32)
        expect = (lv[:, ks] * sval[:, ks // 128]).T
        assert np.array_equal(got, expect), k0
    assert sv.last_device_error() == 0


def test_scales_spanning_a_box(sv, oracle):
    """Group scales 2^e with e spread over 2^+-20 inside each row's box of
    eight groups, and rows whose smallest group scale is 2^-40 of the
    largest.  One-hot activations give y = (nibble - 8) * s for one column of
    each group.  The tcgen05 kernel forms level * s * 2^(137 - E) in fp16 per
    box of eight groups (E the row's largest scale exponent in the box): the
    product is exact whenever s is at least 2^-27 of the box's largest scale,
    and otherwise off by less than 2^-30 of the largest.  The mma.sync kernel
    scales in fp32 and is exact everywhere."""
    K, N, T = 1024, 256, 32
    W = K // 8
    rng = np.random.default_rng(77)
    Wq = rng.integers(0, 2**32, size=(N, W), dtype=np.uint32)
    lv = ((Wq[:, :, None] >> (4 * np.arange(8, dtype=np.uint32))) & 0xF).reshape(N, K).astype(np.int64) - 8
    e = rng.integers(-20, 21, size=(N, K // 128))
    e[N // 2:, 0] = e[N // 2:, 1:].max(axis=1) - 40     # far below the box's largest
    s = gen.f32_to_bf16_bits((2.0 ** e).astype(np.float32))
    sval = gen.bf16_bits_to_f32(s).astype(np.float64)
    one = gen.f32_to_bf16_bits(np.float32(1.0))
    ks = 32 * np.arange(T)                               # four columns of every group
    x = np.zeros((T, K), np.uint16)
    x[np.arange(T), ks] = one
    y = sv.w4a16_gemm(dev_bits16(x), dev_words(Wq), dev_bits16(s))
    torch.cuda.synchronize()
    got = to_f32(y).astype(np.float64)
    expect = (lv[:, ks] * sval[:, ks // 128]).T           # [T][N]
    smax = sval.max(axis=1)                              # one box per row (K = 1024)
    exact = sval[:, ks // 128].T >= smax[None, :] * 2.0 ** -27
    assert np.array_equal(got[exact], expect[exact])
    assert np.all(np.abs(got - expect) <= smax[None, :] * 2.0 ** -30)
    assert sv.last_device_error() == 0


@pytest.mark.parametrize("T,K", [(32, 1024), (24, 5120)])
def test_activation_dynamic_range(sv, oracle, T, K):
    """The wide-range rows (2^100, 2^-100, spread over 2^+-40, outliers),
    repeated to T rows, through the tcgen05 kernel."""
    rng = np.random.default_rng(4400 + K + T)
    N = 700
    Wq, sc = gen.weights(rng, N, K)
    x = np.concatenate([wide_range_activations(rng, K)] * (T // 4))
    y32, _ = oracle.w4a16_gemm(x, Wq, sc, T, K, N)
    y = sv.w4a16_gemm(dev_bits16(x), dev_words(Wq), dev_bits16(sc))
    torch.cuda.synchronize()
    assert_gemm_close(y.view(torch.int16).cpu().numpy().view(np.uint16), y32)


@pytest.mark.parametrize("T,K,N", [
    (17, 1024, 300),     # one real token in the third token tile
    (24, 3072, 1000),
    (32, 5120, 2000),
    (32, 1024, 70),      # one 128-row tile shared by 8 CTAs
    (32, 17408, 70),     # one tile shared by 136 CTAs (one unit each)
])
def test_gemm_matches_oracle(sv, oracle, T, K, N):
    rng = np.random.default_rng(9100 + 31 * T + K + N)
    Wq, sc = gen.weights(rng, N, K)
    x = gen.activations(rng, T, K)
    y32, _ = oracle.w4a16_gemm(x, Wq, sc, T, K, N)
    y = sv.w4a16_gemm(dev_bits16(x), dev_words(Wq), dev_bits16(sc))
    torch.cuda.synchronize()
    assert_gemm_close(y.view(torch.int16).cpu().numpy().view(np.uint16), y32)
    y2 = sv.w4a16_gemm(dev_bits16(x), dev_words(Wq), dev_bits16(sc))
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    assert sv.last_device_error() == 0


@pytest.mark.parametrize("V,K,n_draft,n_streams", [
    (2500, 1024, 15, 2),     # 32 rows
    (5000, 3072, 10, 2),     # 22 rows, ragged third token tile, shares of 3-4 units
    (6000, 1024, 31, 1),
    (3000, 1024, 7, 4),      # four streams of 8 rows
])
def test_verify_matches_oracle(sv, oracle, V, K, n_draft, n_streams):
    run_head_case(sv, oracle, 9900 + V + K + n_draft, V, K, n_draft, n_streams, 0)


@pytest.mark.slow
def test_verify_four_streams_T32_full_size(sv, oracle):
    run_head_case(sv, oracle, 313, gen.VOCAB, gen.HIDDEN, 7, 4, 0)
