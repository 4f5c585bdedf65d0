"""GPU parity: the sm_103a kernels, called through the C ABI, against the CPU
oracle on the same seeded inputs.

Tolerances.  GEMM: |y_gpu - y_oracle| <= 1e-2 * max_n |y_oracle[t][n]| for
every row t (the bound the build is specified to), and the tighter
|y_gpu - y32| <= 2^-8 |y32| + 1e-5 * max|row| (bf16 rounding of the same fp32
sum, plus fp32 reordering).  Verify: argmax ids, accept_len and next_token are
bit-exact wherever the oracle's top-1 fp32 margin of the deciding rows exceeds
1e-3; where a near-tie decides, the outcome must be one of the correct ones
(tests/verify_check.py states the conditions).
"""
import numpy as np
import pytest

import gen
from verify_check import check_verify

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
    assert m.last_device_error() == 0
    return m


def dev_bits16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def dev_words(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).cuda()


def dev_i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def to_f32(t_bf16):
    return gen.bf16_bits_to_f32(t_bf16.view(torch.int16).cpu().numpy().view(np.uint16))


def assert_gemm_close(y_gpu_bits, y32):
    yg = gen.bf16_bits_to_f32(y_gpu_bits).astype(np.float64)
    y32 = y32.astype(np.float64)
    rowmax = np.abs(y32).max(axis=1, keepdims=True)
    err = np.abs(yg - y32)
    assert np.all(err <= 1e-2 * rowmax), "specified tolerance (1e-2 of the row maximum) violated: max rel %.3g" % (
        (err / np.maximum(rowmax, 1e-30)).max())
    assert np.all(err <= 2.0 ** -8 * np.abs(y32) + 1e-5 * rowmax)


# --------------------------------------------------------------------------
# dequantisation and layout on the GPU


def test_gpu_one_hot_pins_nibble_order_and_page_constant(sv, oracle):
    """Every nibble value in every position of a word, through the GPU GEMM:
    x = e_k gives y[n] = (nibble - 8) * s exactly (page: 0x4300 | n is 128+n,
    minus 136 is n - 8, all sixteen exact)."""
    K, N = 256, 18
    W = K // 8
    Wq = np.empty((N, W), np.uint32)
    lv = np.empty((N, K), np.int64)
    for n in range(16):                          # rows 0..15: every nibble = n
        Wq[n, :] = int(("%x" % n) * 8, 16)
        lv[n, :] = n - 8
    Wq[16, :] = 0xFEDCBA98
    lv[16, :] = np.tile(np.arange(8), W)
    Wq[17, :] = 0x76543210
    lv[17, :] = np.tile(np.arange(8) - 8, W)
    s = gen.f32_to_bf16_bits(np.array([[2.0 ** -(n % 5), 2.0 ** (n % 3)] for n in range(N)], np.float32))
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
        assert np.array_equal(got, expect)


@pytest.mark.parametrize("path", ["bf16_stages", "resident"])
def test_gpu_one_hot_at_one_token(sv, oracle, path):
    """The one-hot pin at T = 1 on the two one-token-tile paths: activations
    copied into every stage as bf16 with the bf16 dequantisation (0x4300
    OR, then -136; the QKV and down GEMMs of the step), and resident fp16
    rows with the fp16 dequantisation (enough rows for the resident rule).
    Each call has one nonzero activation, so y[n] = (nibble - 8) * s
    exactly, for every k of two groups and every nibble value."""
    K = 256
    N = 64 if path == "bf16_stages" else resident_rows(K)
    W = K // 8
    rng = np.random.default_rng(62)
    Wq = rng.integers(0, 2**32, size=(N, W), dtype=np.uint32)
    Wq[:16, :] = np.array([int(("%x" % n) * 8, 16) for n in range(16)], np.uint32)[:, None]
    s = gen.f32_to_bf16_bits((2.0 ** rng.integers(-4, 3, size=(N, K // 128))).astype(np.float32))
    sval = gen.bf16_bits_to_f32(s).astype(np.float64)
    one = gen.f32_to_bf16_bits(np.float32(1.0))
    dW, ds = dev_words(Wq), dev_bits16(s)
    for k in range(K):
        x = np.zeros((1, K), np.uint16)
        x[0, k] = one
        y = sv.w4a16_gemm(dev_bits16(x), dW, ds)
        torch.cuda.synchronize()
        got = to_f32(y).astype(np.float64)[0]
        level = ((Wq[:, k // 8] >> np.uint32(4 * (k % 8))) & 0xF).astype(np.int64) - 8
        assert np.array_equal(got, level * sval[:, k // 128]), k
    assert sv.last_device_error() == 0


@pytest.mark.parametrize("T,V,K", [(1, 3000, 1024), (4, "resident", 1024), (8, 5000, 2048)])
def test_gemm_rows_match_the_heads_argmax_values(sv, oracle, T, V, K):
    """Cross-export consistency: w4a16_gemm over the head's rows (N = V)
    computes the same fp32 sums as lmhead_argmax, so at each row's argmax id
    the GEMM's bf16 output is exactly the bf16 rounding of the fp32 logit
    lmhead_argmax returns, and no GEMM output exceeds it after rounding."""
    if V == "resident":
        V = resident_rows(K)
    rng = np.random.default_rng(7100 + T + K)
    Wq, sc = gen.weights(rng, V, K)
    x = gen.activations(rng, T, K)
    dx, dW, ds = dev_bits16(x), dev_words(Wq), dev_bits16(sc)
    ids, vals = sv.lmhead_argmax(dx, dW, ds)
    y = sv.w4a16_gemm(dx, dW, ds)
    torch.cuda.synchronize()
    yb = y.view(torch.int16).cpu().numpy().view(np.uint16)
    ids, vals = ids.cpu().numpy(), vals.cpu().numpy()
    for t in range(T):
        assert yb[t, ids[t]] == gen.f32_to_bf16_bits(np.float32(vals[t])), t
        assert gen.bf16_bits_to_f32(yb[t]).max() == gen.bf16_bits_to_f32(yb[t, ids[t]]), t


# --------------------------------------------------------------------------
# GEMM parity


@pytest.mark.parametrize("T,K,N", [
    (1, 512, 1024),      # the tiny configuration
    (1, 128, 1),
    (2, 128, 64),
    (3, 1152, 1000),     # ragged last tile, 9 groups
    (4, 5120, 200),
    (5, 896, 300),       # uneven warps per token row while staging, 7 groups
    (6, 1664, 129),
    (7, 2432, 65),       # a second token chunk with three real tokens, 19 groups
    (8, 2048, 777),
    (9, 640, 130),       # two n8 token tiles
    (13, 1280, 321),
    (16, 384, 64),
    (32, 1280, 321),     # four n8 token tiles
    (32, 17408, 70),
])
def test_gemm_matches_oracle(sv, oracle, T, K, N):
    rng = np.random.default_rng(7000 + 31 * T + K + N)
    Wq, sc = gen.weights(rng, N, K)
    x = gen.activations(rng, T, K)
    y32, ybf = oracle.w4a16_gemm(x, Wq, sc, T, K, N)
    y = sv.w4a16_gemm(dev_bits16(x), dev_words(Wq), dev_bits16(sc))
    torch.cuda.synchronize()
    yg = y.view(torch.int16).cpu().numpy().view(np.uint16)
    assert_gemm_close(yg, y32)
    # same call again: identical bits (fixed reduction order)
    y2 = sv.w4a16_gemm(dev_bits16(x), dev_words(Wq), dev_bits16(sc))
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


RESIDENT_MIN_UNITS = 80      # the library's threshold for resident activations


def resident_rows(K, ragged=17):
    """A row count whose call keeps the activations resident in shared memory:
    the kernels convert them once per CTA only when each CTA streams at least
    80 units (64 rows x one 128-column group); smaller calls copy bf16 rows
    into every stage.  Ragged last tile."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    G = K // 128
    tiles = (RESIDENT_MIN_UNITS * sms + G - 1) // G + 1
    return tiles * 64 - ragged


@pytest.mark.parametrize("T,K", [(1, 1152), (3, 5120), (5, 2432), (8, 1664)])
def test_gemm_resident_activations_match_oracle(sv, oracle, T, K):
    N = resident_rows(K)
    rng = np.random.default_rng(7300 + 31 * T + K)
    Wq, sc = gen.weights(rng, N, K)
    x = gen.activations(rng, T, K)
    y32, _ = oracle.w4a16_gemm(x, Wq, sc, T, K, N)
    y = sv.w4a16_gemm(dev_bits16(x), dev_words(Wq), dev_bits16(sc))
    torch.cuda.synchronize()
    assert_gemm_close(y.view(torch.int16).cpu().numpy().view(np.uint16), y32)


def test_gemm_resident_activations_two_staging_passes(sv, oracle):
    """Eight token rows of 5,632 columns: each of the two warps per row holds
    fewer chunks than the row has, so the resident rows are staged in two
    passes over global memory (maximum, then conversion)."""
    T, K = 8, 5632
    N = resident_rows(K)
    rng = np.random.default_rng(7411)
    Wq, sc = gen.weights(rng, N, K)
    x = gen.activations(rng, T, K)
    y32, _ = oracle.w4a16_gemm(x, Wq, sc, T, K, N)
    y = sv.w4a16_gemm(dev_bits16(x), dev_words(Wq), dev_bits16(sc))
    torch.cuda.synchronize()
    assert_gemm_close(y.view(torch.int16).cpu().numpy().view(np.uint16), y32)


def test_restricted_head_eight_rows_resident(sv, oracle):
    """Gathered rows with resident activations at T = 8 and K = 5,120: one warp
    per token row, staged in two passes; enough candidate rows that each
    CTA's share keeps the activations resident."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n_map = (RESIDENT_MIN_UNITS * sms + 39) // 40 * 64 + 64
    run_head_case(sv, oracle, 9173, n_map + 4000, 5120, 7, 1, n_map)


def wide_range_activations(rng, K):
    """Four bf16 rows far from N(0,1): scaled by 2^100, by 2^-100, with
    per-element magnitudes spread over 2^-40 .. 2^40, and N(0,1) with a few
    outliers of 2^20.  The kernels keep activations as fp16 scaled by a
    power of two per row; these rows check that the scaling reaches both ends
    of the bf16 range and that a row spanning far more than fp16's range
    stays within tolerance."""
    z = rng.standard_normal((4, K))
    z[0] *= 2.0 ** 100
    z[1] *= 2.0 ** -100
    z[2] *= 2.0 ** rng.uniform(-40, 40, K)
    z[3, rng.choice(K, 5, replace=False)] = 2.0 ** 20 * rng.choice([-1.0, 1.0], 5)
    return gen.f32_to_bf16_bits(z.astype(np.float32))


@pytest.mark.parametrize("K,N", [(1152, 300), (5120, 64), (1152, "resident"), (5120, "resident")])
def test_gemm_activation_dynamic_range(sv, oracle, K, N):
    if N == "resident":
        N = resident_rows(K)
    rng = np.random.default_rng(4100 + K)
    Wq, sc = gen.weights(rng, N, K)
    x = wide_range_activations(rng, K)
    y32, _ = oracle.w4a16_gemm(x, Wq, sc, 4, K, N)
    assert np.all(np.isfinite(y32))
    y = sv.w4a16_gemm(dev_bits16(x), dev_words(Wq), dev_bits16(sc))
    torch.cuda.synchronize()
    assert_gemm_close(y.view(torch.int16).cpu().numpy().view(np.uint16), y32)


@pytest.mark.parametrize("V", [3000, "resident"])
def test_head_argmax_activation_dynamic_range(sv, oracle, V):
    """Rows scaled by 2^30, unscaled, by 2^-30 and the spread row: argmax
    ids bit-exact where the margin allows, chosen logits within reordering."""
    rng = np.random.default_rng(4242)
    K = 768
    if V == "resident":
        V = resident_rows(K, ragged=5)
    Wq, sc = gen.weights(rng, V, K)
    z = rng.standard_normal((4, K))
    z[0] *= 2.0 ** 30
    z[2] *= 2.0 ** -30
    z[3] *= 2.0 ** rng.uniform(-40, 40, K)
    x = gen.f32_to_bf16_bits(z.astype(np.float32))
    lg = oracle.lmhead_logits(x, Wq, sc, K, 4, V)
    a, best, second = oracle.argmax(lg)
    ids, vals = sv.lmhead_argmax(dev_bits16(x), dev_words(Wq), dev_bits16(sc))
    torch.cuda.synchronize()
    ids, vals = ids.cpu().numpy(), vals.cpu().numpy()
    for t in range(4):
        rowmax = np.abs(lg[t]).max()
        if best[t] - second[t] > 1e-3 and best[t] - second[t] > 1e-5 * rowmax:
            assert ids[t] == a[t], t
        assert 0 <= ids[t] < V
        assert abs(float(vals[t]) - float(lg[t, ids[t]])) <= 1e-4 * rowmax
        assert float(lg[t, ids[t]]) >= best[t] - 1e-4 * rowmax


@pytest.mark.slow
@pytest.mark.parametrize("T", [1, 4, 8, 32])
@pytest.mark.parametrize("label,K,N", gen.GEMM_SHAPES)
def test_gemm_full_size_sampled_rows(sv, oracle, label, K, N, T):
    """Full decode shapes in the launch configuration the benchmark times; the
    oracle recomputes 640 sampled output rows (and the last tile)."""
    rng = np.random.default_rng({"qkv": 1, "gate_up": 2, "down": 3}[label] * 100 + T)
    Wq, sc = gen.weights(rng, N, K)
    x = gen.activations(rng, T, K)
    y = sv.w4a16_gemm(dev_bits16(x), dev_words(Wq), dev_bits16(sc))
    torch.cuda.synchronize()
    yg = y.view(torch.int16).cpu().numpy().view(np.uint16)
    rows = np.unique(np.concatenate([rng.choice(N, 576, replace=False), np.arange(N - 64, N)]))
    y32, _ = oracle.w4a16_gemm(x, Wq[rows], sc[rows], T, K, rows.size)
    assert_gemm_close(yg[:, rows], y32)
    assert sv.last_device_error() == 0


# --------------------------------------------------------------------------
# lm_head verify parity


def run_head_case(sv, oracle, seed, V, K, n_draft, n_streams=1, n_map=0, mismatch=None):
    rng = np.random.default_rng(seed)
    Wq, sc = gen.weights(rng, V, K)
    T = n_streams * (n_draft + 1)
    x = gen.activations(rng, T, K)
    vm = gen.vocab_map(rng, V, n_map) if n_map else None
    logits = oracle.lmhead_logits(x, Wq, sc, K, T, V, rows=vm)
    a, best, second = oracle.argmax(logits, ids=vm)
    drafts = np.zeros((n_streams, n_draft), np.int32)
    for s in range(n_streams):
        p = int(rng.integers(0, n_draft + 1)) if mismatch is None else mismatch[s]
        drafts[s] = gen.drafts_with_mismatch(rng, a[s * (n_draft + 1):(s + 1) * (n_draft + 1)], p, V,
                                             pool=vm)
    res = oracle.lmhead_verify(x, Wq, sc, K, V, drafts, n_streams=n_streams, vocab_map=vm)
    dx, dW, ds = dev_bits16(x), dev_words(Wq), dev_bits16(sc)
    dvm = None if vm is None else dev_i32(vm)
    if n_streams == 1:
        acc, nxt = sv.lmhead_verify(dx, dW, ds, dev_i32(drafts[0]), vocab_map=dvm)
    else:
        acc, nxt = sv.lmhead_verify_batched(dx, dW, ds, dev_i32(drafts), vocab_map=dvm)
    ids, vals = sv.lmhead_argmax(dx, dW, ds, vocab_map=dvm)
    torch.cuda.synchronize()
    ids = ids.cpu().numpy()
    vals = vals.cpu().numpy()
    check_verify(res, drafts, acc.cpu().numpy(), nxt.cpu().numpy(), ids, n_draft, n_streams, vm)
    # argmax values: the fp32 logit of the chosen id, within fp32 reordering
    lim = 1e-4 * np.abs(res.logits).max()
    for t in range(T):
        ids_all = np.arange(res.logits.shape[1]) if vm is None else vm
        j = np.where(ids_all == ids[t])[0][0]
        assert abs(float(vals[t]) - float(res.logits[t, j])) <= lim
    assert sv.last_device_error() == 0
    return res, acc.cpu().numpy(), nxt.cpu().numpy()


def test_verify_tiny_configuration(sv, oracle):
    """V=4096, K=512, drafts = oracle argmax of rows 0 and 1, then a different
    token: accept_len 2, next_token = argmax of row 2."""
    rng = np.random.default_rng(0)
    V, K, n_draft = 4096, 512, 3
    Wq, sc = gen.weights(rng, V, K)
    x = gen.activations(rng, n_draft + 1, K)
    lg = oracle.lmhead_logits(x, Wq, sc, K, n_draft + 1, V)
    a, _, _ = oracle.argmax(lg)
    drafts = np.array([a[0], a[1], gen.token_not(rng, V, int(a[2]))], np.int32)
    res = oracle.lmhead_verify(x, Wq, sc, K, V, drafts)
    assert res.accept_len[0] == 2 and res.next_token[0] == a[2]
    dx, dW, ds = dev_bits16(x), dev_words(Wq), dev_bits16(sc)
    acc, nxt = sv.lmhead_verify(dx, dW, ds, dev_i32(drafts))
    ids, _ = sv.lmhead_argmax(dx, dW, ds)
    torch.cuda.synchronize()
    check_verify(res, drafts, acc.cpu().numpy(), nxt.cpu().numpy(), ids.cpu().numpy(), n_draft, 1)


@pytest.mark.parametrize("V,K,n_draft,n_streams,n_map", [
    (4096, 512, 3, 1, 0),
    (1000, 640, 0, 1, 0),        # plain greedy, ragged vocabulary
    (777, 128, 7, 1, 0),
    (3000, 1024, 7, 4, 0),       # 4 streams x 8 rows = 32
    (2500, 1152, 2, 3, 0),
    (5000, 768, 3, 1, 1234),     # restricted
    (5000, 768, 0, 1, 1),        # single-entry map
    (6000, 512, 3, 2, 4000),
    (3333, 896, 4, 1, 0),        # five rows
    (2049, 1664, 6, 1, 0),       # seven rows
    (5000, 768, 7, 1, 2000),     # restricted, eight rows
])
def test_verify_matches_oracle(sv, oracle, V, K, n_draft, n_streams, n_map):
    run_head_case(sv, oracle, 900 + V + K + n_draft, V, K, n_draft, n_streams, n_map)


def test_identity_map_equals_full_head_and_map_order_is_irrelevant(sv, oracle):
    """An identity map is the full head bit for bit (same rows in the same
    positions); a permuted map gives the same ids wherever the oracle margin
    exceeds 1e-3 (a permutation moves rows between tiles, which may change
    the fp32 summation order of a row, not its value beyond rounding)."""
    rng = np.random.default_rng(31)
    V, K, T = 3000, 512, 4
    Wq, sc = gen.weights(rng, V, K)
    x = gen.activations(rng, T, K)
    dx, dW, ds = dev_bits16(x), dev_words(Wq), dev_bits16(sc)
    ids_full, vals_full = sv.lmhead_argmax(dx, dW, ds)
    ids_id, vals_id = sv.lmhead_argmax(dx, dW, ds, vocab_map=dev_i32(np.arange(V)))
    perm = rng.permutation(V).astype(np.int32)
    ids_p, vals_p = sv.lmhead_argmax(dx, dW, ds, vocab_map=dev_i32(perm))
    torch.cuda.synchronize()
    assert torch.equal(ids_full, ids_id) and torch.equal(vals_full, vals_id)
    lg = oracle.lmhead_logits(x, Wq, sc, K, T, V)
    a, best, second = oracle.argmax(lg)
    for t in range(T):
        if best[t] - second[t] > MARGIN:
            assert int(ids_p[t]) == int(a[t]) == int(ids_full[t])
    assert np.allclose(vals_p.cpu().numpy(), vals_full.cpu().numpy(), rtol=0, atol=1e-4 * np.abs(lg).max())
    one = dev_i32(np.array([1234]))
    ids_1, _ = sv.lmhead_argmax(dx, dW, ds, vocab_map=one)
    torch.cuda.synchronize()
    assert ids_1.cpu().tolist() == [1234] * T


def test_exact_tie_goes_to_lowest_id(sv, oracle):
    """Copies of the best row placed in the same 64-row tile (where every row
    is summed in the same order, so the tie is exact on the GPU too): the
    lowest id of the tied set wins, over the full head and over a map that
    lists the tied ids highest first."""
    rng = np.random.default_rng(32)
    V, K = 2000, 512
    Wq, sc = gen.weights(rng, V, K)
    x = gen.activations(rng, 1, K)
    a0 = int(oracle.argmax(oracle.lmhead_logits(x, Wq, sc, K, 1, V))[0][0])
    base = (a0 // 64) * 64
    tied = sorted({base, min(V - 1, base + 63), a0})
    for d in tied:
        Wq[d] = Wq[a0]
        sc[d] = sc[a0]
    lg = oracle.lmhead_logits(x, Wq, sc, K, 1, V)
    a, _, _ = oracle.argmax(lg)
    assert int(a[0]) == tied[0] and len(tied) > 1
    ids, _ = sv.lmhead_argmax(dev_bits16(x), dev_words(Wq), dev_bits16(sc))
    rest = np.setdiff1d(rng.permutation(V), tied)
    vm = np.concatenate([rest[:64], np.array(tied[::-1]), rest[64:]]).astype(np.int32)
    ids_m, _ = sv.lmhead_argmax(dev_bits16(x), dev_words(Wq), dev_bits16(sc), vocab_map=dev_i32(vm))
    torch.cuda.synchronize()
    assert ids.cpu().tolist() == [tied[0]]
    assert ids_m.cpu().tolist() == [tied[0]]


def test_bad_map_id_is_skipped_and_flagged(sv, oracle):
    rng = np.random.default_rng(33)
    V, K, T = 1500, 256, 1
    Wq, sc = gen.weights(rng, V, K)
    x = gen.activations(rng, T, K)
    vm = gen.vocab_map(rng, V, 300)
    bad = vm.copy()
    bad[17] = V + 5
    bad[200] = -3
    good = np.delete(vm, [17, 200])
    ids_b, _ = sv.lmhead_argmax(dev_bits16(x), dev_words(Wq), dev_bits16(sc), vocab_map=dev_i32(bad))
    torch.cuda.synchronize()
    assert sv.last_device_error() & sv.DEVERR_BAD_MAP_ID
    assert sv.last_device_error() == 0            # cleared by the read
    lg = oracle.lmhead_logits(x, Wq, sc, K, T, V, rows=good)
    a, _, _ = oracle.argmax(lg, ids=good)
    assert ids_b.cpu().tolist() == a.tolist()


# --------------------------------------------------------------------------
# full-size configurations (the benchmark's launch configuration)


@pytest.mark.slow
def test_verify_mtp_T4_full_size(sv, oracle):
    run_head_case(sv, oracle, 2, gen.VOCAB, gen.HIDDEN, 3, 1, 0)


@pytest.mark.slow
def test_verify_dflash2_T8_full_size(sv, oracle):
    run_head_case(sv, oracle, 3, gen.VOCAB, gen.HIDDEN, 7, 1, 0)


@pytest.mark.slow
def test_verify_dflash2_4_streams_T32_full_size(sv, oracle):
    run_head_case(sv, oracle, 303, gen.VOCAB, gen.HIDDEN, 7, 4, 0)


@pytest.mark.slow
@pytest.mark.parametrize("n_draft", [0, 3])
def test_restricted_head_full_size(sv, oracle, n_draft):
    run_head_case(sv, oracle, 4 + n_draft, gen.VOCAB, gen.HIDDEN, n_draft, 1, gen.DRAFT_VOCAB)


# --------------------------------------------------------------------------
# calls with more than one n8 token tile (9 <= T <= 32): 64-row tiles, and
# for lm_head-sized calls at 9 <= T <= 16 (at least two 512-row tiles per
# SM, K a multiple of 1024) 512-row tiles


def wide_rows_512(K, ragged=29):
    """A row count for which the library takes 512-row tiles (at least 2 x
    the SM count of them); ragged last tile, whose second 256-row half is
    partly filled."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return 2 * sms * 512 + 3 * 512 - ragged


def wide_rows_512_half(K):
    """As wide_rows_512, with the last tile's second 256-row half empty."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return 2 * sms * 512 + 3 * 512 + 100


@pytest.mark.parametrize("T,K,N", [
    (9, 1024, 777),      # two token tiles, one real token in the second, ragged tile
    (12, 5120, 600),
    (16, 2048, 1500),
    (17, 1024, 300),     # four token tiles, one real token in the third
    (24, 3072, 1000),
    (32, 5120, 2000),
    (32, 1024, 70),      # one tile shared by 16 CTAs
    (32, 17408, 70),     # one tile shared by 136 CTAs (one unit each)
    (16, 17408, 5120),   # the down GEMM's shape at T = 16
])
def test_multi_tile_gemm_matches_oracle(sv, oracle, T, K, N):
    rng = np.random.default_rng(9000 + 31 * T + K + N)
    Wq, sc = gen.weights(rng, N, K)
    x = gen.activations(rng, T, K)
    y32, _ = oracle.w4a16_gemm(x, Wq, sc, T, K, N)
    y = sv.w4a16_gemm(dev_bits16(x), dev_words(Wq), dev_bits16(sc))
    torch.cuda.synchronize()
    assert_gemm_close(y.view(torch.int16).cpu().numpy().view(np.uint16), y32)
    # same call again: identical bits (fixed reduction order of split tiles)
    y2 = sv.w4a16_gemm(dev_bits16(x), dev_words(Wq), dev_bits16(sc))
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    assert sv.last_device_error() == 0


@pytest.mark.slow
@pytest.mark.parametrize("T,K,rows", [(9, 1024, "ragged"), (12, 2048, "ragged"), (16, 1024, "half"),
                                      (16, 3072, "ragged")])
def test_wide_gemm_512_row_tiles_sampled_rows(sv, oracle, T, K, rows):
    """GEMMs with enough rows for 512-row tiles; the oracle recomputes 640
    sampled rows and the last tile; a repeat call gives identical bits."""
    N = wide_rows_512(K) if rows == "ragged" else wide_rows_512_half(K)
    rng = np.random.default_rng(9500 + T + K)
    Wq, sc = gen.weights(rng, N, K)
    x = gen.activations(rng, T, K)
    y = sv.w4a16_gemm(dev_bits16(x), dev_words(Wq), dev_bits16(sc))
    torch.cuda.synchronize()
    yg = y.view(torch.int16).cpu().numpy().view(np.uint16)
    rows = np.unique(np.concatenate([rng.choice(N, 576, replace=False), np.arange(N - 600, N)]))
    y32, _ = oracle.w4a16_gemm(x, Wq[rows], sc[rows], T, K, rows.size)
    assert_gemm_close(yg[:, rows], y32)
    y2 = sv.w4a16_gemm(dev_bits16(x), dev_words(Wq), dev_bits16(sc))
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    assert sv.last_device_error() == 0


@pytest.mark.slow
def test_wide_gemm_activation_dynamic_range(sv, oracle):
    """The wide-range rows (2^100, 2^-100, spread over 2^+-40, outliers),
    repeated to 16 token rows, on 512-row tiles (sampled rows)."""
    K, T = 1024, 16
    N = wide_rows_512(K)
    rng = np.random.default_rng(4300 + K)
    Wq, sc = gen.weights(rng, N, K)
    x = np.concatenate([wide_range_activations(rng, K)] * (T // 4))
    y = sv.w4a16_gemm(dev_bits16(x), dev_words(Wq), dev_bits16(sc))
    torch.cuda.synchronize()
    yg = y.view(torch.int16).cpu().numpy().view(np.uint16)
    rows = np.unique(np.concatenate([rng.choice(N, 400, replace=False), np.arange(N - 100, N)]))
    y32, _ = oracle.w4a16_gemm(x, Wq[rows], sc[rows], T, K, rows.size)
    assert_gemm_close(yg[:, rows], y32)


@pytest.mark.parametrize("V,K,n_draft,n_streams", [
    (4000, 1024, 12, 1),     # 13 rows, two token tiles
    (3000, 2048, 7, 2),      # two streams of 8 rows
    (2500, 1024, 15, 2),     # 32 rows
    (5000, 3072, 10, 2),     # 22 rows, ragged third token tile
    (6000, 1024, 31, 1),     # 32 rows, one stream
])
def test_multi_tile_verify_matches_oracle(sv, oracle, V, K, n_draft, n_streams):
    run_head_case(sv, oracle, 9700 + V + K + n_draft, V, K, n_draft, n_streams, 0)


@pytest.mark.slow
@pytest.mark.parametrize("K,n_draft,n_streams,rows", [
    (1024, 7, 2, "ragged"),      # two streams of 8 rows
    (1024, 8, 1, "half"),        # 9 rows, one real token in the second token tile
    (2048, 12, 1, "ragged"),     # 13 rows
    (1024, 3, 4, "ragged"),      # four streams of 4 rows
    (1024, 15, 1, "half"),       # 16 rows
])
def test_wide_verify_512_row_tiles(sv, oracle, K, n_draft, n_streams, rows):
    """Heads with enough rows for 512-row tiles at 9 <= T <= 16."""
    V = wide_rows_512(K) if rows == "ragged" else wide_rows_512_half(K)
    run_head_case(sv, oracle, 9801 + K + n_draft, V, K, n_draft, n_streams, 0)


@pytest.mark.slow
def test_verify_two_streams_T16_full_size(sv, oracle):
    run_head_case(sv, oracle, 316, gen.VOCAB, gen.HIDDEN, 7, 2, 0)


# --------------------------------------------------------------------------
# bounded waits: a wait that runs out is reported, and later calls are clean


def test_timed_out_wait_is_reported_and_later_calls_are_clean(sv, oracle):
    """The test hook makes one wait of the first thread block run out after
    5 ms (a barrier that nothing completes): the call still finishes, the
    error word carries the time-out bit (and the read clears it and the
    scratch counters), and the next calls give the oracle's results with no
    error."""
    rng = np.random.default_rng(77)
    V, K, n_draft = 3000, 512, 3
    Wq, sc = gen.weights(rng, V, K)
    x = gen.activations(rng, n_draft + 1, K)
    lg = oracle.lmhead_logits(x, Wq, sc, K, n_draft + 1, V)
    a, _, _ = oracle.argmax(lg)
    drafts = gen.drafts_with_mismatch(rng, a, 2, V)
    res = oracle.lmhead_verify(x, Wq, sc, K, V, drafts)
    dx, dW, ds, dd = dev_bits16(x), dev_words(Wq), dev_bits16(sc), dev_i32(drafts)
    assert sv.last_device_error() == 0
    sv.debug_set_wait_stall(5_000_000)
    try:
        sv.lmhead_verify(dx, dW, ds, dd)
        y = sv.w4a16_gemm(dx, dW, ds)
    finally:
        sv.debug_set_wait_stall(0)
    torch.cuda.synchronize()
    assert sv.last_device_error() & sv.DEVERR_TIMEOUT
    assert sv.last_device_error() == 0
    for _ in range(2):
        acc, nxt = sv.lmhead_verify(dx, dW, ds, dd)
        ids, _ = sv.lmhead_argmax(dx, dW, ds)
        y2 = sv.w4a16_gemm(dx, dW, ds)
        torch.cuda.synchronize()
        check_verify(res, drafts, acc.cpu().numpy(), nxt.cpu().numpy(), ids.cpu().numpy(), n_draft, 1)
        assert sv.last_device_error() == 0
    # the stalled GEMM still computed its outputs
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


# --------------------------------------------------------------------------
# the CUDA-core formulation of the consumers (measurement switch) and the
# static-map head


@pytest.mark.parametrize("T,K", [(1, 1152), (4, 5120), (8, 1664)])
def test_fma_consumers_gemm_match_oracle(sv, oracle, T, K):
    """With the CUDA-core consumers switched on, a resident-activation GEMM
    still matches the oracle within the tolerance."""
    N = resident_rows(K)
    rng = np.random.default_rng(7600 + T + K)
    Wq, sc = gen.weights(rng, N, K)
    x = gen.activations(rng, T, K)
    y32, _ = oracle.w4a16_gemm(x, Wq, sc, T, K, N)
    sv.debug_set_fma_consumers(True)
    try:
        y = sv.w4a16_gemm(dev_bits16(x), dev_words(Wq), dev_bits16(sc))
        torch.cuda.synchronize()
    finally:
        sv.debug_set_fma_consumers(False)
    assert_gemm_close(y.view(torch.int16).cpu().numpy().view(np.uint16), y32)
    assert sv.last_device_error() == 0


@pytest.mark.parametrize("n_draft", [0, 3, 7])
def test_fma_consumers_verify_matches_oracle(sv, oracle, n_draft):
    K = 1024
    V = resident_rows(K, ragged=11)
    sv.debug_set_fma_consumers(True)
    try:
        run_head_case(sv, oracle, 7700 + n_draft, V, K, n_draft, 1, 0)
    finally:
        sv.debug_set_fma_consumers(False)


@pytest.mark.parametrize("V,K,n_draft,n_streams,n_map", [
    (5000, 768, 3, 1, 1234),
    (5000, 768, 0, 1, 1),
    (6000, 512, 3, 2, 4000),
    (5000, 768, 7, 1, 2000),
])
def test_static_map_verify_matches_oracle(sv, oracle, V, K, n_draft, n_streams, n_map):
    """lmhead_verify_ex with SV_MAP_STATIC gives the regular call's results."""
    rng = np.random.default_rng(7800 + V + n_map)
    Wq, sc = gen.weights(rng, V, K)
    T = n_streams * (n_draft + 1)
    x = gen.activations(rng, T, K)
    vm = gen.vocab_map(rng, V, n_map)
    a, _, _ = oracle.argmax(oracle.lmhead_logits(x, Wq, sc, K, T, V, rows=vm), ids=vm)
    drafts = np.stack([gen.drafts_with_mismatch(rng, a[s * (n_draft + 1):(s + 1) * (n_draft + 1)],
                                                int(rng.integers(0, n_draft + 1)), V, pool=vm)
                       for s in range(n_streams)]).astype(np.int32).reshape(n_streams, n_draft)
    res = oracle.lmhead_verify(x, Wq, sc, K, V, drafts, n_streams=n_streams, vocab_map=vm)
    dx, dW, ds, dvm = dev_bits16(x), dev_words(Wq), dev_bits16(sc), dev_i32(vm)
    dd = torch.from_numpy(drafts).cuda()
    acc_s, nxt_s = sv.lmhead_verify_ex(dx, dW, ds, dd, vocab_map=dvm, flags=sv.MAP_STATIC)
    acc_r, nxt_r = sv.lmhead_verify_batched(dx, dW, ds, dd, vocab_map=dvm)
    ids, _ = sv.lmhead_argmax(dx, dW, ds, vocab_map=dvm)
    torch.cuda.synchronize()
    assert torch.equal(acc_s, acc_r) and torch.equal(nxt_s, nxt_r)
    check_verify(res, drafts, acc_s.cpu().numpy(), nxt_s.cpu().numpy(), ids.cpu().numpy(), n_draft, n_streams, vm)
    assert sv.last_device_error() == 0


@pytest.mark.slow
@pytest.mark.parametrize("n_draft", [0, 3])
def test_static_map_restricted_head_full_size(sv, oracle, n_draft):
    """The 40,960-id restricted head of a 248,320 x 5,120 lm_head with the
    static-map flag, as the benchmark runs it."""
    rng = np.random.default_rng(7900 + n_draft)
    V, K, n_map = gen.VOCAB, gen.HIDDEN, gen.DRAFT_VOCAB
    Wq, sc = gen.weights(rng, V, K)
    x = gen.activations(rng, n_draft + 1, K)
    vm = gen.vocab_map(rng, V, n_map)
    a, _, _ = oracle.argmax(oracle.lmhead_logits(x, Wq, sc, K, n_draft + 1, V, rows=vm), ids=vm)
    drafts = gen.drafts_with_mismatch(rng, a, min(2, n_draft), V, pool=vm).reshape(1, n_draft)
    res = oracle.lmhead_verify(x, Wq, sc, K, V, drafts, vocab_map=vm)
    dx, dW, ds, dvm = dev_bits16(x), dev_words(Wq), dev_bits16(sc), dev_i32(vm)
    acc, nxt = sv.lmhead_verify_ex(dx, dW, ds, torch.from_numpy(drafts).cuda(), vocab_map=dvm,
                                   flags=sv.MAP_STATIC)
    ids, _ = sv.lmhead_argmax(dx, dW, ds, vocab_map=dvm)
    torch.cuda.synchronize()
    check_verify(res, drafts, acc.cpu().numpy(), nxt.cpu().numpy(), ids.cpu().numpy(), n_draft, 1, vm)
    assert sv.last_device_error() == 0
