"""Pins for the CPU oracle: each test checks it against something other than
itself -- values the pages print, closed forms, exact invariants, a library
matmul on an independently packed matrix, and hand-built argmax / verify
cases.  No GPU needed."""
import os

import numpy as np
import pytest

import gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U = 2.0 ** -24          # fp32 unit roundoff


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def pack_levels(L):
    """Pack signed levels [rows][K] (-8..7) into uint32 words: column 8w+i is
    nibble i (bits 4i..4i+3) of word w, nibble = level + 8.  This is the
    storage format written out in the encoding direction, independent of the
    oracle's decoding."""
    L = np.asarray(L, dtype=np.int64)
    rows, K = L.shape
    nib = (L + 8).astype(np.uint64).reshape(rows, K // 8, 8)
    words = np.zeros((rows, K // 8), dtype=np.uint64)
    for i in range(8):
        words |= nib[:, :, i] << np.uint64(4 * i)
    return words.astype(np.uint32)


def pow2_bf16(e):
    return gen.f32_to_bf16_bits(np.float32(2.0 ** e))


# --------------------------------------------------------------------------
# format and dequantisation


def test_dequant_constant_table_from_page(oracle):
    """Every nibble: bf16 0x4300|n is 128+n and the level is n-8 (page's
    exhaustive check); the oracle's level of nibble n is that same n-8."""
    rows = _read_golden("dequant_bf16_qwen_warp.txt")
    assert len(rows) == 16
    K = 128
    for n_s, bits_s, val_s, lvl_s in rows:
        n, bits, val, lvl = int(n_s), int(bits_s, 16), int(val_s), int(lvl_s)
        assert bits == (0x4300 | n)
        assert float(gen.bf16_bits_to_f32(np.uint16(bits))) == float(val)
        assert val - 136 == lvl == n - 8
        # the oracle on one row whose every nibble is n, x = e_0, scale 1
        word = np.uint32(int("%x" % n * 8, 16))
        Wq = np.full((1, K // 8), word, np.uint32)
        sc = pow2_bf16(0).reshape(1, 1)
        x = np.zeros((1, K), np.uint16)
        x[0, 5] = gen.f32_to_bf16_bits(np.float32(1.0))
        y32, _ = oracle.w4a16_gemm(x, Wq, sc, 1, K, 1)
        assert y32[0, 0] == np.float32(lvl)


def test_one_hot_pins_nibble_order_orientation_and_groups(oracle):
    """x = e_k for every k of a 2-group row: y[n] = level(n,k) * s[n][k//128]
    exactly.  Rows use hand-chosen word patterns so the expected levels are
    known without decoding."""
    K, N = 256, 4
    W = K // 8
    Wq = np.empty((N, W), np.uint32)
    lv = np.empty((N, K), np.int64)
    Wq[0, :] = 0xFEDCBA98            # nibble i = 8 + i  -> level i
    lv[0, :] = np.tile(np.arange(8), W)
    Wq[1, :] = 0x76543210            # nibble i = i      -> level i - 8
    lv[1, :] = np.tile(np.arange(8) - 8, W)
    lv[2, :] = 0
    for w in range(W):               # word w: nibble w%8 holds (5w mod 16), others 8
        i, v = w % 8, (5 * w) % 16
        Wq[2, w] = (0x88888888 & ~(0xF << (4 * i))) | (v << (4 * i))
        lv[2, 8 * w + i] = v - 8
    Wq[3, :] = 0x88888888
    Wq[3, 17] = 0x8F888881           # word 17: nibble 0 -> 1 (-7), nibble 6 -> F (+7)
    lv[3, :] = 0
    lv[3, 8 * 17 + 0] = -7
    lv[3, 8 * 17 + 6] = 7
    scales = np.array([[pow2_bf16(-1), pow2_bf16(-3)],
                       [pow2_bf16(-2), pow2_bf16(2)],
                       [pow2_bf16(0), pow2_bf16(-5)],
                       [pow2_bf16(-4), pow2_bf16(1)]], np.uint16)
    sval = gen.bf16_bits_to_f32(scales).astype(np.float64)
    x = np.zeros((K, K), np.uint16)
    x[np.arange(K), np.arange(K)] = gen.f32_to_bf16_bits(np.float32(1.0))
    y32, ybf = oracle.w4a16_gemm(x, Wq, scales, K, K, N)
    expect = (lv * sval[:, np.arange(K) // 128]).T      # [T=K][N]
    assert np.array_equal(y32.astype(np.float64), expect)
    assert np.array_equal(gen.bf16_bits_to_f32(ybf).astype(np.float64), expect)


# --------------------------------------------------------------------------
# closed forms and exact invariants


def test_level_zero_everywhere_gives_zero(oracle):
    rng = np.random.default_rng(10)
    T, K, N = 3, 640, 37
    Wq = np.full((N, K // 8), 0x88888888, np.uint32)
    _, sc = gen.weights(rng, N, K)
    x = gen.activations(rng, T, K)
    y32, ybf, y64 = oracle.w4a16_gemm(x, Wq, sc, T, K, N, want64=True)
    assert not np.any(y32) and not np.any(y64)
    assert np.all((ybf & 0x7FFF) == 0)


def test_zero_words_closed_form(oracle):
    """Every nibble 0 means level -8: y = -8 * sum_g s_g * sum_{k in g} x_k."""
    rng = np.random.default_rng(11)
    T, K, N = 4, 1024, 9
    Wq = np.zeros((N, K // 8), np.uint32)
    _, sc = gen.weights(rng, N, K)
    x = gen.activations(rng, T, K)
    y32, _, y64 = oracle.w4a16_gemm(x, Wq, sc, T, K, N, want64=True)
    xf = gen.bf16_bits_to_f32(x).astype(np.float64).reshape(T, K // 128, 128)
    gsum = xf.sum(axis=2)                                   # [T][G], exact in fp64
    s = gen.bf16_bits_to_f32(sc).astype(np.float64)         # [N][G]
    closed = -8.0 * gsum @ s.T                              # [T][N]
    assert np.allclose(y64, closed, rtol=1e-13, atol=1e-12)
    absbound = 8.0 * np.abs(xf).sum(axis=2) @ s.T
    assert np.all(np.abs(y32 - closed) <= (128 + K // 128 + 2) * U * absbound + 1e-30)


def test_ones_single_group_closed_form(oracle):
    """x = 1 and K = 128: y[n] = s[n] * sum_k level(n, k), summed exactly."""
    rng = np.random.default_rng(12)
    K, N = 128, 50
    L = rng.integers(-8, 8, size=(N, K))
    Wq = pack_levels(L)
    _, sc = gen.weights(rng, N, K)
    x = np.full((1, K), gen.f32_to_bf16_bits(np.float32(1.0)), np.uint16)
    y32, _ = oracle.w4a16_gemm(x, Wq, sc, 1, K, N)
    s = gen.bf16_bits_to_f32(sc)[:, 0].astype(np.float64)
    # integer sums and one fp32 product: s * sum is rounded once in fp32
    expect = (s * L.sum(axis=1)).astype(np.float32)
    assert np.array_equal(y32[0], expect)


@pytest.mark.parametrize("j", [-3, 5])
def test_power_of_two_scale_is_exact(oracle, j):
    rng = np.random.default_rng(13 + j)
    T, K, N = 2, 768, 33
    Wq, sc = gen.weights(rng, N, K)
    x = gen.activations(rng, T, K)
    y32, ybf = oracle.w4a16_gemm(x, Wq, sc, T, K, N)
    sc2 = gen.f32_to_bf16_bits(gen.bf16_bits_to_f32(sc) * np.float32(2.0 ** j))
    assert np.array_equal(gen.bf16_bits_to_f32(sc2), gen.bf16_bits_to_f32(sc) * np.float32(2.0 ** j))
    y32b, ybfb = oracle.w4a16_gemm(x, Wq, sc2, T, K, N)
    assert np.array_equal(y32b, y32 * np.float32(2.0 ** j))
    assert np.array_equal(gen.bf16_bits_to_f32(ybfb), gen.bf16_bits_to_f32(ybf) * np.float32(2.0 ** j))


def test_one_scale_changes_one_column(oracle):
    rng = np.random.default_rng(14)
    T, K, N = 3, 512, 20
    Wq, sc = gen.weights(rng, N, K)
    x = gen.activations(rng, T, K)
    y32, _ = oracle.w4a16_gemm(x, Wq, sc, T, K, N)
    sc2 = sc.copy()
    sc2[7, 2] = gen.f32_to_bf16_bits(np.float32(0.5))
    y32b, _ = oracle.w4a16_gemm(x, Wq, sc2, T, K, N)
    changed = np.any(y32b != y32, axis=0)
    assert changed[7] and changed.sum() == 1


# --------------------------------------------------------------------------
# against a library matmul on an independently packed matrix


@pytest.mark.parametrize("T,K,N", [(1, 128, 7), (4, 512, 33), (8, 1280, 19), (5, 2048, 3)])
def test_matches_fp64_matmul_of_unpacked_levels(oracle, T, K, N):
    rng = np.random.default_rng(1000 + T * K + N)
    L = rng.integers(-8, 8, size=(N, K))
    Wq = pack_levels(L)
    _, sc = gen.weights(rng, N, K)
    x = gen.activations(rng, T, K)
    s = gen.bf16_bits_to_f32(sc).astype(np.float64)
    Wd = L * np.repeat(s, 128, axis=1)                     # dequantised [N][K]
    xf = gen.bf16_bits_to_f32(x).astype(np.float64)
    ref = xf @ Wd.T                                         # numpy fp64 matmul
    y32, ybf, y64 = oracle.w4a16_gemm(x, Wq, sc, T, K, N, want64=True)
    mag = np.abs(xf) @ np.abs(Wd).T
    assert np.all(np.abs(y64 - ref) <= 1e-12 * mag + 1e-300)
    # rigorous fp32 bound: 127 adds in a group, one product, G adds across groups
    G = K // 128
    assert np.all(np.abs(y32 - ref) <= (127 + G + 2) * U * mag)
    # bf16 output: within half an ulp of bf16 (unit roundoff 2^-8) of the fp32 value
    yb = gen.bf16_bits_to_f32(ybf).astype(np.float64)
    assert np.all(np.abs(yb - y32) <= 2.0 ** -8 * np.abs(y32) + 1e-38)


def test_bf16_output_rounds_to_nearest_even(oracle):
    """Hand cases: y = 1 + 3*2^-8 is a tie between 1+2^-7 (odd) and 1+2^-6
    (even) and must go to 1+2^-6; y = 1 + 2^-8 is a tie that goes to 1."""
    K = 128
    Wq = np.full((1, K // 8), 0x88888888, np.uint32)
    Wq[0, 0] = 0x88888899            # k = 0 and k = 1 have level +1
    sc = pow2_bf16(0).reshape(1, 1)
    x = np.zeros((2, K), np.uint16)
    x[0, 0] = gen.f32_to_bf16_bits(np.float32(1 + 2 ** -7))
    x[0, 1] = gen.f32_to_bf16_bits(np.float32(2 ** -8))
    x[1, 0] = gen.f32_to_bf16_bits(np.float32(1.0))
    x[1, 1] = gen.f32_to_bf16_bits(np.float32(2 ** -8))
    y32, ybf = oracle.w4a16_gemm(x, Wq, sc, 2, K, 1)
    assert y32[0, 0] == np.float32(1 + 3 * 2 ** -8)
    assert float(gen.bf16_bits_to_f32(ybf[0, 0])) == 1 + 2 ** -6
    assert y32[1, 0] == np.float32(1 + 2 ** -8)
    assert float(gen.bf16_bits_to_f32(ybf[1, 0])) == 1.0


def test_bf16_rounding_agrees_with_generator_rounding(oracle):
    """Two independent round-to-nearest-even implementations (the oracle's C
    and the input generator's numpy) agree on a large sample of outputs."""
    rng = np.random.default_rng(15)
    T, K, N = 4, 1024, 257
    Wq, sc = gen.weights(rng, N, K)
    x = gen.activations(rng, T, K)
    y32, ybf = oracle.w4a16_gemm(x, Wq, sc, T, K, N)
    assert np.array_equal(ybf, gen.f32_to_bf16_bits(y32))


# --------------------------------------------------------------------------
# argmax, tie-break and the verify rule


def test_argmax_hand_cases(oracle):
    lg = np.array([[1.0, 3.0, 3.0, 2.0],
                   [-1.0, -1.0, -1.0, -1.0],
                   [0.5, -2.0, 0.25, 0.75]], np.float32)
    a, best, second = oracle.argmax(lg)
    assert list(a) == [1, 0, 3]
    assert list(best) == [3.0, -1.0, 0.75]
    assert list(second) == [3.0, -1.0, 0.5]
    ids = np.array([7, 5, 9, 1], np.int32)
    a2, _, _ = oracle.argmax(lg, ids=ids)
    assert list(a2) == [5, 1, 1]     # tie between ids 5 and 9 -> 5; all equal -> 1


def _planted_head(rng, V, K, T, planted, dup=None):
    """Random head with row planted[t] made the maximiser of token row t: its
    level is +7 where x[t] > 0 and -8 where x[t] < 0 (the largest dot any row
    with the same scales can have), with the largest scale."""
    Wq, sc = gen.weights(rng, V, K)
    x = gen.activations(rng, T, K)
    xf = gen.bf16_bits_to_f32(x)
    for t, v in enumerate(planted):
        L = np.where(xf[t] > 0, 7, -8)[None, :]
        Wq[v] = pack_levels(L)[0]
        sc[v] = gen.f32_to_bf16_bits(np.float32(0.02))
    if dup is not None:
        src, dst = dup
        Wq[dst] = Wq[src]
        sc[dst] = sc[src]
    return x, Wq, sc


def test_planted_unique_maximum_is_found(oracle):
    rng = np.random.default_rng(16)
    V, K, T = 700, 512, 3
    planted = [123, 699, 0]
    x, Wq, sc = _planted_head(rng, V, K, T, planted)
    lg = oracle.lmhead_logits(x, Wq, sc, K, T, V)
    a, best, second = oracle.argmax(lg)
    assert list(a) == planted
    assert np.all(best > second)


def test_exact_tie_goes_to_lowest_token_id_in_any_map_order(oracle):
    rng = np.random.default_rng(17)
    V, K = 600, 256
    x, Wq, sc = _planted_head(rng, V, K, 1, [410], dup=(410, 37))
    lg = oracle.lmhead_logits(x, Wq, sc, K, 1, V)
    assert lg[0, 37] == lg[0, 410]
    a, _, _ = oracle.argmax(lg)
    assert a[0] == 37
    vm = np.array([410, 5, 37, 299], np.int32)          # 410 listed before 37
    lgm = oracle.lmhead_logits(x, Wq, sc, K, 1, V, rows=vm)
    am, _, _ = oracle.argmax(lgm, ids=vm)
    assert am[0] == 37
    am2, _, _ = oracle.argmax(lgm[:, ::-1].copy(), ids=vm[::-1].copy())
    assert am2[0] == 37


def test_restricted_logits_are_full_logits_at_mapped_ids(oracle):
    rng = np.random.default_rng(18)
    V, K, T = 1000, 384, 2
    Wq, sc = gen.weights(rng, V, K)
    x = gen.activations(rng, T, K)
    vm = gen.vocab_map(rng, V, 137)
    full = oracle.lmhead_logits(x, Wq, sc, K, T, V)
    sub = oracle.lmhead_logits(x, Wq, sc, K, T, V, rows=vm)
    assert np.array_equal(sub, full[:, vm])
    a_sub, _, _ = oracle.argmax(sub, ids=vm)
    # the restricted argmax is the full argmax over the subset
    for t in range(T):
        m = full[t, vm].max()
        assert a_sub[t] == np.min(vm[full[t, vm] == m])


def test_verify_rule_hand_cases(oracle):
    a = np.array([11, 22, 33, 44], np.int32)
    assert oracle.verify(a, [11, 22, 33]) == (3, 44)       # all accepted: bonus
    assert oracle.verify(a, [10, 22, 33]) == (0, 11)       # first rejected
    assert oracle.verify(a, [11, 22, 34]) == (2, 33)       # mismatch at 2
    assert oracle.verify(a, [11, 0, 33]) == (1, 22)        # later agreement ignored
    assert oracle.verify(a[:1], []) == (0, 11)             # n_draft = 0: plain greedy


def test_lmhead_verify_per_stream_blocks(oracle):
    rng = np.random.default_rng(19)
    V, K, n_draft, S = 500, 256, 3, 3
    T = S * (n_draft + 1)
    planted = list(rng.choice(V, size=T, replace=False))
    x, Wq, sc = _planted_head(rng, V, K, T, planted)
    a = np.array(planted, np.int32)
    drafts = np.stack([
        a[0:3],                                  # stream 0: all accepted
        np.array([a[4], a[5] ^ 1, a[6]]),        # stream 1: mismatch at 1
        np.array([a[8] ^ 1, a[9], a[10]]),       # stream 2: mismatch at 0
    ]).astype(np.int32)
    r = oracle.lmhead_verify(x, Wq, sc, K, V, drafts, n_streams=S)
    assert list(r.a) == planted
    assert list(r.accept_len) == [3, 1, 0]
    assert list(r.next_token) == [a[3], a[5], a[8]]


# --------------------------------------------------------------------------
# byte accounting printed on the page


def test_lmhead_bytes_match_page():
    (V, K, gb), = _read_golden("lmhead_bytes_qwen_warp.txt")
    V, K = int(V), int(K)
    weights_and_scales = gen.lmhead_bytes(V, K, T=0, n_streams=0)
    assert weights_and_scales == 655_564_800
    assert round(weights_and_scales / 1e9, 3) == float(gb)


def test_gemm_bytes_are_weights_scales_and_activations():
    assert gen.gemm_bytes(0, 5120, 10240) == 10240 * 2560 + 10240 * 40 * 2
    assert gen.gemm_bytes(4, 17408, 5120) == 5120 * 8704 + 5120 * 136 * 2 + 4 * 17408 * 2 + 4 * 5120 * 2


def test_fp32_oracle_within_rounding_of_its_fp64_twin(oracle):
    rng = np.random.default_rng(20)
    T, K, N = 4, 5120, 64
    Wq, sc = gen.weights(rng, N, K)
    x = gen.activations(rng, T, K)
    y32, _, y64 = oracle.w4a16_gemm(x, Wq, sc, T, K, N, want64=True)
    rel = np.abs(y32 - y64).max() / np.abs(y64).max()
    assert rel < 1e-5


# --------------------------------------------------------------------------
# dynamic draft list (list maintenance of the restricted draft head)


def test_draft_list_hand_case(oracle):
    """Static [5, 9, 2], V = 20, cap 4.  Adding 9 (static), 7, 7 (repeat),
    25 and -1 (out of range), 3, 5 (static), 11, 12, 13: the list gains
    7, 3, 11, 12 in that order and 13 finds it full."""
    dl = oracle.draft_list_init([5, 9, 2], 20, 4)
    oracle.draft_list_add(dl, [9, 7, 7, 25, -1, 3, 5, 11, 12, 13])
    assert dl.count == 4
    assert dl.ids().tolist() == [5, 9, 2, 7, 3, 11, 12]


def test_draft_list_unused_slots_repeat_first_static_id(oracle):
    dl = oracle.draft_list_init([8, 1], 10, 3)
    assert dl.ids().tolist() == [8, 1, 8, 8, 8]
    oracle.draft_list_add(dl, [4])
    assert dl.ids().tolist() == [8, 1, 4, 8, 8]
    dl0 = oracle.draft_list_init([8, 1], 10, 0)
    oracle.draft_list_add(dl0, [4, 5])
    assert dl0.ids().tolist() == [8, 1]


def test_draft_list_matches_first_occurrence_definition(oracle):
    """Independent formulation with numpy: the added tokens are the in-range
    tokens of the concatenated sequence outside the static list, at their
    first occurrence, in sequence order, truncated to cap; adding in several
    calls equals adding the concatenation."""
    rng = np.random.default_rng(31)
    for trial in range(20):
        V = int(rng.integers(50, 400))
        static = rng.choice(V, size=int(rng.integers(1, 40)), replace=False)
        cap = int(rng.integers(0, 60))
        seq = rng.integers(-5, V + 5, size=int(rng.integers(0, 300)))
        inr = seq[(seq >= 0) & (seq < V)]
        inr = inr[~np.isin(inr, static)]
        _, first = np.unique(inr, return_index=True)
        expect = inr[np.sort(first)][:cap]
        dl = oracle.draft_list_init(static, V, cap)
        cuts = np.sort(rng.integers(0, seq.size + 1, size=3))
        for a, b in zip(np.r_[0, cuts], np.r_[cuts, seq.size]):
            oracle.draft_list_add(dl, seq[a:b])
        assert dl.count == expect.size
        ids = dl.ids()
        assert ids.size == static.size + cap
        assert ids[:static.size].tolist() == static.tolist()
        assert ids[static.size:static.size + expect.size].tolist() == expect.tolist()
        assert np.all(ids[static.size + expect.size:] == static[0])


# --------------------------------------------------------------------------
# top-k candidates rescored by the bf16 head


def _bf16(a):
    return gen.f32_to_bf16_bits(np.asarray(a, np.float32))


def test_bf16_logits_one_hot_reads_the_weight(oracle):
    rng = np.random.default_rng(40)
    V, K = 50, 64
    Wbf = _bf16(rng.standard_normal((V, K)))
    for k in (0, 17, 63):
        x = np.zeros((1, K), np.uint16)
        x[0, k] = _bf16(1.0)
        lg = oracle.bf16_logits(x, Wbf, K, 1, V)
        assert np.array_equal(lg[0], gen.bf16_bits_to_f32(Wbf[:, k]))


def test_bf16_logits_within_fp32_bound_of_fp64_matmul(oracle):
    rng = np.random.default_rng(41)
    V, K, T = 64, 1000, 3
    Wbf = _bf16(rng.standard_normal((V, K)))
    x = _bf16(rng.standard_normal((T, K)))
    lg = oracle.bf16_logits(x, Wbf, K, T, V).astype(np.float64)
    w = gen.bf16_bits_to_f32(Wbf).astype(np.float64)
    xv = gen.bf16_bits_to_f32(x).astype(np.float64)
    ref = xv @ w.T
    bound = K * 2.0 ** -24 * (np.abs(xv) @ np.abs(w).T)
    assert np.all(np.abs(lg - ref) <= bound)


def test_topk_orders_by_value_then_lowest_id(oracle):
    lg = np.array([[1.0, 3.0, 2.0, 3.0, 0.5, 2.0]], np.float32)
    ids, vals = oracle.topk(lg, 4)
    assert ids[0].tolist() == [1, 3, 2, 5]
    assert vals[0].tolist() == [3.0, 3.0, 2.0, 2.0]
    ids, _ = oracle.topk(lg, 4, ids=np.array([60, 10, 50, 20, 30, 40]))
    assert ids[0].tolist() == [10, 20, 40, 50]


def test_rescoring_with_every_candidate_is_the_bf16_argmax(oracle):
    rng = np.random.default_rng(42)
    V, K = 200, 256
    Wq, sc = gen.weights(rng, V, K)
    Wbf = _bf16(rng.standard_normal((V, K)) * 0.05)
    x = gen.activations(rng, 3, K)
    r = oracle.lmhead_verify_rescored(x, Wq, sc, Wbf, K, V, [0, 0], V)
    full = gen.bf16_bits_to_f32(x).astype(np.float64) @ gen.bf16_bits_to_f32(Wbf).astype(np.float64).T
    for t in range(3):
        s = np.sort(full[t])
        if s[-1] - s[-2] > 1e-3:
            assert r.a[t] == int(np.argmax(full[t]))


def test_rescoring_planted_flip(oracle):
    """Row 5 wins the int4 head by a wide margin, row 9 is second; the bf16
    head gives row 9 the larger logit.  One candidate keeps 5, two or more
    return 9."""
    V, K = 16, 128
    Wq = np.full((V, K // 8), 0x88888888, np.uint32)          # level 0 everywhere
    Wq[5] = 0xFFFFFFFF                                        # level +7
    Wq[9] = 0xEEEEEEEE                                        # level +6
    sc = np.full((V, 1), _bf16(1.0), np.uint16)
    Wbf = np.zeros((V, K), np.uint16)
    Wbf[5] = _bf16(1.0)
    Wbf[9] = _bf16(2.0)
    x = np.full((1, K), _bf16(1.0), np.uint16)
    assert oracle.lmhead_verify_rescored(x, Wq, sc, Wbf, K, V, [], 1).a.tolist() == [5]
    for k in (2, 3, 16):
        r = oracle.lmhead_verify_rescored(x, Wq, sc, Wbf, K, V, [], k)
        assert r.a.tolist() == [9]
        assert r.cand[0][:2].tolist() == [5, 9]


def test_rescoring_agrees_with_int4_when_heads_hold_the_same_weights(oracle):
    """bf16 weights equal to the int4 levels times a power-of-two scale hold
    the same numbers as the int4 head, so the rescored argmax is the int4
    argmax wherever the margin is clear of fp32 reordering."""
    rng = np.random.default_rng(43)
    V, K = 300, 512
    Wq, _ = gen.weights(rng, V, K)
    sc = np.full((V, K // 128), _bf16(2.0 ** -6), np.uint16)
    lv = ((Wq[:, :, None] >> (4 * np.arange(8))) & 0xF).astype(np.int64).reshape(V, K) - 8
    Wbf = _bf16(lv * 2.0 ** -6)
    x = gen.activations(rng, 4, K)
    r = oracle.lmhead_verify_rescored(x, Wq, sc, Wbf, K, V, [0, 0, 0], 8)
    l4 = oracle.lmhead_logits(x, Wq, sc, K, 4, V)
    a4, b4, s4 = oracle.argmax(l4)
    for t in range(4):
        if b4[t] - s4[t] > 1e-3:
            assert r.a[t] == a4[t]
