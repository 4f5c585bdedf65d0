"""CPU oracle for the W4A16 skinny GEMM and the int4 lm_head greedy verify.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  The product library
never imports, links or runs anything here, and this package imports nothing
from the product package.

The arithmetic lives in ``oracle.c`` (plain C, built with gcc, OpenMP over
output rows only, ``-ffp-contract=off``); this module only marshals numpy
arrays through ctypes and composes the three steps of the verify:
logits -> argmax -> first-mismatch comparison.

Sources, by page and section:
  * "qwen-warp and llamAmpere: two RTX 3090 engines for Qwen3.8, and what each one calls the same answer" -- "qwen-warp: keep the activations in bf16"
    (nibble format, level = nibble - 8, fp32 group scale after each
    128-column group) and "What each one calls the same answer" (greedy
    acceptance is argmax equality over the verify rows).
  * "swift-qwen3.8-rtx3090" -- "Body, heads and drafter" (keep drafts up to the
    first disagreement; a restricted draft head is a slice of lm_head rows).
  * "OpenJet Engine: CUDA LLM inference for Qwen3.8-27B" -- "How it works" (verify over T = 1 + n_draft rows),
    "How it gets its speed" (restricted draft vocabulary).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None

_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_u32p = np.ctypeslib.ndpointer(dtype=np.uint32, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    """Compile oracle.c into ``oracle/_build/liboracle.so`` (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    c_int = ctypes.c_int
    lib.or_w4a16_gemm.restype = c_int
    lib.or_w4a16_gemm.argtypes = [_u16p, _u32p, _u16p, c_int, c_int, c_int,
                                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.or_lmhead_logits.restype = c_int
    lib.or_lmhead_logits.argtypes = [_u16p, _u32p, _u16p, c_int, c_int, ctypes.c_void_p,
                                     c_int, c_int, ctypes.c_void_p, ctypes.c_void_p]
    lib.or_bf16_logits.restype = c_int
    lib.or_bf16_logits.argtypes = [_u16p, _u16p, c_int, c_int, ctypes.c_void_p, c_int, c_int,
                                   ctypes.c_void_p]
    lib.or_argmax.restype = c_int
    lib.or_argmax.argtypes = [_f32p, c_int, c_int, ctypes.c_void_p, _i32p,
                              ctypes.c_void_p, ctypes.c_void_p]
    lib.or_verify.restype = c_int
    lib.or_num_threads.restype = c_int
    lib.or_num_threads.argtypes = []
    lib.or_set_num_threads.restype = None
    lib.or_set_num_threads.argtypes = [c_int]
    lib.or_verify.argtypes = [_i32p, ctypes.c_void_p, c_int, ctypes.POINTER(ctypes.c_int32),
                              ctypes.POINTER(ctypes.c_int32)]
    _lib = lib
    return lib


def num_threads() -> int:
    """Threads the oracle's OpenMP regions use."""
    return int(_load().or_num_threads())


def set_num_threads(n: int) -> None:
    """Threads later OpenMP regions of the oracle use (n >= 1)."""
    _load().or_set_num_threads(int(n))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def w4a16_gemm(x, Wq, scales, T, K, N, want64=False):
    """Return (y32 [T][N] float32, ybf [T][N] uint16 bf16 bits[, y64]).

    y[t][n] = sum_g scale[n][g] * sum_{k in g} (nibble(n,k) - 8) * x[t][k],
    fp32 group sums in ascending k, then round-to-nearest-even to bf16.
    """
    lib = _load()
    x = _c(x, np.uint16).reshape(-1)
    Wq = _c(Wq, np.uint32).reshape(-1)
    scales = _c(scales, np.uint16).reshape(-1)
    y32 = np.empty((T, N), np.float32)
    ybf = np.empty((T, N), np.uint16)
    y64 = np.empty((T, N), np.float64) if want64 else None
    rc = lib.or_w4a16_gemm(x, Wq, scales, T, K, N, _ptr(y32), _ptr(y64), _ptr(ybf))
    if rc != 0:
        raise ValueError("oracle w4a16_gemm rejected its arguments")
    return (y32, ybf, y64) if want64 else (y32, ybf)


def lmhead_logits(x, Wq, scales, K, T, V, rows=None, want64=False):
    """fp32 logits [T][n_rows] of the rows listed in ``rows`` (None: all V)."""
    lib = _load()
    x = _c(x, np.uint16).reshape(-1)
    Wq = _c(Wq, np.uint32).reshape(-1)
    scales = _c(scales, np.uint16).reshape(-1)
    rows_a = None if rows is None else _c(rows, np.int32)
    n_rows = V if rows is None else int(rows_a.size)
    l32 = np.empty((T, n_rows), np.float32)
    l64 = np.empty((T, n_rows), np.float64) if want64 else None
    rc = lib.or_lmhead_logits(x, Wq, scales, K, T, _ptr(rows_a), n_rows, V, _ptr(l32), _ptr(l64))
    if rc != 0:
        raise ValueError("oracle lmhead_logits rejected its arguments")
    return (l32, l64) if want64 else l32


def argmax(logits, ids=None):
    """Row argmax with lowest token id on ties.

    Returns (a, best, second): token ids, the top value and the runner-up value.
    """
    lib = _load()
    logits = _c(logits, np.float32)
    T, n = logits.shape
    ids_a = None if ids is None else _c(ids, np.int32)
    a = np.empty(T, np.int32)
    best = np.empty(T, np.float32)
    second = np.empty(T, np.float32)
    rc = lib.or_argmax(logits, T, n, _ptr(ids_a), a, _ptr(best), _ptr(second))
    if rc != 0:
        raise ValueError("oracle argmax rejected its arguments (non-finite logits?)")
    return a, best, second


def verify(a, drafts):
    """(accept_len, next_token) for one block: first mismatch, then a[accept_len]."""
    lib = _load()
    a = _c(a, np.int32)
    d = _c(drafts, np.int32) if len(drafts) else None
    if a.size != (0 if d is None else d.size) + 1:
        raise ValueError("verify needs len(a) == n_draft + 1")
    acc = ctypes.c_int32()
    nxt = ctypes.c_int32()
    rc = lib.or_verify(a, _ptr(d), 0 if d is None else d.size, ctypes.byref(acc), ctypes.byref(nxt))
    if rc != 0:
        raise ValueError("oracle verify rejected its arguments")
    return int(acc.value), int(nxt.value)


def bf16_logits(x, Wbf, K, T, V, rows=None):
    """fp32 logits [T][n_rows] of bf16 weight rows (Wbf [V][K] bf16 bits):
    exact products summed in ascending k."""
    lib = _load()
    x = _c(x, np.uint16).reshape(-1)
    Wbf = _c(Wbf, np.uint16).reshape(-1)
    rows_a = None if rows is None else _c(rows, np.int32)
    n_rows = V if rows is None else int(rows_a.size)
    out = np.empty((T, n_rows), np.float32)
    rc = lib.or_bf16_logits(x, Wbf, K, T, _ptr(rows_a), n_rows, V, _ptr(out))
    if rc != 0:
        raise ValueError("oracle bf16_logits rejected its arguments")
    return out


def topk(logits, k, ids=None):
    """Per row the k candidates of largest logit, ties to the lowest token
    id, ordered best first.  Returns token ids [T][k] and values [T][k]."""
    logits = np.asarray(logits, np.float32)
    T, n = logits.shape
    ids_a = np.arange(n, dtype=np.int64) if ids is None else np.asarray(ids, np.int64)
    out_ids = np.empty((T, k), np.int32)
    out_val = np.empty((T, k), np.float32)
    for t in range(T):
        order = np.lexsort((ids_a, -logits[t].astype(np.float64)))[:k]
        out_ids[t] = ids_a[order]
        out_val[t] = logits[t][order]
    return out_ids, out_val


@dataclass
class RescoredResult:
    accept_len: np.ndarray   # [n_streams] int32
    next_token: np.ndarray   # [n_streams] int32
    a: np.ndarray            # [T] rescored argmax token id per row
    cand: np.ndarray         # [T][k] int4 candidates, best first
    cand_gap: np.ndarray     # [T] k-th minus (k+1)-th int4 logit (inf when k = V)
    bf16: np.ndarray         # [T][k] bf16 logits of the candidates
    margin: np.ndarray       # [T] best - runner-up bf16 logit among the candidates


def lmhead_verify_rescored(x, Wq, scales, Wbf, K, V, drafts, k):
    """Greedy verify with the int4 head's top-k candidates rescored by the
    bf16 head: int4 fp32 logits -> top k per row (ties to the lowest id) ->
    bf16 fp32 logits of those candidates -> argmax among them (ties to the
    lowest id) -> first mismatch with the drafts."""
    drafts = np.asarray(drafts, np.int32).reshape(-1)
    T = drafts.size + 1
    l4 = lmhead_logits(x, Wq, scales, K, T, V)
    cand, cval = topk(l4, k)
    gap = np.full(T, np.inf)
    if k < V:
        _, cval1 = topk(l4, k + 1)
        gap = cval1[:, k - 1].astype(np.float64) - cval1[:, k].astype(np.float64)
    b16 = np.empty((T, k), np.float32)
    a = np.empty(T, np.int32)
    margin = np.empty(T)
    for t in range(T):
        b16[t] = bf16_logits(x[t:t + 1], Wbf, K, 1, V, rows=cand[t])[0]
        at, best, second = argmax(b16[t:t + 1], ids=cand[t])
        a[t] = at[0]
        margin[t] = float(best[0]) - float(second[0])
    acc, nxt = verify(a, drafts)
    return RescoredResult(np.array([acc], np.int32), np.array([nxt], np.int32), a, cand, gap, b16, margin)


@dataclass
class VerifyResult:
    accept_len: np.ndarray   # [n_streams] int32
    next_token: np.ndarray   # [n_streams] int32
    a: np.ndarray            # [T] argmax token id per row
    margin: np.ndarray       # [T] best - runner-up logit per row (fp32)
    logits: np.ndarray       # [T][n_rows] fp32


def lmhead_verify(x, Wq, scales, K, V, drafts, n_streams=1, vocab_map=None):
    """The whole greedy verify: logits -> argmax -> per-stream first mismatch.

    x holds n_streams blocks of (1 + n_draft) rows; drafts is
    [n_streams][n_draft].  With vocab_map the candidate rows are
    Wq[vocab_map[j]] and every id returned is a token id.
    """
    drafts = np.asarray(drafts, np.int32).reshape(n_streams, -1)
    n_draft = drafts.shape[1]
    rows_per = n_draft + 1
    T = n_streams * rows_per
    logits = lmhead_logits(x, Wq, scales, K, T, V, rows=vocab_map)
    a, best, second = argmax(logits, ids=vocab_map)
    acc = np.empty(n_streams, np.int32)
    nxt = np.empty(n_streams, np.int32)
    for s in range(n_streams):
        acc[s], nxt[s] = verify(a[s * rows_per:(s + 1) * rows_per], drafts[s])
    margin = (best.astype(np.float64) - second.astype(np.float64))
    return VerifyResult(acc, nxt, a, margin, logits)



# ----------------------------------------------------------------------------
# Dynamic draft list (list maintenance for the restricted draft head)
#
# Sources: "OpenJet Engine: CUDA LLM inference for Qwen3.8-27B" -- "How it
# gets its speed" (the draft lm_head scores a static list of the most
# frequent tokens plus the tokens of the current sequence missing from it,
# added on the fly); "Tesla P100 (sm_60) llama.cpp patches for
# Qwen3.5/3.6-35B-A3B: ~2x decode and prompt processing over the shinbunbun
# baseline" -- "MTP draft vocabulary (patch 17)" and "The draft vocabulary
# file" (the draft head also scores every token that has appeared in the
# conversation, up to 4096 of them).
#
# The pages fix what the list contains (static ids, then sequence tokens not
# already in it, at most `cap` of them); the order of the added tokens and
# what happens past the cap are readings: added tokens keep their order of
# first appearance, and once `cap` tokens were added, later new tokens are
# not added.  Tokens outside [0, V) are ignored.  The list always has
# n_static + cap entries: unused dynamic slots repeat static_ids[0], which
# changes no argmax (a duplicate candidate ties with itself).


@dataclass
class DraftList:
    V: int
    static: list
    cap: int
    added: list

    def ids(self) -> np.ndarray:
        pad = self.static[0]
        dyn = self.added + [pad] * (self.cap - len(self.added))
        return np.array(self.static + dyn, dtype=np.int32)

    @property
    def count(self) -> int:
        return len(self.added)


def draft_list_init(static_ids, V: int, cap: int) -> DraftList:
    static = [int(t) for t in np.asarray(static_ids).ravel()]
    assert len(static) >= 1 and cap >= 0
    assert all(0 <= t < V for t in static)
    return DraftList(V=V, static=static, cap=cap, added=[])


def draft_list_add(dl: DraftList, tokens) -> DraftList:
    """Append, in order, every token of `tokens` that is in [0, V), not in
    the static list and not already added, while fewer than cap were added."""
    member = set(dl.static) | set(dl.added)
    for t in np.asarray(tokens).ravel():
        t = int(t)
        if len(dl.added) >= dl.cap:
            break
        if 0 <= t < dl.V and t not in member:
            dl.added.append(t)
            member.add(t)
    return dl


# ----------------------------------------------------------------------------
# Exact speculative sampling verify over the 32 best logits of each row
#
# Sources: "OpenJet Engine: CUDA LLM inference for Qwen3.8-27B" -- "How it
# gets its speed" (sampling keeps the 32 best logits of each verified row; a
# draft is accepted with probability p(draft), a rejected one is resampled
# from the rest of the distribution, so the sampled distribution is exact)
# and "Limitations" (temperature, top-k <= 32, top-p and min-p, in
# llama.cpp's order); "qwen-warp and llamAmpere: two RTX 3090 engines for
# Qwen3.8, and what each one calls the same answer" -- "What each one calls
# the same answer" (standard speculative sampling: accept, else draw from the
# residual; that keeps the output distributed exactly as the target).
#
# Readings where the pages leave a step open:
#  * The drafter is a point mass on its draft d, so the acceptance
#    probability min(1, p(d) / q(d)) is p(d) and the residual
#    norm(max(0, p - q)) is p with d removed and renormalised.
#  * llama.cpp's order is top-k, top-p, min-p, then temperature: top-p and
#    min-p see the temperature-1 distribution of the surviving candidates.
#  * All arithmetic is fp32.  The pages fix no summation order, so the
#    plainest one is taken: running sums over the (at most 32) candidates
#    are accumulated one candidate at a time, best first, and a total is
#    the last running sum.  With m the best logit and d_j = l_j - m,
#      top-p keeps the shortest prefix whose running sum of exp(d_j) reaches
#      top_p times the sum over the candidates (all of them if rounding
#      never reaches it);
#      min-p keeps the prefix of candidates with exp(d_j) >= min_p (the best
#      one always);
#      the weights are w_j = exp(d_j / temperature), W their total;
#      accept iff u_accept * W < w_d;
#      a sample takes the first candidate (best first) whose running sum c
#      over the candidates it may take (the rejected draft's weight set to
#      0) satisfies u_sample * W' < c, W' their total (the last of them if
#      rounding never gets there).
#  * temperature <= 0 is greedy: the distribution is the point mass on the
#    best candidate.
#  * Row i uses the uniforms u[2 i] (accept) and u[2 i + 1] (sample), each
#    in [0, 1); they are inputs, drawn by the caller.

SAMPLE_KEEP = 32


@dataclass
class SamplingDist:
    ids: np.ndarray          # [n] token ids of the candidates kept, best first
    logits: np.ndarray       # [n_cand] fp32 logits of all the candidates the chain started from
    w: np.ndarray            # [n] fp32 weights
    W: np.float32            # their fp32 sum, in order
    cut_margin: float        # relative distance of the top-p / min-p cuts from their thresholds
    cut_index: list          # positions after which a cut fell
    n_cand: int              # candidates the chain started from
    sel_gap: float           # the last starting candidate's logit minus the first one left out

    def order_gap(self, j):
        """Logit distance of candidate j from its neighbours in the order."""
        v = self.logits
        g = np.inf
        if j > 0:
            g = min(g, float(v[j - 1]) - float(v[j]))
        if j + 1 < v.size:
            g = min(g, float(v[j]) - float(v[j + 1]))
        return g

    def cut_clear(self, eps_rel, eps_logit):
        """Whether the kept set is the same under any rounding of the logits
        below eps_logit and of the cut sums below eps_rel (a cut after
        position j depends on the order of j and j + 1 only)."""
        if self.cut_margin < eps_rel:
            return False
        v = self.logits
        if any(j + 1 < v.size and float(v[j]) - float(v[j + 1]) < eps_logit for j in self.cut_index):
            return False
        if self.ids.size == self.n_cand and self.sel_gap < eps_logit:
            return False
        return True


def _f32(v):
    return np.float32(v)


def _running_f32(vals):
    """Running sums of fp32 values, added one at a time in the given order
    (c_0 = v_0, c_j = fl(c_{j-1} + v_j))."""
    out = np.zeros(len(vals), np.float32)
    c = _f32(0.0)
    for j, v in enumerate(vals):
        c = _f32(c + _f32(v))
        out[j] = c
    return out


def _sum_f32(vals):
    """Total of fp32 values added one at a time in the given order."""
    return _f32(_running_f32(vals)[-1]) if len(vals) else _f32(0.0)


def sampling_dist(vals, ids, temperature, top_k=0, top_p=1.0, min_p=0.0, sel_gap=np.inf) -> SamplingDist:
    """The sampling distribution of one row from its kept candidates
    (fp32 logits best first, ties to the lowest id)."""
    vals = np.asarray(vals, np.float32)
    ids = np.asarray(ids, np.int32)
    n0 = n = vals.size
    cut_index = []
    if top_k > 0 and top_k < n:
        n = int(top_k)
        cut_index.append(n - 1)
    if temperature <= 0:
        if n0 > 1:
            cut_index = [0]
        return SamplingDist(ids[:1].copy(), vals.copy(), np.ones(1, np.float32), _f32(1.0), np.inf,
                            cut_index, n0, sel_gap)
    m = vals[0]
    d = np.array([_f32(vals[j] - m) for j in range(n)], np.float32)
    e = np.exp(d).astype(np.float32)
    cut_margin = np.inf
    if top_p < 1.0:
        cs = _running_f32(e[:n])
        S = cs[n - 1]
        thr = _f32(_f32(top_p) * S)
        c = _f32(0.0)
        prev = _f32(0.0)
        keep = n
        for j in range(n):
            prev = c
            c = cs[j]
            if c >= thr:
                keep = j + 1
                break
        if keep < n or c >= thr:
            cut_margin = min(cut_margin, float(c - thr) / float(S), float(thr - prev) / float(S) if keep > 1 else np.inf)
            cut_index.append(keep - 1)
        n = keep
    if min_p > 0.0:
        mp = _f32(min_p)
        keep = 1
        while keep < n and e[keep] >= mp:
            keep += 1
        cut_margin = min(cut_margin, float(e[keep - 1] - mp) if keep > 1 else np.inf)
        if keep < n:
            cut_margin = min(cut_margin, float(mp - e[keep]))
            cut_index.append(keep - 1)
        n = keep
    t = _f32(temperature)
    w = np.exp(np.array([_f32(d[j] / t) for j in range(n)], np.float32)).astype(np.float32)
    return SamplingDist(ids[:n].copy(), vals.copy(), w, _sum_f32(w), cut_margin, cut_index, n0,
                        sel_gap)


def sample_from(dist: SamplingDist, u, exclude=None):
    """Inverse-CDF draw over the candidates best first, skipping position
    `exclude`.  Returns (token id, position, relative margin of the draw
    from the nearest boundary of the chosen interval)."""
    order = [j for j in range(dist.ids.size) if j != exclude]
    if not order:
        return int(dist.ids[exclude]), exclude, np.inf
    wx = dist.w.copy()
    if exclude is not None:
        wx[exclude] = 0.0
    cs = _running_f32(wx)
    Wx = cs[-1]
    target = _f32(_f32(u) * Wx)
    c = _f32(0.0)
    for j in order:
        lo = c
        c = cs[j]
        if target < c:
            margin = min(float(c - target), float(target - lo) if j != order[0] else np.inf) / float(Wx)
            return int(dist.ids[j]), j, margin
    return int(dist.ids[order[-1]]), order[-1], float(target - c) / float(Wx) if float(Wx) > 0 else np.inf


@dataclass
class SampledResult:
    accept_len: int
    next_token: int
    dists: list              # [T] SamplingDist
    clear: bool              # every decision that fixed the outcome is clear of rounding
    margin: float            # smallest relative decision margin on the path


def verify_sampled_from_logits(logits, drafts, u, temperature, top_k=0, top_p=1.0, min_p=0.0,
                               eps_rel=1e-4, eps_logit=1e-3) -> SampledResult:
    """Speculative sampling verify of T = 1 + n_draft rows of fp32 logits
    [T][n] with point-mass drafts.  `clear` says whether every decision on
    the path taken (the kept set, the cuts, each accept test and the final
    draw) is at least eps_rel (relative) and every candidate order that
    matters at least eps_logit (logit units) away from flipping."""
    logits = np.asarray(logits, np.float32)
    drafts = np.asarray(drafts, np.int32).reshape(-1)
    u = np.asarray(u, np.float32).reshape(-1)
    T, n = logits.shape
    assert T == drafts.size + 1 and u.size >= 2 * T
    keep = min(SAMPLE_KEEP, n)
    cid, cval = topk(logits, keep)
    sel_gap = np.full(T, np.inf)
    if keep < n:
        _, cval1 = topk(logits, keep + 1)
        sel_gap = cval1[:, keep - 1].astype(np.float64) - cval1[:, keep].astype(np.float64)
    dists = [sampling_dist(cval[i], cid[i], temperature, top_k, top_p, min_p, float(sel_gap[i])) for i in range(T)]
    margin = np.inf
    clear = True

    def draw(i, u_s, exclude=None):
        nonlocal margin, clear
        tok, j, mg = sample_from(dists[i], u_s, exclude)
        margin = min(margin, mg)
        if mg < eps_rel or dists[i].order_gap(j) < eps_logit:
            clear = False
        return tok

    for i in range(T):
        dist = dists[i]
        margin = min(margin, dist.cut_margin)
        if not dist.cut_clear(eps_rel, eps_logit):
            clear = False
        if i == T - 1:
            return SampledResult(i, draw(i, u[2 * i + 1]), dists, clear, margin)
        hit = np.nonzero(dist.ids == drafts[i])[0]
        jd = int(hit[0]) if hit.size else None
        if jd is not None:
            lhs = _f32(u[2 * i] * dist.W)
            mg = abs(float(lhs) - float(dist.w[jd])) / float(dist.W)
            margin = min(margin, mg)
            if mg < eps_rel:
                clear = False
            if lhs < dist.w[jd]:
                continue
        return SampledResult(i, draw(i, u[2 * i + 1], jd), dists, clear, margin)


def lmhead_verify_sampled(x, Wq, scales, K, V, drafts, u, temperature, top_k=0, top_p=1.0, min_p=0.0):
    """The int4 head's fp32 logits, then verify_sampled_from_logits."""
    drafts = np.asarray(drafts, np.int32).reshape(-1)
    T = drafts.size + 1
    logits = lmhead_logits(x, Wq, scales, K, T, V)
    return verify_sampled_from_logits(logits, drafts, u, temperature, top_k, top_p, min_p)
