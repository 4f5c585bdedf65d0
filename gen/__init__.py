"""Seeded synthetic inputs and workload shapes, shared by the tests, the smoke
check and the benchmark.

This module holds none of the verify's arithmetic: it draws random bits,
rounds random reals to bf16 to make *inputs*, names the workload shapes and
counts the bytes a pass must move.  Both the CUDA path and the CPU oracle are
fed from here; neither is imported.

Input recipe (the pages measure on model files and prompts that are not
available, so these stand in for them, with the shapes of a Qwen3.8-27B-class
decoder: hidden 5,120, fused QKV 10,240, fused gate+up 34,816, down 17,408 ->
5,120, lm_head 248,320 x 5,120, draft vocabulary 40,960 ids):
  * packed weights: i.i.d. uniform uint32 words, i.e. eight i.i.d. uniform
    nibbles in [0, 15] per word;
  * scales: U(0.005, 0.02) rounded to bf16 (round to nearest even);
  * activations: N(0, 1) rounded to bf16;
  * vocab_map: distinct ids drawn without replacement from [0, V), unsorted.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# ----------------------------------------------------------------------------
# bf16 bit helpers (input construction only)


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round float32 values to bf16 (nearest even) and return the raw bits."""
    u = np.array(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    """Widen raw bf16 bits to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------
# generators


def weights(rng: np.random.Generator, rows: int, K: int):
    """(Wq [rows][K/8] uint32, scales [rows][K/128] bf16 bits)."""
    if K % 128:
        raise ValueError("K must be a multiple of 128")
    Wq = rng.integers(0, 2**32, size=(rows, K // 8), dtype=np.uint32)
    s = rng.uniform(0.005, 0.02, size=(rows, K // 128)).astype(np.float32)
    return Wq, f32_to_bf16_bits(s)


def activations(rng: np.random.Generator, T: int, K: int) -> np.ndarray:
    """x [T][K] bf16 bits drawn from N(0, 1)."""
    return f32_to_bf16_bits(rng.standard_normal(size=(T, K)).astype(np.float32))


def vocab_map(rng: np.random.Generator, V: int, n_map: int) -> np.ndarray:
    """n_map distinct token ids in [0, V), unsorted, int32."""
    return rng.choice(V, size=n_map, replace=False).astype(np.int32)


def token_not(rng: np.random.Generator, V: int, avoid: int) -> int:
    """A seeded token id in [0, V) different from ``avoid``."""
    while True:
        r = int(rng.integers(0, V))
        if r != avoid:
            return r


def drafts_with_mismatch(rng: np.random.Generator, a: np.ndarray, p: int, V: int,
                         pool=None) -> np.ndarray:
    """Drafts that agree with ``a`` (the verifier's argmax per row, given by the
    caller) before position p and differ from it at p; p == len(a) - 1 means
    every draft agrees.  Drafts after p are copied from ``a`` (they do not
    matter once a draft is rejected).  ``pool`` restricts the replacement token
    to a given id list (a restricted head)."""
    n_draft = len(a) - 1
    d = np.array(a[:n_draft], dtype=np.int32).copy()
    if p < n_draft:
        if pool is None:
            d[p] = token_not(rng, V, int(a[p]))
        else:
            while True:
                r = int(pool[int(rng.integers(0, len(pool)))])
                if r != int(a[p]):
                    d[p] = r
                    break
    return d


# ----------------------------------------------------------------------------
# workload shapes

HIDDEN = 5120
QKV_N = 10240
GATE_UP_N = 34816
FFN = 17408
VOCAB = 248320
DRAFT_VOCAB = 40960

GEMM_SHAPES = (("qkv", HIDDEN, QKV_N), ("gate_up", HIDDEN, GATE_UP_N), ("down", FFN, HIDDEN))


@dataclass
class Config:
    name: str
    seed: int
    gemms: tuple = ()                   # ((label, K, N), ...)
    gemm_T: tuple = ()                  # T values the GEMMs run at
    head: dict = field(default_factory=dict)   # V, K, n_draft, n_streams, n_map


CONFIGS = {
    0: Config("tiny", 0, gemms=(("tiny", 512, 1024),), gemm_T=(1,),
              head=dict(V=4096, K=512, n_draft=3, n_streams=1, n_map=0)),
    1: Config("decode_T1", 1, gemms=GEMM_SHAPES, gemm_T=(1,)),
    2: Config("mtp_T4", 2, gemms=GEMM_SHAPES, gemm_T=(4,),
              head=dict(V=VOCAB, K=HIDDEN, n_draft=3, n_streams=1, n_map=0)),
    3: Config("dflash2_T8_T32", 3, gemms=GEMM_SHAPES, gemm_T=(8, 32),
              head=dict(V=VOCAB, K=HIDDEN, n_draft=7, n_streams=1, n_map=0)),
    4: Config("restricted", 4,
              head=dict(V=VOCAB, K=HIDDEN, n_draft=3, n_streams=1, n_map=DRAFT_VOCAB)),
}


# ----------------------------------------------------------------------------
# algorithmic bytes (what one call must move at minimum)


def gemm_bytes(T: int, K: int, N: int) -> int:
    """Packed weights + scales read once, x read, y written."""
    return N * (K // 2) + N * (K // 128) * 2 + T * K * 2 + T * N * 2


def lmhead_bytes(V: int, K: int, T: int, n_map: int = 0, n_streams: int = 1,
                 n_draft: int = 0) -> int:
    """Packed rows + scales of every scored row read once, x read, the id list
    and the drafts read, two int32 results per stream written."""
    rows = n_map if n_map else V
    return (rows * (K // 2) + rows * (K // 128) * 2 + T * K * 2 + n_map * 4
            + n_streams * n_draft * 4 + n_streams * 8)


def gemm_flops(T: int, K: int, N: int) -> int:
    return 2 * T * K * N
