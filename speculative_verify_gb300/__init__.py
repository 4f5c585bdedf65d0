"""Python binding of the C ABI in ``include/specverify.h``.

Argument marshalling only: every step of the GEMM and of the verify runs in
the sm_103a kernels of ``libspecverify.so``.  Tensors are torch CUDA tensors
(torch supplies device memory and streams); each call passes their
``data_ptr()`` and the current CUDA stream through ctypes.  There is no CPU
fallback: if the library is missing the import of the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

from . import build as _build

SV_OK = 0
STATUS = {0: "SV_OK", -1: "SV_ERR_NULL", -2: "SV_ERR_SHAPE", -3: "SV_ERR_ALIGN",
          -4: "SV_ERR_CUDA", -5: "SV_ERR_NOMEM", -6: "SV_ERR_DEVICE"}
DEVERR_BAD_MAP_ID = 0x1
DEVERR_TIMEOUT = 0x2

_lib = None


class GemmCall(ctypes.Structure):
    """sv_gemm_call of include/specverify.h."""
    _fields_ = [("x", ctypes.c_void_p), ("Wq", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("T", ctypes.c_int), ("K", ctypes.c_int), ("N", ctypes.c_int), ("y", ctypes.c_void_p)]


class VerifyCall(ctypes.Structure):
    """sv_verify_call of include/specverify.h."""
    _fields_ = [("x", ctypes.c_void_p), ("Wq", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("K", ctypes.c_int), ("drafts", ctypes.c_void_p), ("n_draft", ctypes.c_int),
                ("n_streams", ctypes.c_int), ("vocab_map", ctypes.c_void_p), ("n_map", ctypes.c_int),
                ("V", ctypes.c_int), ("accept_len", ctypes.c_void_p), ("next_token", ctypes.c_void_p)]


class SpecVerifyError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s failed: %s (%d): %s" % (fn, STATUS.get(status, "?"), status,
                                                     status_string(status)))


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None):
    """Load libspecverify.so (building it first only if asked via
    SPECVERIFY_AUTOBUILD=1) and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB_PATH
    if not os.path.exists(path):
        if os.environ.get("SPECVERIFY_AUTOBUILD") == "1":
            _build.build()
        else:
            raise RuntimeError("libspecverify.so is not built (%s); run "
                               "speculative_verify_gb300.build.build() or __graft_entry__.build()" % path)
    lib = ctypes.CDLL(path)
    vp, ci = ctypes.c_void_p, ctypes.c_int
    lib.w4a16_gemm.argtypes = [vp, vp, vp, ci, ci, ci, vp, vp]
    lib.w4a16_gemm.restype = ci
    lib.lmhead_verify.argtypes = [vp, vp, vp, ci, vp, ci, vp, ci, ci, vp, vp, vp]
    lib.lmhead_verify.restype = ci
    lib.lmhead_verify_batched.argtypes = [vp, vp, vp, ci, vp, ci, ci, vp, ci, ci, vp, vp, vp]
    lib.lmhead_verify_batched.restype = ci
    lib.lmhead_verify_ex.argtypes = [vp, vp, vp, ci, vp, ci, ci, vp, ci, ci, ci, vp, vp, vp]
    lib.lmhead_verify_ex.restype = ci
    lib.lmhead_verify_noalloc.argtypes = [vp, vp, vp, ci, vp, ci, vp, ci, ci, vp, vp, vp]
    lib.lmhead_verify_noalloc.restype = ci
    lib.lmhead_argmax.argtypes = [vp, vp, vp, ci, ci, vp, ci, ci, vp, vp, vp]
    lib.lmhead_argmax.restype = ci
    lib.lmhead_verify_rescored.argtypes = [vp, vp, vp, vp, ci, vp, ci, ci, ci, vp, vp, vp]
    lib.lmhead_verify_rescored.restype = ci
    lib.lmhead_argmax_rescored.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, vp, vp, vp]
    lib.lmhead_argmax_rescored.restype = ci
    cf = ctypes.c_float
    lib.lmhead_verify_sampled.argtypes = [vp, vp, vp, ci, vp, ci, ci, cf, ci, cf, cf, vp, vp, vp, vp]
    lib.lmhead_verify_sampled.restype = ci
    lib.lmhead_sampling_dist.argtypes = [vp, vp, vp, ci, ci, ci, cf, ci, cf, cf, vp, vp, vp]
    lib.lmhead_sampling_dist.restype = ci
    lib.draft_list_bytes.argtypes = [ci, ci, ci]
    lib.draft_list_bytes.restype = ctypes.c_size_t
    lib.draft_list_ids.argtypes = [vp, ci]
    lib.draft_list_ids.restype = vp
    lib.draft_list_init.argtypes = [vp, vp, ci, ci, ci, vp]
    lib.draft_list_init.restype = ci
    lib.draft_list_add.argtypes = [vp, vp, ci, vp]
    lib.draft_list_add.restype = ci
    lib.draft_list_count.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
    lib.draft_list_count.restype = ci
    lib.sv_status_string.argtypes = [ci]
    lib.sv_status_string.restype = ctypes.c_char_p
    lib.sv_last_device_error.argtypes = [ctypes.POINTER(ctypes.c_int32)]
    lib.sv_last_device_error.restype = ci
    lib.sv_hbm_read.argtypes = [vp, ctypes.c_size_t, vp, vp]
    lib.sv_hbm_read.restype = ci
    lib.sv_verify_cycle.argtypes = [ctypes.POINTER(GemmCall), ci, ctypes.POINTER(VerifyCall), vp]
    lib.sv_verify_cycle.restype = ci
    lib.sv_debug_set_fma_consumers.argtypes = [ci]
    lib.sv_debug_set_fma_consumers.restype = ci
    lib.sv_debug_set_tcgen05.argtypes = [ci]
    lib.sv_debug_set_tcgen05.restype = ci
    lib.sv_debug_set_wait_stall.argtypes = [ctypes.c_uint32]
    lib.sv_debug_set_wait_stall.restype = ci
    _lib = lib
    return lib


def header_symbols() -> list[str]:
    """Every function the public header declares."""
    hdr = os.path.join(_build.INCLUDE, "specverify.h")
    text = open(hdr).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)


def status_string(status: int) -> str:
    return load().sv_status_string(int(status)).decode()


# --------------------------------------------------------------------------
# torch-facing wrappers


def _torch():
    import torch
    return torch


def _check(fn, rc):
    if rc != SV_OK:
        raise SpecVerifyError(fn, rc)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _bits16(t, name):
    torch = _torch()
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError("%s must hold bf16 values (bfloat16, or int16/uint16 raw bits)" % name)
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA tensor" % name)
    return t


def _words(t, name):
    torch = _torch()
    if t.dtype not in (torch.int32, torch.uint32):
        raise TypeError("%s must be int32/uint32 packed nibble words" % name)
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA tensor" % name)
    return t


def _i32(t, name):
    torch = _torch()
    if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
        raise TypeError("%s must be a contiguous int32 CUDA tensor" % name)
    return t


def w4a16_gemm(x, Wq, scales, y=None, stream=None):
    """y[T][N] (bf16) = W4A16 group-128 GEMM of x[T][K] with Wq[N][K/8] and
    scales[N][K/128]; see ``w4a16_gemm`` in include/specverify.h."""
    torch = _torch()
    _bits16(x, "x"), _words(Wq, "Wq"), _bits16(scales, "scales")
    T, K = x.shape
    N = Wq.shape[0]
    if Wq.shape[1] * 8 != K or tuple(scales.shape) != (N, K // 128):
        raise ValueError("shape mismatch: x %s, Wq %s, scales %s" % (tuple(x.shape), tuple(Wq.shape),
                                                                      tuple(scales.shape)))
    if y is None:
        y = torch.empty((T, N), dtype=torch.bfloat16, device=x.device)
    _bits16(y, "y")
    _check("w4a16_gemm", load().w4a16_gemm(_ptr(x), _ptr(Wq), _ptr(scales), T, K, N, _ptr(y),
                                           _stream(stream)))
    return y


def lmhead_verify_batched(x, Wq, scales, drafts, vocab_map=None, accept_len=None,
                          next_token=None, stream=None):
    """One head pass for n_streams verify blocks: drafts is [n_streams][n_draft]
    int32, x is [n_streams*(1+n_draft)][K].  Returns (accept_len, next_token),
    int32 CUDA tensors of n_streams entries."""
    torch = _torch()
    _bits16(x, "x"), _words(Wq, "Wq"), _bits16(scales, "scales")
    T, K = x.shape
    V = Wq.shape[0]
    if drafts.dim() != 2:
        raise ValueError("drafts must be [n_streams][n_draft]")
    S, n_draft = drafts.shape
    if S * (n_draft + 1) != T:
        raise ValueError("x must have n_streams * (1 + n_draft) rows")
    if Wq.shape[1] * 8 != K or tuple(scales.shape) != (V, K // 128):
        raise ValueError("shape mismatch between x, Wq and scales")
    if n_draft:
        _i32(drafts, "drafts")
    if vocab_map is not None:
        _i32(vocab_map, "vocab_map")
    if accept_len is None:
        accept_len = torch.empty(S, dtype=torch.int32, device=x.device)
    if next_token is None:
        next_token = torch.empty(S, dtype=torch.int32, device=x.device)
    n_map = 0 if vocab_map is None else vocab_map.numel()
    _check("lmhead_verify_batched", load().lmhead_verify_batched(
        _ptr(x), _ptr(Wq), _ptr(scales), K, _ptr(drafts) if n_draft else None, n_draft, S,
        _ptr(vocab_map), n_map, V, _ptr(accept_len), _ptr(next_token), _stream(stream)))
    return accept_len, next_token


MAP_STATIC = 0x1


def lmhead_verify_ex(x, Wq, scales, drafts, vocab_map=None, flags=0, accept_len=None, next_token=None,
                     stream=None):
    """lmhead_verify_batched with flags (lmhead_verify_ex): MAP_STATIC for a
    vocab_map that no preceding kernel writes.  drafts: [n_streams][n_draft]."""
    torch = _torch()
    _bits16(x, "x"), _words(Wq, "Wq"), _bits16(scales, "scales")
    T, K = x.shape
    V = Wq.shape[0]
    if drafts.dim() != 2:
        raise ValueError("drafts must be [n_streams][n_draft]")
    S, n_draft = drafts.shape
    if S * (n_draft + 1) != T:
        raise ValueError("x must have n_streams * (1 + n_draft) rows")
    if Wq.shape[1] * 8 != K or tuple(scales.shape) != (V, K // 128):
        raise ValueError("shape mismatch between x, Wq and scales")
    if n_draft:
        _i32(drafts, "drafts")
    if vocab_map is not None:
        _i32(vocab_map, "vocab_map")
    if accept_len is None:
        accept_len = torch.empty(S, dtype=torch.int32, device=x.device)
    if next_token is None:
        next_token = torch.empty(S, dtype=torch.int32, device=x.device)
    n_map = 0 if vocab_map is None else vocab_map.numel()
    _check("lmhead_verify_ex", load().lmhead_verify_ex(
        _ptr(x), _ptr(Wq), _ptr(scales), K, _ptr(drafts) if n_draft else None, n_draft, S,
        _ptr(vocab_map), n_map, V, int(flags), _ptr(accept_len), _ptr(next_token), _stream(stream)))
    return accept_len, next_token


def lmhead_verify(x, Wq, scales, drafts, vocab_map=None, accept_len=None, next_token=None,
                  stream=None):
    """Greedy verify of one block of 1 + n_draft rows (drafts: [n_draft] int32).
    Returns (accept_len, next_token) as one-element int32 CUDA tensors."""
    torch = _torch()
    _bits16(x, "x"), _words(Wq, "Wq"), _bits16(scales, "scales")
    T, K = x.shape
    V = Wq.shape[0]
    n_draft = drafts.numel()
    if T != n_draft + 1:
        raise ValueError("x must have 1 + n_draft rows")
    if Wq.shape[1] * 8 != K or tuple(scales.shape) != (V, K // 128):
        raise ValueError("shape mismatch between x, Wq and scales")
    if n_draft:
        _i32(drafts, "drafts")
    if vocab_map is not None:
        _i32(vocab_map, "vocab_map")
    if accept_len is None:
        accept_len = torch.empty(1, dtype=torch.int32, device=x.device)
    if next_token is None:
        next_token = torch.empty(1, dtype=torch.int32, device=x.device)
    n_map = 0 if vocab_map is None else vocab_map.numel()
    _check("lmhead_verify", load().lmhead_verify(
        _ptr(x), _ptr(Wq), _ptr(scales), K, _ptr(drafts) if n_draft else None, n_draft,
        _ptr(vocab_map), n_map, V, _ptr(accept_len), _ptr(next_token), _stream(stream)))
    return accept_len, next_token


def lmhead_verify_noalloc(x, Wq, scales, drafts, vocab_map=None, accept_len=None,
                          next_token=None, stream=None):
    """lmhead_verify for callers that cannot allocate device memory: the
    kernel's scratch is a fixed array inside the library.  Pass accept_len and
    next_token (one-element int32 CUDA tensors) to keep the call itself free of
    allocations."""
    torch = _torch()
    _bits16(x, "x"), _words(Wq, "Wq"), _bits16(scales, "scales")
    T, K = x.shape
    V = Wq.shape[0]
    n_draft = drafts.numel()
    if T != n_draft + 1:
        raise ValueError("x must have 1 + n_draft rows")
    if Wq.shape[1] * 8 != K or tuple(scales.shape) != (V, K // 128):
        raise ValueError("shape mismatch between x, Wq and scales")
    if n_draft:
        _i32(drafts, "drafts")
    if vocab_map is not None:
        _i32(vocab_map, "vocab_map")
    if accept_len is None:
        accept_len = torch.empty(1, dtype=torch.int32, device=x.device)
    if next_token is None:
        next_token = torch.empty(1, dtype=torch.int32, device=x.device)
    n_map = 0 if vocab_map is None else vocab_map.numel()
    _check("lmhead_verify_noalloc", load().lmhead_verify_noalloc(
        _ptr(x), _ptr(Wq), _ptr(scales), K, _ptr(drafts) if n_draft else None, n_draft,
        _ptr(vocab_map), n_map, V, _ptr(accept_len), _ptr(next_token), _stream(stream)))
    return accept_len, next_token


def verify_cycle(gemms, verify=None, stream=None):
    """One verify cycle's weight reads in one call (sv_verify_cycle).

    gemms: a list of (x [T][K], Wq [N][K/8], scales [N][K/128], y [T][N])
    CUDA tensors; verify: None or a dict with x, Wq, scales, drafts
    [n_streams][n_draft], accept_len and next_token ([n_streams] int32), and
    optionally vocab_map.  Outputs are written in place."""
    arr = (GemmCall * max(1, len(gemms)))()
    for i, (x, Wq, scales, y) in enumerate(gemms):
        _bits16(x, "x"), _words(Wq, "Wq"), _bits16(scales, "scales"), _bits16(y, "y")
        T, K = x.shape
        N = Wq.shape[0]
        if Wq.shape[1] * 8 != K or tuple(scales.shape) != (N, K // 128) or tuple(y.shape) != (T, N):
            raise ValueError("shape mismatch in GEMM %d" % i)
        arr[i] = GemmCall(x.data_ptr(), Wq.data_ptr(), scales.data_ptr(), T, K, N, y.data_ptr())
    vptr = None
    if verify is not None:
        x, Wq, scales, drafts = verify["x"], verify["Wq"], verify["scales"], verify["drafts"]
        _bits16(x, "x"), _words(Wq, "Wq"), _bits16(scales, "scales")
        S, n_draft = drafts.shape
        if n_draft:
            _i32(drafts, "drafts")
        vm = verify.get("vocab_map")
        if vm is not None:
            _i32(vm, "vocab_map")
        acc, nxt = _i32(verify["accept_len"], "accept_len"), _i32(verify["next_token"], "next_token")
        K = x.shape[1]
        v = VerifyCall(x.data_ptr(), Wq.data_ptr(), scales.data_ptr(), K,
                       drafts.data_ptr() if n_draft else None, n_draft, S,
                       None if vm is None else vm.data_ptr(), 0 if vm is None else vm.numel(), Wq.shape[0],
                       acc.data_ptr(), nxt.data_ptr())
        vptr = ctypes.byref(v)
    _check("sv_verify_cycle", load().sv_verify_cycle(arr, len(gemms), vptr, _stream(stream)))


def hbm_read(src, sink, nbytes=None, stream=None):
    """Read nbytes (default: all) of the CUDA tensor src in one launch of the
    read-ceiling kernel (sv_hbm_read); sink: an int32/uint32 CUDA tensor with
    one entry per SM."""
    n = src.numel() * src.element_size() if nbytes is None else int(nbytes)
    _check("sv_hbm_read", load().sv_hbm_read(_ptr(src), n, _ptr(sink), _stream(stream)))


def lmhead_argmax(x, Wq, scales, vocab_map=None, ids=None, vals=None, stream=None):
    """Per-row argmax token id (lowest id on ties) and its fp32 logit."""
    torch = _torch()
    _bits16(x, "x"), _words(Wq, "Wq"), _bits16(scales, "scales")
    T, K = x.shape
    V = Wq.shape[0]
    if Wq.shape[1] * 8 != K or tuple(scales.shape) != (V, K // 128):
        raise ValueError("shape mismatch between x, Wq and scales")
    if vocab_map is not None:
        _i32(vocab_map, "vocab_map")
    if ids is None:
        ids = torch.empty(T, dtype=torch.int32, device=x.device)
    if vals is None:
        vals = torch.empty(T, dtype=torch.float32, device=x.device)
    n_map = 0 if vocab_map is None else vocab_map.numel()
    _check("lmhead_argmax", load().lmhead_argmax(
        _ptr(x), _ptr(Wq), _ptr(scales), K, T, _ptr(vocab_map), n_map, V, _ptr(ids), _ptr(vals),
        _stream(stream)))
    return ids, vals


def lmhead_verify_rescored(x, Wq, scales, Wbf, drafts, top_k=16, accept_len=None, next_token=None,
                           stream=None):
    """Greedy verify whose ids are the bf16 head's: the int4 head's top_k
    candidates of every row rescored with Wbf [V][K] bf16."""
    torch = _torch()
    _bits16(x, "x"), _words(Wq, "Wq"), _bits16(scales, "scales"), _bits16(Wbf, "Wbf")
    T, K = x.shape
    V = Wq.shape[0]
    n_draft = drafts.numel()
    if T != n_draft + 1:
        raise ValueError("x must have 1 + n_draft rows")
    if tuple(Wbf.shape) != (V, K):
        raise ValueError("Wbf must be [V][K]")
    if n_draft:
        _i32(drafts, "drafts")
    if accept_len is None:
        accept_len = torch.empty(1, dtype=torch.int32, device=x.device)
    if next_token is None:
        next_token = torch.empty(1, dtype=torch.int32, device=x.device)
    _check("lmhead_verify_rescored", load().lmhead_verify_rescored(
        _ptr(x), _ptr(Wq), _ptr(scales), _ptr(Wbf), K, _ptr(drafts) if n_draft else None, n_draft, int(top_k),
        V, _ptr(accept_len), _ptr(next_token), _stream(stream)))
    return accept_len, next_token


def lmhead_argmax_rescored(x, Wq, scales, Wbf, top_k=16, ids=None, vals=None, stream=None):
    """Per-row argmax among the int4 head's top_k candidates by bf16 logit."""
    torch = _torch()
    _bits16(x, "x"), _words(Wq, "Wq"), _bits16(scales, "scales"), _bits16(Wbf, "Wbf")
    T, K = x.shape
    V = Wq.shape[0]
    if tuple(Wbf.shape) != (V, K):
        raise ValueError("Wbf must be [V][K]")
    if ids is None:
        ids = torch.empty(T, dtype=torch.int32, device=x.device)
    if vals is None:
        vals = torch.empty(T, dtype=torch.float32, device=x.device)
    _check("lmhead_argmax_rescored", load().lmhead_argmax_rescored(
        _ptr(x), _ptr(Wq), _ptr(scales), _ptr(Wbf), K, T, int(top_k), V, _ptr(ids), _ptr(vals), _stream(stream)))
    return ids, vals


def lmhead_verify_sampled(x, Wq, scales, drafts, u, temperature=1.0, top_k=0, top_p=1.0, min_p=0.0,
                          accept_len=None, next_token=None, stream=None):
    """Exact speculative sampling verify over the 32 best logits of each
    row; u holds 2 (n_draft + 1) fp32 uniforms in [0, 1) on the device."""
    torch = _torch()
    _bits16(x, "x"), _words(Wq, "Wq"), _bits16(scales, "scales")
    T, K = x.shape
    V = Wq.shape[0]
    n_draft = drafts.numel()
    if T != n_draft + 1:
        raise ValueError("x must have 1 + n_draft rows")
    if n_draft:
        _i32(drafts, "drafts")
    if not (u.is_cuda and u.dtype == torch.float32 and u.is_contiguous() and u.numel() >= 2 * T):
        raise ValueError("u must be a contiguous CUDA float32 tensor of 2 (n_draft + 1) uniforms")
    if accept_len is None:
        accept_len = torch.empty(1, dtype=torch.int32, device=x.device)
    if next_token is None:
        next_token = torch.empty(1, dtype=torch.int32, device=x.device)
    _check("lmhead_verify_sampled", load().lmhead_verify_sampled(
        _ptr(x), _ptr(Wq), _ptr(scales), K, _ptr(drafts) if n_draft else None, n_draft, V, float(temperature),
        int(top_k), float(top_p), float(min_p), _ptr(u), _ptr(accept_len), _ptr(next_token), _stream(stream)))
    return accept_len, next_token


def lmhead_sampling_dist(x, Wq, scales, temperature=1.0, top_k=0, top_p=1.0, min_p=0.0, stream=None):
    """The rows' sampling distributions: ids [T][32] (-1 past the kept
    candidates) and probs [T][32]."""
    torch = _torch()
    _bits16(x, "x"), _words(Wq, "Wq"), _bits16(scales, "scales")
    T, K = x.shape
    V = Wq.shape[0]
    ids = torch.empty((T, 32), dtype=torch.int32, device=x.device)
    probs = torch.empty((T, 32), dtype=torch.float32, device=x.device)
    _check("lmhead_sampling_dist", load().lmhead_sampling_dist(
        _ptr(x), _ptr(Wq), _ptr(scales), K, T, V, float(temperature), int(top_k), float(top_p), float(min_p),
        _ptr(ids), _ptr(probs), _stream(stream)))
    return ids, probs


class DraftList:
    """A dynamic draft list in a device workspace (see draft_list_* in
    include/specverify.h).  ``ids`` is the n_static + cap entry int32 view
    to pass as vocab_map."""

    def __init__(self, static_ids, V, cap, stream=None):
        torch = _torch()
        _i32(static_ids, "static_ids")
        self.V, self.n_static, self.cap = int(V), static_ids.numel(), int(cap)
        nbytes = load().draft_list_bytes(self.V, self.n_static, self.cap)
        if nbytes == 0:
            raise ValueError("invalid draft list sizes")
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=static_ids.device)
        _check("draft_list_init", load().draft_list_init(_ptr(self.ws), _ptr(static_ids), self.n_static,
                                                         self.V, self.cap, _stream(stream)))
        off = load().draft_list_ids(_ptr(self.ws), self.V) - self.ws.data_ptr()
        self.ids = self.ws[off:off + 4 * (self.n_static + self.cap)].view(torch.int32)

    def add(self, tokens, stream=None):
        if tokens.numel():
            _i32(tokens, "tokens")
        _check("draft_list_add", load().draft_list_add(_ptr(self.ws), _ptr(tokens) if tokens.numel() else None,
                                                       tokens.numel(), _stream(stream)))

    def count(self) -> int:
        out = ctypes.c_int32(0)
        _check("draft_list_count", load().draft_list_count(_ptr(self.ws), ctypes.byref(out)))
        return int(out.value)


def last_device_error() -> int:
    """The sticky device error word (SV_DEVERR_* bits), cleared by the read."""
    out = ctypes.c_int32(0)
    _check("sv_last_device_error", load().sv_last_device_error(ctypes.byref(out)))
    return int(out.value)


def debug_set_wait_stall(ns: int) -> None:
    """Test hook of the bounded waits (sv_debug_set_wait_stall): with ns > 0
    every later stream-kernel launch makes one wait run out after ns
    nanoseconds and report SV_DEVERR_TIMEOUT; 0 turns it off."""
    _check("sv_debug_set_wait_stall", load().sv_debug_set_wait_stall(int(ns)))


def debug_set_fma_consumers(on: bool) -> None:
    """Measurement switch (sv_debug_set_fma_consumers): CUDA-core fma
    consumers instead of tensor-core mma for resident-activation launches."""
    _check("sv_debug_set_fma_consumers", load().sv_debug_set_fma_consumers(1 if on else 0))


def debug_set_tcgen05(on: bool) -> None:
    """Measurement switch (sv_debug_set_tcgen05): calls with 17 <= T <= 32
    run on the tcgen05 kernel (the default, True) or on mma.sync (False)."""
    _check("sv_debug_set_tcgen05", load().sv_debug_set_tcgen05(1 if on else 0))
