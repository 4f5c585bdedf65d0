"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every function the header declares, and rejects bad arguments with the
documented status before touching CUDA."""
import ctypes

import pytest

import speculative_verify_gb300 as sv
from speculative_verify_gb300 import build as svbuild


@pytest.fixture(scope="module")
def lib():
    svbuild.build()
    return sv.load()


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def test_library_exports_every_header_symbol(lib):
    names = sv.header_symbols()
    assert set(names) >= {"w4a16_gemm", "lmhead_verify", "lmhead_verify_batched",
                          "lmhead_argmax", "sv_status_string", "sv_last_device_error"}
    for name in names:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in sv.STATUS.items():
        s = sv.status_string(code)
        assert isinstance(s, str) and s
    assert sv.status_string(12345) == "unknown status"


def test_binding_has_same_names_as_abi():
    for name in ("w4a16_gemm", "lmhead_verify", "lmhead_verify_batched", "lmhead_argmax", "DraftList",
                 "lmhead_verify_rescored", "lmhead_argmax_rescored", "lmhead_verify_sampled",
                 "lmhead_sampling_dist"):
        assert callable(getattr(sv, name))


# Fake, never-dereferenced addresses.  Every call below must fail argument
# checking before any CUDA call; skipped where a GPU is present so that a
# checking bug could never turn into a launch on fake pointers.
A = ctypes.c_void_p(0x10000)          # 16-byte aligned
A2 = ctypes.c_void_p(0x20000)
A3 = ctypes.c_void_p(0x30000)
MIS = ctypes.c_void_p(0x10008)        # 8-byte aligned only
NUL = None

nogpu = pytest.mark.skipif(_has_gpu(), reason="fake-pointer checks run only where no GPU exists")


@nogpu
@pytest.mark.parametrize("args,code", [
    ((NUL, A, A2, 1, 512, 64, A3, None), -1),
    ((A, NUL, A2, 1, 512, 64, A3, None), -1),
    ((A, A, NUL, 1, 512, 64, A3, None), -1),
    ((A, A2, A3, 1, 512, 64, NUL, None), -1),
    ((A, A2, A3, 0, 512, 64, A, None), -2),
    ((A, A2, A3, 33, 512, 64, A, None), -2),
    ((A, A2, A3, 1, 500, 64, A, None), -2),
    ((A, A2, A3, 1, 0, 64, A, None), -2),
    ((A, A2, A3, 1, 512, 0, A, None), -2),
    ((MIS, A2, A3, 1, 512, 64, A, None), -3),
    ((A, MIS, A3, 1, 512, 64, A, None), -3),
    ((A, A2, A3, 1, 512, 64, MIS, None), -3),
])
def test_gemm_rejects_bad_arguments(lib, args, code):
    assert lib.w4a16_gemm(*args) == code


@nogpu
@pytest.mark.parametrize("kw,code", [
    (dict(n_draft=32), -2),
    (dict(n_draft=-1), -2),
    (dict(n_streams=0), -2),
    (dict(n_streams=9, n_draft=3), -2),         # T = 36 > 32
    (dict(V=0), -2),
    (dict(vmap=A, n_map=0), -2),
    (dict(vmap=A, n_map=5000, V=4096), -2),
    (dict(drafts=NUL), -1),
    (dict(acc=NUL), -1),
    (dict(nxt=NUL), -1),
    (dict(K=100), -2),
    (dict(x=MIS), -3),
    (dict(vmap=ctypes.c_void_p(0x10002), n_map=10), -3),
])
def test_verify_rejects_bad_arguments(lib, kw, code):
    a = dict(x=A, W=A2, s=A3, K=512, drafts=A, n_draft=3, n_streams=1, vmap=NUL, n_map=0,
             V=4096, acc=A, nxt=A2)
    a.update(kw)
    rc = lib.lmhead_verify_batched(a["x"], a["W"], a["s"], a["K"], a["drafts"], a["n_draft"],
                                   a["n_streams"], a["vmap"], a["n_map"], a["V"], a["acc"],
                                   a["nxt"], None)
    assert rc == code


@nogpu
def test_argmax_rejects_bad_arguments(lib):
    assert lib.lmhead_argmax(A, A2, A3, 512, 4, NUL, 0, 4096, NUL, NUL, None) == -1
    assert lib.lmhead_argmax(A, A2, A3, 512, 40, NUL, 0, 4096, A, NUL, None) == -2
    assert lib.lmhead_argmax(A, A2, A3, 512, 4, NUL, 0, 4096, ctypes.c_void_p(0x10001), NUL, None) == -3


def test_last_device_error_rejects_null(lib):
    assert lib.sv_last_device_error(None) == -1


def test_draft_list_sizes_and_ids_address(lib):
    """Workspace size = 32-byte header + membership bitmap (V bits, padded
    to 16 bytes) + 4 bytes per list entry; the id array follows the bitmap."""
    assert lib.draft_list_bytes(0, 1, 1) == 0
    assert lib.draft_list_bytes(100, 0, 1) == 0
    assert lib.draft_list_bytes(100, 1, -1) == 0
    V = 248320
    words = (V + 31) // 32                       # 7760, already a multiple of 4
    assert lib.draft_list_bytes(V, 32768, 4096) == 32 + 4 * words + 4 * (32768 + 4096)
    assert lib.draft_list_bytes(33, 1, 0) == 32 + 16 + 4
    assert lib.draft_list_ids(ctypes.c_void_p(0x10000), V) == 0x10000 + 32 + 4 * words
    assert lib.draft_list_ids(None, V) is None


@nogpu
def test_draft_list_rejects_bad_arguments(lib):
    assert lib.draft_list_init(NUL, A, 4, 100, 8, None) == -1
    assert lib.draft_list_init(A, NUL, 4, 100, 8, None) == -1
    assert lib.draft_list_init(A, A2, 0, 100, 8, None) == -2
    assert lib.draft_list_init(A, A2, 4, 0, 8, None) == -2
    assert lib.draft_list_init(MIS, A2, 4, 100, 8, None) == -3
    assert lib.draft_list_init(A, ctypes.c_void_p(0x20002), 4, 100, 8, None) == -3
    assert lib.draft_list_add(NUL, A2, 4, None) == -1
    assert lib.draft_list_add(A, NUL, 4, None) == -1
    assert lib.draft_list_add(A, A2, -1, None) == -2
    assert lib.draft_list_add(A, A2, 0, None) == 0          # nothing to add: no launch
    assert lib.draft_list_add(MIS, A2, 4, None) == -3
    assert lib.draft_list_count(NUL, None) == -1


NAN = float("nan")


@nogpu
@pytest.mark.parametrize("kw,code", [
    (dict(n_draft=8), -2),
    (dict(n_draft=-1), -2),
    (dict(top_k=33), -2),
    (dict(temp=NAN), -2),
    (dict(top_p=NAN), -2),
    (dict(min_p=1.5), -2),
    (dict(V=0), -2),
    (dict(K=200), -2),
    (dict(u=NUL), -1),
    (dict(drafts=NUL), -1),
    (dict(acc=NUL), -1),
    (dict(u=ctypes.c_void_p(0x10002)), -3),
    (dict(x=MIS), -3),
])
def test_sampled_verify_rejects_bad_arguments(lib, kw, code):
    a = dict(x=A, W=A2, s=A3, K=512, drafts=A, n_draft=3, V=4096, temp=1.0, top_k=0, top_p=1.0, min_p=0.0,
             u=A2, acc=A, nxt=A2)
    a.update(kw)
    rc = lib.lmhead_verify_sampled(a["x"], a["W"], a["s"], a["K"], a["drafts"], a["n_draft"], a["V"], a["temp"],
                                   a["top_k"], a["top_p"], a["min_p"], a["u"], a["acc"], a["nxt"], None)
    assert rc == code


@nogpu
def test_sampling_dist_rejects_bad_arguments(lib):
    assert lib.lmhead_sampling_dist(A, A2, A3, 512, 4, 4096, 1.0, 0, 1.0, 0.0, NUL, A, None) == -1
    assert lib.lmhead_sampling_dist(A, A2, A3, 512, 9, 4096, 1.0, 0, 1.0, 0.0, A, A2, None) == -2
    assert lib.lmhead_sampling_dist(A, A2, A3, 512, 4, 4096, 1.0, 0, 1.0, 0.0, A, ctypes.c_void_p(0x20001),
                                    None) == -3


@nogpu
def test_rescored_rejects_bad_arguments(lib):
    assert lib.lmhead_verify_rescored(A, A2, A3, NUL, 512, A, 3, 16, 4096, A, A2, None) == -1
    assert lib.lmhead_verify_rescored(A, A2, A3, A, 512, A, 3, 65, 4096, A, A2, None) == -2
    assert lib.lmhead_verify_rescored(A, A2, A3, A, 512, A, 3, 16, 8, A, A2, None) == -2
    assert lib.lmhead_verify_rescored(A, A2, A3, MIS, 512, A, 3, 16, 4096, A, A2, None) == -3
    assert lib.lmhead_argmax_rescored(A, A2, A3, A, 512, 9, 16, 4096, A, A2, None) == -2
