"""The C ABI without a GPU: the library loads, exports every function that
include/csa.h declares, and rejects bad arguments before touching a device."""
import ctypes
import os
import re

import pytest

from long_context_sparse_23_b300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa.h")

A16 = 1 << 20  # a fake, 16-byte aligned "device pointer" (never dereferenced on these paths)


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|csa_status|int|void)\s+(\w+)\s*\(", src, re.M)))


@pytest.fixture(scope="module")
def L():
    from long_context_sparse_23_b300 import build
    build.build()
    return _lib.lib()


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 15, names
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(_lib.SIGNATURES), set(names) ^ set(_lib.SIGNATURES)


def test_status_strings_and_version(L):
    for code, name in enumerate(["CSA_OK", "CSA_ERR_INVALID", "CSA_ERR_UNSUPPORTED", "CSA_ERR_WORKSPACE",
                                 "CSA_ERR_CUDA", "CSA_ERR_TIMEOUT", "CSA_ERR_DEVICE_INDEX"]):
        assert L.csa_status_string(code).decode() == name
    assert L.csa_status_string(99).decode() == "CSA_ERR_UNKNOWN"
    assert L.csa_version() >= 100


def test_workspace_sizes(L):
    need = ctypes.c_size_t(0)
    assert L.csa_index_topk_workspace(4, 1, 262144, 64, 128, 1024, ctypes.byref(need)) == 0
    # long rows: three bucket histograms (4096, 4096, 256 bins), then per 4096-key chunk a count,
    # and candidate lists of (key, index) pairs for every visible entry
    topk_scratch = (4 * (2 * 4096 + 256) * 4 + 4 * 64 * 4 + 4 * 262144 * 8 + 255) // 256 * 256
    assert need.value == 256 + 4 * 262144 * 4 + topk_scratch
    assert L.csa_topk_workspace(4, 1, 262144, 1024, ctypes.byref(need)) == 0
    assert need.value == 256 + topk_scratch
    assert L.csa_topk_workspace(8192, 1, 2048, 1024, ctypes.byref(need)) == 0
    assert need.value == 256                       # short rows: selected in shared memory
    assert L.csa_index_topk_workspace(1, 1, 5, 64, 128, 4, ctypes.byref(need)) == 0
    assert need.value == 256 + 256                # 8 floats rounded up to 256 bytes
    # decode, H = 64, d = 128 (tensor-core kernel): 1024 + 128 slots = 9 tiles -> 2
    # ranges, merged inside their cluster: no partials
    assert L.csa_attend_workspace(64, 1, 64, 128, 1024, 128, ctypes.byref(need)) == 0
    assert need.value == 256
    # 5200 + 128 slots = 42 tiles -> 9 ranges of 5 tiles, beyond a cluster:
    # H x (d + 1) floats of partials per range
    assert L.csa_attend_workspace(64, 1, 64, 128, 5200, 128, ctypes.byref(need)) == 0
    assert need.value == 256 + (64 * 9 * 64 * 129 * 4 + 255) // 256 * 256
    # one range (up to 5 tiles): no partials
    assert L.csa_attend_workspace(64, 1, 64, 128, 384, 128, ctypes.byref(need)) == 0
    assert need.value == 256
    # other head counts: the general decode kernel merges its splits inside a cluster
    assert L.csa_attend_workspace(64, 1, 32, 128, 1024, 128, ctypes.byref(need)) == 0
    assert need.value == 256
    assert L.csa_attend_workspace(1, 8192, 16, 128, 1024, 128, ctypes.byref(need)) == 0
    assert need.value == 256                       # prefill: no split partials
    # HCA decode, H = 64, d = 128 (tensor-core kernel): ranges of 4 128-key tiles,
    # partials (H x (d + 1) floats per range) in the workspace; 8192 + 128 keys
    # -> 65 tiles -> 17 ranges
    assert L.hca_attend_workspace(8, 1, 8192, 64, 128, 128, ctypes.byref(need)) == 0
    assert need.value == 256 + (8 * 17 * 64 * 129 * 4 + 255) // 256 * 256
    # one range: no partials
    assert L.hca_attend_workspace(8, 1, 300, 64, 128, 128, ctypes.byref(need)) == 0
    assert need.value == 256
    # other head counts keep the general kernel: one cluster per query up to
    # 131072 keys, 8192-key splits with partials in the workspace beyond
    assert L.hca_attend_workspace(8, 1, 8192, 32, 128, 128, ctypes.byref(need)) == 0
    assert need.value == 256
    # batch-invariant: per-sequence bytes scale linearly with B
    a, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    L.hca_attend_workspace(1, 1, 140000, 64, 128, 128, ctypes.byref(a))
    L.hca_attend_workspace(8, 1, 140000, 64, 128, 128, ctypes.byref(b))
    assert a.value == 256 + (274 * 64 * 129 * 4 + 255) // 256 * 256
    assert b.value - 256 == (8 * 274 * 64 * 129 * 4 + 255) // 256 * 256
    L.hca_attend_workspace(1, 1, 140000, 16, 128, 128, ctypes.byref(a))
    assert a.value == 256 + (18 * 16 * 129 * 4 + 255) // 256 * 256
    assert L.csa_attend_workspace(0, 1, 64, 128, 16, 8, ctypes.byref(need)) == _lib.CSA_ERR_INVALID


def test_layer_workspace_holds_the_attention_partials(L):
    """csa_layer's workspace = header + scores + top-k scratch + index lists +
    attention partials; only the last part depends on H.  At the 128K decode
    shape (B = 64, 32768 entries, W = 128) H = 64, d = 128 runs the
    tensor-core attention: top-1024 gives 2 ranges per query, merged inside
    their cluster (no partials), top-5200 gives 9 ranges, which keep their
    partials in the workspace; H = 32 merges its splits inside a cluster and
    needs none."""
    def size(H, k):
        la = _lib.csa_layer_args()
        for name, v in dict(B=64, Tq=1, N=32768, m=4, H=H, d=128, H_I=64, d_I=128, k=k, W=128).items():
            setattr(la, name, v)
        need = ctypes.c_size_t(0)
        assert L.csa_layer_workspace(ctypes.byref(la), ctypes.byref(need)) == 0
        return need.value
    assert size(64, 1024) == size(32, 1024)
    assert size(64, 5200) - size(32, 5200) == (64 * 9 * 64 * 129 * 4 + 255) // 256 * 256


def test_validation_before_any_launch(L):
    P3 = ctypes.c_void_p * 3
    D = (ctypes.c_int * 3)(64, 64, 32)
    ok = P3(A16, A16, A16)
    # compress: stream count, null pointer, misalignment, channel count, dtype
    assert L.csa_compress(0, ok, ok, ok, D, 1, 256, 4, 0, None) == _lib.CSA_ERR_INVALID
    assert L.csa_compress(1, P3(None, A16, A16), ok, ok, D, 1, 256, 4, 0, None) == _lib.CSA_ERR_INVALID
    assert L.csa_compress(1, P3(A16 + 2, 0, 0), ok, ok, D, 1, 256, 4, 0, None) == _lib.CSA_ERR_INVALID
    assert L.csa_compress(1, ok, ok, ok, (ctypes.c_int * 3)(12, 0, 0), 1, 256, 4, 0, None) == _lib.CSA_ERR_INVALID
    assert L.csa_compress(1, ok, ok, ok, D, 1, 256, 4, 7, None) == _lib.CSA_ERR_INVALID
    assert L.csa_compress(1, ok, ok, ok, D, 1, 256, 0, 0, None) == _lib.CSA_ERR_INVALID
    # indexer: unsupported head count / width, bad leading dimension, workspace
    args = [A16, A16, A16, 0, A16, 1, 4, 64, 64, 128, 4, A16, 64, A16, 256, None]
    a = list(args); a[8] = 48
    assert L.csa_index_scores(*a) == _lib.CSA_ERR_UNSUPPORTED
    a = list(args); a[9] = 96
    assert L.csa_index_scores(*a) == _lib.CSA_ERR_UNSUPPORTED
    a = list(args); a[12] = 62
    assert L.csa_index_scores(*a) == _lib.CSA_ERR_INVALID
    a = list(args); a[14] = 100
    assert L.csa_index_scores(*a) == _lib.CSA_ERR_WORKSPACE
    a = list(args); a[13] = A16 + 16
    assert L.csa_index_scores(*a) == _lib.CSA_ERR_WORKSPACE
    a = list(args); a[0] = None
    assert L.csa_index_scores(*a) == _lib.CSA_ERR_INVALID
    # per-query weights: the stride must cover the H_I heads
    a = list(args); a[3] = 32
    assert L.csa_index_scores(*a) == _lib.CSA_ERR_INVALID
    a = list(args); a[3] = -64
    assert L.csa_index_scores(*a) == _lib.CSA_ERR_INVALID
    # top-k: k range, too many entries
    targs = [A16, 64, A16, 1, 1, 64, 4, 16, A16, None, A16, 256, None]
    t = list(targs); t[7] = 5000
    assert L.csa_topk(*t) == _lib.CSA_ERR_UNSUPPORTED
    t = list(targs); t[5] = (1 << 24) + 1; t[1] = (1 << 24) + 4
    assert L.csa_topk(*t) == _lib.CSA_ERR_UNSUPPORTED
    t = list(targs); t[7] = 0
    assert L.csa_topk(*t) == _lib.CSA_ERR_INVALID
    # attention: head width, head count, window buffer, workspace
    at = [A16, A16, A16, A16, A16, A16, A16, A16, 1, 1, 64, 256, 64, 128, 16, 32, 0.0, A16, 0, None,
          A16, 1 << 20, None]
    x = list(at); x[13] = 96
    assert L.csa_attend(*x) == _lib.CSA_ERR_UNSUPPORTED
    x = list(at); x[12] = 65
    assert L.csa_attend(*x) == _lib.CSA_ERR_UNSUPPORTED
    x = list(at); x[4] = None
    assert L.csa_attend(*x) == _lib.CSA_ERR_INVALID
    x = list(at); x[21] = 100
    assert L.csa_attend(*x) == _lib.CSA_ERR_WORKSPACE
    x = list(at); x[18] = 3
    assert L.csa_attend(*x) == _lib.CSA_ERR_INVALID
    # layer: missing struct, partial gate set
    assert L.csa_layer(None, A16, 1 << 20, None) == _lib.CSA_ERR_INVALID
    la = _lib.csa_layer_args()
    la.g_k = A16
    assert L.csa_layer(ctypes.byref(la), A16, 1 << 20, None) == _lib.CSA_ERR_INVALID
    # workspace init / check with a bad pointer
    assert L.csa_workspace_init(None, 1024, None) == _lib.CSA_ERR_WORKSPACE
    assert L.csa_check_error(A16 + 8, None, 0, None) == _lib.CSA_ERR_WORKSPACE


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(ImportError):
        _lib.lib()


def test_stack_validation_before_any_launch(L):
    """csa_stack_decode refuses, before anything is enqueued, an unknown layer
    kind, a CSA layer whose indexer query shape is not the activation's, and
    layers of different activation shapes (fake device pointers: nothing runs)."""
    def layer(kind, **kw):
        la = _lib.csa_layer_args()
        for n, v in dict(B=1, Tq=1, N=1024, m=4, H=64, d=128, H_I=64, d_I=128, k=64, W=8, T=0, T_raw=16).items():
            setattr(la, n, v)
        for n in ("k_cmp", "v_cmp", "i_cmp", "k_win", "v_win", "raw_base", "w", "q_pos"):
            setattr(la, n, A16)
        for n, v in kw.items():
            setattr(la, n, v)
        st = _lib.csa_stack_layer()
        st.kind, st.a = kind, la
        return st

    def run(*ls):
        arr = (_lib.csa_stack_layer * len(ls))(*ls)
        need = ctypes.c_size_t(0)
        assert L.csa_stack_workspace(arr, len(ls), ctypes.byref(need)) == 0
        return L.csa_stack_decode(arr, len(ls), A16, A16, 0, A16, need.value, None)

    assert run(layer(_lib.CSA_STACK_SWA), layer(7)) == _lib.CSA_ERR_INVALID
    assert run(layer(_lib.CSA_STACK_SWA), layer(_lib.CSA_STACK_CSA, d_I=64)) == _lib.CSA_ERR_INVALID
    assert run(layer(_lib.CSA_STACK_SWA), layer(_lib.CSA_STACK_HCA, H=32)) == _lib.CSA_ERR_INVALID
    assert run(layer(_lib.CSA_STACK_HCA, m=0)) == _lib.CSA_ERR_INVALID
    assert L.csa_stack_decode(None, 1, A16, A16, 0, A16, 1 << 20, None) == _lib.CSA_ERR_INVALID
