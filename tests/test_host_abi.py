"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/varlen_attn.h declares, validates arguments with the
documented status codes before touching a device, and its host tile count
matches the page values.  Pointers passed here are never dereferenced: every
call either fails validation or stops at the device query, which fails for
want of a GPU; where a GPU is visible the tests that call the library skip
themselves rather than launch on fake pointers."""
import ctypes
import json
import os
import pathlib
import re

import numpy as np
import pytest

from packed_variable_length_varlen_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "varlen_attn.h")
GOLDEN = os.path.join(ROOT, "tests", "golden", "page_values.json")


def _gpu_visible() -> bool:
    try:
        import torch
        return bool(torch.cuda.is_available())
    except Exception:
        return False


@pytest.fixture(scope="module")
def va():
    # Every call below passes fake device pointers and relies on the device
    # query failing.  Where a GPU is visible, a call that passes validation
    # would launch kernels on those addresses, so these checks run only on a
    # machine without one (the GPU tests cover the calls that reach a device).
    if _gpu_visible():
        pytest.skip("fake-pointer ABI checks run only where no GPU is visible")
    from packed_variable_length_varlen_gb300 import build
    build.build()
    from packed_variable_length_varlen_gb300 import varlen_attn
    return varlen_attn


def _declared():
    src = pathlib.Path(HEADER).read_text()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(varlen_attn_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(va):
    names = _declared()
    assert len(names) >= 9
    for n in names:
        assert hasattr(va.LIB, n), n
    assert sorted(va.EXPORTED) == names


def test_status_strings(va):
    for code in range(0, -11, -1):
        s = va.varlen_attn_status_string(code)
        assert s and s != "unknown status"
    assert va.varlen_attn_status_string(5) == "unknown status"


def test_tile_count_page_values(va):
    g = json.loads(pathlib.Path(GOLDEN).read_text())["windowed_tile_count"]
    cu = g["cu_seqlens_q"]
    assert va.varlen_attn_tile_count(cu, len(cu) - 1, cu[-1], g["num_heads"], g["tile_m"]) == g["valid_tiles"]


def test_tile_count_edge_cases(va):
    # empty, one-row, tile multiples +-1, trailing empty pair
    cu = [0, 0, 1, 128, 256, 385, 385, 385]
    assert va.varlen_attn_tile_count(cu, 7, 385, 2, 128) == 2 * (0 + 1 + 1 + 1 + 2 + 0 + 0)
    # clamping: entries beyond total or decreasing count as empty
    assert va.varlen_attn_tile_count([0, 500, 100, 2 ** 30, -5, 260], 5, 260, 1, 128) == 3 + 0 + 2 + 0 + 3
    rng = np.random.default_rng(3)
    for _ in range(50):
        lens = rng.integers(0, 1000, size=int(rng.integers(1, 30)))
        cu = [0] + list(np.cumsum(lens))
        for tile in (64, 128):
            exp = sum(-(-int(x) // tile) for x in lens) * 3
            assert va.varlen_attn_tile_count(cu, len(lens), int(cu[-1]), 3, tile) == exp
    assert va.varlen_attn_tile_count([0, 1], 1, 1, 1, 0) == -1


def test_workspace_size(va):
    n = va.varlen_attn_bwd_workspace_size(2, 410923, 16, 96)
    r = lambda x: (x + 255) // 256 * 256
    pad = 4 * ((410923 + 3) // 4) + 4 * 2 + 128  # segment-padded delta / LSE rows
    assert n == r(410923 * 16 * 96 * 4) + 2 * r(pad * 16 * 4)
    assert n > 2 ** 31  # a 64-bit size
    assert va.varlen_attn_bwd_workspace_size(-1, 10, 1, 64) == 0


class _Fake:
    """Stands in for a tensor: a data pointer and (row, head, 1) strides."""

    def __init__(self, ptr, row, head, rows=10, H=2, D=64):
        self._p, self._s, self.shape = ptr, (row, head, 1), (rows, H, D)

    def data_ptr(self):
        return self._p

    def stride(self, i=None):
        return self._s if i is None else self._s[i]

    def dim(self):
        return 3


def _fwd(va, q=None, cu=0x2000, B=1, tq=10, tk=10, H=2, D=64, scale=0.125, out=None, lse=0x3000, stride=None):
    st = stride or (H * D, D)
    q = q or _Fake(0x1000, *st)
    out = out or _Fake(0x1000, *st)

    class _P:
        def __init__(self, p):
            self._p = p

        def data_ptr(self):
            return self._p
    return va.varlen_attn_fwd(q, q, q, _P(cu), _P(cu), B, tq, tk, H, D, 0, 0, scale, out, _P(lse), 0)


def test_validation_codes(va):
    assert _fwd(va, D=80) == va.VARLEN_ERR_HEAD_DIM
    assert _fwd(va, B=0) == va.VARLEN_ERR_SHAPE
    assert _fwd(va, scale=0.0) == va.VARLEN_ERR_SHAPE
    assert _fwd(va, scale=float("nan")) == va.VARLEN_ERR_SHAPE
    assert _fwd(va, H=0) == va.VARLEN_ERR_SHAPE
    assert _fwd(va, tq=-1) == va.VARLEN_ERR_SHAPE
    assert _fwd(va, q=_Fake(0x1008, 128, 64)) == va.VARLEN_ERR_ALIGN
    assert _fwd(va, stride=(130, 64)) == va.VARLEN_ERR_STRIDE
    assert _fwd(va, stride=(128, -8)) == va.VARLEN_ERR_STRIDE
    assert _fwd(va, stride=(1 << 40, 64)) == va.VARLEN_ERR_STRIDE
    assert _fwd(va, lse=0) == va.VARLEN_ERR_NULL
    assert _fwd(va, q=_Fake(0, 128, 64)) == va.VARLEN_ERR_NULL


def test_large_strides_pass_validation(va):
    """The strided-dout layout of the "[FA4] cute varlen backward: int32
    overflow" issue (row stride 9728, 410923 rows: offsets past 2^31) is
    accepted; without a GPU the call stops at the device query."""
    st = _fwd(va, tq=410923, tk=410923, H=16, D=96, stride=(9728, 96))
    assert st in (va.VARLEN_ERR_CUDA, va.VARLEN_ERR_ARCH)


def test_int64_offsets_page_value():
    g = json.loads(pathlib.Path(GOLDEN).read_text())["dout_offset_wrap"]
    # the library's offsets are int64 products of row index and row stride
    off = np.int64(g["coord"]) * np.int64(g["dout_stride"][0])
    assert int(off) == g["true_offset"] and int(off) != g["off_signed_i32"]


class _Fake4:
    """A [batch, seqlen, H, D] stand-in: data pointer and element strides."""

    def __init__(self, ptr, batch_stride, row, head):
        self._p, self._s = ptr, (batch_stride, row, head, 1)

    def data_ptr(self):
        return self._p

    def stride(self, i=None):
        return self._s if i is None else self._s[i]

    def dim(self):
        return 4


def test_dense_validation_codes(va):
    """The dense entry points check that each tensor is the packed
    [batch * seqlen, H, D] layout (batch stride = seqlen row strides) and
    that batch * seqlen fits int32, before touching a device."""
    B, Sq, Sk, H, D = 3, 10, 12, 2, 64
    good_q = _Fake4(0x1000, Sq * H * D, H * D, D)
    good_k = _Fake4(0x1000, Sk * H * D, H * D, D)

    class _P:
        def __init__(self, p):
            self._p = p

        def data_ptr(self):
            return self._p

    def fwd(q=good_q, k=good_k, B=B, Sq=Sq, Sk=Sk, causal=0):
        return va.varlen_attn_fwd_dense(q, k, k, B, Sq, Sk, H, D, 0.125, causal, q, _P(0x3000), 0)

    assert fwd(q=_Fake4(0x1000, Sq * H * D + 8, H * D, D)) == va.VARLEN_ERR_STRIDE
    assert fwd(k=_Fake4(0x1000, Sq * H * D, H * D, D)) == va.VARLEN_ERR_STRIDE   # k uses seqlen_k
    assert fwd(B=2 ** 16, Sq=2 ** 16) == va.VARLEN_ERR_SHAPE                        # 2^32 rows
    # the Python wrapper passes bool(causal); a C caller's causal must be 0 or 1
    ds = va.VarlenDenseStride(Sq * H * D, H * D, D)
    dk = va.VarlenDenseStride(Sk * H * D, H * D, D)
    assert va.LIB.varlen_attn_fwd_dense(0x1000, ds, 0x1000, dk, 0x1000, dk, B, Sq, Sk, H, D, 0.125, 2, 0x1000, ds,
                                        0x3000, None) == va.VARLEN_ERR_SHAPE
    assert fwd(B=0) == va.VARLEN_ERR_SHAPE
    # one batch: the batch stride is never used, so it is not checked
    assert fwd(q=_Fake4(0x1000, 7, H * D, D), B=1) in (va.VARLEN_ERR_CUDA, va.VARLEN_ERR_ARCH)
    assert fwd() in (va.VARLEN_ERR_CUDA, va.VARLEN_ERR_ARCH)
    assert va.varlen_attn_bwd_dense_workspace_size(B, Sq, H, D) == va.varlen_attn_bwd_workspace_size(B, B * Sq, H, D)
    assert va.varlen_attn_bwd_dense_workspace_size(2 ** 16, 2 ** 16, H, D) == 0
    # the dense E4M3 forward: the same layout checks, head size 128, its workspace that of the packed call
    q8 = _Fake4(0x1000, Sq * H * 128, H * 128, 128)
    k8 = _Fake4(0x1000, Sk * H * 128, H * 128, 128)
    nb = va.varlen_attn_fwd_fp8_dense_workspace_size(B, Sq, Sk, H, 128)
    assert nb == va.varlen_attn_fwd_fp8_workspace_size(B, B * Sq, B * Sk, H, 128) > 0
    assert va.varlen_attn_fwd_fp8_dense_workspace_size(2 ** 16, 2 ** 16, 1, H, 128) == 0
    assert va.varlen_attn_fwd_fp8_dense_workspace_size(B, Sq, Sk, H, 64) == 0

    def fwd8(q=q8, k=k8, D=128, causal=0, B=B, Sq=Sq, nbytes=nb, ws=0x10000):
        return va.varlen_attn_fwd_fp8_dense(q, k, k, B, Sq, Sk, H, D, 0.125, causal, q, _P(0x3000), _P(ws), nbytes,
                                            0)

    assert fwd8(q=_Fake4(0x1000, Sq * H * 128 + 16, H * 128, 128)) == va.VARLEN_ERR_STRIDE
    assert fwd8(D=64, q=_Fake4(0x1000, Sq * H * 64, H * 64, 64), k=_Fake4(0x1000, Sk * H * 64, H * 64, 64)) \
        == va.VARLEN_ERR_HEAD_DIM
    assert fwd8(B=2 ** 16, Sq=2 ** 16) == va.VARLEN_ERR_SHAPE
    assert fwd8(nbytes=nb - 1) == va.VARLEN_ERR_WORKSPACE
    assert fwd8(ws=0x10010) == va.VARLEN_ERR_WORKSPACE
    for causal in (0, 1):
        assert fwd8(causal=causal) in (va.VARLEN_ERR_CUDA, va.VARLEN_ERR_ARCH)
    assert va.LIB.varlen_attn_fwd_fp8_dense(0x1000, va.VarlenDenseStride(Sq * H * 128, H * 128, 128), 0x1000,
                                            va.VarlenDenseStride(Sk * H * 128, H * 128, 128), 0x1000,
                                            va.VarlenDenseStride(Sk * H * 128, H * 128, 128), B, Sq, Sk, H, 128,
                                            0.125, 2, 0x1000, va.VarlenDenseStride(Sq * H * 128, H * 128, 128),
                                            0x3000, 0x10000, nb, None) == va.VARLEN_ERR_SHAPE


def test_visible_pairs_band_by_brute_force():
    """The pair count the benchmark credits for a mask, against a double loop
    over (query, key) with the band written as two comparisons."""
    w = W.custom("band", [7, 0, 5, 9, 1], [7, 4, 9, 3, 0], 1, 64)
    for causal, window in ((False, (-1, -1)), (True, (-1, -1)), (False, (2, 1)), (False, (0, 0)),
                           (True, (3, 7)), (False, (-1, 2)), (False, (4, -1))):
        left, right = window[0], 0 if causal else window[1]
        n = 0
        for sq, sk in zip(w.seqlens_q(), w.seqlens_k()):
            for i in range(sq):
                for j in range(sk):
                    d = i + sk - sq
                    n += (left < 0 or j >= d - left) and (right < 0 or j <= d + right)
        assert w.visible_pairs(causal, window) == n, (causal, window)


def test_window_and_deterministic_validation_codes(va):
    """The window and deterministic entry points validate like the plain
    ones (any window side is accepted: negative means unbounded) and check
    the workspace before touching a device."""
    H, D, tq = 2, 64, 10
    q = _Fake(0x1000, H * D, D)

    class _P:
        def __init__(self, p):
            self._p = p

        def data_ptr(self):
            return self._p

    cu, lse = _P(0x2000), _P(0x3000)
    for window in ((-1, -1), (0, 0), (5, -1), (-7, 3), (2 ** 31 - 1, 2 ** 31 - 1)):
        st = va.varlen_attn_fwd(q, q, q, cu, cu, 1, tq, tq, H, D, 0, 0, 0.125, q, lse, 0, window=window)
        assert st in (va.VARLEN_ERR_CUDA, va.VARLEN_ERR_ARCH), window
    assert va.varlen_attn_fwd_window(q, q, q, cu, cu, 1, tq, tq, H, D, 0, 0, 0.125, 3, 1, q, lse, 0) in (
        va.VARLEN_ERR_CUDA, va.VARLEN_ERR_ARCH)
    assert va.varlen_attn_fwd_window(q, q, q, cu, cu, 1, tq, tq, 2, 80, 0, 0, 0.125, 3, 1, q, lse, 0) == \
        va.VARLEN_ERR_HEAD_DIM
    assert va.varlen_attn_fwd_window(q, q, q, _P(0), cu, 1, tq, tq, H, D, 0, 0, 0.125, 3, 1, q, lse, 0) == \
        va.VARLEN_ERR_NULL
    need = va.varlen_attn_bwd_workspace_size(1, tq, H, D)
    for det in (False, True):
        def bwd(ws_ptr=0x10000, ws_bytes=need, window=(-1, -1)):
            return va.varlen_attn_bwd(q, q, q, q, q, lse, cu, cu, 1, tq, tq, H, D, 0, 0, 0.125, q, q, q,
                                      _P(ws_ptr), ws_bytes, 0, window=window, deterministic=det)
        assert bwd(ws_bytes=need - 1) == va.VARLEN_ERR_WORKSPACE
        assert bwd(ws_ptr=0x10010) == va.VARLEN_ERR_WORKSPACE   # not 256-byte aligned
        assert bwd(ws_ptr=0) == va.VARLEN_ERR_WORKSPACE
        assert bwd(window=(4, 0)) in (va.VARLEN_ERR_CUDA, va.VARLEN_ERR_ARCH)
        assert bwd() in (va.VARLEN_ERR_CUDA, va.VARLEN_ERR_ARCH)


def test_fp8_workspace_layout_and_validation(va):
    """The E4M3 forward's workspace sections (256-byte aligned, in order, V^T
    rows long enough for every segment's padded start) and its argument
    checks before touching a device."""
    B, tq, tk, H = 3, 1000, 777, 4
    st, off, cols = va.varlen_attn_fwd_fp8_workspace_layout(B, tq, tk, H, 128)
    assert st == va.VARLEN_OK
    r = lambda x: (x + 255) // 256 * 256
    assert cols == 128 * (B + -(-tk // 128) + 1)
    assert off == [0, r(3 * B * H * 4), r(3 * B * H * 4) + r(tq * H * 128),
                   r(3 * B * H * 4) + r(tq * H * 128) + r(tk * H * 128)]
    assert va.varlen_attn_fwd_fp8_workspace_size(B, tq, tk, H, 128) == off[3] + r(H * 128 * cols)
    assert va.varlen_attn_fwd_fp8_workspace_size(B, tq, tk, H, 64) == 0
    assert va.varlen_attn_fwd_fp8_workspace_layout(B, tq, tk, H, 64)[0] == va.VARLEN_ERR_HEAD_DIM
    # every segment's padded V^T block ends inside the rows (the layout's bound)
    cu = [0, 5, 300, 777]
    for b in range(B):
        start = 128 * (b + -(-cu[b] // 128))
        assert start + 128 * -(-(cu[b + 1] - cu[b]) // 128) <= cols

    class _P:
        def __init__(self, p):
            self._p = p

        def data_ptr(self):
            return self._p

    q = _Fake(0x1000, H * 128, 128, H=H, D=128)
    need = va.varlen_attn_fwd_fp8_workspace_size(1, 10, 10, H, 128)
    fwd = lambda D=128, ws=0x10000, nbytes=need: va.varlen_attn_fwd_fp8(
        q, q, q, _P(0x2000), _P(0x2000), 1, 10, 10, H, D, 0, 0, 0.1, q, _P(0x3000), _P(ws), nbytes, 0)
    assert fwd(D=64) == va.VARLEN_ERR_HEAD_DIM
    # V^T columns (128 (batch + ceil(total_k / 128) + 1)) must fit a 32-bit TMA coordinate
    assert va.varlen_attn_fwd_fp8(q, q, q, _P(0x2000), _P(0x2000), 2 ** 24, 10, 2 ** 31 - 1, H, 128, 0, 0, 0.1, q,
                                  _P(0x3000), _P(0x10000), 1 << 62, 0) == va.VARLEN_ERR_SHAPE
    assert fwd(nbytes=need - 1) == va.VARLEN_ERR_WORKSPACE
    assert fwd(ws=0x10010) == va.VARLEN_ERR_WORKSPACE
    assert fwd() in (va.VARLEN_ERR_CUDA, va.VARLEN_ERR_ARCH)
    # the window form: the same checks, then the same device query
    win = lambda D=128, ws=0x10000, nbytes=need, cu=0x2000, band=(-1, 0): va.varlen_attn_fwd_fp8_window(
        q, q, q, _P(cu), _P(0x2000), 1, 10, 10, H, D, 0, 0, 0.1, *band, q, _P(0x3000), _P(ws), nbytes, 0)
    assert win(D=96) == va.VARLEN_ERR_HEAD_DIM
    assert win(cu=0) == va.VARLEN_ERR_NULL
    assert win(nbytes=need - 1) == va.VARLEN_ERR_WORKSPACE
    assert win(ws=0x10008) == va.VARLEN_ERR_WORKSPACE
    for band in ((-1, 0), (4, 0), (0, 0), (-1, -1), (3, 7)):
        assert win(band=band) in (va.VARLEN_ERR_CUDA, va.VARLEN_ERR_ARCH)


def test_prep_roofline_arithmetic():
    """The preprocess roofline in bench.py: 4 D + 12 algorithmic bytes per
    (q row, head), plus 4 D of accumulator zeroing moved on the default path."""
    import bench
    r = bench.prep_roofline(1000, 4, 128, prep_ms=0.5, hbm_gbs=5000.0)
    alg = 1000 * 4 * (4 * 128 + 12)
    assert r["algorithmic_bytes"] == alg and r["moved_bytes"] == alg + 1000 * 4 * 512
    assert abs(r["achieved"] - alg / 0.5e-3 / 1e9) < 1e-9 and abs(r["frac"] - r["achieved"] / 5000.0) < 1e-12
    assert bench.prep_roofline(1000, 4, 128, 0.5, 5000.0, zero_accumulator=False)["moved_bytes"] == alg


def test_bench_helpers():
    """bench.py's CPU-side helpers: the kernel's cpulist syntax and the metric
    name of each timed variant."""
    import argparse
    import bench
    assert bench._parse_cpulist("0-3,8,10-11\n") == {0, 1, 2, 3, 8, 10, 11}
    assert bench._parse_cpulist("5") == {5}
    base = bench.METRIC
    ns = lambda **kw: argparse.Namespace(**{"causal": False, "window": None, **kw})
    assert bench._metric(ns()) == base
    assert bench._metric(ns(causal=True)).startswith("varlen attention TFLOP/s (fwd, bwd) bf16 causal H=56")
    assert "window(128,0)" in bench._metric(ns(window=[128, 0]))
    assert bench._metric(ns(window=[-1, -1])) == base


def test_output_overlap_rejected(va):
    """An output layout whose (row, head) vectors overlap is refused before
    a device is touched; inputs may alias (a zero head stride broadcasts)."""
    H, D = 2, 64
    good = (H * D, D)
    # out with head stride < D: heads overlap
    assert _fwd(va, out=_Fake(0x1000, 128, 32)) == va.VARLEN_ERR_STRIDE
    # out with row stride 0: every row at one address
    assert _fwd(va, out=_Fake(0x1000, 0, 64)) == va.VARLEN_ERR_STRIDE
    # rows inner (head stride = rows * row stride) is a valid layout
    assert _fwd(va, out=_Fake(0x1000, 64, 10 * 64)) in (va.VARLEN_ERR_CUDA, va.VARLEN_ERR_ARCH)
    # ... but not when the head stride is one row short of the rows' extent
    assert _fwd(va, out=_Fake(0x1000, 64, 9 * 64)) == va.VARLEN_ERR_STRIDE
    # an input broadcasting one head (head stride 0) is accepted
    assert _fwd(va, q=_Fake(0x1000, 64, 0)) in (va.VARLEN_ERR_CUDA, va.VARLEN_ERR_ARCH)
    # one row, one head: no overlap possible whatever the strides
    assert _fwd(va, tq=1, H=1, out=_Fake(0x1000, 0, 0), stride=(0, 0)) in (va.VARLEN_ERR_CUDA,
                                                                          va.VARLEN_ERR_ARCH)
    assert _fwd(va, stride=good) in (va.VARLEN_ERR_CUDA, va.VARLEN_ERR_ARCH)


def test_noalloc_scratch_size_matches_header(va):
    """The scratch limit the binding reports comes from the library and
    equals the header's VARLEN_NOALLOC_SCRATCH_BYTES."""
    m = re.search(r"#define\s+VARLEN_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*\*\s*(\d+)u\s*\*\s*(\d+)u\)",
                  pathlib.Path(HEADER).read_text())
    assert m, "VARLEN_NOALLOC_SCRATCH_BYTES not found in the header"
    want = int(m.group(1)) * int(m.group(2)) * int(m.group(3))
    assert va.NOALLOC_SCRATCH_BYTES == want == va.LIB.varlen_attn_bwd_noalloc_scratch_bytes()


def test_noalloc_without_gpu_reports_cuda_error(va):
    """With no usable GPU the allocation-free backward fails like the
    workspace entry point (device check first), and the failing CUDA call
    is reported by varlen_attn_last_cuda_error."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: the non-GPU path is not reachable")
    q = _Fake(0x1000, 128, 64)

    class _P:
        def __init__(self, p):
            self._p = p

        def data_ptr(self):
            return self._p

    st = va.varlen_attn_bwd_noalloc(q, q, q, q, q, _P(0x3000), _P(0x2000), _P(0x2000), 1, 10, 10, 2, 64, 0, 0,
                                    0.125, q, q, q, 0)
    assert st == va.VARLEN_ERR_CUDA
    assert va.varlen_attn_last_cuda_error() != "no error"
    st2, addr, ctx = va.varlen_attn_debug_noalloc_scratch()
    assert st2 == va.VARLEN_ERR_CUDA and addr == 0 and ctx == 0


def test_debug_knobs_validate_without_a_gpu(va):
    """The bounds-checking query and the debug knobs answer on the host: the
    normal build carries no checks, a negative span slack and an unknown
    producer are refused, and every knob can be reset."""
    assert va.varlen_attn_bounds_checked() is False
    assert va.varlen_attn_debug_set_span_slack(-1) == va.VARLEN_ERR_SHAPE
    assert va.varlen_attn_debug_set_span_slack(16) == va.VARLEN_OK
    assert va.varlen_attn_debug_set_span_slack(0) == va.VARLEN_OK
    assert va.varlen_attn_debug_skip_load(2, 1) == va.VARLEN_ERR_SHAPE
    for which in (0, 1):
        assert va.varlen_attn_debug_skip_load(which, 3) == va.VARLEN_OK
        assert va.varlen_attn_debug_skip_load(which, -1) == va.VARLEN_OK


def test_bounds_build_is_separate():
    """The bounds-checking variant builds into its own directory from the
    same sources with -DVARLEN_DEBUG_BOUNDS (compiled here, not loaded)."""
    from packed_variable_length_varlen_gb300 import build
    assert build.BOUNDS_LIB != build.LIB
    assert os.path.dirname(build.BOUNDS_LIB).endswith(os.path.join("_build", "bounds"))


def test_mma_probe_argument_checks():
    """The issue-rate probe rejects its bad arguments before touching a device."""
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    fake = ctypes.c_void_p(16)
    assert va.LIB.varlen_attn_debug_mma_cycles(256, 128, 0, None, None) == va.VARLEN_ERR_NULL
    for n_mma, n_cols, mode in ((0, 128, 0), (6, 128, 0), (1 << 21, 128, 0), (256, 96, 0), (256, 128, 8), (256, 256, 5),
                                (256, 128, -1)):
        assert va.LIB.varlen_attn_debug_mma_cycles(n_mma, n_cols, mode, fake, None) == va.VARLEN_ERR_SHAPE
