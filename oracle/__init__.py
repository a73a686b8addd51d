"""fp64 CPU oracle for packed variable-length multi-head attention.

TEST INFRASTRUCTURE ONLY.  This package is the independent checker for the CUDA
library in ``packed_variable_length_varlen_gb300``: only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import it.  The product path never calls it, and it
imports nothing from the product package.

The arithmetic lives in ``varlen_oracle.c`` (plain fp64 loops, OpenMP over
independent (row, head) pairs); this module compiles it with the host C
compiler, loads it with ctypes and marshals torch CPU tensors (bf16 or fp64,
any row / head stride, unit innermost stride) into it.

What it computes is the packed ``cu_seqlens`` attention of the flash-attention
issue pages ("[FA4] cute varlen backward: int32 overflow in _bwd_preprocess",
sections "Summary" and "Minimal repro"; "[FA4][SM120] flash_attn_varlen_func
... illegal memory access", section "Bug 2 details"):

    O_b = softmax(scale * Q_b K_b^T) V_b  per segment b,
    LSE_i = ln sum_j exp(s_ij)            (natural log; -inf for no keys),

and the gradients dQ, dK, dV of sum(O * dO).  Every function takes explicit
(row, head) pairs so that large problems can be checked on samples.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py`` and,
for the FP8 (E4M3) codec and forward, ``tests/test_oracle_fp8_pins.py``
(torch fp64 SDPA + autograd per segment, closed forms, central finite
differences, gradient invariants, planted-mistake detection).
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "varlen_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIB = None


class _Problem(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p), ("dout", ctypes.c_void_p),
        ("q_rs", ctypes.c_int64), ("q_hs", ctypes.c_int64),
        ("k_rs", ctypes.c_int64), ("k_hs", ctypes.c_int64),
        ("v_rs", ctypes.c_int64), ("v_hs", ctypes.c_int64),
        ("do_rs", ctypes.c_int64), ("do_hs", ctypes.c_int64),
        ("cu_q", ctypes.c_void_p), ("cu_k", ctypes.c_void_p),
        ("batch", ctypes.c_int32), ("num_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("scale", ctypes.c_double),
        ("window_left", ctypes.c_int32), ("window_right", ctypes.c_int32),
    ]


class _Fp8Problem(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("q_rs", ctypes.c_int64), ("q_hs", ctypes.c_int64),
        ("k_rs", ctypes.c_int64), ("k_hs", ctypes.c_int64),
        ("v_rs", ctypes.c_int64), ("v_hs", ctypes.c_int64),
        ("cu_q", ctypes.c_void_p), ("cu_k", ctypes.c_void_p),
        ("batch", ctypes.c_int32), ("num_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("scale", ctypes.c_double),
        ("q_descale", ctypes.c_void_p), ("k_descale", ctypes.c_void_p), ("v_descale", ctypes.c_void_p),
        ("quantize_p", ctypes.c_int32),
        ("window_left", ctypes.c_int32), ("window_right", ctypes.c_int32),
    ]


def library_path(src: str = _SRC, tag: str = "") -> str:
    name = "liboracle%s_%s.so" % (tag, platform.machine())
    return os.path.join(_BUILD_DIR, name)


def build(src: str = _SRC, out: str | None = None, extra_flags=()) -> str:
    """Compile the C oracle into a shared library; returns its path."""
    out = out or library_path(src)
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src) and not extra_flags:
        return out
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC",
           *extra_flags, "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _declare(lib):
    P = ctypes.POINTER(_Problem)
    for name in ("oracle_fwd", "oracle_bwd_q", "oracle_bwd_kv"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        f.argtypes = [P, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                      ctypes.c_void_p, ctypes.c_void_p]
    lib.oracle_bwd_kv_stats.restype = ctypes.c_int
    lib.oracle_bwd_kv_stats.argtypes = [P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_fwd_fp8.restype = ctypes.c_int
    lib.oracle_fwd_fp8.argtypes = [ctypes.POINTER(_Fp8Problem), ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_void_p]
    for name in ("oracle_e4m3_round", "oracle_e4m3_decode", "oracle_e4m3_encode"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    return lib


def load_library(path: str | None = None):
    """Load (building if needed) the oracle library.  ``path`` loads a
    specific build, e.g. a planted-mistake variant compiled by a test."""
    global _LIB
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _LOCK:
        if _LIB is None:
            _LIB = _declare(ctypes.CDLL(build()))
        return _LIB


def num_threads() -> int:
    return int(load_library().oracle_num_threads())


def _view_args(t: torch.Tensor | None, H: int, D: int):
    if t is None:
        return None, 0, 0
    if t.device.type != "cpu":
        raise ValueError("oracle inputs must be CPU tensors")
    if t.dim() != 3 or t.shape[1] != H or t.shape[2] != D or t.stride(2) != 1:
        raise ValueError("oracle inputs must be [rows, H, D] with unit innermost stride")
    return t.data_ptr(), t.stride(0), t.stride(1)


class Problem:
    """One packed-attention problem, held as CPU tensors (no copies)."""

    def __init__(self, q, k, v, cu_q, cu_k, scale, dout=None, causal=False, window=(-1, -1)):
        """``window = (left, right)``: q row ii of a segment sees the keys jj
        with ii + Sk - Sq - left <= jj <= ii + Sk - Sq + right, a negative
        side unbounded; ``causal`` sets right = 0."""
        dt = q.dtype
        if dt not in (torch.bfloat16, torch.float64):
            raise ValueError("oracle supports bf16 or fp64 inputs")
        for t in (k, v, dout):
            if t is not None and t.dtype != dt:
                raise ValueError("all oracle inputs must share one dtype")
        self.H, self.D = int(q.shape[1]), int(q.shape[2])
        self.cu_q = torch.as_tensor(cu_q, dtype=torch.int32).contiguous()
        self.cu_k = torch.as_tensor(cu_k, dtype=torch.int32).contiguous()
        if self.cu_q.numel() != self.cu_k.numel() or self.cu_q.numel() < 1:
            raise ValueError("cu_seqlens_q and cu_seqlens_k need batch+1 entries each")
        self._keep = (q, k, v, dout, self.cu_q, self.cu_k)
        self._t = {"q": q, "k": k, "v": v, "dout": dout}
        self.scale = float(scale)
        self.masked = bool(causal) or int(window[0]) >= 0 or int(window[1]) >= 0
        s = _Problem()
        s.q, s.q_rs, s.q_hs = _view_args(q, self.H, self.D)
        s.k, s.k_rs, s.k_hs = _view_args(k, self.H, self.D)
        s.v, s.v_rs, s.v_hs = _view_args(v, self.H, self.D)
        s.dout, s.do_rs, s.do_hs = _view_args(dout, self.H, self.D)
        s.cu_q, s.cu_k = self.cu_q.data_ptr(), self.cu_k.data_ptr()
        s.batch = self.cu_q.numel() - 1
        s.num_heads, s.head_dim = self.H, self.D
        s.dtype = 0 if dt == torch.bfloat16 else 1
        s.scale = float(scale)
        wl, wr = int(window[0]), int(window[1])
        if causal:
            wr = 0
        s.window_left, s.window_right = (min(max(w, -1), 2**31 - 1) for w in (wl, wr))
        self._s = s
        self.has_dout = dout is not None

    def _pairs(self, rows, heads):
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        heads = np.ascontiguousarray(np.asarray(heads, dtype=np.int32).reshape(-1))
        if rows.shape != heads.shape:
            raise ValueError("rows and heads must pair up")
        if heads.size and (heads.min() < 0 or heads.max() >= self.H):
            raise ValueError("head index out of range")
        return rows, heads

    def _call(self, fn, rows, heads, width_a, width_b):
        rows, heads = self._pairs(rows, heads)
        n = rows.size
        a = np.empty((n, width_a), dtype=np.float64)
        b = np.empty((n, width_b) if width_b > 1 else (n,), dtype=np.float64)
        if n:
            fn(ctypes.byref(self._s), n, rows.ctypes.data, heads.ctypes.data,
               a.ctypes.data, b.ctypes.data)
        return a, b

    def fwd(self, rows, heads, lib=None):
        """O rows [n, D] and LSE [n] for (q row, head) pairs."""
        lib = lib or load_library()
        return self._call(lib.oracle_fwd, rows, heads, self.D, 1)

    def bwd_q(self, rows, heads, lib=None):
        """dQ rows [n, D] and delta [n] for (q row, head) pairs."""
        if not self.has_dout:
            raise ValueError("backward needs dout")
        lib = lib or load_library()
        return self._call(lib.oracle_bwd_q, rows, heads, self.D, 1)

    def bwd_kv(self, rows, heads, lib=None):
        """dK rows [n, D] and dV rows [n, D] for (kv row, head) pairs."""
        if not self.has_dout:
            raise ValueError("backward needs dout")
        lib = lib or load_library()
        return self._call(lib.oracle_bwd_kv, rows, heads, self.D, self.D)


    def segment_stats(self, b: int, h: int, chunk: int = 256):
        """LSE_i and delta_i = dO_i . o_i (fp64) of every q row i of segment b,
        head h (no mask), by the definition: s_ij = scale q_i . k_j over the
        segment's keys, m_i = max_j s_ij, l_i = sum_j exp(s_ij - m_i),
        LSE_i = m_i + ln l_i, o_i = sum_j P_ij v_j with P_ij = exp(s_ij - m_i)
        / l_i (= exp(s_ij - LSE_i)).  The sums over j are fp64 matrix
        products (a library primitive) over chunks of `chunk` q rows; each
        row's result depends on that row alone.  Returns two fp64 arrays of
        Sq_b entries; an empty key set gives LSE = -inf and delta = 0.  This
        is the same quantity oracle_fwd / oracle_bwd_q compute row by row,
        at a cost a long segment (10^5 rows) allows."""
        if self.masked:
            raise ValueError("segment_stats covers the unmasked problem only")
        if not self.has_dout:
            raise ValueError("delta needs dout")
        cu_q, cu_k = self.cu_q.tolist(), self.cu_k.tolist()
        q0, q1, k0, k1 = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        sq, sk = max(q1 - q0, 0), max(k1 - k0, 0)
        lse = np.empty(sq, dtype=np.float64)
        delta = np.empty(sq, dtype=np.float64)
        if sq == 0:
            return lse, delta
        if sk == 0:
            lse[:] = -np.inf
            delta[:] = 0.0
            return lse, delta
        t = self._t
        kt = t["k"][k0:k1, h].to(torch.float64).t().contiguous()   # [D, Sk]
        vv = t["v"][k0:k1, h].to(torch.float64).contiguous()       # [Sk, D]
        c = min(chunk, sq)
        s = torch.empty(c, sk, dtype=torch.float64)
        o = torch.empty(c, self.D, dtype=torch.float64)
        for i0 in range(0, sq, c):
            n = min(c, sq - i0)
            qc = t["q"][q0 + i0:q0 + i0 + n, h].to(torch.float64)
            sc, oc = s[:n], o[:n]
            torch.matmul(qc, kt, out=sc)
            sc.mul_(self.scale)
            m = sc.max(dim=1, keepdim=True).values
            sc.sub_(m).exp_()
            l = sc.sum(dim=1, keepdim=True)
            lse[i0:i0 + n] = (m + torch.log(l)).reshape(-1).numpy()
            sc.div_(l)
            torch.matmul(sc, vv, out=oc)
            g = t["dout"][q0 + i0:q0 + i0 + n, h].to(torch.float64)
            delta[i0:i0 + n] = (g * oc).sum(dim=1).numpy()
        return lse, delta

    def rows_block(self, b: int, h: int, rows, chunk: int = 128):
        """Forward and query-side backward of the q rows ``rows`` (packed
        indices, all in segment b) of head h, no mask, by the definition:
        s_ij = scale q_i . k_j over the segment's keys, m_i = max_j s_ij,
        LSE_i = m_i + ln sum_j exp(s_ij - m_i), P_ij = exp(s_ij - LSE_i),
        o_i = sum_j P_ij v_j, delta_i = dO_i . o_i, dS_ij = P_ij (dO_i . v_j -
        delta_i), dq_i = scale sum_j dS_ij k_j.  The sums over j are fp64
        matrix products (a library primitive) over chunks of rows; each
        row's result depends on that row alone.  Returns o [n, D], lse [n],
        dq [n, D] and delta [n] (dq and delta None without dout).  An empty
        key set gives o = 0, LSE = -inf, dq = 0, delta = 0.  The same
        quantities as fwd / bwd_q, at a cost long segments allow."""
        if self.masked:
            raise ValueError("rows_block covers the unmasked problem only")
        cu_q, cu_k = self.cu_q.tolist(), self.cu_k.tolist()
        rows = np.asarray(rows, dtype=np.int64).reshape(-1)
        q0, q1, k0, k1 = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        if rows.size and (rows.min() < q0 or rows.max() >= q1):
            raise ValueError("rows outside segment %d" % b)
        n, D, sk = rows.size, self.D, max(k1 - k0, 0)
        o = np.zeros((n, D), dtype=np.float64)
        lse = np.full(n, -np.inf, dtype=np.float64)
        dq = np.zeros((n, D), dtype=np.float64) if self.has_dout else None
        delta = np.zeros(n, dtype=np.float64) if self.has_dout else None
        if n == 0 or sk == 0:
            return o, lse, dq, delta
        t = self._t
        kk = t["k"][k0:k1, h].to(torch.float64).contiguous()   # [Sk, D]
        vv = t["v"][k0:k1, h].to(torch.float64).contiguous()   # [Sk, D]
        kt, vt = kk.t().contiguous(), vv.t().contiguous()      # [D, Sk]
        ridx = torch.from_numpy(rows)
        for i0 in range(0, n, chunk):
            r = ridx[i0:i0 + chunk]
            qc = t["q"][r, h].to(torch.float64)
            sc = torch.matmul(qc, kt).mul_(self.scale)
            m = sc.max(dim=1, keepdim=True).values
            l = torch.exp(sc - m).sum(dim=1, keepdim=True)
            lc = m + torch.log(l)
            p = torch.exp(sc.sub_(lc))                           # P = exp(s - LSE)
            oc = torch.matmul(p, vv)
            o[i0:i0 + r.numel()] = oc.numpy()
            lse[i0:i0 + r.numel()] = lc.reshape(-1).numpy()
            if self.has_dout:
                g = t["dout"][r, h].to(torch.float64)
                dl = (g * oc).sum(dim=1, keepdim=True)
                ds = torch.matmul(g, vt).sub_(dl).mul_(p)       # P (dP - delta)
                dq[i0:i0 + r.numel()] = (torch.matmul(ds, kk) * self.scale).numpy()
                delta[i0:i0 + r.numel()] = dl.reshape(-1).numpy()
        return o, lse, dq, delta

    def bwd_kv_block(self, b: int, h: int, rows, stats=None, lib=None):
        """dK rows [n, D] and dV rows [n, D] for kv rows of segment b, head h,
        with the per-q-row LSE and delta of that segment taken from
        ``stats`` (default: ``segment_stats(b, h)``); the sums over q rows are
        those of bwd_kv (oracle_bwd_kv_stats)."""
        if not self.has_dout:
            raise ValueError("backward needs dout")
        lib = lib or load_library()
        lse, delta = stats if stats is not None else self.segment_stats(b, h)
        lse = np.ascontiguousarray(lse, dtype=np.float64)
        delta = np.ascontiguousarray(delta, dtype=np.float64)
        sq = int(self.cu_q[b + 1]) - int(self.cu_q[b])
        if lse.size != max(sq, 0) or delta.size != max(sq, 0):
            raise ValueError("stats need one entry per q row of the segment")
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        n = rows.size
        dk = np.empty((n, self.D), dtype=np.float64)
        dv = np.empty((n, self.D), dtype=np.float64)
        if n:
            st = lib.oracle_bwd_kv_stats(ctypes.byref(self._s), int(b), int(h), n, rows.ctypes.data,
                                         lse.ctypes.data, delta.ctypes.data, dk.ctypes.data, dv.ctypes.data)
            if st != 0:
                raise ValueError("segment or head out of range")
        return dk, dv


def all_pairs(total_rows: int, num_heads: int):
    """Every (row, head) pair of a [total_rows, num_heads, D] tensor."""
    rows = np.repeat(np.arange(total_rows, dtype=np.int64), num_heads)
    heads = np.tile(np.arange(num_heads, dtype=np.int32), total_rows)
    return rows, heads


# ---------------------------------------------------------------- FP8 (E4M3)

def e4m3_round(x, lib=None) -> np.ndarray:
    """Nearest OCP FP8 E4M3 value of each element (ties to even, saturating at
    +-448), as fp64."""
    lib = lib or load_library()
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty_like(a)
    lib.oracle_e4m3_round(a.size, a.ctypes.data, out.ctypes.data)
    return out


def e4m3_decode(codes, lib=None) -> np.ndarray:
    """Values of E4M3 codes (uint8), as fp64."""
    lib = lib or load_library()
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(c.shape, dtype=np.float64)
    lib.oracle_e4m3_decode(c.size, c.ctypes.data, out.ctypes.data)
    return out


def e4m3_encode(x, lib=None) -> np.ndarray:
    """E4M3 codes (uint8) of the values nearest to x."""
    lib = lib or load_library()
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(a.shape, dtype=np.uint8)
    lib.oracle_e4m3_encode(a.size, a.ctypes.data, out.ctypes.data)
    return out


def quantize_e4m3(x: torch.Tensor, cu_seqlens, lib=None):
    """Per-(segment, head) E4M3 quantisation of a [rows, H, D] tensor, in fp32
    arithmetic (the precision that decides each code): the descale of (b, h)
    is fp32(amax) / 448 over the segment's rows of head h (1 for an all-zero
    block), the code of x is e4m3(fp32(x) / descale) with an IEEE fp32
    division.  Returns the codes as a uint8 [rows, H, D] tensor and the
    descales [batch * H] (fp32 values held in fp64)."""
    xs = x.float().numpy()
    cu = [int(c) for c in cu_seqlens]
    B, H = len(cu) - 1, xs.shape[1]
    desc = np.ones(B * H, dtype=np.float32)
    scaled = np.zeros(xs.shape, dtype=np.float32)
    for b in range(B):
        blk = xs[cu[b]:cu[b + 1]]
        for h in range(H):
            amax = np.float32(np.abs(blk[:, h]).max()) if blk.shape[0] else np.float32(0)
            if amax > 0:
                desc[b * H + h] = amax / np.float32(448.0)
            scaled[cu[b]:cu[b + 1], h] = blk[:, h] / desc[b * H + h]
    return torch.from_numpy(e4m3_encode(scaled.astype(np.float64), lib)), desc.astype(np.float64)


class Fp8Problem:
    """One FP8 (E4M3) forward problem: codes as uint8 [rows, H, D] CPU tensors
    (unit innermost stride) and fp64 descales [batch * H] per tensor."""

    def __init__(self, q8, k8, v8, cu_q, cu_k, scale, q_descale, k_descale, v_descale, quantize_p=True,
                 causal=False, window=(-1, -1)):
        """``causal`` and ``window = (left, right)`` as in ``Problem``."""
        for t in (q8, k8, v8):
            if t.dtype != torch.uint8 or t.dim() != 3 or t.stride(2) != 1:
                raise ValueError("FP8 operands are uint8 [rows, H, D] tensors with unit innermost stride")
        self.H, self.D = int(q8.shape[1]), int(q8.shape[2])
        self.cu_q = torch.as_tensor(cu_q, dtype=torch.int32).contiguous()
        self.cu_k = torch.as_tensor(cu_k, dtype=torch.int32).contiguous()
        B = self.cu_q.numel() - 1
        self.desc = [np.ascontiguousarray(np.asarray(d, dtype=np.float64).reshape(-1)) for d in
                     (q_descale, k_descale, v_descale)]
        if any(d.size != B * self.H for d in self.desc):
            raise ValueError("descales need batch * num_heads entries")
        self._keep = (q8, k8, v8, self.cu_q, self.cu_k, self.desc)
        s = _Fp8Problem()
        s.q, s.k, s.v = q8.data_ptr(), k8.data_ptr(), v8.data_ptr()
        s.q_rs, s.q_hs = q8.stride(0), q8.stride(1)
        s.k_rs, s.k_hs = k8.stride(0), k8.stride(1)
        s.v_rs, s.v_hs = v8.stride(0), v8.stride(1)
        s.cu_q, s.cu_k = self.cu_q.data_ptr(), self.cu_k.data_ptr()
        s.batch, s.num_heads, s.head_dim = B, self.H, self.D
        s.scale = float(scale)
        s.q_descale, s.k_descale, s.v_descale = (d.ctypes.data for d in self.desc)
        s.quantize_p = 1 if quantize_p else 0
        wl, wr = int(window[0]), int(window[1])
        if causal:
            wr = 0
        s.window_left, s.window_right = (min(max(w, -1), 2**31 - 1) for w in (wl, wr))
        self._s = s

    def fwd(self, rows, heads, lib=None):
        """O rows [n, D] and LSE [n] for (q row, head) pairs."""
        lib = lib or load_library()
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        heads = np.ascontiguousarray(np.asarray(heads, dtype=np.int32).reshape(-1))
        n = rows.size
        o = np.empty((n, self.D), dtype=np.float64)
        l = np.empty(n, dtype=np.float64)
        if n:
            lib.oracle_fwd_fp8(ctypes.byref(self._s), n, rows.ctypes.data, heads.ctypes.data, o.ctypes.data,
                               l.ctypes.data)
        return o, l

