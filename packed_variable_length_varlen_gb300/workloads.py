"""Seeded synthetic workloads for packed variable-length attention.

This module holds no attention arithmetic: it only decides segment lengths,
tensor layouts (row strides, padding, strided views) and draws random inputs.
Both the CUDA path's tests / benchmark and the CPU oracle consume what it
makes, so the two sides see bit-identical inputs.

The shapes follow the workloads on the pages:

* ``tiny``      -- 2 segments cu=[0,37,100], H=2, D=64, inputs N(0,1)*0.5.
* ``windowed``  -- the packed windowed video-DiT call captured on the
  flash-attention issue "[FA4][SM120] flash_attn_varlen_func ... >=4 varlen
  segments" (section "Bug 2 details"): cu_seqlens_q=[0,4032,...,35280],
  17580 kv rows per window, H=56, D=128.
* ``long``      -- one dense 77000-token segment, H=56, D=128, the length of
  the minimal reproduction on the ffpa-attn pull request "NVFP4 ... int32
  extents" (section "Minimal reproduction").
* ``strided_dout`` -- cu=[0,225304,410923], H=16, D=96, inputs *0.1, dout a
  [410923,16,96] view with row stride 9728 into a wider buffer, as in the
  "[FA4] cute varlen backward: int32 overflow in _bwd_preprocess" issue
  (sections "Root cause", "Real-world trigger").
* ``ragged``    -- 64 segments with lengths drawn uniformly in [0, 8192] and
  forced 0 / 1 / 127 / 129 / 8191 / 8192 / trailing-empty entries, H=32,
  D=128, inputs *2, every row padded by 64 elements.

Inputs are drawn from ``torch.Generator('cpu')`` seeded with ``seed`` in the
order q, k, v, dout (after the segment lengths where those are random), as
float32 N(0,1) times the workload's amplitude, then rounded to bf16.  Padding
elements of padded / strided layouts hold NaN so that a stray read shows.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

TILE_ROWS = 128  # rows of one q or kv tile in the CUDA kernels' tile grid


@dataclass(frozen=True)
class Workload:
    name: str
    cu_q: tuple
    cu_k: tuple
    num_heads: int
    head_dim: int
    amplitude: float = 1.0
    dout_amplitude: float = 1.0
    row_pad: int = 0                 # extra elements after H*D in every row
    dout_row_stride: int | None = None  # dout as a view into a wider buffer
    max_seqlen_q: int | None = None  # None: the true maximum
    max_seqlen_k: int | None = None
    backward: bool = True
    lengths_from_seed: bool = False  # lengths were drawn from the generator
    scale: float | None = None       # None: 1/sqrt(head_dim)

    @property
    def batch(self) -> int:
        return len(self.cu_q) - 1

    @property
    def total_q(self) -> int:
        return int(self.cu_q[-1])

    @property
    def total_k(self) -> int:
        return int(self.cu_k[-1])

    @property
    def softmax_scale(self) -> float:
        # float32 value, as the C-ABI takes it
        s = self.scale if self.scale is not None else 1.0 / math.sqrt(self.head_dim)
        return float(np.float32(s))

    @property
    def row_stride(self) -> int:
        return self.num_heads * self.head_dim + self.row_pad

    def seqlens_q(self):
        return [self.cu_q[b + 1] - self.cu_q[b] for b in range(self.batch)]

    def seqlens_k(self):
        return [self.cu_k[b + 1] - self.cu_k[b] for b in range(self.batch)]

    def max_q(self) -> int:
        return self.max_seqlen_q if self.max_seqlen_q is not None else max(self.seqlens_q() + [0])

    def max_k(self) -> int:
        return self.max_seqlen_k if self.max_seqlen_k is not None else max(self.seqlens_k() + [0])

    def pair_products(self) -> int:
        """sum_b Sq_b * Sk_b (per head)."""
        return sum(a * b for a, b in zip(self.seqlens_q(), self.seqlens_k()))

    def visible_pairs(self, causal: bool = False, window=(-1, -1)) -> int:
        """(query, key) pairs that take part, per head: sum_b Sq_b * Sk_b, or
        with a mask the sum over rows of row_keys (the keys in each row's
        band)."""
        if not causal and window[0] < 0 and window[1] < 0:
            return self.pair_products()
        tot = 0
        for sq, sk in zip(self.seqlens_q(), self.seqlens_k()):
            if sq > 0 and sk > 0:
                tot += int(row_keys(np.arange(sq, dtype=np.int64), sq, sk, causal, window).sum())
        return tot

    def fwd_flops(self, causal: bool = False, window=(-1, -1)) -> float:
        """4 * (visible pairs) * H * D: two matmuls of 2 flops per MAC."""
        return 4.0 * self.visible_pairs(causal, window) * self.num_heads * self.head_dim

    def bwd_flops(self, causal: bool = False, window=(-1, -1)) -> float:
        """2.5 x the forward count (five matmuls instead of two)."""
        return 2.5 * self.fwd_flops(causal, window)

    def q_tiles(self, tile: int = TILE_ROWS) -> int:
        """Exact tile count H * sum_b ceil(Sq_b / tile)."""
        return self.num_heads * sum(-(-max(0, s) // tile) for s in self.seqlens_q())

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


def row_keys(ii, sq, sk, causal: bool = False, window=(-1, -1)):
    """Number of keys q rows `ii` (0-based within a segment of sq rows and sk
    keys) see: row i sees the keys j with i + sk - sq - left <= j <=
    i + sk - sq + right, a negative side unbounded, causal setting right = 0
    (all sk without a mask).  Array arguments broadcast."""
    left, right = int(window[0]), int(window[1])
    if causal:
        right = 0
    ii = np.asarray(ii, dtype=np.int64)
    sq, sk = np.asarray(sq, dtype=np.int64), np.asarray(sk, dtype=np.int64)
    diag = ii + (sk - sq)
    lo = np.clip(diag - left, 0, sk) if left >= 0 else np.zeros_like(diag)
    hi = np.clip(diag + right + 1, 0, sk) if right >= 0 else np.broadcast_to(sk, diag.shape)
    return np.maximum(hi - lo, 0)


def _cu(lengths):
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return tuple(cu)


def _ragged_lengths(g: torch.Generator, n: int = 64, hi: int = 8192):
    lens = torch.randint(0, hi + 1, (n,), generator=g).tolist()
    forced = {0: 0, 1: 1, 2: 127, 3: 129, 4: 8191, 5: 8192, n - 2: 0, n - 1: 0}
    for i, v in forced.items():
        lens[i] = v
    return lens


def tiny() -> Workload:
    return Workload("tiny", (0, 37, 100), (0, 37, 100), 2, 64,
                    amplitude=0.5, dout_amplitude=0.5)


def windowed() -> Workload:
    cu_q = (0, 4032, 9072, 14112, 19152, 24292, 29232, 34272, 35280)
    cu_k = tuple(17580 * i for i in range(9))
    return Workload("windowed", cu_q, cu_k, 56, 128, max_seqlen_q=5140, max_seqlen_k=17580)


def long_dense() -> Workload:
    return Workload("long", (0, 77000), (0, 77000), 56, 128)


def strided_dout() -> Workload:
    cu = (0, 225304, 410923)
    return Workload("strided_dout", cu, cu, 16, 96, amplitude=0.1, dout_amplitude=0.1,
                    dout_row_stride=9728)


def ragged(seed: int = 0) -> Workload:
    g = torch.Generator().manual_seed(seed)
    cu = _cu(_ragged_lengths(g))
    return Workload("ragged", cu, cu, 32, 128, amplitude=2.0, dout_amplitude=2.0,
                    row_pad=64, lengths_from_seed=True)


def dense_batched() -> Workload:
    """Uniform segments for the dense batched entry points: 8 x (4096 q, 16384
    kv), H=56, D=128 -- the windowed workload's size class with equal lengths."""
    return Workload("dense", _cu([4096] * 8), _cu([16384] * 8), 56, 128)


WORKLOADS = {
    "tiny": tiny,
    "dense": dense_batched,
    "windowed": windowed,
    "long": long_dense,
    "strided_dout": strided_dout,
    "ragged": ragged,
}


def get(name: str) -> Workload:
    return WORKLOADS[name]()


def custom(name, seqlens_q, seqlens_k, num_heads, head_dim, **kw) -> Workload:
    """A workload from explicit per-segment lengths (tests' small cases)."""
    return Workload(name, _cu(seqlens_q), _cu(seqlens_k), num_heads, head_dim, **kw)


# --------------------------------------------------------------------------
# tensors

def _layout(total: int, H: int, D: int, row_stride: int, fill: float,
            dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """A [total, H, D] view with the given row stride into a NaN-padded (or
    ``fill``-padded) buffer; contiguous when row_stride == H*D."""
    if row_stride == H * D:
        return torch.empty(total, H, D, dtype=dtype, device=device)
    buf = torch.full((max(total, 1), row_stride), fill, dtype=dtype, device=device)
    return buf[:total, :H * D].unflatten(1, (H, D))


@dataclass
class Inputs:
    workload: Workload
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    dout: torch.Tensor | None
    cu_q: torch.Tensor
    cu_k: torch.Tensor
    extra: dict = field(default_factory=dict)

    def to(self, device) -> "Inputs":
        """Copy to ``device`` keeping every stride and the padding bytes."""
        def mv(t):
            if t is None:
                return None
            if t._base is None:
                return t.to(device)
            base = t._base  # a contiguous padded buffer with storage offset 0
            return base.to(device).as_strided(t.shape, t.stride(), t.storage_offset())
        return Inputs(self.workload, mv(self.q), mv(self.k), mv(self.v), mv(self.dout),
                      self.cu_q.to(device), self.cu_k.to(device), dict(self.extra))


def make_inputs(w: Workload, seed: int = 0, with_dout: bool | None = None) -> Inputs:
    """Draw the workload's inputs on the CPU (see the module docstring)."""
    g = torch.Generator().manual_seed(seed)
    if w.lengths_from_seed:
        _ragged_lengths(g)  # advance the generator exactly as the lengths did
    H, D = w.num_heads, w.head_dim
    rs = w.row_stride

    def draw(total, amp, row_stride):
        t = _layout(total, H, D, row_stride, float("nan"))
        x = torch.randn(total, H, D, generator=g, dtype=torch.float32)
        x.mul_(amp)
        t.copy_(x)
        return t

    q = draw(w.total_q, w.amplitude, rs)
    k = draw(w.total_k, w.amplitude, rs)
    v = draw(w.total_k, w.amplitude, rs)
    need_dout = w.backward if with_dout is None else with_dout
    dout = None
    if need_dout:
        drs = w.dout_row_stride if w.dout_row_stride is not None else rs
        dout = draw(w.total_q, w.dout_amplitude, drs)
    cu_q = torch.tensor(w.cu_q, dtype=torch.int32)
    cu_k = torch.tensor(w.cu_k, dtype=torch.int32)
    return Inputs(w, q, k, v, dout, cu_q, cu_k)


def output_like(w: Workload, which: str, device, canary: float = 12345.0) -> torch.Tensor:
    """Output buffer for ``which`` in {'out','dq','dk','dv'} with the
    workload's row stride; padding holds ``canary`` so tests can check that
    it is left untouched."""
    total = w.total_q if which in ("out", "dq") else w.total_k
    return _layout(total, w.num_heads, w.head_dim, w.row_stride, canary, device=device)


# --------------------------------------------------------------------------
# row sampling for checks on large workloads

def offset_crossing_row(row_stride_elems: int, elem_bytes: int, limit: int = 2 ** 31) -> int:
    """First row whose starting offset (row * stride, in elements times
    elem_bytes) reaches ``limit``."""
    per_row = row_stride_elems * elem_bytes
    return -(-limit // per_row)


def sample_rows(cu, n_target: int = 4096, seed: int = 1, extra_rows=()) -> np.ndarray:
    """Rows spanning every segment: per segment the first two and last two
    rows and rows at tile multiples +-1 (subsampled), the ``extra_rows``
    (e.g. where an offset first crosses 2^31), then uniform random rows from
    ``seed`` up to ``n_target``, all within [cu[0], cu[-1]) (a slice of
    cu_seqlens, e.g. one segment's bounds, samples that slice only).  Sorted
    and unique."""
    cu = [int(c) for c in cu]
    first, total = cu[0], cu[-1]
    rng = np.random.default_rng(seed)
    picked = set()
    for b in range(len(cu) - 1):
        a, e = cu[b], cu[b + 1]
        if e <= a:
            continue
        for r in (a, a + 1, e - 2, e - 1):
            if a <= r < e:
                picked.add(r)
        mult = list(range(a + TILE_ROWS, e, TILE_ROWS))
        if len(mult) > 16:
            mult = list(rng.choice(mult, 16, replace=False))
        for m in mult:
            for r in (m - 1, m, m + 1):
                if a <= r < e:
                    picked.add(int(r))
    for r in extra_rows:
        if first <= r < total:
            picked.add(int(r))
            if r + 1 < total:
                picked.add(int(r) + 1)
    if total > first:
        while len(picked) < min(n_target, total - first):
            picked.update(int(x) for x in rng.integers(first, total, size=n_target - len(picked)))
    return np.array(sorted(picked), dtype=np.int64)


def sample_pairs(rows: np.ndarray, num_heads: int, heads_per_row: int, seed: int = 2,
                 all_heads_rows=()):
    """(row, head) pairs: ``heads_per_row`` random heads for each row, all
    heads for the rows in ``all_heads_rows``."""
    rng = np.random.default_rng(seed)
    full = set(int(r) for r in all_heads_rows)
    R, Hs = [], []
    for r in rows:
        r = int(r)
        if r in full or heads_per_row >= num_heads:
            hs = range(num_heads)
        else:
            hs = sorted(rng.choice(num_heads, heads_per_row, replace=False).tolist())
        for h in hs:
            R.append(r)
            Hs.append(int(h))
    return np.array(R, dtype=np.int64), np.array(Hs, dtype=np.int32)
