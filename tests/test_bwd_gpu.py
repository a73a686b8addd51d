"""GPU parity of the backward (preprocess + dQ/dK/dV kernels + dQ conversion)
against the fp64 oracle, through the C ABI.  The GPU backward consumes the
GPU forward's O and LSE, as a training step would; the oracle computes every
quantity from the inputs in fp64.  Tolerance: relative Frobenius error
<= 1e-2 per tensor over the compared (row, head) pairs, exact zeros where
the oracle is exactly zero (empty segments).

Full-size workloads compare dQ on sampled rows (the oracle computes each q
row alone) and check dK / dV through the exact invariants
sum_j dk_j = 0 and sum_j dv_j = sum_i dO_i per (segment, head), which hold at
any size; dK / dV rows are compared directly on same-shaped smaller cases and
on sampled (segment, head) blocks of the full windowed workload."""
import numpy as np
import pytest
import torch

import oracle
from packed_variable_length_varlen_gb300 import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run_gpu(w: W.Workload, cpu: W.Inputs, canary=12345.0):
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    dev = cpu.to(DEV)
    H, D = w.num_heads, w.head_dim
    out = W.output_like(w, "out", DEV, canary=canary)
    lse = torch.empty(H, w.total_q, dtype=torch.float32, device=DEV)
    P.run_fwd(dev, out, lse)
    dq = W.output_like(w, "dq", DEV, canary=canary)
    dk = W.output_like(w, "dk", DEV, canary=canary)
    dv = W.output_like(w, "dv", DEV, canary=canary)
    nbytes = va.varlen_attn_bwd_workspace_size(w.batch, w.total_q, H, D)
    wsp = torch.full((max(nbytes, 1),), 0x7F, dtype=torch.uint8, device=DEV)  # garbage on entry
    st = va.varlen_attn_bwd(dev.q, dev.k, dev.v, out, dev.dout, lse, dev.cu_q, dev.cu_k, w.batch, w.total_q,
                            w.total_k, H, D, w.max_q(), w.max_k(), w.softmax_scale, dq, dk, dv, wsp, nbytes)
    assert st == 0, va.varlen_attn_status_string(st)
    st = va.varlen_attn_get_device_status()
    assert st == 0, va.varlen_attn_status_string(st)
    for t in (dq, dk, dv):
        assert P.padding_untouched(t, w, canary)
    return out, lse, dq, dk, dv


def _compare(w, cpu, dq, dk, dv, qpairs=None, kpairs=None, tag="", kblock=None, rows_path=False):
    """Relative Frobenius error of dQ over the q pairs and of dK, dV over the
    kv pairs (all pairs by default).  ``kblock = (b, h, rows)`` compares the
    kv rows `rows` of one long (segment, head) block instead, with the
    oracle's per-segment statistics path (LSE and delta of every q row of
    the segment computed once).  ``rows_path`` computes the sampled dQ rows
    with the oracle's matrix-product path (long unmasked segments)."""
    pb = P.oracle_problem(cpu)
    rows, heads = qpairs if qpairs is not None else oracle.all_pairs(w.total_q, w.num_heads)
    if kblock is not None:
        krows, kheads = (np.zeros(0, np.int64), np.zeros(0, np.int32))
    else:
        krows, kheads = kpairs if kpairs is not None else oracle.all_pairs(w.total_k, w.num_heads)
    res = {}
    if rows.size:
        dq_ref = P.oracle_rows(pb, w, rows, heads)[2] if rows_path else pb.bwd_q(rows, heads)[0]
        res["dq"] = P.rel_fro(P.gather(dq.cpu(), rows, heads), dq_ref)
        res["dq_rows"] = int(np.unique(rows).size)
    if krows.size:
        dk_ref, dv_ref = pb.bwd_kv(krows, kheads)
        res["dk"] = P.rel_fro(P.gather(dk.cpu(), krows, kheads), dk_ref)
        res["dv"] = P.rel_fro(P.gather(dv.cpu(), krows, kheads), dv_ref)
        res["kv_rows"] = int(np.unique(krows).size)
    if kblock is not None:
        b, h, brows = kblock
        brows = np.asarray(brows, dtype=np.int64)
        dk_ref, dv_ref = pb.bwd_kv_block(b, h, brows)
        hh = np.full(brows.size, h, np.int32)
        res["dk"] = P.rel_fro(P.gather(dk.cpu(), brows, hh), dk_ref)
        res["dv"] = P.rel_fro(P.gather(dv.cpu(), brows, hh), dv_ref)
        res["kv_block"] = (int(b), int(h), int(brows.size))
    print(w.name, tag, res)
    for k_ in ("dq", "dk", "dv"):
        if k_ in res:
            assert res[k_] <= P.GRAD_REL_FRO, (k_, res)
    return res


def _invariants(w, cpu, dk, dv, tol=1e-2):
    """sum_j dk_j = 0 and sum_j dv_j = sum_i dO_i per (segment, head), exact
    in exact arithmetic.  The residual is compared, per (segment, head, d),
    with tol times the size of the terms summed, plus a noise floor of
    sqrt(Sk) times the tensor's rms (a one-key segment has dk = 0 exactly,
    so its terms are pure rounding noise)."""
    dkc, dvc = dk.cpu().double(), dv.cpu().double()
    doc = cpu.dout.double()
    rms_k = float(dkc.pow(2).mean().sqrt()) + 1e-30
    rms_v = float(dvc.pow(2).mean().sqrt()) + 1e-30
    worst = 0.0
    for b in range(w.batch):
        k0, k1 = w.cu_k[b], w.cu_k[b + 1]
        q0, q1 = w.cu_q[b], w.cu_q[b + 1]
        if k1 <= k0:
            continue
        if q1 <= q0:
            assert torch.all(dkc[k0:k1] == 0) and torch.all(dvc[k0:k1] == 0)
            continue
        floor = (k1 - k0) ** 0.5
        sk = dkc[k0:k1].sum(0)
        ak = dkc[k0:k1].abs().sum(0) + floor * rms_k
        sv = dvc[k0:k1].sum(0) - doc[q0:q1].sum(0)
        av = dvc[k0:k1].abs().sum(0) + doc[q0:q1].abs().sum(0) + floor * rms_v
        worst = max(worst, float((sk.abs() / ak).max()), float((sv.abs() / av).max()))
    print(w.name, "invariants worst", worst)
    assert worst <= tol


def test_bwd_tiny():
    w = W.tiny()
    cpu = W.make_inputs(w, 0)
    _, _, dq, dk, dv = _run_gpu(w, cpu)
    _compare(w, cpu, dq, dk, dv)


@pytest.mark.parametrize("D", [64, 96, 128])
def test_bwd_ragged_small(D):
    w = W.custom("bwd_ragged_d%d" % D, [0, 1, 127, 128, 129, 300, 0, 517, 3, 65],
                 [5, 0, 200, 128, 1, 700, 40, 517, 1000, 64], 2, D)
    cpu = W.make_inputs(w, 0)
    _, _, dq, dk, dv = _run_gpu(w, cpu)
    _compare(w, cpu, dq, dk, dv)
    _invariants(w, cpu, dk, dv)


def test_bwd_strided_dout_small():
    """The strided-dout layout at reduced size: dout is a view with row
    stride 9728 into a NaN-filled buffer; outputs are padded with canaries."""
    w = W.custom("strided_small", [2253, 1856], [2253, 1856], 16, 96, amplitude=0.1, dout_amplitude=0.1,
                 dout_row_stride=9728)
    cpu = W.make_inputs(w, 0)
    _, _, dq, dk, dv = _run_gpu(w, cpu)
    rows = W.sample_rows(w.cu_q, 600, seed=1)
    qp = W.sample_pairs(rows, 16, 4, seed=2)
    krows = W.sample_rows(w.cu_k, 300, seed=3)
    kp = W.sample_pairs(krows, 16, 1, seed=4)
    _compare(w, cpu, dq, dk, dv, qp, kp)
    _invariants(w, cpu, dk, dv)


def test_bwd_padded_and_isolation():
    w = W.custom("bwd_pad", [130, 70, 5, 200], [129, 61, 40, 0], 2, 128, row_pad=64, amplitude=2.0,
                 dout_amplitude=2.0)
    cpu = W.make_inputs(w, 0)
    # plant NaN in segment 1 (q, k, v, dout rows); the others must stay exact
    cpu.q[w.cu_q[1]:w.cu_q[2]] = float("nan")
    cpu.k[w.cu_k[1]:w.cu_k[2]] = float("nan")
    cpu.v[w.cu_k[1]:w.cu_k[2]] = float("nan")
    cpu.dout[w.cu_q[1]:w.cu_q[2]] = float("nan")
    _, _, dq, dk, dv = _run_gpu(w, cpu)
    qrows = np.array([r for r in range(w.total_q) if not (w.cu_q[1] <= r < w.cu_q[2])], dtype=np.int64)
    krows = np.array([r for r in range(w.total_k) if not (w.cu_k[1] <= r < w.cu_k[2])], dtype=np.int64)
    qp = (np.repeat(qrows, 2), np.tile(np.arange(2, dtype=np.int32), qrows.size))
    kp = (np.repeat(krows, 2), np.tile(np.arange(2, dtype=np.int32), krows.size))
    _compare(w, cpu, dq, dk, dv, qp, kp)
    # segment 3 has no keys: dQ = 0 exactly
    assert torch.all(dq[w.cu_q[3]:w.cu_q[4]] == 0)


def test_bwd_deterministic_dk_dv():
    w = W.custom("bwd_det", [300, 64], [257, 64], 2, 128)
    cpu = W.make_inputs(w, 0)
    a = _run_gpu(w, cpu)
    b = _run_gpu(w, cpu)
    assert torch.equal(a[3], b[3]) and torch.equal(a[4], b[4])  # dK, dV: no atomics
    assert (a[2].float() - b[2].float()).abs().max().item() < 1e-2  # dQ: atomic order may differ


# ---------------------------------------------------------------- full size

def _qpairs(w, n=4096, hpr=1, extra=()):
    rows = W.sample_rows(w.cu_q, n, seed=1, extra_rows=extra)
    return W.sample_pairs(rows, w.num_heads, hpr, seed=2)


def _kv_block_rows(w, b, n=128, seed=5):
    """Sampled kv rows of segment b: its first and last rows, tile
    multiples +-1 and random rows (at least n)."""
    return W.sample_rows([w.cu_k[b], w.cu_k[b + 1]], n, seed=seed)


@pytest.mark.slow
def test_bwd_strided_dout_full():
    """410923 tokens, H=16, D=96, dout row stride 9728: the dout offset of
    segment 1's first row is 225304 * 9728 = 2,191,757,312 elements, past
    2^31 (the page's failing case).  dQ on 4096 sampled rows spanning both
    segments, including the rows where the dout element offset and the dQ
    accumulator byte offset cross 2^31; dK / dV element-wise on sampled kv
    rows of segment 1 (every one of its q rows, whose dout the gradients sum
    over, lies past the 2^31 element offset) and through the invariants over
    every row."""
    w = W.strided_dout()
    cpu = W.make_inputs(w, 0)
    _, _, dq, dk, dv = _run_gpu(w, cpu)
    extra = [225304, W.offset_crossing_row(9728, 1), W.offset_crossing_row(16 * 96, 4),
             W.offset_crossing_row(16 * 96, 2)]
    _compare(w, cpu, dq, dk, dv, _qpairs(w, 4096, 1, extra), kblock=(1, 11, _kv_block_rows(w, 1)), rows_path=True)
    _invariants(w, cpu, dk, dv)


@pytest.mark.slow
def test_bwd_long_full():
    """One 77000-row segment, H=56, D=128: dQ on 4096 sampled rows
    (including where the accumulator byte offset crosses 2^31), dK / dV
    element-wise on sampled kv rows of one head, invariants over all rows."""
    w = W.long_dense()
    cpu = W.make_inputs(w, 0)
    _, _, dq, dk, dv = _run_gpu(w, cpu)
    extra = [W.offset_crossing_row(56 * 128, 4)]
    _compare(w, cpu, dq, dk, dv, _qpairs(w, 4096, 1, extra), kblock=(0, 37, _kv_block_rows(w, 0)), rows_path=True)
    _invariants(w, cpu, dk, dv)


@pytest.mark.slow
def test_bwd_ragged_full():
    w = W.ragged()
    cpu = W.make_inputs(w, 0)
    _, _, dq, dk, dv = _run_gpu(w, cpu)
    # dK / dV rows of a few (segment, head) blocks, compared directly
    rng = np.random.default_rng(7)
    segs = [b for b in range(w.batch) if 0 < w.cu_k[b + 1] - w.cu_k[b] <= 3000][:3] + [4, 5]
    kr, kh = [], []
    for b in segs:
        h = int(rng.integers(0, w.num_heads))
        rows = W.sample_rows([w.cu_k[b], w.cu_k[b + 1]], 64, seed=b)
        kr.append(rows)
        kh.append(np.full(rows.size, h, np.int32))
    kp = (np.concatenate(kr), np.concatenate(kh))
    extra = [W.offset_crossing_row(w.row_stride, 2)]
    _compare(w, cpu, dq, dk, dv, _qpairs(w, 4096, 1, extra), kp)
    _invariants(w, cpu, dk, dv)


@pytest.mark.slow
def test_bwd_windowed_full():
    w = W.windowed()
    cpu = W.make_inputs(w, 0)
    _, _, dq, dk, dv = _run_gpu(w, cpu)
    b, h = 3, 17
    rows = W.sample_rows([w.cu_k[b], w.cu_k[b + 1]], 128, seed=9)
    kp = (rows, np.full(rows.size, h, np.int32))
    _compare(w, cpu, dq, dk, dv, _qpairs(w, 4096, 1), kp)
    _invariants(w, cpu, dk, dv)
