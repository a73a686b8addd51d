"""Pins of the oracle's per-segment statistics path (``Problem.segment_stats``
and ``Problem.bwd_kv_block``), which the GPU parity tests use for dK / dV on
long segments (10^5 q rows), where running the row forward of every q row in
plain C would take many minutes.

It computes the same definition as the row-by-row oracle (LSE_i, delta_i =
dO_i . o_i, then dk_j, dv_j as sums over the segment's q rows) with fp64
matrix products over chunks of rows.  It is pinned here to the row-by-row
oracle functions, which are themselves pinned by tests/test_oracle_pins.py
(torch fp64 SDPA and autograd, closed forms, finite differences, planted
mistakes), and to closed forms of its own."""
import math

import numpy as np
import pytest
import torch

import oracle
from packed_variable_length_varlen_gb300 import workloads as W


def _problem(w, cpu, **kw):
    return oracle.Problem(cpu.q, cpu.k, cpu.v, cpu.cu_q, cpu.cu_k, w.softmax_scale, dout=cpu.dout, **kw)


def _close(a, b, rtol=1e-11):
    a, b = np.asarray(a), np.asarray(b)
    fa, fb = np.isfinite(a), np.isfinite(b)
    assert np.array_equal(fa, fb) and np.array_equal(a[~fa], b[~fb])
    scale = max(1.0, float(np.abs(b[fb]).max())) if fb.any() else 1.0
    assert float(np.abs(a[fa] - b[fb]).max(initial=0.0)) <= rtol * scale


@pytest.mark.parametrize("D,amp", [(64, 1.0), (96, 0.1), (128, 2.0)])
def test_stats_equal_row_by_row_oracle(D, amp):
    """LSE and delta of every q row, and dK / dV of every kv row, of every
    (segment, head): empty q, empty k, one-key and one-query segments,
    Sq != Sk."""
    w = W.custom("stats_d%d" % D, [0, 1, 37, 129, 5, 200], [4, 0, 1, 130, 77, 64], 2, D,
                 amplitude=amp, dout_amplitude=amp)
    cpu = W.make_inputs(w, 0)
    pb = _problem(w, cpu)
    for b in range(w.batch):
        q0, q1 = w.cu_q[b], w.cu_q[b + 1]
        k0, k1 = w.cu_k[b], w.cu_k[b + 1]
        for h in range(w.num_heads):
            lse, delta = pb.segment_stats(b, h)
            assert lse.shape == (q1 - q0,) and delta.shape == (q1 - q0,)
            if q1 > q0:
                rows = np.arange(q0, q1, dtype=np.int64)
                heads = np.full(rows.size, h, np.int32)
                _, lse_ref = pb.fwd(rows, heads)
                _, delta_ref = pb.bwd_q(rows, heads)
                _close(lse, lse_ref)
                _close(delta, delta_ref)
            if k1 > k0:
                krows = np.arange(k0, k1, dtype=np.int64)
                dk, dv = pb.bwd_kv_block(b, h, krows)
                dk_ref, dv_ref = pb.bwd_kv(krows, np.full(krows.size, h, np.int32))
                _close(dk, dk_ref)
                _close(dv, dv_ref)


def test_stats_chunking_is_row_local():
    """Each row's statistics depend on that row alone: any chunk size gives
    the same values."""
    w = W.custom("chunks", [61], [45], 3, 64)
    pb = _problem(w, W.make_inputs(w, 0))
    ref = pb.segment_stats(0, 1, chunk=256)
    for c in (1, 7, 60, 61):
        got = pb.segment_stats(0, 1, chunk=c)
        _close(got[0], ref[0], 1e-13)
        _close(got[1], ref[1], 1e-13)


def test_stats_closed_form_zero_queries():
    """Q = 0: every score is 0, so LSE_i = ln Sk and o_i = mean_j v_j, hence
    delta_i = dO_i . mean_j v_j; dv_j = (1/Sk) sum_i dO_i and dk_j = 0 (all
    P_ij equal, and sum_i dS_ij q_i with q_i = 0)."""
    w = W.custom("zeroq", [33], [50], 2, 64)
    cpu = W.make_inputs(w, 0)
    cpu.q.zero_()
    pb = _problem(w, cpu)
    for h in range(2):
        lse, delta = pb.segment_stats(0, h)
        assert np.allclose(lse, math.log(50), rtol=0, atol=1e-14)
        vbar = cpu.v[:, h].double().mean(0)
        want = (cpu.dout[:, h].double() * vbar).sum(1).numpy()
        assert np.allclose(delta, want, rtol=1e-12, atol=1e-14)
        dk, dv = pb.bwd_kv_block(0, h, np.arange(50))
        assert np.all(dk == 0.0)
        assert np.allclose(dv, np.broadcast_to(cpu.dout[:, h].double().sum(0).numpy() / 50, dv.shape),
                           rtol=1e-12, atol=1e-14)


def test_stats_strided_dout_layout():
    """dout as a view with a large row stride into a NaN-filled buffer (the
    strided-dout layout): only the view's elements are read."""
    w = W.custom("strided_stats", [70, 33], [70, 33], 2, 96, amplitude=0.1, dout_amplitude=0.1,
                 dout_row_stride=9728)
    cpu = W.make_inputs(w, 0)
    pb = _problem(w, cpu)
    for b in range(2):
        lse, delta = pb.segment_stats(b, 1)
        rows = np.arange(w.cu_q[b], w.cu_q[b + 1])
        _close(delta, pb.bwd_q(rows, np.full(rows.size, 1, np.int32))[1])
        assert np.all(np.isfinite(delta))


def test_stats_refuse_masks_and_bad_blocks():
    w = W.custom("m", [5], [5], 1, 64)
    cpu = W.make_inputs(w, 0)
    with pytest.raises(ValueError):
        _problem(w, cpu, causal=True).segment_stats(0, 0)
    pb = _problem(w, cpu)
    with pytest.raises(ValueError):
        pb.bwd_kv_block(0, 0, [0], stats=(np.zeros(4), np.zeros(4)))
    dk, dv = pb.bwd_kv_block(0, 0, [7])  # a row outside the segment
    assert np.all(np.isnan(dk)) and np.all(np.isnan(dv))


@pytest.mark.parametrize("D,amp", [(64, 1.0), (96, 0.1), (128, 2.0)])
def test_rows_block_equals_row_by_row_oracle(D, amp):
    """O, LSE, dQ and delta of every q row of every (segment, head) by the
    matrix-product path equal the row-by-row oracle's."""
    w = W.custom("rows_d%d" % D, [0, 1, 37, 129, 5, 200], [4, 0, 1, 130, 77, 64], 2, D,
                 amplitude=amp, dout_amplitude=amp)
    cpu = W.make_inputs(w, 0)
    pb = _problem(w, cpu)
    for b in range(w.batch):
        q0, q1 = w.cu_q[b], w.cu_q[b + 1]
        for h in range(w.num_heads):
            rows = np.arange(q0, q1, dtype=np.int64)[::-1].copy()  # any order
            o, lse, dq, delta = pb.rows_block(b, h, rows, chunk=16)
            heads = np.full(rows.size, h, np.int32)
            o_ref, lse_ref = pb.fwd(rows, heads)
            dq_ref, delta_ref = pb.bwd_q(rows, heads)
            for a, ref in ((o, o_ref), (lse, lse_ref), (dq, dq_ref), (delta, delta_ref)):
                _close(a, ref)


def test_rows_block_closed_forms():
    """Q = 0 gives LSE = ln Sk and o = mean_j v_j; a one-key segment gives
    o = v exactly, LSE = scale q . k and dq = 0."""
    w = W.custom("rows_cf", [9, 4], [21, 1], 2, 64)
    cpu = W.make_inputs(w, 0)
    cpu.q[:9].zero_()
    pb = _problem(w, cpu)
    o, lse, _, _ = pb.rows_block(0, 1, np.arange(9))
    assert np.allclose(lse, math.log(21), rtol=0, atol=1e-14)
    assert np.allclose(o, np.broadcast_to(cpu.v[:21, 1].double().mean(0).numpy(), o.shape), rtol=1e-12,
                       atol=1e-14)
    o, lse, dq, _ = pb.rows_block(1, 0, np.arange(9, 13))
    assert np.array_equal(o, np.broadcast_to(cpu.v[21, 0].double().numpy(), o.shape))
    want = w.softmax_scale * (cpu.q[9:13, 0].double() * cpu.k[21, 0].double()).sum(1).numpy()
    assert np.allclose(lse, want, rtol=1e-13, atol=1e-15)
    assert np.allclose(dq, 0.0, atol=1e-15)
    with pytest.raises(ValueError):
        pb.rows_block(0, 0, [9])  # row of another segment
