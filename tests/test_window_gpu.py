"""GPU parity of the sliding-window forward and backward
(varlen_attn_fwd_window / varlen_attn_bwd_window) against the fp64 oracle
with the same band: q row i of a segment sees the kv rows j with
i + Sk - Sq - left <= j <= i + Sk - Sq + right (a negative side unbounded).
Bands narrower than a tile, one-sided bands, bands wider than every segment,
Sq != Sk and empty sides.  Tolerances as for the unmasked path."""
import numpy as np
import pytest
import torch

import oracle
from packed_variable_length_varlen_gb300 import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu
DEV = "cuda"

SQ = [300, 129, 517, 1, 5, 0, 40, 255, 256, 2, 700]
SK = [300, 517, 129, 5, 1, 40, 0, 256, 255, 2, 130]


def _run(w: W.Workload, cpu: W.Inputs, window, canary=12345.0, causal=False):
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    dev = cpu.to(DEV)
    H, D = w.num_heads, w.head_dim
    out = W.output_like(w, "out", DEV, canary=canary)
    lse = torch.full((H, w.total_q), 777.0, dtype=torch.float32, device=DEV)
    P.run_fwd(dev, out, lse, causal=causal, window=window)
    dq, dk, dv = (W.output_like(w, n, DEV, canary=canary) for n in ("dq", "dk", "dv"))
    nbytes = va.varlen_attn_bwd_workspace_size(w.batch, w.total_q, H, D)
    wsp = torch.full((max(nbytes, 1),), 0x7F, dtype=torch.uint8, device=DEV)
    st = va.varlen_attn_bwd(dev.q, dev.k, dev.v, out, dev.dout, lse, dev.cu_q, dev.cu_k, w.batch, w.total_q,
                            w.total_k, H, D, w.max_q(), w.max_k(), w.softmax_scale, dq, dk, dv, wsp, nbytes,
                            causal=causal, window=window)
    assert st == 0, va.varlen_attn_status_string(st)
    st = va.varlen_attn_get_device_status()
    assert st == 0, va.varlen_attn_status_string(st)
    res = {"out": out, "lse": lse, "dq": dq, "dk": dk, "dv": dv}
    for t in res.values():
        if t.dim() == 3:
            assert P.padding_untouched(t, w, canary)
    return res


def _check(w, cpu, res, window, qpairs=None, kpairs=None):
    pb = P.oracle_problem(cpu, window=window)
    rows, heads = qpairs if qpairs is not None else oracle.all_pairs(w.total_q, w.num_heads)
    o_ref, lse_ref = pb.fwd(rows, heads)
    o_gpu = P.gather(res["out"].cpu(), rows, heads)
    lse_gpu = res["lse"].cpu().numpy()[heads, rows].astype(np.float64)
    m = P.fwd_metrics(o_gpu, lse_gpu, o_ref, lse_ref)
    print(w.name, window, m)
    # A narrow band averages few rows of V, so |O| reaches |v| (beyond 2 for
    # unit-variance inputs), where one bf16 ulp exceeds the 1e-2 bound:
    # elements past it may differ from bf16(exact) by one ulp.
    P.assert_fwd(m, allow_one_ulp_above=True, ulps=1)
    dead = np.isneginf(lse_ref)
    assert np.all(o_gpu[dead] == 0)  # rows whose band holds no key: exactly zero
    r = {}
    dq_ref, _ = pb.bwd_q(rows, heads)
    dq_gpu = P.gather(res["dq"].cpu(), rows, heads)
    r["dq"] = P.rel_fro(dq_gpu, dq_ref)
    assert np.all(dq_gpu[dead] == 0)
    krows, kheads = kpairs if kpairs is not None else oracle.all_pairs(w.total_k, w.num_heads)
    if krows.size:
        dk_ref, dv_ref = pb.bwd_kv(krows, kheads)
        dk_gpu, dv_gpu = P.gather(res["dk"].cpu(), krows, kheads), P.gather(res["dv"].cpu(), krows, kheads)
        r["dk"] = P.rel_fro(dk_gpu, dk_ref)
        r["dv"] = P.rel_fro(dv_gpu, dv_ref)
        unseen = np.all(dv_ref == 0, axis=1) & np.all(dk_ref == 0, axis=1)  # keys no query sees
        assert np.all(dk_gpu[unseen] == 0) and np.all(dv_gpu[unseen] == 0)
    print(w.name, window, r)
    for k_, v_ in r.items():
        if v_ == np.inf:
            # The band holds one key per row (window (0, 0)), so dS = P (dP - delta)
            # cancels exactly: dQ = dK = 0 in the oracle.  The kernel's delta uses
            # O rounded to bf16 (relative error <= 2^-9 per element), so
            # |dS| <= 2^-9 |dO| |o| and |dQ|, |dK| <= scale 2^-9 |dO| |o| max(|k|, |q|):
            # checked with a factor 8 of margin.
            g = {"dq": dq_gpu, "dk": dk_gpu if krows.size else None}[k_]
            nrm = lambda t: t.float().norm(dim=-1).max().item()
            bound = 2.0 ** -6 * w.softmax_scale * nrm(cpu.dout) * float(np.linalg.norm(o_ref, axis=1).max()) * max(
                nrm(cpu.k), nrm(cpu.q))
            assert float(np.abs(g).max()) <= bound, (k_, float(np.abs(g).max()), bound)
        else:
            assert v_ <= P.GRAD_REL_FRO, (k_, r)
    return dead


@pytest.mark.parametrize("window", [(3, 5), (0, 0), (200, 0), (0, 200), (130, 129), (-1, 5), (5, -1), (64, 64)])
def test_window_ragged_small(window):
    w = W.custom("window_ragged", SQ, SK, 2, 128)
    cpu = W.make_inputs(w, 0)
    res = _run(w, cpu, window)
    _check(w, cpu, res, window)


@pytest.mark.parametrize("D", [64, 96])
def test_window_head_dims(D):
    w = W.custom("window_d%d" % D, SQ, SK, 2, D)
    cpu = W.make_inputs(w, 1)
    res = _run(w, cpu, (17, 3))
    _check(w, cpu, res, (17, 3))


def test_window_causal_combination():
    """causal=True with a left side: the band (left, 0)."""
    w = W.custom("window_causal", SQ, SK, 2, 128)
    cpu = W.make_inputs(w, 2)
    res = _run(w, cpu, (100, 7), causal=True)
    _check(w, cpu, res, (100, 0))


def test_window_unbounded_and_wide_match_other_entry_points():
    """(-1, -1) runs the unmasked kernels and (-1, 0) the causal ones: bit
    for bit the same forward and dK / dV.  A band wider than every segment
    runs the masked kernel over every tile: the same forward bits as the
    unmasked kernel (same tiles, same arithmetic order)."""
    w = W.custom("window_same", [200, 64, 129, 1], [333, 64, 500, 7], 2, 128)
    cpu = W.make_inputs(w, 3)
    unmasked = _run(w, cpu, (-1, -1))
    causal = _run(w, cpu, (-1, -1), causal=True)
    for window, ref in (((-1, 0), causal), ((10 ** 6, 10 ** 6), unmasked)):
        got = _run(w, cpu, window)
        for n in ("out", "lse", "dk", "dv"):
            assert torch.equal(got[n].cpu(), ref[n].cpu()), (window, n)
        torch.testing.assert_close(got["dq"].cpu().float(), ref["dq"].cpu().float(), rtol=2e-2, atol=1e-3)


def test_window_long_segments_sampled():
    """Segments of several thousand rows (Sq < Sk and Sq > Sk) with a band of
    a few tiles: sampled rows of the forward and dQ, and dK / dV on sampled
    rows of two (segment, head) blocks."""
    w = W.custom("window_long", [4032, 5040, 300, 2049], [8000, 3000, 4500, 2049], 4, 128)
    cpu = W.make_inputs(w, 4)
    window = (777, 255)
    res = _run(w, cpu, window)
    rows = W.sample_rows(w.cu_q, 768, seed=5)
    qp = W.sample_pairs(rows, w.num_heads, 1, seed=6)
    kr, kh = [], []
    for b, h in ((0, 1), (3, 2)):
        rr = W.sample_rows([w.cu_k[b], w.cu_k[b + 1]], 96, seed=b)
        kr.append(rr)
        kh.append(np.full(rr.size, h, np.int32))
    _check(w, cpu, res, window, qp, (np.concatenate(kr), np.concatenate(kh)))


@pytest.mark.slow
def test_window_windowed_full():
    """The windowed workload (8 segments, H=56, D=128, Sq < Sk) with the band
    (1024, 0) that the benchmark times: forward and dQ on 4096 sampled rows
    over every segment; dK / dV on sampled kv rows of two (segment, head)
    blocks that start a little before the first key any query sees; and, over
    the whole dK / dV outputs, exact zeros for every key no query sees (with
    this band most of each segment's keys)."""
    w = W.windowed()
    cpu = W.make_inputs(w, 0)
    window = (1024, 0)
    res = _run(w, cpu, window)
    qp = W.sample_pairs(W.sample_rows(w.cu_q, 4096, seed=1), w.num_heads, 1, seed=2)
    first_seen = []  # per segment: the first key (0-based) some query's band holds
    for b in range(w.batch):
        sq, sk = w.cu_q[b + 1] - w.cu_q[b], w.cu_k[b + 1] - w.cu_k[b]
        first_seen.append(max(0, sk - sq - window[0]))
    kr, kh = [], []
    for b, h in ((2, 7), (5, 44)):
        lo = w.cu_k[b] + max(0, first_seen[b] - 64)
        rr = W.sample_rows([lo, w.cu_k[b + 1]], 128, seed=b)
        kr.append(rr)
        kh.append(np.full(rr.size, h, np.int32))
    _check(w, cpu, res, window, qp, (np.concatenate(kr), np.concatenate(kh)))
    dk, dv = res["dk"].cpu(), res["dv"].cpu()
    unseen = 0
    for b in range(w.batch):
        k0 = w.cu_k[b]
        assert first_seen[b] > 0
        assert int(torch.count_nonzero(dk[k0:k0 + first_seen[b]])) == 0, b
        assert int(torch.count_nonzero(dv[k0:k0 + first_seen[b]])) == 0, b
        assert int(torch.count_nonzero(dv[k0 + first_seen[b]])) > 0, b  # the first seen key has gradients
        unseen += first_seen[b]
    print("window (1024, 0) full size: %d of %d keys seen by no query, dK = dV = 0 there" % (unseen, w.total_k))
