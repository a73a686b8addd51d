"""GPU parity of the causal forward and backward (varlen_attn_fwd_causal /
varlen_attn_bwd_causal) against the fp64 oracle with the causal mask: q row i
of a segment sees kv rows j <= i + Sk - Sq.  Segments cover Sq = Sk, Sq < Sk
(the diagonal enters late), Sq > Sk (rows that see no key: O = 0,
LSE = -inf, dQ = 0), tile multiples +-1, one row, and empty sides.
Tolerances as for the unmasked path."""
import numpy as np
import pytest
import torch

import oracle
from packed_variable_length_varlen_gb300 import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu
DEV = "cuda"

SQ = [300, 129, 517, 1, 5, 0, 40, 255, 256, 2, 130]
SK = [300, 517, 129, 5, 1, 40, 0, 256, 255, 2, 700]


def _run(w: W.Workload, cpu: W.Inputs, backward=True, canary=12345.0):
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    dev = cpu.to(DEV)
    H, D = w.num_heads, w.head_dim
    out = W.output_like(w, "out", DEV, canary=canary)
    lse = torch.full((H, w.total_q), 777.0, dtype=torch.float32, device=DEV)
    P.run_fwd(dev, out, lse, causal=True)
    res = {"out": out, "lse": lse}
    if backward:
        dq, dk, dv = (W.output_like(w, n, DEV, canary=canary) for n in ("dq", "dk", "dv"))
        nbytes = va.varlen_attn_bwd_workspace_size(w.batch, w.total_q, H, D)
        wsp = torch.full((max(nbytes, 1),), 0x7F, dtype=torch.uint8, device=DEV)
        st = va.varlen_attn_bwd_causal(dev.q, dev.k, dev.v, out, dev.dout, lse, dev.cu_q, dev.cu_k, w.batch,
                                       w.total_q, w.total_k, H, D, w.max_q(), w.max_k(), w.softmax_scale, dq, dk,
                                       dv, wsp, nbytes)
        assert st == 0, va.varlen_attn_status_string(st)
        res.update(dq=dq, dk=dk, dv=dv)
    st = va.varlen_attn_get_device_status()
    assert st == 0, va.varlen_attn_status_string(st)
    for t in res.values():
        if t.dim() == 3:
            assert P.padding_untouched(t, w, canary)
    return res


def _check_fwd(w, cpu, res, pairs=None):
    rows, heads = pairs if pairs is not None else oracle.all_pairs(w.total_q, w.num_heads)
    pb = P.oracle_problem(cpu, causal=True)
    o_ref, lse_ref = pb.fwd(rows, heads)
    o_gpu = P.gather(res["out"].cpu(), rows, heads)
    lse_gpu = res["lse"].cpu().numpy()[heads, rows].astype(np.float64)
    m = P.fwd_metrics(o_gpu, lse_gpu, o_ref, lse_ref)
    print(w.name, m)
    P.assert_fwd(m)
    dead = np.isneginf(lse_ref)
    assert np.all(o_gpu[dead] == 0)  # rows that see no key: exactly zero
    return dead


def _check_bwd(w, cpu, res, qpairs=None, kpairs=None):
    pb = P.oracle_problem(cpu, causal=True)
    rows, heads = qpairs if qpairs is not None else oracle.all_pairs(w.total_q, w.num_heads)
    krows, kheads = kpairs if kpairs is not None else oracle.all_pairs(w.total_k, w.num_heads)
    r = {}
    if rows.size:
        dq_ref, _ = pb.bwd_q(rows, heads)
        r["dq"] = P.rel_fro(P.gather(res["dq"].cpu(), rows, heads), dq_ref)
    if krows.size:
        dk_ref, dv_ref = pb.bwd_kv(krows, kheads)
        r["dk"] = P.rel_fro(P.gather(res["dk"].cpu(), krows, kheads), dk_ref)
        r["dv"] = P.rel_fro(P.gather(res["dv"].cpu(), krows, kheads), dv_ref)
    print(w.name, r)
    for k_, v_ in r.items():
        assert v_ <= P.GRAD_REL_FRO, (k_, r)


@pytest.mark.parametrize("D", [64, 96, 128])
def test_causal_ragged_small(D):
    w = W.custom("causal_ragged_d%d" % D, SQ, SK, 2, D)
    cpu = W.make_inputs(w, 0)
    res = _run(w, cpu)
    dead = _check_fwd(w, cpu, res)
    assert dead.any()  # the Sq > Sk segments have rows that see no key
    _check_bwd(w, cpu, res)
    rows, heads = oracle.all_pairs(w.total_q, w.num_heads)
    dq = P.gather(res["dq"].cpu(), rows, heads)
    assert np.all(dq[dead] == 0)


def test_causal_matches_unmasked_on_rows_that_see_everything():
    """The last row of each segment sees every key: its output equals the
    unmasked kernel's bit for bit (same tiles, same arithmetic order)."""
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    w = W.custom("causal_vs_full", [200, 64, 129], [333, 64, 500], 2, 128)
    cpu = W.make_inputs(w, 1, with_dout=False)
    dev = cpu.to(DEV)
    outs = []
    for causal in (False, True):
        out = W.output_like(w, "out", DEV)
        lse = torch.empty(w.num_heads, w.total_q, dtype=torch.float32, device=DEV)
        P.run_fwd(dev, out, lse, causal=causal)
        outs.append((out.cpu(), lse.cpu()))
    last = [w.cu_q[b + 1] - 1 for b in range(w.batch)]
    for r in last:
        assert torch.equal(outs[0][0][r], outs[1][0][r]) and torch.equal(outs[0][1][:, r], outs[1][1][:, r])


@pytest.mark.slow
def test_causal_windowed_full():
    """The windowed workload (H=56, D=128, Sq < Sk) with the causal mask:
    forward on sampled rows of every segment, dQ on sampled rows, dK / dV on
    sampled rows of two (segment, head) blocks, and the exact invariant
    sum_j dk_j = 0 per (segment, head) (no row of this workload is dead)."""
    w = W.windowed()
    cpu = W.make_inputs(w, 0)
    res = _run(w, cpu)
    rows = W.sample_rows(w.cu_q, 4096, seed=1)
    _check_fwd(w, cpu, res, W.sample_pairs(rows, w.num_heads, 1, seed=2))
    qp = W.sample_pairs(W.sample_rows(w.cu_q, 4096, seed=3), w.num_heads, 1, seed=4)
    kr, kh = [], []
    for b, h in ((1, 5), (6, 40)):
        rr = W.sample_rows([w.cu_k[b], w.cu_k[b + 1]], 64, seed=b)
        kr.append(rr)
        kh.append(np.full(rr.size, h, np.int32))
    _check_bwd(w, cpu, res, qp, (np.concatenate(kr), np.concatenate(kh)))
    dkc = res["dk"].cpu().double()
    rms = float(dkc.pow(2).mean().sqrt())
    for b in range(w.batch):
        k0, k1 = w.cu_k[b], w.cu_k[b + 1]
        s = dkc[k0:k1].sum(0)
        a = dkc[k0:k1].abs().sum(0) + (k1 - k0) ** 0.5 * rms
        assert float((s.abs() / a).max()) <= 1e-2
