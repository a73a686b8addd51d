"""GPU checks of the deterministic backward (varlen_attn_bwd_deterministic):
dQ from the q-major kernel without atomics, dK / dV from the main kernel
without its dQ products.

* parity with the fp64 oracle on ragged segments (empty sides, Sq != Sk,
  tile multiples +-1) at D = 64 / 96 / 128, unmasked, causal and windowed;
* repeated calls return the same bits for dQ, dK and dV;
* dK and dV are bit for bit those of varlen_attn_bwd (same kernel and
  arithmetic order), and dQ matches it within the gradient tolerance."""
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


def _bwd(w, dev, out, lse, deterministic, causal=False, window=(-1, -1), canary=12345.0):
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    H, D = w.num_heads, w.head_dim
    dq, dk, dv = (W.output_like(w, n, DEV, canary=canary) for n in ("dq", "dk", "dv"))
    nbytes = va.varlen_attn_bwd_workspace_size(w.batch, w.total_q, H, D)
    wsp = torch.full((max(nbytes, 1),), 0x7F, dtype=torch.uint8, device=DEV)
    st = va.varlen_attn_bwd(dev.q, dev.k, dev.v, out, dev.dout, lse, dev.cu_q, dev.cu_k, w.batch, w.total_q,
                            w.total_k, H, D, w.max_q(), w.max_k(), w.softmax_scale, dq, dk, dv, wsp, nbytes,
                            causal=causal, window=window, deterministic=deterministic)
    assert st == 0, va.varlen_attn_status_string(st)
    st = va.varlen_attn_get_device_status()
    assert st == 0, va.varlen_attn_status_string(st)
    for t in (dq, dk, dv):
        assert P.padding_untouched(t, w, canary)
    return dq, dk, dv


def _fwd(w, dev, causal=False, window=(-1, -1)):
    out = W.output_like(w, "out", DEV)
    lse = torch.empty(w.num_heads, w.total_q, dtype=torch.float32, device=DEV)
    P.run_fwd(dev, out, lse, causal=causal, window=window)
    return out, lse


@pytest.mark.parametrize("D,causal,window", [(128, False, (-1, -1)), (64, False, (-1, -1)), (96, False, (-1, -1)),
                                             (128, True, (-1, -1)), (128, False, (77, 20)), (64, True, (300, 0))])
def test_deterministic_parity(D, causal, window):
    w = W.custom("det_d%d" % D, SQ, SK, 2, D)
    cpu = W.make_inputs(w, 0)
    dev = cpu.to(DEV)
    out, lse = _fwd(w, dev, causal, window)
    dq, dk, dv = _bwd(w, dev, out, lse, True, causal, window)
    band = (window[0], 0) if causal else window
    pb = P.oracle_problem(cpu, window=band)
    rows, heads = oracle.all_pairs(w.total_q, w.num_heads)
    krows, kheads = oracle.all_pairs(w.total_k, w.num_heads)
    dq_ref, _ = pb.bwd_q(rows, heads)
    dk_ref, dv_ref = pb.bwd_kv(krows, kheads)
    r = {"dq": P.rel_fro(P.gather(dq.cpu(), rows, heads), dq_ref),
         "dk": P.rel_fro(P.gather(dk.cpu(), krows, kheads), dk_ref),
         "dv": P.rel_fro(P.gather(dv.cpu(), krows, kheads), dv_ref)}
    print(D, causal, window, r)
    for k_, v_ in r.items():
        assert v_ <= P.GRAD_REL_FRO, (k_, r)
    # rows that see no key (empty-key segments, empty bands): exactly zero
    _, lse_ref = pb.fwd(rows, heads)
    dead = np.isneginf(lse_ref)
    assert dead.any()
    assert np.all(P.gather(dq.cpu(), rows, heads)[dead] == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_deterministic_repeats_bitwise(causal):
    """Many kv tiles per segment (so the atomic path's dQ has many adds per
    element): three deterministic runs agree bit for bit; dK / dV equal the
    atomic path's bits; dQ agrees with it within the gradient tolerance."""
    w = W.custom("det_rep", [3000, 1500, 4100], [9000, 2600, 4100], 4, 128)
    cpu = W.make_inputs(w, 7)
    dev = cpu.to(DEV)
    out, lse = _fwd(w, dev, causal)
    runs = [_bwd(w, dev, out, lse, True, causal) for _ in range(3)]
    for other in runs[1:]:
        for a, b in zip(runs[0], other):
            assert torch.equal(a, b)
    dq_a, dk_a, dv_a = _bwd(w, dev, out, lse, False, causal)
    assert torch.equal(runs[0][1], dk_a) and torch.equal(runs[0][2], dv_a)
    a = runs[0][0].double()
    b = dq_a.double()
    assert float((a - b).norm() / b.norm()) <= P.GRAD_REL_FRO


@pytest.mark.slow
def test_deterministic_windowed_sampled():
    """The windowed workload (H=56, D=128): dQ on sampled rows of every
    segment against the oracle, and dK / dV equal to the atomic path."""
    w = W.windowed()
    cpu = W.make_inputs(w, 0)
    dev = cpu.to(DEV)
    out, lse = _fwd(w, dev)
    dq, dk, dv = _bwd(w, dev, out, lse, True)
    qp = W.sample_pairs(W.sample_rows(w.cu_q, 4096, seed=3), w.num_heads, 1, seed=4)
    dq_ref, _ = P.oracle_problem(cpu).bwd_q(*qp)
    r = P.rel_fro(P.gather(dq.cpu(), *qp), dq_ref)
    print("windowed deterministic dq", r)
    assert r <= P.GRAD_REL_FRO
    _, dk_a, dv_a = _bwd(w, dev, out, lse, False)
    assert torch.equal(dk, dk_a) and torch.equal(dv, dv_a)


@pytest.mark.parametrize("sq,sk", [([0, 0, 0], [5, 130, 0]), ([7, 129, 3], [0, 0, 0]), ([0, 200, 0], [1, 0, 257])])
def test_deterministic_empty_sides(sq, sk):
    """No queries at all, no keys at all, and alternating empty segments: the
    deterministic form returns what the default one does (dK / dV bit for
    bit; dQ = 0 wherever a row sees no key) and never touches padding."""
    w = W.custom("det_empty", sq, sk, 2, 64)
    cpu = W.make_inputs(w, 9)
    dev = cpu.to(DEV)
    out, lse = _fwd(w, dev)
    dq, dk, dv = _bwd(w, dev, out, lse, True)
    dq_a, dk_a, dv_a = _bwd(w, dev, out, lse, False)
    assert torch.equal(dk, dk_a) and torch.equal(dv, dv_a)
    if w.total_q:
        pb = P.oracle_problem(cpu)
        rows, heads = oracle.all_pairs(w.total_q, w.num_heads)
        dq_ref, _ = pb.bwd_q(rows, heads)
        _, lse_ref = pb.fwd(rows, heads)
        dead = np.isneginf(lse_ref)
        got = P.gather(dq.cpu(), rows, heads)
        assert np.all(got[dead] == 0)
        if (~dead).any():
            assert P.rel_fro(got[~dead], dq_ref[~dead]) <= P.GRAD_REL_FRO
