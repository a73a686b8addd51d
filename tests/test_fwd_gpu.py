"""GPU parity of the forward kernel against the fp64 oracle (through the C
ABI).  Small cases compare every (row, head); the full-size workloads compare
sampled rows that span every segment and the rows where a byte offset first
crosses 2^31."""
import numpy as np
import pytest
import torch

import oracle
from packed_variable_length_varlen_gb300 import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _fwd_case(w: W.Workload, seed=0, pairs=None, plant=None, max_seqlen=None, allow_ulp=None, ulps=1,
              canary=12345.0, rows_path=False):
    cpu = W.make_inputs(w, seed, with_dout=False)
    if plant is not None:
        plant(cpu)
    dev = cpu.to(DEV)
    out = W.output_like(w, "out", DEV, canary=canary)
    lse = torch.full((w.num_heads, w.total_q), 777.0, dtype=torch.float32, device=DEV)
    ms = max_seqlen if max_seqlen is not None else (None, None)
    P.run_fwd(dev, out, lse, *ms)
    torch.cuda.synchronize()
    assert P.padding_untouched(out, w, canary)
    if pairs is None:
        rows, heads = oracle.all_pairs(w.total_q, w.num_heads)
    else:
        rows, heads = pairs
    pb = P.oracle_problem(cpu)
    if rows_path:  # long unmasked segments: the oracle's matrix-product path
        o_ref, lse_ref = P.oracle_rows(pb, w, rows, heads)[:2]
    else:
        o_ref, lse_ref = pb.fwd(rows, heads)
    out_c = out.cpu()
    o_gpu = P.gather(out_c, rows, heads)
    lse_gpu = lse.cpu().numpy()[heads, rows].astype(np.float64)
    m = P.fwd_metrics(o_gpu, lse_gpu, o_ref, lse_ref)
    print(w.name, m)
    print(w.name, "worst (row, head, d, gpu, exact):", P.worst_elements(o_gpu, o_ref, rows, heads))
    P.assert_fwd(m, allow_one_ulp_above=allow_ulp, ulps=ulps)
    return out, lse, m


def test_fwd_tiny():
    _fwd_case(W.tiny())


@pytest.mark.parametrize("D", [64, 96, 128])
def test_fwd_ragged_small(D):
    # empty q, empty k, one-key, one-query, tile multiples +-1, Sq != Sk
    w = W.custom("ragged_small_d%d" % D, [0, 1, 127, 128, 129, 300, 0, 517, 3, 2],
                 [5, 0, 200, 128, 1, 700, 40, 517, 1000, 129], 3, D)
    _fwd_case(w)


def test_fwd_padded_strides_canary():
    w = W.custom("padded", [200, 0, 77, 256], [130, 9, 0, 300], 2, 128, row_pad=64)
    _fwd_case(w)


RESCALE_AMP = (0.05, 3.0, 10.0, 30.0)  # K amplitude per 128-key tile of a segment (last one onwards)


def _plant_rising_scores(w):
    """K rows scaled up tile by tile, so that a row's running max of
    S * scale * log2(e) grows by more than 8 at tiles 1, 2 and 3: the
    forward must rescale O (exactly, by alpha = 2^(m_old - m_new))."""
    def plant(cpu):
        for b in range(w.batch):
            k0, k1 = w.cu_k[b], w.cu_k[b + 1]
            for t, r in enumerate(range(k0, k1, 128)):
                cpu.k[r:min(r + 128, k1)] *= RESCALE_AMP[min(t, len(RESCALE_AMP) - 1)]
    return plant


def _rescale_rows(cpu, w):
    """Fraction of (row, head) pairs whose running tile max of S * c grows by
    more than 8 at some tile (unmasked)."""
    c = w.softmax_scale / np.log(2.0)
    hits = total = 0
    for b in range(w.batch):
        q0, q1, k0, k1 = w.cu_q[b], w.cu_q[b + 1], w.cu_k[b], w.cu_k[b + 1]
        if q1 == q0 or k1 - k0 <= 128:
            continue
        for h in range(w.num_heads):
            s = (cpu.q[q0:q1, h].double() @ cpu.k[k0:k1, h].double().T).numpy() * c
            m = np.maximum.accumulate(np.stack([s[:, t:t + 128].max(1) for t in range(0, k1 - k0, 128)], 1), 1)
            hits += int((np.diff(m, axis=1) > 8).any(1).sum())
            total += q1 - q0
    return hits / max(total, 1)


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_rescale_path(causal):
    """Scores that rise by more than 2^8 from one key tile to the next: every
    such step has O rescaled in TMEM before the step's P V is added; O and LSE
    match the oracle."""
    w = W.custom("rising_scores", [300, 129, 600, 1], [640, 300, 1100, 513], 2, 128)
    cpu = W.make_inputs(w, 5, with_dout=False)
    _plant_rising_scores(w)(cpu)
    if not causal:
        assert _rescale_rows(cpu, w) > 0.9
    dev = cpu.to(DEV)
    out = W.output_like(w, "out", DEV, canary=12345.0)
    lse = torch.full((w.num_heads, w.total_q), 777.0, dtype=torch.float32, device=DEV)
    P.run_fwd(dev, out, lse, causal=causal)
    torch.cuda.synchronize()
    assert P.padding_untouched(out, w, 12345.0)
    rows, heads = oracle.all_pairs(w.total_q, w.num_heads)
    o_ref, lse_ref = P.oracle_problem(cpu, causal=causal).fwd(rows, heads)
    o_gpu = P.gather(out.cpu(), rows, heads)
    lse_gpu = lse.cpu().numpy()[heads, rows].astype(np.float64)
    m = P.fwd_metrics(o_gpu, lse_gpu, o_ref, lse_ref)
    print("rescale", causal, m)
    # near one-hot rows: O is close to single V rows, |O| reaches 2 and more,
    # where one bf16 ulp (>= 1.6e-2) is above 1e-2: one ulp from bf16(exact)
    P.assert_fwd(m, allow_one_ulp_above=True, ulps=1)


def test_fwd_segment_isolation_nan():
    """NaN in the rows of the segment after a ragged tail must not reach the
    tail's outputs (rows past a segment end are masked / cleared)."""
    w = W.custom("isolation", [130, 70, 5], [129, 61, 40], 2, 128)

    def plant(cpu):
        # segment 1's kv rows and q rows hold NaN; segment 0 and 2 must be clean
        k0, k1 = w.cu_k[1], w.cu_k[2]
        cpu.k[k0:k1] = float("nan")
        cpu.v[k0:k1] = float("nan")
        q0, q1 = w.cu_q[1], w.cu_q[2]
        cpu.q[q0:q1] = float("nan")

    rows = np.array([r for r in range(w.total_q) if not (w.cu_q[1] <= r < w.cu_q[2])], dtype=np.int64)
    rr = np.repeat(rows, w.num_heads)
    hh = np.tile(np.arange(w.num_heads, dtype=np.int32), rows.size)
    _fwd_case(w, plant=plant, pairs=(rr, hh))


def test_fwd_max_seqlen_is_advisory():
    """A too-small max_seqlen (as in the captured call: 5040 passed while a
    5140-row segment exists) gives bit-identical output."""
    w = W.custom("advisory", [300, 129, 517], [200, 700, 128], 2, 128)
    out1, lse1, _ = _fwd_case(w)
    out2, lse2, _ = _fwd_case(w, max_seqlen=(5, 7))
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_fwd_no_keys_anywhere():
    w = W.custom("nokeys", [5, 130], [0, 0], 2, 64)
    out, lse, _ = _fwd_case(w)
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_fwd_deterministic():
    w = W.custom("det", [1000, 3], [2000, 5], 2, 128)
    cpu = W.make_inputs(w, 0, with_dout=False).to(DEV)
    outs = []
    for _ in range(2):
        out = W.output_like(w, "out", DEV)
        lse = torch.empty(w.num_heads, w.total_q, device=DEV)
        P.run_fwd(cpu, out, lse)
        outs.append((out.clone(), lse.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


# ---------------------------------------------------------------- full size

def _sampled_pairs(w: W.Workload, heads_per_row: int, extra=()):
    rows = W.sample_rows(w.cu_q, 4096, seed=1, extra_rows=extra)
    firsts = [w.cu_q[b] for b in range(w.batch) if w.cu_q[b + 1] > w.cu_q[b]]
    return W.sample_pairs(rows, w.num_heads, heads_per_row, seed=2, all_heads_rows=firsts[:4])


@pytest.mark.slow
def test_fwd_windowed_full():
    w = W.windowed()
    _fwd_case(w, pairs=_sampled_pairs(w, 2))


@pytest.mark.slow
def test_fwd_ragged_full():
    w = W.ragged()
    extra = [W.offset_crossing_row(w.row_stride, 2)]
    # amplitude-2 inputs: |O| reaches 8; see parity.assert_fwd for the ulp bound
    _fwd_case(w, pairs=_sampled_pairs(w, 2, extra), allow_ulp=1.28, ulps=2)


@pytest.mark.slow
def test_fwd_long_full():
    w = W.long_dense()
    extra = [W.offset_crossing_row(w.row_stride, 2)]
    rows = W.sample_rows(w.cu_q, 4096, seed=1, extra_rows=extra)
    _fwd_case(w, pairs=W.sample_pairs(rows, w.num_heads, 1, seed=2, all_heads_rows=[0, 76999]), rows_path=True)


@pytest.mark.slow
def test_fwd_strided_dout_workload_full():
    """Forward of the 410923-token, H=16, D=96 workload (inputs * 0.1)."""
    w = W.strided_dout()
    rows = W.sample_rows(w.cu_q, 4096, seed=1, extra_rows=[225304])
    _fwd_case(w, pairs=W.sample_pairs(rows, w.num_heads, 1, seed=2, all_heads_rows=[0, 225304, 410922]),
              rows_path=True)
