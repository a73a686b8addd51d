"""GPU checks of the E4M3 (FP8) forward (varlen_attn_fwd_fp8) against the
oracle's FP8 reading:

* the quantiser is integer work decided in fp32 on both sides: amax per
  (segment, head), the Q / K codes and the transposed V codes (with code 0
  past each segment's end) equal the oracle's bit for bit;
* O matches the oracle's FP8 forward within the rounding of P: the kernel
  rounds P from a running row maximum, the oracle from the final one, each
  within 2^-4 relative per weight, so |dO| <= 2^-3 vd sum_j p_j |v8_j| / l
  (computed by the oracle with |V| and unrounded P) plus the bf16 rounding of
  O; LSE within 1e-3 (P's rounding does not enter it);
* against the fp64 oracle on the bf16 inputs, cosine >= 0.998 (the method's
  own envelope);
* under causal and sliding-window bands (varlen_attn_fwd_fp8_window), the
  same bounds against the oracle's masked FP8 forward, rows that see no key
  exactly O = 0 and LSE = -inf;
* Q and K small enough (~1e-22) that scale * qd * kd underflows fp32: finite
  results within the same bounds;
* at full size (the windowed workload, H=56), unmasked and causal, one head
  per segment: the segment's amax and codes bit for bit, and O / LSE on
  4096 sampled rows spanning every segment; on the long-sequence workload
  (one 77000-row segment) the same for four heads on 2048 rows."""
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


def _run(w, cpu, scale=None, causal=False, window=(-1, -1)):
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    dev = cpu.to(DEV)
    H = w.num_heads
    out = W.output_like(w, "out", DEV, canary=12345.0)
    lse = torch.full((H, w.total_q), 777.0, dtype=torch.float32, device=DEV)
    nbytes = va.varlen_attn_fwd_fp8_workspace_size(w.batch, w.total_q, w.total_k, H, 128)
    ws = torch.full((nbytes,), 0x7F, dtype=torch.uint8, device=DEV)  # NaN codes: every used byte is written
    st = va.varlen_attn_fwd_fp8(dev.q, dev.k, dev.v, dev.cu_q, dev.cu_k, w.batch, w.total_q, w.total_k, H, 128,
                                w.max_q(), w.max_k(), w.softmax_scale if scale is None else scale, out, lse, ws,
                                nbytes, causal=causal, window=window)
    assert st == 0, va.varlen_attn_status_string(st)
    st = va.varlen_attn_get_device_status()
    assert st == 0, va.varlen_attn_status_string(st)
    assert P.padding_untouched(out, w, 12345.0)
    st, off, cols = va.varlen_attn_fwd_fp8_workspace_layout(w.batch, w.total_q, w.total_k, H, 128)
    assert st == 0
    wsc = ws.cpu()
    nbh = w.batch * H
    amax = wsc[off[0]:off[0] + 3 * nbh * 4].view(torch.float32).view(3, nbh)
    q8 = wsc[off[1]:off[1] + w.total_q * H * 128].view(w.total_q, H, 128)
    k8 = wsc[off[2]:off[2] + w.total_k * H * 128].view(w.total_k, H, 128)
    vt = wsc[off[3]:off[3] + H * 128 * cols].view(H, 128, cols)
    return out, lse, amax, q8, k8, vt


def _amax_ref(x, cu, H):
    a = np.zeros(((len(cu) - 1) * H,), dtype=np.float32)
    xs = x.float().numpy()
    for b in range(len(cu) - 1):
        if cu[b + 1] > cu[b]:
            a[b * H:(b + 1) * H] = np.abs(xs[cu[b]:cu[b + 1]]).max(axis=(0, 2))
    return a


def _check_codes(w, cpu, amax, q8, k8, vt):
    """amax, Q / K codes and the transposed V codes equal the oracle's bit for
    bit; returns the oracle's codes and descales."""
    H = w.num_heads
    for i, (x, cu) in enumerate(((cpu.q, w.cu_q), (cpu.k, w.cu_k), (cpu.v, w.cu_k))):
        assert np.array_equal(amax[i].numpy(), _amax_ref(x, cu, H)), i
    q8r, qd = oracle.quantize_e4m3(cpu.q, w.cu_q)
    k8r, kd = oracle.quantize_e4m3(cpu.k, w.cu_k)
    v8r, vd = oracle.quantize_e4m3(cpu.v, w.cu_k)
    for name, got, ref, x, d, cu in (("q", q8, q8r, cpu.q, qd, w.cu_q), ("k", k8, k8r, cpu.k, kd, w.cu_k)):
        bad = (got != ref).nonzero()
        if len(bad):
            r, h, e = (int(t) for t in bad[0])
            b = int(np.searchsorted(np.asarray(cu), r, side="right")) - 1
            raise AssertionError("%s codes: %d differ; first at row %d head %d d %d: x %r descale %r gpu %d oracle %d"
                                 % (name, len(bad), r, h, e, float(x[r, h, e].float()), float(d[b * H + h]),
                                    int(got[r, h, e]), int(ref[r, h, e])))
    for b in range(w.batch):
        k0, k1 = w.cu_k[b], w.cu_k[b + 1]
        base = 128 * (b + -(-k0 // 128))
        n = k1 - k0
        if n == 0:
            continue
        blk = vt[:, :, base:base + n]                       # [H, 128, n]
        assert torch.equal(blk, v8r[k0:k1].permute(1, 2, 0)), b
        pad = -(-n // 128) * 128 - n
        assert bool((vt[:, :, base + n:base + n + pad] == 0).all()), b
    return q8r, k8r, v8r, qd, kd, vd


def _check_forward(w, cpu, out, lse, codes, causal=False, window=(-1, -1), min_cos=0.998):
    """O within the P-rounding bound of the oracle's FP8 forward (under the
    same band), LSE within 1e-3, rows without keys exactly O = 0 and
    LSE = -inf, and the fp64 forward on the bf16 inputs within the method's
    cosine envelope."""
    H = w.num_heads
    q8r, k8r, v8r, qd, kd, vd = codes
    band = dict(causal=causal, window=window)
    rows, heads = oracle.all_pairs(w.total_q, H)
    pf = oracle.Fp8Problem(q8r, k8r, v8r, w.cu_q, w.cu_k, w.softmax_scale, qd, kd, vd, quantize_p=True, **band)
    o_ref, l_ref = pf.fwd(rows, heads)
    pa = oracle.Fp8Problem(q8r, k8r, v8r & 0x7F, w.cu_q, w.cu_k, w.softmax_scale, qd, kd, vd, quantize_p=False,
                           **band)
    o_abs, _ = pa.fwd(rows, heads)
    o_gpu = P.gather(out.cpu(), rows, heads)
    l_gpu = lse.cpu().numpy()[heads, rows].astype(np.float64)
    bound = 2.0 ** -3 * o_abs + 2.0 ** -8 * np.abs(o_ref) + 1e-3
    excess = np.abs(o_gpu - o_ref) - bound
    fin = np.isfinite(l_ref)
    print("fp8 %s: max |dO| %.4g, max excess %.4g, %d rows without keys"
          % (band, np.abs(o_gpu - o_ref).max(), excess.max(), int((~fin).sum())))
    assert (excess <= 0).all()
    assert np.array_equal(np.isneginf(l_gpu), ~fin)
    assert np.abs(l_gpu[fin] - l_ref[fin]).max() <= 1e-3
    assert np.all(o_gpu[~fin] == 0)
    o64, _ = P.oracle_problem(cpu, **band).fwd(rows, heads)
    cos = float((o_gpu * o64).sum() / np.linalg.norm(o_gpu) / np.linalg.norm(o64))
    print("fp8 cosine vs fp64", cos)
    assert cos >= min_cos
    return int((~fin).sum())


# Bands for the masked E4M3 forward: causal, windows whose edges cross key
# tiles on one or both sides, the diagonal alone, and causal with a left
# width (SQ / SK include segments with Sq > Sk, whose first causal rows see
# no key).
FP8_BANDS = [(True, (-1, -1)), (False, (200, 0)), (False, (0, 0)), (False, (130, 257)), (False, (-1, 40)),
             (True, (300, -1))]


@pytest.mark.parametrize("causal,window", FP8_BANDS, ids=["causal", "w200_0", "w0_0", "w130_257", "w-1_40",
                                                          "causal_w300"])
def test_fp8_masked_forward(causal, window):
    """The E4M3 forward under a band: codes as unmasked (the quantisation
    does not depend on the band), O / LSE against the oracle's masked FP8
    forward."""
    w = W.custom("fp8_masked", SQ, SK, 2, 128)
    cpu = W.make_inputs(w, 2, with_dout=False)
    out, lse, amax, q8, k8, vt = _run(w, cpu, causal=causal, window=window)
    codes = _check_codes(w, cpu, amax, q8, k8, vt)
    empty = _check_forward(w, cpu, out, lse, codes, causal=causal, window=window)
    if causal:
        assert empty > 0  # segments with Sq > Sk start with rows that see no key


@pytest.mark.parametrize("causal", [False, True], ids=["unmasked", "causal"])
def test_fp8_padded_rows(causal):
    """Inputs and output with rows padded past H * D (NaN in the inputs'
    padding, a canary in the output's): the quantiser reads only each row's
    H * D elements, the codes and O / LSE match the oracle as for packed
    rows, and the output's padding is untouched."""
    w = W.custom("fp8_padded", SQ[:7], SK[:7], 2, 128, row_pad=64)
    cpu = W.make_inputs(w, 8, with_dout=False)
    assert cpu.q._base is not None and bool(torch.isnan(cpu.q._base[:, 256:]).all())
    out, lse, amax, q8, k8, vt = _run(w, cpu, causal=causal)
    codes = _check_codes(w, cpu, amax, q8, k8, vt)
    _check_forward(w, cpu, out, lse, codes, causal=causal)


@pytest.mark.parametrize("causal", [False, True], ids=["unmasked", "causal"])
def test_fp8_tiny_descales(causal):
    """Q and K of magnitude ~1e-22, so that scale * log2(e) * qd * kd rounds
    to 0 in fp32: the scores are ~0, P is 1 for every visible key, and the
    keys past a segment's end (or outside the band) must still count as
    -inf, not NaN."""
    w = W.custom("fp8_tiny", [300, 129, 40], [300, 517, 5], 2, 128)
    cpu = W.make_inputs(w, 6, with_dout=False)
    cpu.q.mul_(1e-22)
    cpu.k.mul_(1e-22)
    out, lse, amax, q8, k8, vt = _run(w, cpu, causal=causal)
    codes = _check_codes(w, cpu, amax, q8, k8, vt)
    assert float(codes[3].max()) * float(codes[4].max()) * w.softmax_scale * 1.4427 < 2.0 ** -150
    assert bool(torch.isfinite(out.float()).all())
    _check_forward(w, cpu, out, lse, codes, causal=causal)


@pytest.mark.parametrize("seed", [0, 1])
def test_fp8_codes_and_forward(seed):
    w = W.custom("fp8", SQ, SK, 2, 128)
    cpu = W.make_inputs(w, seed, with_dout=False)
    out, lse, amax, q8, k8, vt = _run(w, cpu)
    H = w.num_heads
    # quantiser: bit for bit
    q8r, k8r, v8r, qd, kd, vd = _check_codes(w, cpu, amax, q8, k8, vt)
    # forward against the oracle's FP8 reading
    rows, heads = oracle.all_pairs(w.total_q, H)
    pf = oracle.Fp8Problem(q8r, k8r, v8r, w.cu_q, w.cu_k, w.softmax_scale, qd, kd, vd, quantize_p=True)
    o_ref, l_ref = pf.fwd(rows, heads)
    pa = oracle.Fp8Problem(q8r, k8r, v8r & 0x7F, w.cu_q, w.cu_k, w.softmax_scale, qd, kd, vd, quantize_p=False)
    o_abs, _ = pa.fwd(rows, heads)
    o_gpu = P.gather(out.cpu(), rows, heads)
    l_gpu = lse.cpu().numpy()[heads, rows].astype(np.float64)
    bound = 2.0 ** -3 * o_abs + 2.0 ** -8 * np.abs(o_ref) + 1e-3
    excess = np.abs(o_gpu - o_ref) - bound
    print("fp8 max |dO| %.4g, max excess %.4g" % (np.abs(o_gpu - o_ref).max(), excess.max()))
    assert (excess <= 0).all()
    fin = np.isfinite(l_ref)
    assert np.array_equal(np.isneginf(l_gpu), ~fin)
    assert np.abs(l_gpu[fin] - l_ref[fin]).max() <= 1e-3
    assert np.all(o_gpu[~fin] == 0)
    # the method's envelope against fp64 on the bf16 inputs
    o64, _ = P.oracle_problem(cpu).fwd(rows, heads)
    cos = float((o_gpu * o64).sum() / np.linalg.norm(o_gpu) / np.linalg.norm(o64))
    print("fp8 cosine vs fp64", cos)
    assert cos >= 0.998


# Segment maxima (bf16 bit patterns) for the every-value test: a subnormal,
# the smallest normal, the three around a descale of 2^-100 (448 * 2^-100 is
# 0x11E0), 1, 448, 2^63 and the largest finite bf16.
ALL_VALUE_AMAX = [0x0005, 0x0080, 0x11DF, 0x11E0, 0x11E1, 0x3F80, 0x43E0, 0x5F00, 0x7F7F]


def _every_value_rows(amax_bits, rows):
    """[rows, 128] bf16 holding every finite bf16 of magnitude <= the bf16
    amax_bits, both signs, then zeros."""
    pos = torch.arange(amax_bits + 1, dtype=torch.int32)
    vals = torch.cat([pos, pos | 0x8000]).to(torch.int16).view(torch.bfloat16)
    out = torch.zeros(rows * 128, dtype=torch.bfloat16)
    out[:vals.numel()] = vals
    return out.view(rows, 128)


# 32 more maxima drawn over the whole positive finite bf16 range (seeded)
SPREAD_AMAX = sorted(int(a) for a in np.random.default_rng(11).integers(1, 0x7F80, 32))


@pytest.mark.parametrize("maxima", [ALL_VALUE_AMAX, SPREAD_AMAX], ids=["edges", "spread"])
def test_fp8_codes_every_bf16_value(maxima):
    """Q and V segments whose heads hold every finite bf16 value up to their
    maximum, for maxima from a subnormal to the largest finite bf16 (descales
    on both sides of 2^-100 among them, and 32 spread over the range): every
    code equals the oracle's IEEE fp32 division and conversion.  K is
    ordinary data; the softmax scale is small enough that S stays finite."""
    lens = [-(-2 * (a + 1) // 128) for a in maxima]
    w = W.custom("fp8_every_value", lens, lens, 2, 128)
    cpu = W.make_inputs(w, 3, with_dout=False)
    for b, a in enumerate(maxima):
        r0, r1 = w.cu_q[b], w.cu_q[b + 1]
        blk = _every_value_rows(a, r1 - r0)
        cpu.q[r0:r1, 0] = blk
        cpu.q[r0:r1, 1] = blk.flip(0)
        cpu.v[r0:r1, 0] = blk.flip(0)
        cpu.v[r0:r1, 1] = blk
    _, _, amax, q8, k8, vt = _run(w, cpu, scale=1e-37)
    _check_codes(w, cpu, amax, q8, k8, vt)


@pytest.mark.slow
@pytest.mark.parametrize("causal", [False, True], ids=["unmasked", "causal"])
def test_fp8_windowed_full_size_sampled(causal):
    """The E4M3 forward on the windowed workload (8 segments, H=56, D=128, the
    size the benchmark times), unmasked and causal.  Per segment b one head
    h_b: the oracle quantises that (segment, head) block on its own (its
    descale depends on nothing else), the block's amax and Q, K and
    transposed V codes must equal the kernel's bit for bit, and 512 sampled
    rows of it (4096 in all) must match the oracle's FP8 forward (under the
    same band, which is per segment) within the P-rounding bound, LSE within
    1e-3, and the fp64 forward on the bf16 inputs with cosine >= 0.998."""
    w = W.windowed()
    H = w.num_heads
    cpu = W.make_inputs(w, 0, with_dout=False)
    out, lse, amax, q8, k8, vt = _run(w, cpu, causal=causal)
    out_c, lse_c = out.cpu(), lse.cpu().numpy()
    pb64 = P.oracle_problem(cpu, causal=causal)
    rng = np.random.default_rng(7)
    all_gpu, all_64 = [], []
    for b in range(w.batch):
        h = (5 + 7 * b) % H
        q0, q1, k0, k1 = w.cu_q[b], w.cu_q[b + 1], w.cu_k[b], w.cu_k[b + 1]
        blk = [t[r0:r1, h:h + 1] for t, r0, r1 in ((cpu.q, q0, q1), (cpu.k, k0, k1), (cpu.v, k0, k1))]
        codes, desc = [], []
        for i, x in enumerate(blk):
            assert np.float32(amax[i][b * H + h]) == np.float32(x.float().abs().max()), (b, h, i)
            c, d = oracle.quantize_e4m3(x, [0, x.shape[0]])
            codes.append(c)
            desc.append(d)
        assert torch.equal(q8[q0:q1, h], codes[0][:, 0]), (b, h)
        assert torch.equal(k8[k0:k1, h], codes[1][:, 0]), (b, h)
        base = 128 * (b + -(-k0 // 128))
        assert torch.equal(vt[h, :, base:base + (k1 - k0)], codes[2][:, 0].T), (b, h)
        rows = np.sort(np.concatenate([1 + rng.choice(q1 - q0 - 2, 510, replace=False), [0, q1 - q0 - 1]]))
        zeros = np.zeros(rows.size, dtype=np.int64)
        pf = oracle.Fp8Problem(*codes, [0, q1 - q0], [0, k1 - k0], w.softmax_scale, *desc, quantize_p=True,
                               causal=causal)
        o_ref, l_ref = pf.fwd(rows, zeros)
        pa = oracle.Fp8Problem(codes[0], codes[1], codes[2] & 0x7F, [0, q1 - q0], [0, k1 - k0], w.softmax_scale,
                               *desc, quantize_p=False, causal=causal)
        o_abs, _ = pa.fwd(rows, zeros)
        grow, gh = q0 + rows, np.full(rows.size, h)
        o_gpu = P.gather(out_c, grow, gh)
        l_gpu = lse_c[gh, grow].astype(np.float64)
        excess = np.abs(o_gpu - o_ref) - (2.0 ** -3 * o_abs + 2.0 ** -8 * np.abs(o_ref) + 1e-3)
        assert (excess <= 0).all(), (b, h, excess.max())
        assert np.abs(l_gpu - l_ref).max() <= 1e-3, (b, h)
        # the matrix-product path covers unmasked problems; the band takes the row-by-row oracle
        o64 = pb64.fwd(grow, gh)[0] if causal else P.oracle_rows(pb64, w, grow, gh)[0]
        all_gpu.append(o_gpu)
        all_64.append(o64)
    o_gpu, o64 = np.concatenate(all_gpu), np.concatenate(all_64)
    assert o_gpu.shape[0] >= 4096
    cos = float((o_gpu * o64).sum() / np.linalg.norm(o_gpu) / np.linalg.norm(o64))
    print("fp8 full size (causal=%s): %d rows, cosine vs fp64 %.6f" % (causal, o_gpu.shape[0], cos))
    assert cos >= 0.998


@pytest.mark.slow
def test_fp8_long_full_size_sampled():
    """The E4M3 forward on the long-sequence workload: one 77000-row segment,
    H=56, D=128, the size at which the ffpa-attn NVFP4 launcher aborted
    ("Minimal reproduction").  For four heads: amax and the Q, K and
    transposed V codes of the head's block bit for bit (code 0 past the
    segment end), and 512 sampled rows each (2048 in all; the oracle decodes
    every key's codes per row, about 35 ms a row on one core) within the
    P-rounding bound of the oracle's FP8 forward, LSE within 1e-3, and the
    fp64 forward on the bf16 inputs with cosine >= 0.998."""
    w = W.long_dense()
    H, n = w.num_heads, w.total_q
    cpu = W.make_inputs(w, 0, with_dout=False)
    out, lse, amax, q8, k8, vt = _run(w, cpu)
    out_c, lse_c = out.cpu(), lse.cpu().numpy()
    pb64 = P.oracle_problem(cpu)
    rng = np.random.default_rng(9)
    all_gpu, all_64 = [], []
    for h in (0, 19, 38, 55):
        codes, desc = [], []
        for i, x in enumerate((cpu.q[:, h:h + 1], cpu.k[:, h:h + 1], cpu.v[:, h:h + 1])):
            assert np.float32(amax[i][h]) == np.float32(x.float().abs().max()), (h, i)
            c, d = oracle.quantize_e4m3(x, [0, n])
            codes.append(c)
            desc.append(d)
        assert torch.equal(q8[:, h], codes[0][:, 0]), h
        assert torch.equal(k8[:, h], codes[1][:, 0]), h
        assert torch.equal(vt[h, :, :n], codes[2][:, 0].T), h
        assert bool((vt[h, :, n:-(-n // 128) * 128] == 0).all()), h
        rows = np.sort(np.concatenate([1 + rng.choice(n - 2, 510, replace=False), [0, n - 1]]))
        zeros = np.zeros(rows.size, dtype=np.int64)
        o_ref, l_ref = oracle.Fp8Problem(*codes, [0, n], [0, n], w.softmax_scale, *desc,
                                         quantize_p=True).fwd(rows, zeros)
        o_abs, _ = oracle.Fp8Problem(codes[0], codes[1], codes[2] & 0x7F, [0, n], [0, n], w.softmax_scale, *desc,
                                     quantize_p=False).fwd(rows, zeros)
        gh = np.full(rows.size, h)
        o_gpu = P.gather(out_c, rows, gh)
        l_gpu = lse_c[gh, rows].astype(np.float64)
        excess = np.abs(o_gpu - o_ref) - (2.0 ** -3 * o_abs + 2.0 ** -8 * np.abs(o_ref) + 1e-3)
        assert (excess <= 0).all(), (h, excess.max())
        assert np.abs(l_gpu - l_ref).max() <= 1e-3, h
        all_gpu.append(o_gpu)
        all_64.append(P.oracle_rows(pb64, w, rows, gh)[0])
    o_gpu, o64 = np.concatenate(all_gpu), np.concatenate(all_64)
    cos = float((o_gpu * o64).sum() / np.linalg.norm(o_gpu) / np.linalg.norm(o64))
    print("fp8 long: %d rows, cosine vs fp64 %.6f" % (o_gpu.shape[0], cos))
    assert cos >= 0.998


@pytest.mark.parametrize("causal,window", [(False, (-1, -1)), (True, (-1, -1)), (False, (64, 0))],
                         ids=["unmasked", "causal", "window"])
def test_fp8_python_wrapper_matches_raw_call(causal, window):
    """attention_fwd_fp8 (argument marshalling only) returns the raw call's
    bits; the window form with (-1, -1) is the unmasked call."""
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    w = W.custom("fp8_wrap", [200, 3, 129], [150, 300, 1], 2, 128)
    cpu = W.make_inputs(w, 4, with_dout=False)
    out, lse, *_ = _run(w, cpu, causal=causal, window=window)
    dev = cpu.to(DEV)
    o2, l2, ws = va.attention_fwd_fp8(dev.q, dev.k, dev.v, dev.cu_q, dev.cu_k, w.softmax_scale, causal=causal,
                                      window=window)
    assert torch.equal(o2.cpu(), out.cpu()) and torch.equal(l2.cpu(), lse.cpu())
    if not causal and window == (-1, -1):
        o3 = torch.empty_like(out)
        l3 = torch.empty_like(lse)
        st = va.varlen_attn_fwd_fp8_window(dev.q, dev.k, dev.v, dev.cu_q, dev.cu_k, w.batch, w.total_q, w.total_k,
                                           2, 128, 0, 0, w.softmax_scale, -1, -1, o3, l3, ws, ws.numel())
        assert st == 0
        assert torch.equal(o3.cpu(), out.cpu()) and torch.equal(l3.cpu(), lse.cpu())
