"""GPU parity of the dense batched entry points (varlen_attn_fwd_dense /
varlen_attn_bwd_dense) against the fp64 oracle run on the packed view with
cu_seqlens = {0, S, 2S, ...}, unmasked and causal, through padded row
strides; and bit-identity with the packed entry points on the same data."""
import numpy as np
import pytest
import torch

import oracle
from packed_variable_length_varlen_gb300 import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _dense(B, S, H, D, seed, pad=24, amp=1.0):
    """A [B, S, H, D] bf16 view with row stride H*D + pad (NaN in the pad)."""
    g = torch.Generator().manual_seed(seed)
    base = torch.full((B, S, H * D + pad), float("nan"), dtype=torch.bfloat16)
    t = base[:, :, :H * D].unflatten(2, (H, D))
    t.copy_((torch.randn(B, S, H, D, generator=g) * amp).to(torch.bfloat16))
    return t


def _packed(t):
    """The [B*S, H, D] view of a dense tensor (same memory)."""
    B, S, H, D = t.shape
    return t.as_strided((B * S, H, D), (t.stride(1), t.stride(2), 1), t.storage_offset())


def _dev(t):
    base = t._base if t._base is not None else t
    return base.to(DEV).as_strided(t.shape, t.stride(), t.storage_offset())


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_dense_matches_oracle(D, causal):
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    B, Sq, Sk, H = 3, 130, 257, 2
    q, k, v = _dense(B, Sq, H, D, 1), _dense(B, Sk, H, D, 2), _dense(B, Sk, H, D, 3)
    do = _dense(B, Sq, H, D, 4)
    qd, kd, vd, dod = (_dev(t) for t in (q, k, v, do))
    out, lse = va.attention_fwd_dense(qd, kd, vd, causal=causal)
    dq, dk, dv = va.attention_bwd_dense(qd, kd, vd, out, dod, lse, causal=causal)
    assert va.varlen_attn_get_device_status() == 0
    cu_q, cu_k = [b * Sq for b in range(B + 1)], [b * Sk for b in range(B + 1)]
    pb = oracle.Problem(_packed(q), _packed(k), _packed(v), cu_q, cu_k, D ** -0.5, dout=_packed(do), causal=causal)
    rows, heads = oracle.all_pairs(B * Sq, H)
    krows, kheads = oracle.all_pairs(B * Sk, H)
    o_ref, lse_ref = pb.fwd(rows, heads)
    m = P.fwd_metrics(P.gather(out.reshape(B * Sq, H, D).cpu(), rows, heads),
                      lse.cpu().numpy()[heads, rows].astype(np.float64), o_ref, lse_ref)
    print("dense", D, causal, m)
    P.assert_fwd(m)
    dq_ref, _ = pb.bwd_q(rows, heads)
    dk_ref, dv_ref = pb.bwd_kv(krows, kheads)
    r = {"dq": P.rel_fro(P.gather(dq.reshape(B * Sq, H, D).cpu(), rows, heads), dq_ref),
         "dk": P.rel_fro(P.gather(dk.reshape(B * Sk, H, D).cpu(), krows, kheads), dk_ref),
         "dv": P.rel_fro(P.gather(dv.reshape(B * Sk, H, D).cpu(), krows, kheads), dv_ref)}
    print("dense", D, causal, r)
    assert all(x <= P.GRAD_REL_FRO for x in r.values()), r


def test_dense_bit_identical_to_packed():
    """Same data through the dense and the packed entry points: the same
    kernels on the same segments give the same bits (dQ up to reduction
    order, so it is compared with a tolerance)."""
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    B, Sq, Sk, H, D = 4, 200, 129, 2, 128
    q, k, v, do = (_dev(_dense(B, s, H, D, i)) for i, s in enumerate((Sq, Sk, Sk, Sq)))
    out_d, lse_d = va.attention_fwd_dense(q, k, v)
    dq_d, dk_d, dv_d = va.attention_bwd_dense(q, k, v, out_d, do, lse_d)
    cu_q = torch.arange(B + 1, dtype=torch.int32, device=DEV) * Sq
    cu_k = torch.arange(B + 1, dtype=torch.int32, device=DEV) * Sk
    pq, pk, pv, pdo = (_packed(t) for t in (q, k, v, do))
    out_p, lse_p = va.attention_fwd(pq, pk, pv, cu_q, cu_k)
    dq_p, dk_p, dv_p = va.attention_bwd(pq, pk, pv, out_p, pdo, lse_p, cu_q, cu_k)
    torch.cuda.synchronize()
    assert torch.equal(out_d.reshape(B * Sq, H, D), out_p) and torch.equal(lse_d, lse_p)
    assert torch.equal(dk_d.reshape(B * Sk, H, D), dk_p) and torch.equal(dv_d.reshape(B * Sk, H, D), dv_p)
    assert (dq_d.reshape(B * Sq, H, D).float() - dq_p.float()).abs().max().item() < 1e-2


@pytest.mark.parametrize("causal", [False, True], ids=["unmasked", "causal"])
def test_fp8_dense_matches_packed_fp8(causal):
    """varlen_attn_fwd_fp8_dense on [B, S, H, 128] (padded rows) returns the
    packed E4M3 call's bits on cu_seqlens = {0, S, 2S, ...} over the same
    memory (same kernels, segment bounds computed on the device), codes
    included; the packed E4M3 call is checked against the oracle in
    tests/test_fp8_gpu.py."""
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    B, Sq, Sk, H, D = 3, 200, 333, 2, 128
    q, k, v = _dense(B, Sq, H, D, 11), _dense(B, Sk, H, D, 12), _dense(B, Sk, H, D, 13)
    qd, kd, vd = (_dev(t) for t in (q, k, v))
    n = va.varlen_attn_fwd_fp8_dense_workspace_size(B, Sq, Sk, H, D)
    assert n == va.varlen_attn_fwd_fp8_workspace_size(B, B * Sq, B * Sk, H, D) > 0
    # zero-filled workspaces: the V^T columns between segment blocks and the
    # sections' alignment padding are neither written nor read, so they
    # compare equal only if they start equal
    ws, ws2 = (torch.zeros(n, dtype=torch.uint8, device=DEV) for _ in range(2))
    out, lse, _ = va.attention_fwd_fp8_dense(qd, kd, vd, causal=causal, workspace=ws)
    assert va.varlen_attn_get_device_status() == 0
    cu_q = torch.tensor([b * Sq for b in range(B + 1)], dtype=torch.int32, device=DEV)
    cu_k = torch.tensor([b * Sk for b in range(B + 1)], dtype=torch.int32, device=DEV)
    o2, l2, _ = va.attention_fwd_fp8(_packed(qd), _packed(kd), _packed(vd), cu_q, cu_k, causal=causal, workspace=ws2)
    assert va.varlen_attn_get_device_status() == 0
    assert torch.equal(out.reshape(B * Sq, H, D).cpu(), o2.cpu())
    assert torch.equal(lse.cpu(), l2.cpu())
    assert torch.equal(ws.cpu(), ws2.cpu())
    assert bool(torch.isfinite(out.float()).all())
