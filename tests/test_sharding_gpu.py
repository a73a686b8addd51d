"""The multi-GPU split of the packed problem, run through the kernels on one
GPU: every (segment, head) pair is independent, so a rank that passes its
head range as views ``t[:, h0:h1]`` (pointer offset h0 * head_stride, same
strides) with rows h0:h1 of lse, or its run of segments as row slices with
rebased cu_seqlens, computes exactly the unsharded call's values for its
slice.  The shards run one after another here (one GPU); together they
must reproduce the unsharded forward and backward: O, LSE, dK and dV bit for
bit, dQ within the tolerance its reduction order allows."""
import pytest
import torch

from packed_variable_length_varlen_gb300 import sharding as S
from packed_variable_length_varlen_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(va, w, q, k, v, dout, cu_q, cu_k, batch, total_q, total_k, H, out, lse, bwd=True, grads=None):
    D = w.head_dim
    mq = max(int(x) for x in torch.diff(cu_q.cpu()).tolist() + [0])
    mk = max(int(x) for x in torch.diff(cu_k.cpu()).tolist() + [0])
    assert va.varlen_attn_fwd(q, k, v, cu_q, cu_k, batch, total_q, total_k, H, D, mq, mk, w.softmax_scale,
                              out, lse) == 0
    if not bwd:
        return out, lse
    dq, dk, dv = grads
    nb = va.varlen_attn_bwd_workspace_size(batch, total_q, H, D)
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=DEV)
    assert va.varlen_attn_bwd(q, k, v, out, dout, lse, cu_q, cu_k, batch, total_q, total_k, H, D, mq, mk,
                              w.softmax_scale, dq, dk, dv, ws, nb) == 0
    return out, lse


def _full(va, w, d):
    H = w.num_heads
    out = torch.empty_like(d.q)
    lse = torch.empty(H, w.total_q, device=DEV)
    grads = (torch.empty_like(d.q), torch.empty_like(d.k), torch.empty_like(d.v))
    _run(va, w, d.q, d.k, d.v, d.dout, d.cu_q, d.cu_k, w.batch, w.total_q, w.total_k, H, out, lse, True, grads)
    assert va.varlen_attn_get_device_status() == 0
    return out, lse, grads


def _dq_close(a, b):
    a, b = a.double(), b.double()
    assert float((a - b).norm() / max(float(b.norm()), 1e-30)) <= 1e-3


@pytest.mark.parametrize("D", [64, 128])
def test_head_shards_reproduce_the_unsharded_call(D):
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    w = W.custom("shard_heads", [300, 0, 129, 517, 1], [257, 5, 300, 517, 64], 6, D)
    d = W.make_inputs(w, 0).to(DEV)
    out, lse, (dq, dk, dv) = _full(va, w, d)
    for world in (2, 3, 4):
        o2, l2 = torch.full_like(out, float("nan")), torch.full_like(lse, float("nan"))
        g2 = [torch.full_like(t, float("nan")) for t in (dq, dk, dv)]
        for rank in range(world):
            h0, h1 = S.head_range(w.num_heads, world, rank)
            if h1 == h0:
                continue
            sl = slice(h0, h1)
            _run(va, w, d.q[:, sl], d.k[:, sl], d.v[:, sl], d.dout[:, sl], d.cu_q, d.cu_k, w.batch, w.total_q,
                 w.total_k, h1 - h0, o2[:, sl], l2[sl], True, [g[:, sl] for g in g2])
            assert va.varlen_attn_get_device_status() == 0
        assert torch.equal(o2, out) and torch.equal(l2, lse), world
        assert torch.equal(g2[1], dk) and torch.equal(g2[2], dv), world
        _dq_close(g2[0], dq)


def test_segment_shards_reproduce_the_unsharded_call():
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    w = W.custom("shard_segs", [300, 0, 129, 517, 1, 77], [257, 5, 300, 517, 64, 0], 3, 128)
    d = W.make_inputs(w, 0).to(DEV)
    out, lse, (dq, dk, dv) = _full(va, w, d)
    for world in (2, 3, 4):
        o2, l2 = torch.full_like(out, float("nan")), torch.full_like(lse, float("nan"))
        g2 = [torch.full_like(t, float("nan")) for t in (dq, dk, dv)]
        for rank in range(world):
            sh = S.segment_range(w.cu_q, w.cu_k, world, rank)
            if sh.empty:
                continue
            qs, ks = slice(sh.q0, sh.q1), slice(sh.k0, sh.k1)
            cu_q = torch.tensor(sh.cu_q, dtype=torch.int32, device=DEV)
            cu_k = torch.tensor(sh.cu_k, dtype=torch.int32, device=DEV)
            tq, tk = sh.q1 - sh.q0, sh.k1 - sh.k0
            # lse of a shard is [H, its q rows]: computed into its own buffer, then placed
            lse_sh = torch.empty(w.num_heads, tq, device=DEV)
            _run(va, w, d.q[qs], d.k[ks], d.v[ks], d.dout[qs], cu_q, cu_k, sh.b1 - sh.b0, tq, tk, w.num_heads,
                 o2[qs], lse_sh, True, [g2[0][qs], g2[1][ks], g2[2][ks]])
            assert va.varlen_attn_get_device_status() == 0
            l2[:, qs] = lse_sh
        assert torch.equal(o2, out) and torch.equal(l2, lse), world
        assert torch.equal(g2[1], dk) and torch.equal(g2[2], dv), world
        _dq_close(g2[0], dq)


@pytest.mark.parametrize("causal", [False, True], ids=["unmasked", "causal"])
def test_fp8_shards_reproduce_the_unsharded_call(causal):
    """The E4M3 forward split by heads (views t[:, h0:h1], lse rows h0:h1) and
    by segments (row slices, rebased cu_seqlens): each shard quantises its
    own (segment, head) blocks, whose descales depend on nothing else, so
    together the shards reproduce the unsharded O and LSE bit for bit."""
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    w = W.custom("shard_fp8", [300, 0, 129, 517, 1, 77], [257, 5, 300, 517, 64, 0], 4, 128)
    H = w.num_heads
    d = W.make_inputs(w, 0, with_dout=False).to(DEV)
    out, lse, _ = va.attention_fwd_fp8(d.q, d.k, d.v, d.cu_q, d.cu_k, w.softmax_scale, causal=causal)
    assert va.varlen_attn_get_device_status() == 0
    for world in (2, 4):
        o2, l2 = torch.full_like(out, float("nan")), torch.full_like(lse, float("nan"))
        for rank in range(world):
            h0, h1 = S.head_range(H, world, rank)
            if h1 == h0:
                continue
            sl = slice(h0, h1)
            va.attention_fwd_fp8(d.q[:, sl], d.k[:, sl], d.v[:, sl], d.cu_q, d.cu_k, w.softmax_scale, out=o2[:, sl],
                                 lse=l2[sl], causal=causal)
            assert va.varlen_attn_get_device_status() == 0
        assert torch.equal(o2, out) and torch.equal(l2, lse), ("heads", world)
    for world in (2, 3):
        o2, l2 = torch.full_like(out, float("nan")), torch.full_like(lse, float("nan"))
        for rank in range(world):
            sh = S.segment_range(w.cu_q, w.cu_k, world, rank)
            if sh.empty:
                continue
            qs, ks = slice(sh.q0, sh.q1), slice(sh.k0, sh.k1)
            cu_q = torch.tensor(sh.cu_q, dtype=torch.int32, device=DEV)
            cu_k = torch.tensor(sh.cu_k, dtype=torch.int32, device=DEV)
            lse_sh = torch.empty(H, sh.q1 - sh.q0, device=DEV)
            va.attention_fwd_fp8(d.q[qs], d.k[ks], d.v[ks], cu_q, cu_k, w.softmax_scale, out=o2[qs], lse=lse_sh,
                                 causal=causal)
            assert va.varlen_attn_get_device_status() == 0
            l2[:, qs] = lse_sh
        assert torch.equal(o2, out) and torch.equal(l2, lse), ("segments", world)
