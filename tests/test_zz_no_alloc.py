"""The allocation-free backward entry point (varlen_attn_bwd_noalloc), for
callers that cannot allocate device memory: it must give the same gradients
as varlen_attn_bwd with a caller-provided workspace, on two calls in a row
(the second call finds the first call's leftovers in the shared scratch
array), and refuse problems larger than its fixed scratch.  Collected last
so that a failure here never hides the other tests."""
import pytest
import torch

from packed_variable_length_varlen_gb300 import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _rel(a, b):
    return P.rel_fro(a.double().cpu().numpy(), b.double().cpu().numpy())


def test_noalloc_matches_workspace_entry_point_twice():
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    w = W.custom("noalloc", [300, 0, 129, 77, 1], [257, 5, 128, 0, 64], 4, 128)
    cpu = W.make_inputs(w, 0)
    d = cpu.to(DEV)
    H, D = w.num_heads, w.head_dim
    out = torch.empty_like(d.q)
    lse = torch.empty(H, w.total_q, dtype=torch.float32, device=DEV)
    P.run_fwd(d, out, lse)
    args = (d.q, d.k, d.v, out, d.dout, lse, d.cu_q, d.cu_k, w.batch, w.total_q, w.total_k, H, D, w.max_q(),
            w.max_k(), w.softmax_scale)
    nbytes = va.varlen_attn_bwd_workspace_size(w.batch, w.total_q, H, D)
    assert nbytes <= va.NOALLOC_SCRATCH_BYTES
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    ref = [torch.empty_like(d.q), torch.empty_like(d.k), torch.empty_like(d.v)]
    assert va.varlen_attn_bwd(*args, *ref, ws, nbytes) == 0
    assert va.varlen_attn_get_device_status() == 0
    for _ in range(2):
        got = [torch.full_like(d.q, float("nan")), torch.full_like(d.k, float("nan")),
               torch.full_like(d.v, float("nan"))]
        assert va.varlen_attn_bwd_noalloc(*args, *got) == 0
        assert va.varlen_attn_get_device_status() == 0
        for a, b in zip(got, ref):
            assert bool(torch.isfinite(a).all())
            assert _rel(a, b) <= P.GRAD_REL_FRO
        # dK and dV involve no atomics: identical bits
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])


def test_noalloc_refuses_problems_beyond_its_scratch():
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    big = 1 << 20  # rows: 16 heads x 96 dims needs far more than the fixed array
    assert va.varlen_attn_bwd_workspace_size(1, big, 16, 96) > va.NOALLOC_SCRATCH_BYTES
    st = va.varlen_attn_bwd_noalloc(None, None, None, None, None, None, None, None, 1, big, big, 16, 96, 0, 0,
                                    0.1, None, None, None)
    assert st == va.VARLEN_ERR_WORKSPACE
