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


def test_noalloc_scratch_address_follows_the_context():
    """The scratch array's device address belongs to a CUDA context.  With a
    second context made current on the same device, the address the next
    call would use is looked up in that context (its identity is the new
    context's); back in the first context, the first context's address is
    used again.  Nothing is launched in the second context."""
    import ctypes
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    torch.zeros(1, device=DEV)
    torch.cuda.synchronize()
    cuda = ctypes.CDLL("libcuda.so.1")

    def ctx_id(ctx):
        v = ctypes.c_ulonglong(0)
        assert cuda.cuCtxGetId(ctx, ctypes.byref(v)) == 0
        return v.value

    st, a0, c0 = va.varlen_attn_debug_noalloc_scratch()
    assert st == 0 and a0 != 0
    cur = ctypes.c_void_p()
    assert cuda.cuCtxGetCurrent(ctypes.byref(cur)) == 0 and cur.value
    assert c0 == ctx_id(cur)
    dev = ctypes.c_int(0)
    assert cuda.cuCtxGetDevice(ctypes.byref(dev)) == 0
    params = ctypes.create_string_buffer(64)  # CUctxCreateParams, all fields null
    new = ctypes.c_void_p()
    assert cuda.cuCtxCreate_v4(ctypes.byref(new), params, 0, dev) == 0  # made current
    try:
        st, a1, c1 = va.varlen_attn_debug_noalloc_scratch()
        assert st == 0 and a1 != 0
        assert c1 == ctx_id(new) and c1 != c0
    finally:
        popped = ctypes.c_void_p()
        assert cuda.cuCtxPopCurrent_v2(ctypes.byref(popped)) == 0
        assert cuda.cuCtxDestroy_v2(new) == 0
    st, a2, c2 = va.varlen_attn_debug_noalloc_scratch()
    assert st == 0 and (a2, c2) == (a0, c0)
