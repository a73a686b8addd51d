"""Failure detection without a GPU fault: a kernel whose bounded mbarrier wait
is never satisfied gives up after its budget, records a timeout in the
device error word and returns; the context stays usable."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    assert va.varlen_attn_get_device_status() == 0
    t0 = time.time()
    assert va.varlen_attn_selftest_wait_timeout(50_000_000) == 0  # 50 ms budget
    st = va.varlen_attn_get_device_status()
    assert st == va.VARLEN_ERR_TIMEOUT
    assert time.time() - t0 < 10
    # the error word is cleared by the read, and the context still works
    assert va.varlen_attn_get_device_status() == 0
    x = torch.ones(4, device="cuda")
    assert float((x * 2).sum()) == 8.0


def _case():
    from packed_variable_length_varlen_gb300 import workloads as W
    # CTA 0's first unit walks 6 kv tiles (12 K/V loads); its first kv tile 3 q steps
    return W.custom("skip", [300, 77], [700, 129], 2, 128)


def _fwd_call(va, w, d, out, lse):
    return va.varlen_attn_fwd(d.q, d.k, d.v, d.cu_q, d.cu_k, w.batch, w.total_q, w.total_k, w.num_heads,
                              w.head_dim, w.max_q(), w.max_k(), w.softmax_scale, out, lse)


@pytest.mark.parametrize("which", ["fwd", "bwd"])
def test_skipped_load_times_out_unwinds_and_context_survives(which):
    """A real kernel's bounded wait runs out: the forward's (or the
    backward's) producer in CTA 0 leaves one TMA load out, the waits for it
    give up after their 2 s budget, every role unwinds (producer drains its
    copies in flight, the MMA issuer its products, TMEM is freed) and the
    call reports VARLEN_ERR_TIMEOUT.  The next normal call on the same
    context then matches the oracle."""
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    from packed_variable_length_varlen_gb300 import workloads as W
    from tests import parity as P
    w = _case()
    cpu = W.make_inputs(w, 0)
    d = cpu.to("cuda")
    H, D = w.num_heads, w.head_dim
    out = torch.empty_like(d.q)
    lse = torch.empty(H, w.total_q, device="cuda")
    nb = va.varlen_attn_bwd_workspace_size(w.batch, w.total_q, H, D)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    grads = [torch.empty_like(d.q), torch.empty_like(d.k), torch.empty_like(d.v)]

    def bwd_call():
        return va.varlen_attn_bwd(d.q, d.k, d.v, out, d.dout, lse, d.cu_q, d.cu_k, w.batch, w.total_q, w.total_k,
                                  H, D, w.max_q(), w.max_k(), w.softmax_scale, *grads, ws, nb)

    assert va.varlen_attn_get_device_status() == 0
    if which == "bwd":
        assert _fwd_call(va, w, d, out, lse) == 0
        assert va.varlen_attn_get_device_status() == 0
    assert va.varlen_attn_debug_skip_load(0 if which == "fwd" else 1, 1) == 0
    try:
        t0 = time.time()
        assert (_fwd_call(va, w, d, out, lse) if which == "fwd" else bwd_call()) == 0
        st = va.varlen_attn_get_device_status()
        elapsed = time.time() - t0
    finally:
        va.varlen_attn_debug_skip_load(0, -1)
        va.varlen_attn_debug_skip_load(1, -1)
    assert st == va.VARLEN_ERR_TIMEOUT, va.varlen_attn_status_string(st)
    assert 1.5 < elapsed < 30
    assert va.varlen_attn_get_device_status() == 0
    # the same context runs the full path again, and it is right
    assert _fwd_call(va, w, d, out, lse) == 0
    assert bwd_call() == 0
    assert va.varlen_attn_get_device_status() == 0
    pb = P.oracle_problem(cpu)
    import oracle
    rows, heads = oracle.all_pairs(w.total_q, H)
    o_ref, lse_ref = pb.fwd(rows, heads)
    m = P.fwd_metrics(P.gather(out.cpu(), rows, heads), lse.cpu().numpy()[heads, rows].astype("float64"), o_ref,
                      lse_ref)
    P.assert_fwd(m)
    dq_ref, _ = pb.bwd_q(rows, heads)
    assert P.rel_fro(P.gather(grads[0].cpu(), rows, heads), dq_ref) <= P.GRAD_REL_FRO
    krows, kheads = oracle.all_pairs(w.total_k, H)
    dk_ref, dv_ref = pb.bwd_kv(krows, kheads)
    assert P.rel_fro(P.gather(grads[1].cpu(), krows, kheads), dk_ref) <= P.GRAD_REL_FRO
    assert P.rel_fro(P.gather(grads[2].cpu(), krows, kheads), dv_ref) <= P.GRAD_REL_FRO
