"""Small cases for the bounds-checking build (shared by
tests/test_bounds_gpu.py and the child process it starts with
VARLEN_ATTN_LIB pointing at that build).  Every entry point's kernels run on
ragged, padded and strided layouts; ``run_cases`` returns the outputs and the
device status after each call.

    python -m tests.bounds_cases OUT.pt   # run with the library the binding loads
"""
from __future__ import annotations

import sys

import torch

from packed_variable_length_varlen_gb300 import workloads as W

DEV = "cuda"

CASES = {
    # name: (seqlens_q, seqlens_k, H, D, extra workload arguments)
    "ragged_d64": ([0, 1, 127, 128, 129, 300, 0, 517, 3, 65], [5, 0, 200, 128, 1, 700, 40, 517, 1000, 64], 2, 64, {}),
    "ragged_d96": ([0, 1, 127, 129, 300, 3], [5, 0, 200, 1, 700, 1000], 2, 96, {}),
    "padded_d128": ([130, 70, 5, 200], [129, 61, 40, 0], 2, 128, {"row_pad": 64}),
    "strided_dout": ([253, 186], [253, 186], 4, 96, {"dout_row_stride": 9728, "amplitude": 0.1,
                                                      "dout_amplitude": 0.1}),
}


def run_cases(va) -> dict:
    res = {"bounds_checked": va.varlen_attn_bounds_checked()}
    for name, (sq, sk, H, D, kw) in CASES.items():
        w = W.custom(name, sq, sk, H, D, **kw)
        d = W.make_inputs(w, 0).to(DEV)
        out = W.output_like(w, "out", DEV)
        lse = torch.full((H, w.total_q), 777.0, device=DEV)
        grads = [W.output_like(w, n, DEV) for n in ("dq", "dk", "dv")]
        nb = va.varlen_attn_bwd_workspace_size(w.batch, w.total_q, H, D)
        ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=DEV)
        for mask, kwm in (("none", {}), ("causal", {"causal": True}), ("window", {"window": (40, 7)})):
            for det in (False, True):
                st = va.varlen_attn_fwd(d.q, d.k, d.v, d.cu_q, d.cu_k, w.batch, w.total_q, w.total_k, H, D,
                                        w.max_q(), w.max_k(), w.softmax_scale, out, lse, **kwm)
                st2 = va.varlen_attn_get_device_status()
                st3 = va.varlen_attn_bwd(d.q, d.k, d.v, out, d.dout, lse, d.cu_q, d.cu_k, w.batch, w.total_q,
                                         w.total_k, H, D, w.max_q(), w.max_k(), w.softmax_scale, *grads, ws, nb,
                                         deterministic=det, **kwm)
                st4 = va.varlen_attn_get_device_status()
                key = "%s/%s/%s" % (name, mask, "det" if det else "atomic")
                res[key] = {"status": (st, st2, st3, st4), "out": out.clone().cpu(), "lse": lse.clone().cpu(),
                            "dq": grads[0].clone().cpu(), "dk": grads[1].clone().cpu(),
                            "dv": grads[2].clone().cpu()}
    # the E4M3 forward (head size 128)
    w = W.custom("fp8", [130, 70, 5, 200], [129, 61, 40, 0], 2, 128, row_pad=64)
    d = W.make_inputs(w, 0, with_dout=False).to(DEV)
    out = W.output_like(w, "out", DEV)
    lse = torch.full((2, w.total_q), 777.0, device=DEV)
    nb = va.varlen_attn_fwd_fp8_workspace_size(w.batch, w.total_q, w.total_k, 2, 128)
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
    for mask, kwm in (("none", {}), ("causal", {"causal": True}), ("window", {"window": (40, 7)})):
        st = va.varlen_attn_fwd_fp8(d.q, d.k, d.v, d.cu_q, d.cu_k, w.batch, w.total_q, w.total_k, 2, 128,
                                    w.max_q(), w.max_k(), w.softmax_scale, out, lse, ws, nb, **kwm)
        res["fp8" if mask == "none" else "fp8/" + mask] = {
            "status": (st, va.varlen_attn_get_device_status()), "out": out.clone().cpu(), "lse": lse.clone().cpu()}
    # the dense batched E4M3 forward (uniform segments, bounds computed on the device), rows padded
    B, Sq, Sk, H = 2, 130, 77, 2
    w = W.custom("fp8_dense", [Sq] * B, [Sk] * B, H, 128, row_pad=32)
    d = W.make_inputs(w, 1, with_dout=False).to(DEV)
    out = W.output_like(w, "out", DEV)
    lse = torch.full((H, w.total_q), 777.0, device=DEV)
    nb = va.varlen_attn_fwd_fp8_dense_workspace_size(B, Sq, Sk, H, 128)
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV)

    def as4(t, S):
        return t.as_strided((B, S, H, 128), (S * t.stride(0), t.stride(0), t.stride(1), 1), t.storage_offset())

    for causal in (0, 1):
        st = va.varlen_attn_fwd_fp8_dense(as4(d.q, Sq), as4(d.k, Sk), as4(d.v, Sk), B, Sq, Sk, H, 128,
                                          w.softmax_scale, causal, as4(out, Sq), lse, ws, nb)
        res["fp8_dense/%d" % causal] = {"status": (st, va.varlen_attn_get_device_status()),
                                        "out": out.clone().cpu(), "lse": lse.clone().cpu()}
    # the checker's self test: extents 16 bytes short make the last accesses fail
    w = W.custom("slack", [70], [90], 2, 64)
    d = W.make_inputs(w, 0).to(DEV)
    out = W.output_like(w, "out", DEV)
    lse = torch.empty(2, w.total_q, device=DEV)
    va.varlen_attn_debug_set_span_slack(16)
    try:
        st = va.varlen_attn_fwd(d.q, d.k, d.v, d.cu_q, d.cu_k, w.batch, w.total_q, w.total_k, 2, 64, w.max_q(),
                                w.max_k(), w.softmax_scale, out, lse)
        res["slack"] = {"status": (st, va.varlen_attn_get_device_status())}
    finally:
        va.varlen_attn_debug_set_span_slack(0)
    res["after_slack"] = va.varlen_attn_get_device_status()
    return res


if __name__ == "__main__":
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    torch.save(run_cases(va), sys.argv[1])
