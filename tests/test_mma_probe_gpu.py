"""The tcgen05 issue-rate probe (varlen_attn_debug_mma_cycles) runs on every
shape and issue form it accepts, completes within its bounded wait and
reports a cycle count; one M=128 K=16 bf16 MMA cannot take fewer cycles than
the tensor core's dense rate allows (8192 flops per cycle per SM would put
N=128 at 64 cycles)."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("n_cols", [64, 128, 256])
def test_mma_probe_runs(mode, n_cols):
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    cyc = torch.zeros(1, dtype=torch.int64, device="cuda")
    st = va.varlen_attn_debug_mma_cycles(256, n_cols, mode, cyc)
    assert st == 0, va.varlen_attn_status_string(st)
    torch.cuda.synchronize()
    assert va.varlen_attn_get_device_status() == 0
    per = int(cyc.item()) / 256
    assert per >= 2 * 128 * n_cols * 16 / 16384 - 1e-9, per   # not above twice the dense bf16 rate
    assert per < 1e5, per
