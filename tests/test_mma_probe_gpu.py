"""The tcgen05 issue-rate probe (varlen_attn_debug_mma_cycles) runs on every
shape and issue form it accepts, completes within its bounded wait and
reports a cycle count; one M=128 K=16 bf16 MMA cannot take fewer cycles than
the tensor core's dense rate allows (8192 flops per cycle per SM would put
N=128 at 64 cycles)."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode,n_cols", [(m, n) for m in (0, 1, 2) for n in (64, 128, 256)] + [(5, 64), (5, 128), (6, 128), (7, 128)])
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


@pytest.mark.parametrize("mode", [3, 4])
def test_tmem_traffic_probe_runs(mode):
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    cyc = torch.zeros(1, dtype=torch.int64, device="cuda")
    st = va.varlen_attn_debug_mma_cycles(256, 128, mode, cyc)
    assert st == 0, va.varlen_attn_status_string(st)
    torch.cuda.synchronize()
    assert va.varlen_attn_get_device_status() == 0
    assert 0 < int(cyc.item()) < 256 * 100000
