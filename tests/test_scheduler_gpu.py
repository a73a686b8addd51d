"""The device tile scheduler run on its own: every (segment, row-block, head)
tile is visited exactly once, by the CTA the static persistent order assigns,
in the longest-processing-time-first order of the segments, and the count
equals H * sum_b ceil(len_b / tile) -- 15680 for the windowed workload, the
valid-tile count printed on the "[FA4][SM120] ... >=4 varlen segments" issue
(section "Interpretation")."""
import json
import os
import pathlib

import numpy as np
import pytest
import torch

from packed_variable_length_varlen_gb300 import workloads as W

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_values.json")


def _lpt(cu):
    """The walk order of the segments: longest processing time first, by
    ceil(len / 128) descending (each tile of a segment iterates over 128-row
    steps of its length), ties by index; the index order for one segment."""
    B = len(cu) - 1
    cost = [-(-max(0, cu[b + 1] - cu[b]) // 128) for b in range(B)]
    return sorted(range(B), key=lambda b: (-cost[b], b)) if B > 1 else list(range(B))


def _expected(cu, H, tile):
    recs = []
    for b in _lpt(cu):
        n = -(-max(0, cu[b + 1] - cu[b]) // tile)
        for h in range(H):
            for m in range(n):
                recs.append((b, m, h))
    return recs


def _run(cu, H, tile, grid, guard=64):
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    cu = [int(c) for c in cu]
    B, total = len(cu) - 1, max(cu[-1], 0)
    exp = _expected(cu, H, tile)
    assert va.varlen_attn_tile_count(cu, B, total, H, tile) == len(exp)
    # cu_seqlens sits at the very end of a guarded buffer whose tail holds a
    # poison value: a read past index B would decode a huge segment.
    buf = torch.full((B + 1 + guard,), 1 << 30, dtype=torch.int32)
    buf[:B + 1] = torch.tensor(cu, dtype=torch.int32)
    dbuf = buf.cuda()
    n = max(len(exp), 1) + 4096
    out = torch.full((n, 4), -1, dtype=torch.int32, device="cuda")
    st = va.varlen_attn_debug_schedule(dbuf[:B + 1], B, total, H, tile, grid, out, n)
    assert st == 0
    assert va.varlen_attn_get_device_status() == 0
    got = out.cpu().numpy()
    recs = [tuple(r[:3]) for r in got[:len(exp)]]
    assert recs == exp
    assert np.all(got[len(exp):] == -1), "tiles visited past the exact count"
    ctas = got[:len(exp), 3]
    assert np.array_equal(ctas, np.arange(len(exp)) % grid)


def test_windowed_tile_count_pin():
    g = json.loads(pathlib.Path(GOLDEN).read_text())["windowed_tile_count"]
    _run(g["cu_seqlens_q"], g["num_heads"], g["tile_m"], 152)


@pytest.mark.parametrize("grid", [1, 7, 152, 1000])
def test_ragged_with_empty_segments(grid):
    lens = [0, 1, 127, 128, 129, 0, 0, 300, 5, 0, 0, 256, 257, 511]
    cu = [0] + list(np.cumsum(lens))
    _run(cu, 3, 256, grid)
    _run(cu, 3, 128, grid)
    _run(cu, 3, 64, grid)


def test_page_grid_sweep():
    """Segments x lengths like the synthetic W x S grid of the issue page
    (section "Bug 2 details"), at a few heads."""
    for nseg in (1, 3, 4, 8, 16):
        for S in (1024, 5040, 5140, 17580):
            for H in (8, 56):
                cu = [S * i for i in range(nseg + 1)]
                _run(cu, H, 128, 152)


def test_random_ragged():
    rng = np.random.default_rng(0)
    for _ in range(20):
        B = int(rng.integers(1, 40))
        lens = rng.integers(0, 700, size=B)
        lens[rng.random(B) < 0.2] = 0
        cu = [0] + list(np.cumsum(lens))
        _run(cu, int(rng.integers(1, 5)), int(rng.choice([64, 128, 256])), int(rng.integers(1, 300)))


def test_malformed_cu_is_clamped():
    """Decreasing or out-of-range entries are clamped into [0, total]: the
    schedule stays finite and in range."""
    from packed_variable_length_varlen_gb300 import varlen_attn as va
    cu = torch.tensor([0, 500, 100, 2 ** 30, -5, 260], dtype=torch.int32)
    total = 260
    n = va.varlen_attn_tile_count(cu.tolist(), 5, total, 2, 128)
    out = torch.full((n + 100, 4), -1, dtype=torch.int32, device="cuda")
    assert va.varlen_attn_debug_schedule(cu.cuda(), 5, total, 2, 128, 3, out, n + 100) == 0
    got = out.cpu().numpy()
    assert np.all(got[n:] == -1) and np.all(got[:n, 0] >= 0) and np.all(got[:n, 0] < 5)
    # clamped lengths 260, 0, 160, 0, 260: the walk takes segments 0, 4, 2
    segs = [int(b) for b in got[:n, 0]]
    assert [b for i, b in enumerate(segs) if i == 0 or segs[i - 1] != b] == [0, 4, 2]


def test_lpt_order_many_segments():
    """Hundreds of segments of mixed lengths: exact coverage in the LPT walk
    (the order table holds up to 4096 segments)."""
    rng = np.random.default_rng(5)
    lens = rng.integers(0, 3000, size=600)
    cu = [0] + list(np.cumsum(lens))
    _run(cu, 2, 128, 152)
