"""Splitting packed variable-length attention across GPUs.

Every (segment, head) pair of packed attention is independent in both the
forward and the backward, so the work splits across ranks with no exchange
of data:

* by heads: every rank passes the same cu_seqlens and, for each of q, k, v,
  out, dout, dq, dk, dv, the view ``t[:, h0:h1]`` (same strides, pointer
  offset h0 * head_stride), with num_heads = h1 - h0 and the rows h0:h1 of
  lse;
* by segments: a rank takes a contiguous run of segments [b0, b1), the
  packed rows they own (``t[q0:q1]``, ``t[k0:k1]``) and cu_seqlens rebased to
  start at 0.

Either way the outputs land in disjoint slices, so no collective is needed;
the only cross-rank operation of a benchmark is the max of the ranks' step
times (``max_over_ranks``).

A shard can be empty: more ranks than heads (``head_range`` gives h0 == h1)
or than segments, or one segment holding most of the cost
(``SegmentShard.empty``).  The library refuses num_heads = 0 and batch = 0
(VARLEN_ERR_SHAPE), so a rank with an empty shard has no call to make: it
skips the work and still takes part in ``max_over_ranks``.
"""
from dataclasses import dataclass
from typing import List, Sequence, Tuple


def head_range(num_heads: int, world: int, rank: int) -> Tuple[int, int]:
    """Contiguous heads [h0, h1) of `rank`; sizes differ by at most one.
    With world > num_heads some ranks get h0 == h1 (nothing to launch)."""
    if world < 1 or not 0 <= rank < world or num_heads < 0:
        raise ValueError("bad world / rank / num_heads")
    base, extra = divmod(num_heads, world)
    h0 = rank * base + min(rank, extra)
    return h0, h0 + base + (1 if rank < extra else 0)


@dataclass
class SegmentShard:
    b0: int            # segments [b0, b1)
    b1: int
    q0: int            # packed q rows [q0, q1)
    q1: int
    k0: int            # packed k / v rows [k0, k1)
    k1: int
    cu_q: List[int]    # cu_seqlens of the shard, starting at 0
    cu_k: List[int]

    @property
    def empty(self) -> bool:
        """No segment: the rank has nothing to launch (batch would be 0)."""
        return self.b1 <= self.b0


def segment_cost(sq: int, sk: int) -> float:
    """Relative work of one segment: the attention products scale with
    Sq * Sk; the Sq + Sk term accounts for the per-row reads and writes (and
    keeps segments without queries or keys from costing nothing)."""
    return float(sq) * float(sk) + float(sq) + float(sk)


def segment_range(cu_q: Sequence[int], cu_k: Sequence[int], world: int, rank: int) -> SegmentShard:
    """Contiguous segments of `rank`, split where the running cost crosses
    rank / world of the total (so every rank's share is within one segment's
    cost of total / world).  cu_seqlens must be non-decreasing."""
    cu_q, cu_k = [int(x) for x in cu_q], [int(x) for x in cu_k]
    if len(cu_q) != len(cu_k) or len(cu_q) < 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k need batch + 1 entries each")
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world / rank")
    if any(b < a for a, b in zip(cu_q, cu_q[1:])) or any(b < a for a, b in zip(cu_k, cu_k[1:])):
        raise ValueError("cu_seqlens must be non-decreasing to split by segments")
    B = len(cu_q) - 1
    cost = [segment_cost(cu_q[b + 1] - cu_q[b], cu_k[b + 1] - cu_k[b]) for b in range(B)]
    total = sum(cost)

    def boundary(r: int) -> int:
        # first segment index whose prefix cost reaches r / world of the total
        if r <= 0:
            return 0
        if r >= world:
            return B
        target, acc = total * r / world, 0.0
        for b in range(B):
            if acc >= target:
                return b
            acc += cost[b]
        return B

    b0, b1 = boundary(rank), boundary(rank + 1)
    return SegmentShard(b0, b1, cu_q[b0], cu_q[b1], cu_k[b0], cu_k[b1],
                        [x - cu_q[b0] for x in cu_q[b0:b1 + 1]], [x - cu_k[b0] for x in cu_k[b0:b1 + 1]])


def max_over_ranks(x: float, group=None) -> float:
    """The maximum of `x` over the ranks of `group` (x itself without a
    process group).  Runs on the backend's device: CPU for gloo, the current
    GPU for nccl."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size(group) == 1:
        return float(x)
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())
