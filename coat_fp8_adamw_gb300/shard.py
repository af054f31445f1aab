"""Data-parallel sharding of the flat optimizer state (ZeRO / FSDP layout)
and the sharded step that follows the gradient reduce-scatter.

COAT's optimizer states are quantized per group and the expansion needs no
statistic wider than one group (COAT review page, section 4, table of
FP8 methods: the FSDP row).  A rank can therefore own a group-aligned slice of
w, m, v and the group records and step it alone; the only exchange is the
gradient reduce-scatter that hands each rank the summed gradient of its slice.

Layout (bucket-interleaved, like FSDP's per-layer flat parameters).  The flat
buffer of n parameters is padded to ``buckets * world * cap`` elements.
Bucket b covers global indices ``[b * world * cap, (b + 1) * world * cap)`` and
gives rank r the piece ``[b * world * cap + r * cap, ... + cap)``; a rank's
local state is its pieces of every bucket, back to back (``buckets * cap``
elements).  ``cap`` is a multiple of ``max(G, 16)``, so every piece holds whole
groups and every piece's w, g, m, v and group-record pointers stay 16-byte
aligned.  With one bucket this is the plain contiguous split.

The padding is zeros (w = g = 0, codes 0x00, records (0, 1, 0, 1)).  A zero
element stays zero through the step, and the group statistics ignore it (the
group minimum runs over non-zero magnitudes), so a padded group steps its real
elements exactly as the unpadded ragged group does.

A gradient bucket is one contiguous slice of the padded flat gradient, so its
reduce-scatter needs no gather: the collective of bucket b+1 runs while the
step kernel works on bucket b.  This module is host-side orchestration only:
the step is whatever callable the caller passes (the library's
``coat_fp8_adamw_step`` on a GPU), and the collective is torch.distributed's.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, Optional, Sequence


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


@dataclass(frozen=True)
class ShardLayout:
    """Where each rank's slice of an ``n``-parameter flat state lives."""

    n: int
    G: int
    world: int
    buckets: int = 1

    def __post_init__(self):
        if self.n < 1 or self.world < 1 or self.buckets < 1:
            raise ValueError("n, world and buckets must be positive")
        if self.G < 1 or self.G > 256 or self.G & (self.G - 1):
            raise ValueError("G must be a power of two in [1, 256]")

    @property
    def unit(self) -> int:
        """Piece granularity: whole groups and 16-byte aligned code buffers."""
        return max(self.G, 16)

    @property
    def cap(self) -> int:
        """Elements of one rank's piece of one bucket."""
        return _ceil_div(_ceil_div(self.n, self.buckets * self.world), self.unit) * self.unit

    @property
    def padded(self) -> int:
        """Length of the padded flat buffers (w, g, m, v)."""
        return self.buckets * self.world * self.cap

    @property
    def local(self) -> int:
        """Elements of one rank's local state."""
        return self.buckets * self.cap

    def bucket(self, b: int) -> slice:
        """Global (padded) index range of bucket b, the input of its reduce-scatter."""
        span = self.world * self.cap
        return slice(b * span, (b + 1) * span)

    def piece(self, rank: int, b: int) -> slice:
        """Global (padded) index range of rank ``rank``'s piece of bucket b."""
        lo = b * self.world * self.cap + rank * self.cap
        return slice(lo, lo + self.cap)

    def local_piece(self, b: int) -> slice:
        """Local index range of bucket b's piece."""
        return slice(b * self.cap, (b + 1) * self.cap)

    def groups(self, s: slice) -> slice:
        """Group-record rows of an element range whose ends are piece boundaries."""
        return slice(s.start // self.G, s.stop // self.G)

    def real(self, rank: int, b: int) -> int:
        """Elements of rank's piece of bucket b that are real parameters (< n)."""
        p = self.piece(rank, b)
        return max(0, min(p.stop, self.n) - p.start)


def to_local(x_padded, layout: ShardLayout, rank: int, per_group: bool = False):
    """Rank's local slice of a padded flat tensor (or of the group records when
    ``per_group``): its pieces of every bucket, concatenated.  Used to lay out
    the state once, not on the step's path."""
    import torch
    sl = [layout.piece(rank, b) for b in range(layout.buckets)]
    if per_group:
        sl = [layout.groups(s) for s in sl]
    return torch.cat([x_padded[s] for s in sl]).contiguous()


def from_locals(locals_: Sequence, layout: ShardLayout, per_group: bool = False):
    """The padded flat tensor rebuilt from every rank's local slice."""
    import torch
    first = locals_[0]
    rows = layout.padded // layout.G if per_group else layout.padded
    out = torch.empty((rows,) + tuple(first.shape[1:]), dtype=first.dtype, device=first.device)
    for r, loc in enumerate(locals_):
        for b in range(layout.buckets):
            g, l = layout.piece(r, b), layout.local_piece(b)
            if per_group:
                g, l = layout.groups(g), layout.groups(l)
            out[g] = loc[l]
    return out


def sharded_step(step: Callable, layout: ShardLayout, rank: int, w, m_q, v_q, meta, g_padded,
                 g_local, beta1: float, beta2: float, lr: float, eps: float,
                 weight_decay: float, t: int, group=None) -> None:
    """One data-parallel step on this rank's slice.

    ``g_padded`` is this rank's own (unreduced) gradient over the padded flat
    buffer; ``g_local`` (``layout.local`` elements) receives the reduce-scatter
    (SUM) of every rank's gradient for this rank's pieces.  All bucket
    collectives are issued asynchronously first; the step of bucket b runs as
    soon as bucket b's collective has completed (on a GPU, ``wait`` orders the
    current stream after the collective, so later buckets' transfers overlap
    earlier buckets' steps).  w, m_q, v_q (``layout.local`` elements) and meta
    (``layout.local // G`` records) are updated in place.  A caller that wants
    the mean gradient scales its loss by 1 / world.
    """
    import torch.distributed as dist
    works = []
    for b in range(layout.buckets):
        works.append(dist.reduce_scatter_tensor(g_local[layout.local_piece(b)],
                                                g_padded[layout.bucket(b)],
                                                op=dist.ReduceOp.SUM, group=group,
                                                async_op=True))
    for b, work in enumerate(works):
        work.wait()
        s = layout.local_piece(b)
        step(w[s], g_local[s], m_q[s], v_q[s], meta[layout.groups(s)], layout.G, beta1, beta2,
             lr, eps, weight_decay, t)


def all_gather_padded(x_local, layout: ShardLayout, group=None, per_group: bool = False,
                      out: Optional[object] = None):
    """The padded flat tensor from every rank's local slice, by one all-gather
    per bucket (e.g. the updated weights for the next forward pass)."""
    import torch
    import torch.distributed as dist
    rows = layout.padded // layout.G if per_group else layout.padded
    if out is None:
        out = torch.empty((rows,) + tuple(x_local.shape[1:]), dtype=x_local.dtype,
                          device=x_local.device)
    for b in range(layout.buckets):
        src, dst = layout.local_piece(b), layout.bucket(b)
        if per_group:
            src, dst = layout.groups(src), layout.groups(dst)
        dist.all_gather_into_tensor(out[dst], x_local[src].contiguous(), group=group)
    return out
