"""Expert parallelism for the routed W4A16 MoE layer across the ranks of a
process group: each rank owns a contiguous range of the experts and the
tokens of its own batch; one all-to-all exchange each way moves the routed
rows to the experts' owners and the results back.

The layer's data path stays in the library's kernels (`LibraryOps`); this
module only plans the exchange on the host:

  1. route and permute the rank's own tokens: the permutation groups the
     assignments by expert, so the rows bound for each owner are one
     contiguous slice, and the expert histogram gives the send counts;
  2. exchange the per-expert counts of each owner's experts (a small
     all-to-all), then the rows themselves (all_to_all_single);
  3. regroup the received rows (source-major, expert-minor) by local expert
     with the permutation kernel itself, run the grouped expert FFN on the
     local experts, and undo the regrouping with the combine kernel at k = 1
     and weight 1 (an exact gather of bf16 rows);
  4. send the rows back in the order they came and combine them with the
     router weights in slot order.

"Performance and verification" (bloomery docs/performance.md), section "Why
it is fast": grouping a batch's tokens by expert is what lets each expert's
weights be read once per batch; here the grouping also decides what crosses
the wire.  The exchange needs one GPU per rank (NCCL); it is exercised on the
CPU with gloo and a stand-in for the kernels.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch
import torch.distributed as dist


@dataclass(frozen=True)
class ExpertShard:
    """Experts [lo(r), hi(r)) belong to rank r: lo(r) = r E // W."""
    E: int
    world: int
    rank: int

    def lo(self, r: int) -> int:
        return r * self.E // self.world

    def hi(self, r: int) -> int:
        return (r + 1) * self.E // self.world

    @property
    def n_local(self) -> int:
        return self.hi(self.rank) - self.lo(self.rank)

    @property
    def block(self) -> int:
        """Largest expert range of any rank (the width of the count exchange)."""
        return max(self.hi(r) - self.lo(r) for r in range(self.world))


def send_counts(counts, shard: ExpertShard) -> list[int]:
    """Rows this rank sends to each owner: its assignments per owner's experts."""
    c = [int(v) for v in counts]
    return [sum(c[shard.lo(r):shard.hi(r)]) for r in range(shard.world)]


def count_blocks(counts, shard: ExpertShard) -> torch.Tensor:
    """[world, block] int64: row r holds this rank's counts for owner r's
    experts, zero-padded to the widest range."""
    c = torch.as_tensor([int(v) for v in counts], dtype=torch.int64)
    out = torch.zeros((shard.world, shard.block), dtype=torch.int64)
    for r in range(shard.world):
        out[r, :shard.hi(r) - shard.lo(r)] = c[shard.lo(r):shard.hi(r)]
    return out


def received_local_ids(recv_blocks: torch.Tensor, n_local: int) -> torch.Tensor:
    """Local expert of every received row.  Rows arrive source by source, and
    each source's rows are grouped by expert in ascending order, so source s
    contributes recv_blocks[s, e] rows of local expert e, e = 0, 1, ..."""
    counts = recv_blocks[:, :n_local].reshape(-1)
    experts = torch.arange(n_local, dtype=torch.int32).repeat(recv_blocks.shape[0])
    return torch.repeat_interleave(experts, counts)


class LibraryOps:
    """The layer's steps through the library's C ABI (CUDA device tensors)."""

    def __init__(self, M=None):
        if M is None:
            import bit_quantized_expert_moe_gb300 as M
        self.M = M

    def route_topk(self, logits, k):
        return self.M.route_topk(logits, k)

    def permute(self, ids, E, x):
        out = self.M.permute(ids, E, x=x, want_x_perm=True)
        return out["counts"], out["offsets"], out["inv"], out["x_perm"]

    def expert_ffn(self, local_layer, x_local, offsets):
        return self.M.expert_ffn_w4a16(local_layer, x_local, offsets)

    def gather_rows(self, y, inv):
        ones = torch.ones((inv.numel(), 1), dtype=torch.float32, device=y.device)
        return self.M.combine(y, inv, ones)

    def combine(self, y_perm, inv, w):
        return self.M.combine(y_perm, inv, w)


def ep_layer_forward(ops, shard: ExpertShard, x, logits, k: int, local_layer, group=None):
    """The layer for this rank's tokens x [T, d] with router logits [T, E];
    `local_layer` holds the weights of experts [shard.lo(rank), shard.hi(rank)).
    Returns out [T, d] and the per-rank send and receive row counts."""
    T, d = x.shape
    ids, w = ops.route_topk(logits, k)
    counts, offsets, inv, x_perm = ops.permute(ids, shard.E, x)
    blocks = count_blocks(counts.cpu(), shard)
    send = [int(v) for v in blocks.sum(1)]
    rb = torch.empty(blocks.shape, dtype=blocks.dtype, device=x.device)
    _all_to_all(rb, blocks.to(x.device), None, None, group)
    recv_blocks = rb.cpu()
    recv = [int(v) for v in recv_blocks[:, :shard.n_local].sum(1)]
    x_recv = x_perm.new_empty((sum(recv), d))
    _all_to_all(x_recv, x_perm[:T * k], recv, send, group)
    local_ids = received_local_ids(recv_blocks, shard.n_local).to(x.device)
    if local_ids.numel():
        _, loc_offsets, loc_inv, x_local = ops.permute(local_ids.view(-1, 1), shard.n_local, x_recv)
        y_local = ops.expert_ffn(local_layer, x_local, loc_offsets)
        y_recv = ops.gather_rows(y_local, loc_inv)
    else:
        y_recv = x_recv.new_empty((0, d))
    y_perm = x_perm.new_empty((T * k, d))
    _all_to_all(y_perm, y_recv, send, recv, group)
    return ops.combine(y_perm, inv, w), send, recv


def _all_to_all(out, inp, out_splits, in_splits, group):
    """all_to_all_single with per-rank row counts (None: equal blocks)."""
    dist.all_to_all_single(out, inp, output_split_sizes=out_splits, input_split_sizes=in_splits, group=group)


def local_layer(layer, shard: ExpertShard):
    """The weights of this rank's experts as a layer of their own (views into
    the full layer's tensors, no copy; each expert's arrays stay 16-byte
    aligned because d_model and d_ff are multiples of 256)."""
    lo, hi = shard.lo(shard.rank), shard.hi(shard.rank)
    return type(layer)(E=hi - lo, d_model=layer.d_model, d_ff=layer.d_ff, w13_q=layer.w13_q[lo:hi],
                       w13_s=layer.w13_s[lo:hi], w13_z=layer.w13_z[lo:hi], w2_q=layer.w2_q[lo:hi],
                       w2_s=layer.w2_s[lo:hi], w2_z=layer.w2_z[lo:hi])
