"""Expert parallelism (bit_quantized_expert_moe_gb300/ep.py) on the CPU with
gloo ranks: the exchange plan, and the whole layer split over 2 ranks (experts
7 = 3 + 4, each rank with its own tokens) against the oracle's single-process
layer.  The kernel steps are stood in for by the oracle here (no GPU); the
GPU path runs the same plan through the library (LibraryOps) and is not
measured on hardware (one GPU per box)."""
import os
import socket

import numpy as np
import pytest

import moe_synth as S
from bit_quantized_expert_moe_gb300 import ep


def test_shard_ranges_and_count_blocks():
    torch = pytest.importorskip("torch")
    sh = ep.ExpertShard(E=7, world=2, rank=0)
    assert [(sh.lo(r), sh.hi(r)) for r in range(2)] == [(0, 3), (3, 7)] and sh.block == 4
    counts = [5, 0, 2, 1, 3, 0, 4]
    assert ep.send_counts(counts, sh) == [7, 8]
    b = ep.count_blocks(counts, sh)
    assert b.tolist() == [[5, 0, 2, 0], [1, 3, 0, 4]]
    # rows received by rank 1 from two sources, source-major then expert-minor
    recv = torch.tensor([[1, 3, 0, 4], [2, 0, 1, 0]])
    ids = ep.received_local_ids(recv, 4)
    assert ids.tolist() == [0, 1, 1, 1, 3, 3, 3, 3, 0, 0, 2]


class _OracleOps:
    """The layer's steps on the CPU, from the oracle (fp64), on torch tensors."""

    def __init__(self, d, f):
        from oracle import moe_oracle as OM
        self.OM, self.d, self.f = OM, d, f

    def route_topk(self, logits, k):
        ids, w = self.OM.route_topk(logits.numpy(), k)
        return torch_from(ids), torch_from(w)

    def permute(self, ids, E, x):
        counts, offsets, sorted_, inv = self.OM.permute(ids.numpy(), E)
        kk = ids.shape[1]
        return torch_from(counts), torch_from(offsets), torch_from(inv), x[torch_from(sorted_ // kk).long()]

    def expert_ffn(self, getter, x_local, offsets):
        return torch_from(self.OM.expert_ffn(x_local.numpy(), offsets.numpy(), getter, self.d, self.f))

    def gather_rows(self, y, inv):
        return y[inv.long()]

    def combine(self, y_perm, inv, w):
        T, k = w.shape
        return torch_from(self.OM.combine(y_perm.numpy(), inv.numpy(), w.numpy(), T, k))


def torch_from(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


CFG = dict(T=9, d=256, f=512, E=7, k=2)


def _rank(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.join(os.path.dirname(__file__), ".."))
    import torch
    import torch.distributed as dist
    from oracle import moe_oracle as OM
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = S.custom("ep", cfg_id=60, **CFG)
        W = S.layer_weights(cfg, 0)                    # the same layer on every rank
        mine = S.custom("ep", cfg_id=61 + rank, **CFG)  # each rank's own tokens
        x_bits, lg = S.activations(mine), S.router_logits(mine)
        sh = ep.ExpertShard(E=cfg.E, world=world, rank=rank)
        lo = sh.lo(rank)
        getter = lambda e: {key: v[lo + e] for key, v in W.items()}  # noqa: E731
        x = torch.from_numpy(OM.bf16_bits_to_f64(x_bits))
        out, send, recv = ep.ep_layer_forward(_OracleOps(cfg.d, cfg.f), sh, x, torch.from_numpy(lg), cfg.k, getter)
        ref = OM.layer_forward(x_bits, lg, lambda e: {key: v[e] for key, v in W.items()}, cfg.E, cfg.d, cfg.f, cfg.k)
        q.put((rank, float(np.abs(out.numpy() - ref).max() / np.abs(ref).max()), send, recv))
    finally:
        dist.destroy_process_group()


def test_two_rank_expert_parallel_layer_matches_the_oracle():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, rel, send, recv in got:
        assert rel < 1e-12, (rank, rel)
        assert sum(send) == CFG["T"] * CFG["k"]       # every assignment leaves once
    # what rank a sends to rank b is what b receives from a
    (_, _, s0, r0), (_, _, s1, r1) = got
    assert s0[1] == r1[0] and s1[0] == r0[1] and s0[0] == r0[0] and s1[1] == r1[1]
