"""Two CPU ranks (gloo): the device-local re-layout equals a real exchange between processes.

The pages' Ulysses Anything path pads every rank's sequence shard for transport,
exchanges shards between ranks, trims each received shard to its true length
before concatenating ("[attention] Add Ulysses Anything backward", What does
this PR do), and restores the sequence-sharded layout with the inverse exchange.
Here two processes run that exchange with torch.distributed (gloo, all-gather of
the padded shards) and compare what each rank ends up holding with the oracle's
seq->head / head->seq permutations and key-mask assembly -- the same functions
the GPU re-layout kernels are checked against bit for bit.  The bench's
multi-rank helpers (barrier, max over ranks) run on the same process group.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle

P = 2
B, H, D = 2, 4, 8
LENS = (5, 4)  # uneven final shard, transport capacity 5
CAP = 5


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=P)
    try:
        rng = np.random.default_rng(7)
        N = sum(LENS)
        x = rng.standard_normal((B, N, H, D))
        mask = rng.random((B, N)) < 0.7
        shards = oracle.shard_sequence(x, LENS, CAP)  # (P, B, cap, H, D), zero padding
        hg = H // P

        # forward exchange: every rank contributes its padded shard, keeps head group `rank`
        gathered = [torch.empty((B, CAP, H, D), dtype=torch.float64) for _ in range(P)]
        dist.all_gather(gathered, torch.from_numpy(shards[rank]))
        group = np.concatenate([gathered[p].numpy()[:, :LENS[p], rank * hg:(rank + 1) * hg] for p in range(P)],
                               axis=1)
        want = oracle.seq_to_head(shards, LENS, CAP)[rank]
        assert np.array_equal(group, want)

        # inverse exchange: every rank contributes its head group, rebuilds its own padded shard
        groups = [torch.empty((B, N, hg, D), dtype=torch.float64) for _ in range(P)]
        dist.all_gather(groups, torch.from_numpy(np.ascontiguousarray(group)))
        off = sum(LENS[:rank])
        back = np.zeros((B, CAP, H, D))
        for g in range(P):
            back[:, :LENS[rank], g * hg:(g + 1) * hg] = groups[g].numpy()[:, off:off + LENS[rank]]
        assert np.array_equal(back, shards[rank])
        assert np.array_equal(back, oracle.head_to_seq(oracle.seq_to_head(shards, LENS, CAP), LENS, CAP)[rank])

        # key mask: gather the padded mask shards, trim each, concatenate
        msh = oracle.split_key_mask(mask, LENS, CAP)
        mg = [torch.empty((B, CAP), dtype=torch.uint8) for _ in range(P)]
        dist.all_gather(mg, torch.from_numpy(msh[rank].astype(np.uint8)))
        got = oracle.assemble_key_mask(np.stack([t.numpy() for t in mg]), LENS)
        assert np.array_equal(got.astype(bool), mask)
        untrimmed = oracle.assemble_key_mask_untrimmed(np.stack([t.numpy() for t in mg]))
        assert untrimmed.shape[1] != mask.shape[1]  # the defect the trim fixes

        # bench helpers on the same group: barrier, slowest-rank time
        import bench
        bench.barrier(P)
        assert bench.max_over_ranks(P, 1.0 + rank, device="cpu") == float(P)
    finally:
        dist.destroy_process_group()


def test_two_rank_exchange_matches_the_emulated_relayout():
    if not dist.is_available() or not dist.is_gloo_available():
        pytest.skip("torch.distributed with gloo is not available")
    mp.spawn(_worker, args=(_free_port(),), nprocs=P, join=True)
