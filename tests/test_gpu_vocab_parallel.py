"""Vocabulary tensor parallelism across processes ("Tensor Parallel": TP=1, 2
and 4 bit-identical).  Two and four processes share the one GPU; each holds
only its own shard of the vocabulary, computes its tiles' partials, exchanges
them with a bytes-only all_gather (gloo) and merges.  Every rank must return
the single-device forward's bits.  No kernel waits on another process."""
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, layout, out):
    import os

    import torch
    import torch.distributed as dist

    import invariant_token_log_gb300 as bil
    import workloads as wl
    from gpu_helpers import device_logits, f32_bits
    from invariant_token_log_gb300.vocab_parallel import vocab_parallel_logp
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    v, tile = 151936, 4096
    w = wl.random_rows(seed=31, n_rows=300, vocab=v, dtype="bfloat16", tile_v=tile, ignore_every=7)
    nt = -(-v // tile)
    if layout == "contiguous":
        b = [(r * nt) // world for r in range(world + 1)]
        lo, hi = b[rank], b[rank + 1]
    else:  # uneven ranges, ranks in reverse order of their tiles
        cuts = [0, 5, 20, 33, nt][: world + 1] if world == 4 else [0, 11, nt]
        k = world - 1 - rank
        lo, hi = cuts[k], cuts[k + 1]
    c0, c1 = lo * tile, min(hi * tile, v)
    shard = device_logits(np.ascontiguousarray(w.logits[:, c0:c1]), "bfloat16")   # this rank's memory only
    t = torch.from_numpy(w.target_ids).cuda()
    logp, lse, ent = vocab_parallel_logp(shard, t, v, lo, hi, tile, temperature=0.9, return_entropy=True)
    full = device_logits(w.logits, "bfloat16")
    ref = bil.logp_fwd(full, t, -100, tile, temperature=0.9, return_entropy=True)
    torch.cuda.synchronize()
    out[rank] = all(np.array_equal(f32_bits(a), f32_bits(b)) for a, b in zip((logp, lse, ent), ref))
    dist.destroy_process_group()


@pytest.mark.timeout(600)
@pytest.mark.parametrize("world,layout", [(2, "contiguous"), (4, "contiguous"), (2, "uneven"), (4, "uneven")])
def test_vocab_parallel_ranks_match_single_device_bits(world, layout):
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, _free_port(), layout, out), nprocs=world, start_method="spawn", join=True)
    assert [out[r] for r in range(world)] == [True] * world
