"""Host logic of the vocabulary-parallel forward on two gloo CPU ranks: the
exchange of tile ranges, the assembly of the [N, T] partials in global tile
order (and its coverage check), and the owner's copy of the target logit."""
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import os

    import torch.distributed as dist

    from invariant_token_log_gb300 import vocab_parallel as vp
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    num_tiles, tile_v, n = 7, 8, 5
    mine = [(4, 7), (0, 4)][rank]                      # ranks own ranges out of order
    ranges = vp.tile_ranges(None, *mine)
    # each rank's block holds its global tile index + 100 * row, padded (as the
    # forward pads them) to the longest range so that every rank sends one shape
    pad = max(e - b for b, e in ranges)
    blk = torch.tensor([[100.0 * r + t for t in range(mine[0], mine[1])] + [-1.0] * (pad - (mine[1] - mine[0]))
                        for r in range(n)])
    blocks = vp._gather(blk, None)
    full = vp.assemble(blocks, ranges, num_tiles)
    targets = torch.tensor([0, 31, 32, 55, -100])
    tl = torch.tensor([float(rank * 1000 + r) for r in range(n)])
    owner = vp.owner_target_logit(vp._gather(tl, None), ranges, targets, tile_v)
    bad = None
    try:
        vp.assemble(blocks, [(0, 4), (3, 7)], num_tiles)
    except ValueError as e:
        bad = str(e)
    out[rank] = (ranges, full.tolist(), owner.tolist(), bad)
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_ranks_assemble_partials_and_pick_owners():
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(2, _free_port(), out), nprocs=2, start_method="spawn", join=True)
    for r in range(2):
        ranges, full, owner, bad = out[r]
        assert ranges == [(4, 7), (0, 4)]
        assert full == [[100.0 * row + t for t in range(7)] for row in range(5)]
        # targets 0, 31 sit in tiles 0, 3 (rank 1); 32, 55 in tiles 4, 6 (rank 0); -100 has no owner
        assert owner[:4] == [1000.0, 1001.0, 2.0, 3.0]
        assert owner[4] != owner[4]  # NaN
        assert bad is not None and "exactly once" in bad
