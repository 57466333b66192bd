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


def _rank_linear(rank, world, port, layout, out):
    import os

    import torch
    import torch.distributed as dist

    import invariant_token_log_gb300 as bil
    import workloads as wl
    from gpu_helpers import device_logits, f32_bits
    from invariant_token_log_gb300.vocab_parallel import vocab_parallel_linear_logp, vocab_parallel_linear_logp_bwd
    from test_gpu_linear_backward import tolerances
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    n, h, v, tile = 96, 128, 3000, bil.LINEAR_TILE_V
    nt = -(-v // tile)  # 12 tiles, the last one ragged
    x = wl.linear_hidden(n, h, seed=41)
    w = wl.linear_weight(v, h, seed=41)
    t = wl.rng(41, 1).integers(0, v, n, dtype=np.int64)
    t[::9] = -100
    g = wl.rng(41, 2).standard_normal(n).astype(np.float32)
    gh = wl.rng(41, 3).standard_normal(n).astype(np.float32)
    if layout == "contiguous":
        b = [(r * nt) // world for r in range(world + 1)]
        lo, hi = b[rank], b[rank + 1]
    else:  # uneven ranges, ranks in reverse order of their tiles
        cuts = [0, 1, 5, 9, nt][: world + 1] if world == 4 else [0, 7, nt]
        k = world - 1 - rank
        lo, hi = cuts[k], cuts[k + 1]
    c0, c1 = lo * tile, min(hi * tile, v)
    xd = device_logits(x, "bfloat16")
    wshard = device_logits(np.ascontiguousarray(w[c0:c1]), "bfloat16")   # this rank's rows only
    td = torch.from_numpy(t).cuda()
    gd, ghd = torch.from_numpy(g).cuda(), torch.from_numpy(gh).cuda()
    logp, lse, ent = vocab_parallel_linear_logp(xd, wshard, td, v, lo, hi, temperature=0.9, return_entropy=True)
    dh, dw = vocab_parallel_linear_logp_bwd(xd, wshard, td, lse, gd, v, lo, hi, temperature=0.9, entropy=ent,
                                            grad_entropy=ghd)
    wfull = device_logits(w, "bfloat16")
    ref = bil.linear_logp(xd, wfull, td, temperature=0.9, return_entropy=True)
    rdh, rdw = bil.linear_logp_bwd(xd, wfull, td, ref[1], gd, temperature=0.9, entropy=ref[2], grad_entropy=ghd,
                                   out_dtype=torch.float32)
    torch.cuda.synchronize()
    fwd_ok = all(np.array_equal(f32_bits(a), f32_bits(b)) for a, b in zip((logp, lse, ent), ref))
    dw_ok = np.array_equal(f32_bits(dw), f32_bits(rdw[c0:c1]))
    odx, _, _, tol_dz, tol_dx, _ = tolerances(x, w, "bfloat16", t, g, gh, 0.9)
    dh_ok = bool(np.all(np.abs(dh.cpu().numpy().astype(np.float64) - odx) <= tol_dx))
    out[rank] = (fwd_ok, dw_ok, dh_ok, f32_bits(dh).tobytes())
    dist.destroy_process_group()


@pytest.mark.timeout(600)
@pytest.mark.parametrize("world,layout", [(2, "contiguous"), (4, "contiguous"), (2, "uneven"), (4, "uneven")])
def test_vocab_parallel_fused_lm_head(world, layout):
    """The fused LM-head + logp with the LM head split by vocabulary tiles across
    processes: the forward is bit for bit the single-device one on every rank;
    each rank's dweight rows are the single-device rows; dhidden (the ranks'
    parts added in rank order) is the same on every rank and within the
    backward's derived bound of the oracle."""
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_linear, args=(world, _free_port(), layout, out), nprocs=world, start_method="spawn",
                       join=True)
    res = [out[r] for r in range(world)]
    assert all(r[0] for r in res), "forward"
    assert all(r[1] for r in res), "dweight rows"
    assert all(r[2] for r in res), "dhidden vs oracle"
    assert len({r[3] for r in res}) == 1, "dhidden differs between ranks"
