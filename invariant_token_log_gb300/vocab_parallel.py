"""Vocabulary-parallel selected-token log-probability across processes.

"Batch-Invariant LogP" operator page, section "Tensor Parallel", steps 1-6:
every rank reduces the fixed vocabulary tiles it owns to float32 (max,
sumexp) partials; the partials are shared with an all_gather, which moves
bytes and never does arithmetic; every rank merges all tiles in the same
fixed order over the same [n, num_vocab_tiles] shape; the target logit is
copied from the rank that owns it, never summed.  So TP=1, 2, 4, ... give the
same bits as the single-device forward.

Each rank holds its own shard of the logits: the global columns
[tile_begin * tile_v, min(tile_end * tile_v, vocab)).  Ranks may own ranges
of different lengths, in any order; together they must cover every tile
exactly once.  The reductions and the merge run in the CUDA library; this
module only moves bytes between ranks (torch.distributed all_gather; with
the gloo backend through host memory).
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from .logp import DEFAULT_TILE_V, IGNORE_INDEX, logp_merge, logp_tile_partials


def _gather(t: torch.Tensor, group) -> list[torch.Tensor]:
    """all_gather of equal-shaped tensors; through the host for gloo."""
    world = dist.get_world_size(group)
    via_host = dist.get_backend(group) == "gloo" and t.is_cuda
    src = t.cpu() if via_host else t.contiguous()
    out = [torch.empty_like(src) for _ in range(world)]
    dist.all_gather(out, src, group=group)
    return [o.to(t.device) for o in out] if via_host else out


def tile_ranges(group=None, tile_begin: int = 0, tile_end: int = 0) -> list[tuple[int, int]]:
    """Every rank's (tile_begin, tile_end), in rank order."""
    mine = torch.tensor([tile_begin, tile_end], dtype=torch.int64)
    return [tuple(int(v) for v in r.tolist()) for r in _gather(mine, group)]


def assemble(blocks: list[torch.Tensor], ranges: list[tuple[int, int]], num_tiles: int) -> torch.Tensor:
    """Place each rank's [N, >= its tile count] block at its global tile columns of an [N, num_tiles] buffer.

    Raises if the ranges do not cover every tile exactly once."""
    cover = [0] * num_tiles
    for b, e in ranges:
        for t in range(b, e):
            cover[t] += 1
    if any(c != 1 for c in cover):
        raise ValueError(f"tile ranges {ranges} do not cover tiles [0, {num_tiles}) exactly once")
    n = blocks[0].shape[0]
    out = torch.empty((n, num_tiles), dtype=blocks[0].dtype, device=blocks[0].device)
    for blk, (b, e) in zip(blocks, ranges):
        out[:, b:e] = blk[:, : e - b]
    return out


def owner_target_logit(target_logits: list[torch.Tensor], ranges: list[tuple[int, int]], target_ids: torch.Tensor,
                       tile_v: int, ignore_index: int = IGNORE_INDEX) -> torch.Tensor:
    """Each row's target logit taken from the rank whose tiles hold the target
    (a copy; rows with no owner -- ignored or out of range -- get NaN)."""
    t = target_ids.reshape(-1).to(torch.int64)
    tile = torch.div(t, tile_v, rounding_mode="floor")
    out = torch.full_like(target_logits[0], float("nan"))
    valid = (t != ignore_index) & (t >= 0)
    for tl, (b, e) in zip(target_logits, ranges):
        own = valid & (tile >= b) & (tile < e)
        out = torch.where(own, tl, out)
    return out


def vocab_parallel_logp(local_logits: torch.Tensor, target_ids: torch.Tensor, vocab: int, tile_begin: int,
                        tile_end: int, tile_v: int = DEFAULT_TILE_V, group=None, ignore_index: int = IGNORE_INDEX,
                        temperature: float = 1.0, return_entropy: bool = False):
    """(logp, lse[, entropy]) for rows whose vocabulary is split across the ranks of `group`.

    local_logits  [N, >= shard columns] this rank's shard; column 0 is global
                  column tile_begin * tile_v.
    target_ids    [N] global target columns (the same on every rank).
    Every rank returns the same float32 results, bit for bit those of
    logp_fwd on the unsplit rows with the same tile_v."""
    num_tiles = -(-vocab // tile_v)
    n = target_ids.numel()
    t_local = tile_end - tile_begin
    dev = local_logits.device
    # 1-2. this rank's tile partials (columns [tile_begin, tile_end) of [N, num_tiles])
    width = num_tiles
    pm = torch.empty((n, width), dtype=torch.float32, device=dev)
    ps = torch.empty_like(pm)
    pe = torch.empty_like(pm) if return_entropy else None
    tl = torch.full((n,), float("nan"), dtype=torch.float32, device=dev)
    logp_tile_partials(local_logits, target_ids, vocab, tile_v, tile_begin, tile_end, pm, ps, tl, ignore_index,
                       temperature=temperature, part_ent=pe)
    # 3. all_gather: bytes only.  Blocks are padded to the longest range so that
    # every rank sends the same shape.
    ranges = tile_ranges(group, tile_begin, tile_end)
    pad = max(e - b for b, e in ranges)
    mine = torch.zeros((3 if return_entropy else 2, n, pad), dtype=torch.float32, device=dev)
    mine[0, :, :t_local] = pm[:, tile_begin:tile_end]
    mine[1, :, :t_local] = ps[:, tile_begin:tile_end]
    if return_entropy:
        mine[2, :, :t_local] = pe[:, tile_begin:tile_end]
    blocks = _gather(mine, group)
    tls = _gather(tl, group)
    # 4-6. the same fixed-order merge on every rank; the target logit from its owner
    full_m = assemble([blk[0] for blk in blocks], ranges, num_tiles).contiguous()
    full_s = assemble([blk[1] for blk in blocks], ranges, num_tiles).contiguous()
    full_e = assemble([blk[2] for blk in blocks], ranges, num_tiles).contiguous() if return_entropy else None
    tl_owner = owner_target_logit(tls, ranges, target_ids, tile_v, ignore_index).contiguous()
    return logp_merge(full_m, full_s, num_tiles, tl_owner, target_ids, vocab, ignore_index, part_ent=full_e)
