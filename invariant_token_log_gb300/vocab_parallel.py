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

from .linear import LINEAR_TILE_V, linear_logp_bwd, linear_logp_partials, sum_f32
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
    dev = local_logits.device
    # 1-2. this rank's tile partials (columns [tile_begin, tile_end) of [N, num_tiles])
    pm = torch.empty((n, num_tiles), dtype=torch.float32, device=dev)
    ps = torch.empty_like(pm)
    pe = torch.empty_like(pm) if return_entropy else None
    tl = torch.full((n,), float("nan"), dtype=torch.float32, device=dev)
    logp_tile_partials(local_logits, target_ids, vocab, tile_v, tile_begin, tile_end, pm, ps, tl, ignore_index,
                       temperature=temperature, part_ent=pe)
    return _exchange_and_merge(pm, ps, pe, tl, tile_begin, tile_end, num_tiles, tile_v, target_ids, vocab, group,
                               ignore_index)


def _exchange_and_merge(pm, ps, pe, tl, tile_begin, tile_end, num_tiles, tile_v, target_ids, vocab, group,
                        ignore_index):
    """Steps 3-6 of "Tensor Parallel": all_gather this rank's partials (bytes
    only; blocks padded to the longest range so that every rank sends one
    shape), place every block at its tile columns, take the target logit from
    its owner and merge all tiles in the fixed order."""
    n = pm.shape[0]
    t_local = tile_end - tile_begin
    ranges = tile_ranges(group, tile_begin, tile_end)
    pad = max(e - b for b, e in ranges)
    mine = torch.zeros((3 if pe is not None else 2, n, pad), dtype=torch.float32, device=pm.device)
    mine[0, :, :t_local] = pm[:, tile_begin:tile_end]
    mine[1, :, :t_local] = ps[:, tile_begin:tile_end]
    if pe is not None:
        mine[2, :, :t_local] = pe[:, tile_begin:tile_end]
    blocks = _gather(mine, group)
    tls = _gather(tl, group)
    full_m = assemble([blk[0] for blk in blocks], ranges, num_tiles).contiguous()
    full_s = assemble([blk[1] for blk in blocks], ranges, num_tiles).contiguous()
    full_e = assemble([blk[2] for blk in blocks], ranges, num_tiles).contiguous() if pe is not None else None
    tl_owner = owner_target_logit(tls, ranges, target_ids, tile_v, ignore_index).contiguous()
    return logp_merge(full_m, full_s, num_tiles, tl_owner, target_ids, vocab, ignore_index, part_ent=full_e)


def vocab_parallel_linear_logp(hidden: torch.Tensor, weight_shard: torch.Tensor, target_ids: torch.Tensor,
                               vocab: int, tile_begin: int, tile_end: int, group=None,
                               ignore_index: int = IGNORE_INDEX, temperature: float = 1.0,
                               return_entropy: bool = False):
    """The fused LM-head + logp with the LM head split by vocabulary tiles across
    the ranks of `group` ("[RFC][ROCm] End-to-end optimization of bitwise VIME
    R/R beyond native P/P", "Workstream 3": merge vocabulary tiles and TP ranks
    with an explicit fixed tree).

    hidden        [N, H] the same on every rank.
    weight_shard  this rank's LM-head rows: global vocabulary columns
                  [tile_begin * 256, min(tile_end * 256, vocab)).
    Every rank returns (logp, lse[, entropy]), bit for bit those of
    linear_logp on the whole LM head."""
    num_tiles = -(-vocab // LINEAR_TILE_V)
    n = target_ids.numel()
    dev = hidden.device
    pm = torch.empty((n, num_tiles), dtype=torch.float32, device=dev)
    ps = torch.empty_like(pm)
    pe = torch.empty_like(pm) if return_entropy else None
    tl = torch.full((n,), float("nan"), dtype=torch.float32, device=dev)
    linear_logp_partials(hidden, weight_shard, target_ids, vocab, tile_begin, tile_end, pm, ps, tl, ignore_index,
                         temperature=temperature, part_ent=pe)
    return _exchange_and_merge(pm, ps, pe, tl, tile_begin, tile_end, num_tiles, LINEAR_TILE_V, target_ids, vocab,
                               group, ignore_index)


def vocab_parallel_linear_logp_bwd(hidden: torch.Tensor, weight_shard: torch.Tensor, target_ids: torch.Tensor,
                                   lse: torch.Tensor, grad_logp: torch.Tensor, vocab: int, tile_begin: int,
                                   tile_end: int, group=None, ignore_index: int = IGNORE_INDEX,
                                   temperature: float = 1.0, entropy: torch.Tensor | None = None,
                                   grad_entropy: torch.Tensor | None = None):
    """Backward of vocab_parallel_linear_logp: (dhidden [N, H], dweight_shard).

    Each rank computes its shard's dZ, its dweight rows (bit for bit the
    single-device rows: the sum runs over the batch, not the vocabulary) and
    its part of dhidden = dZ . W; the parts are all-gathered (bytes only) and
    added in rank order by bil_sum_f32, so every rank holds the same dhidden
    (not the single-device bits: the sum over the vocabulary is split at the
    shard boundaries)."""
    dh, dw = linear_logp_bwd(hidden, weight_shard, target_ids, lse, grad_logp, ignore_index, temperature, entropy,
                             grad_entropy, out_dtype=torch.float32, vocab=vocab,
                             tile_begin=tile_begin, tile_end=tile_end)
    parts = _gather(dh.contiguous(), group)
    return sum_f32(parts), dw
