"""Bitwise invariance on the GPU ("Batch-Invariance" section of the operator
page; "Tensor Parallel": TP=1/2/4 bit-identical).

A row's logp and lse bits must not change with the number of rows, its
position, its neighbours, the row stride, or how the vocabulary tiles are
split between partial calls (emulated tensor-parallel ranks); the gradient
row's bits must not change with the batch either.
"""
import numpy as np
import pytest
import torch

import invariant_token_log_gb300 as bil
import workloads as wl
from gpu_helpers import check_watchdog, device_logits, f32_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _watchdog():
    yield
    check_watchdog()


@pytest.fixture(scope="module")
def bank():
    return wl.decode_bank()


@pytest.fixture(scope="module")
def packed():
    return wl.packed()


def tp_ranges(num_tiles, k, how, seed=0):
    """Tile ownership of k emulated ranks, as lists of single-tile or contiguous ranges."""
    if how == "contiguous":
        b = [(r * num_tiles) // k for r in range(k + 1)]
        return [[(b[r], b[r + 1])] for r in range(k)]
    if how == "round_robin":
        return [[(t, t + 1) for t in range(r, num_tiles, k)] for r in range(k)]
    perm = wl.rng(seed, 77, k).permutation(num_tiles)
    return [[(int(t), int(t) + 1) for t in perm[r::k]] for r in range(k)]


def split_forward(x, t, vocab, tile, ranks, ignore_index=-100, own_shards=False):
    """Emulated TP: every rank fills its tiles of one [N, T] buffer; then one merge."""
    n = x.shape[0]
    nt = -(-vocab // tile)
    pm = torch.full((n, nt), float("nan"), device="cuda")
    ps = torch.full((n, nt), float("nan"), device="cuda")
    tl = torch.full((n,), float("nan"), device="cuda")
    streams = [torch.cuda.Stream() for _ in ranks]
    torch.cuda.synchronize()
    for r, rr in enumerate(reversed(ranks)):  # ranks finish in any order
        with torch.cuda.stream(streams[r]):
            for b, e in rr:
                c0, c1 = b * tile, min(e * tile, vocab)
                shard = x[:, c0:c1].contiguous() if own_shards else x[:, c0:]
                bil.logp_tile_partials(shard, t, vocab, tile, b, e, pm, ps, tl, ignore_index)
    torch.cuda.synchronize()
    return bil.logp_merge(pm, ps, nt, tl, t, vocab, ignore_index)


def test_decode_rows_bitwise_across_batch_sizes_and_positions(bank):
    w = bank
    x = device_logits(w.logits, w.dtype)
    t = torch.from_numpy(w.target_ids).cuda()
    ref_logp, ref_lse = bil.logp_fwd(x, t, -100, w.tile_v)
    x_pad = torch.full((256, wl.PADDED_VOCAB), float("-inf"), dtype=x.dtype, device="cuda")
    x_pad[:, :w.vocab] = x
    torch.cuda.synchronize()
    rl, rs = f32_bits(ref_logp), f32_bits(ref_lse)
    checked = 0
    for n in (1, 2, 3, 7, 64, 256):
        for draw in wl.decode_draws(n, draws=8):
            idx = torch.from_numpy(draw).cuda()
            for xs, vocab in ((x, None), (x_pad, w.vocab)):
                logp, lse = bil.logp_fwd(xs.index_select(0, idx), t.index_select(0, idx), -100, w.tile_v,
                                         vocab=vocab)
                assert np.array_equal(f32_bits(logp), rl[draw]), (n, "logp")
                assert np.array_equal(f32_bits(lse), rs[draw]), (n, "lse")
                checked += n
    assert checked > 2 * 8 * (1 + 2 + 3 + 7 + 64 + 256) - 1


def test_decode_rows_through_partials(bank):
    w = bank
    x = device_logits(w.logits, w.dtype)
    t = torch.from_numpy(w.target_ids).cuda()
    ref_logp, ref_lse = bil.logp_fwd(x, t, -100, w.tile_v)
    nt = -(-w.vocab // w.tile_v)
    for n in (1, 3, 7):
        draw = wl.decode_draws(n, draws=1)[0]
        idx = torch.from_numpy(draw).cuda()
        logp, lse = split_forward(x.index_select(0, idx), t.index_select(0, idx), w.vocab, w.tile_v,
                                  tp_ranges(nt, 2, "contiguous"))
        assert np.array_equal(f32_bits(logp), f32_bits(ref_logp)[draw])
        assert np.array_equal(f32_bits(lse), f32_bits(ref_lse)[draw])


@pytest.mark.parametrize("k", [1, 2, 4])
@pytest.mark.parametrize("how", ["contiguous", "round_robin", "permuted"])
def test_packed_emulated_tp_is_bitwise_fused(packed, k, how):
    w = packed
    x = device_logits(w.logits, w.dtype)
    t = torch.from_numpy(w.target_ids).cuda()
    fused = bil.logp_fwd(x, t, -100, w.tile_v)
    nt = -(-w.vocab // w.tile_v)
    split = split_forward(x, t, w.vocab, w.tile_v, tp_ranges(nt, k, how, seed=k),
                          own_shards=(how == "contiguous" and k == 4))
    torch.cuda.synchronize()
    assert np.array_equal(f32_bits(split[0]), f32_bits(fused[0]))
    assert np.array_equal(f32_bits(split[1]), f32_bits(fused[1]))


def test_packed_sequences_alone_match_the_packed_batch(packed):
    """Each packed sequence evaluated on its own gives the packed batch's bits,
    forward and backward; padding rows are exactly zero."""
    w = packed
    x = device_logits(w.logits, w.dtype)
    t = torch.from_numpy(w.target_ids).cuda()
    g = torch.from_numpy(wl.rng(4, 9).standard_normal(w.n_rows).astype(np.float32)).cuda()
    logp, lse = bil.logp_fwd(x, t, -100, w.tile_v)
    d = bil.logp_bwd(x, t, lse, g, -100)
    torch.cuda.synchronize()
    T = w.meta["T"]
    for b, start, length in w.meta["seqs"]:
        r0, r1 = b * T + start, b * T + start + length
        lp, ls = bil.logp_fwd(x[r0:r1], t[r0:r1], -100, w.tile_v)
        dd = bil.logp_bwd(x[r0:r1], t[r0:r1], ls, g[r0:r1], -100)
        torch.cuda.synchronize()
        assert np.array_equal(f32_bits(lp), f32_bits(logp[r0:r1]))
        assert np.array_equal(f32_bits(ls), f32_bits(lse[r0:r1]))
        assert torch.equal(dd.view(torch.int16), d[r0:r1].view(torch.int16))  # bitwise, on the device
    pad = (w.target_ids == -100)
    assert pad.any()
    assert np.all(f32_bits(logp)[pad] == 0)
    pad_rows = torch.from_numpy(np.flatnonzero(pad)).cuda()
    assert not torch.any(d.index_select(0, pad_rows).view(torch.int16) != 0)  # +0.0 bit patterns


@pytest.mark.parametrize("temperature", [1.0, 0.8])
def test_small_batches_take_the_cluster_path_with_the_same_bits(bank, temperature):
    """Up to 128 rows (16-bit, 16-byte aligned rows, tiles of at most 4096), the
    forward shares each row among a cluster of blocks instead of streaming it
    through one; the bits must not change: every row of a small batch (1, 5,
    128 rows; 129 takes the streaming path) equals that row in the full
    256-row batch, with the entropy, ignored rows and an out-of-range target
    among them."""
    w = bank
    x = device_logits(w.logits, w.dtype)
    t = torch.from_numpy(w.target_ids).cuda()
    t[7] = -100
    t[12] = w.vocab + 3  # invalid: NaN logp, lse still computed
    ref = bil.logp_fwd(x, t, -100, w.tile_v, temperature=temperature, return_entropy=True)
    torch.cuda.synchronize()
    refb = [f32_bits(r) for r in ref]
    r = wl.rng(11, 3)
    for n in (1, 5, 128, 129):
        for draw in range(3):
            idx = r.permutation(256)[:n]
            if draw == 0:
                idx[: min(n, 2)] = [7, 12][: min(n, 2)]
            sel = torch.from_numpy(idx).cuda()
            got = bil.logp_fwd(x.index_select(0, sel), t.index_select(0, sel), -100, w.tile_v,
                               temperature=temperature, return_entropy=True)
            torch.cuda.synchronize()
            for g, rb in zip(got, refb):
                assert np.array_equal(f32_bits(g), rb[idx]), (n, draw)
