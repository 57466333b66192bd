"""The fused LM-head + logp on the GPU, against the CPU oracle and for bit-invariance.

"[RFC][ROCm] End-to-end optimization of bitwise VIME R/R beyond native P/P",
section "Workstream 3: fused ROCm LM-head and linear logp": the projection
z = hidden . weight^T and the operator's tile statistics are one operation;
logp and lse must be the same bits whether or not the logits are also stored;
the vocabulary tiles and tensor-parallel ranks are merged in one fixed order.

Tolerances: logp, lse 1e-4 and entropy 1e-4 absolute against the float64
oracle (the operator's bounds).  The stored float32 logits against the
oracle's float64 projection: |dz| <= 2^-20 * sum_k |x_k w_k| + 1e-6 per
element.  The products of two 16-bit values are exact in float32, so the
error is the accumulation's; a float32 sum of H terms in any order errs by at
most about log2(H) * 2^-24 * sum |terms| with pairwise blocks and H * 2^-24
sequentially, and 2^-20 covers the tensor cores' K = 16 steps over H <= 4096
with a margin of 4 over the sequential bound at H = 4096.  bf16 logits must
be the round-to-nearest-even of the float32 ones.
"""
import numpy as np
import pytest
import torch

import invariant_token_log_gb300 as bil
import oracle
import workloads as wl
from gpu_helpers import ENTROPY_ATOL, LOGP_ATOL, assert_close_abs, check_watchdog, device_logits, f32_bits

pytestmark = pytest.mark.gpu

TILE = bil.LINEAR_TILE_V


@pytest.fixture(autouse=True)
def _watchdog():
    yield
    check_watchdog()


def make_case(n, h, v, dtype="bfloat16", seed=11, ignore_every=5):
    x = wl.linear_hidden(n, h, seed=seed, dtype=dtype)
    w = wl.linear_weight(v, h, seed=seed, dtype=dtype)
    t = wl.rng(seed, 1, n, v).integers(0, v, n, dtype=np.int64)
    if ignore_every:
        t[::ignore_every] = wl.IGNORE_INDEX
    return x, w, t


def to_dev(x, w, t, dtype):
    return device_logits(x, dtype), device_logits(w, dtype), torch.from_numpy(t).cuda()


def z_bound(x, w, dtype):
    """Per-element bound on the float32 projection's error: 2^-20 * sum |x w| + 1e-6."""
    ax, aw = np.abs(oracle.widen(x, dtype)), np.abs(oracle.widen(w, dtype))
    return (ax @ aw.T) * 2.0 ** -20 + 1e-6


SHAPES = [
    (128, 64, 256),     # one row tile, one K block, one vocabulary tile
    (300, 200, 1000),   # ragged rows (3 row tiles), ragged K (200 = 3 x 64 + 8), ragged last tile (232)
    (257, 512, 3000),   # 3 row tiles with one row in the last, 12 tiles
    (64, 1024, 777),
]


@pytest.mark.parametrize("dtype", ["bfloat16", "float16"])
@pytest.mark.parametrize("n,h,v", SHAPES)
def test_linear_vs_oracle(n, h, v, dtype):
    x, w, t = make_case(n, h, v, dtype, seed=n + h + v)
    xd, wd, td = to_dev(x, w, t, dtype)
    logp, lse, ent, z = bil.linear_logp(xd, wd, td, return_entropy=True, return_logits=True)
    torch.cuda.synchronize()
    rl, rs, bad, rh = oracle.linear_logp_fwd(x, w, dtype, t, entropy=True)
    assert bad == 0
    assert_close_abs(logp.cpu().numpy(), rl, LOGP_ATOL, "logp")
    assert_close_abs(lse.cpu().numpy(), rs, LOGP_ATOL, "lse")
    assert_close_abs(ent.cpu().numpy(), rh, ENTROPY_ATOL, "entropy")
    ign = t == wl.IGNORE_INDEX
    assert np.all(f32_bits(logp)[ign] == 0) and np.all(f32_bits(lse)[ign] == 0) and np.all(f32_bits(ent)[ign] == 0)
    zr = oracle.linear_logits(x, w, dtype)
    err = np.abs(z.cpu().numpy().astype(np.float64) - zr)
    assert np.all(err <= z_bound(x, w, dtype)), float(err.max())


def test_logits_output_does_not_change_the_bits():
    n, h, v = 300, 256, 2000
    x, w, t = make_case(n, h, v, seed=5)
    xd, wd, td = to_dev(x, w, t, "bfloat16")
    plain = bil.linear_logp(xd, wd, td, return_entropy=True)
    with32 = bil.linear_logp(xd, wd, td, return_entropy=True, return_logits=True)
    with16 = bil.linear_logp(xd, wd, td, return_entropy=True, return_logits=True, logits_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    for a, b, c in zip(plain, with32[:3], with16[:3]):
        assert np.array_equal(f32_bits(a), f32_bits(b)) and np.array_equal(f32_bits(a), f32_bits(c))
    # bf16 logits are the correctly rounded float32 logits
    assert torch.equal(with16[3].view(torch.int16), with32[3].to(torch.bfloat16).view(torch.int16))


def test_rows_bitwise_across_batch_sizes_and_positions():
    n, h, v = 256, 512, 1500
    x, w, t = make_case(n, h, v, seed=6, ignore_every=0)
    xd, wd, td = to_dev(x, w, t, "bfloat16")
    ref = bil.linear_logp(xd, wd, td, return_entropy=True, return_logits=True)
    torch.cuda.synchronize()
    refb = [f32_bits(r) for r in ref]
    r = wl.rng(6, 2)
    for size in (1, 2, 3, 7, 64, 129, 256):
        for _ in range(3):
            idx = r.permutation(n)[:size]
            sel = torch.from_numpy(idx).cuda()
            got = bil.linear_logp(xd.index_select(0, sel), wd, td.index_select(0, sel), return_entropy=True,
                                  return_logits=True)
            torch.cuda.synchronize()
            for g, rb in zip(got, refb):
                assert np.array_equal(f32_bits(g), rb[idx]), size
    # a row placed among other rows in a larger, padded batch
    big = torch.cat([xd, xd.flip(0), xd[:100]])
    tb = torch.cat([td, td.flip(0), td[:100]])
    got = bil.linear_logp(big, wd, tb, return_entropy=True)
    torch.cuda.synchronize()
    for g, rb in zip(got, refb[:3]):
        gb = f32_bits(g)
        assert np.array_equal(gb[:n], rb) and np.array_equal(gb[n:2 * n], rb[::-1]) and np.array_equal(gb[2 * n:],
                                                                                                       rb[:100])


@pytest.mark.parametrize("k", [2, 3])
def test_vocab_split_is_bitwise_fused(k):
    """Emulated tensor-parallel ranks each hold a weight shard of whole tiles and fill
    their tiles' partials (in reverse rank order, on their own streams); one merge."""
    n, h, v = 200, 384, 2900
    x, w, t = make_case(n, h, v, seed=7)
    xd, wd, td = to_dev(x, w, t, "bfloat16")
    fused = bil.linear_logp(xd, wd, td, return_entropy=True, temperature=0.9)
    nt = -(-v // TILE)
    pm = torch.full((n, nt), float("nan"), device="cuda")
    ps = torch.full((n, nt), float("nan"), device="cuda")
    pe = torch.full((n, nt), float("nan"), device="cuda")
    tl = torch.full((n,), float("nan"), device="cuda")
    bounds = [(r * nt) // k for r in range(k + 1)]
    streams = [torch.cuda.Stream() for _ in range(k)]
    torch.cuda.synchronize()
    for r in reversed(range(k)):
        b, e = bounds[r], bounds[r + 1]
        shard = wd[b * TILE: min(e * TILE, v)].clone()
        with torch.cuda.stream(streams[r]):
            bil.linear_logp_partials(xd, shard, td, v, b, e, pm, ps, tl, temperature=0.9, part_ent=pe)
    torch.cuda.synchronize()
    logp, lse, ent = bil.logp_merge(pm, ps, nt, tl, td, v, part_ent=pe)
    torch.cuda.synchronize()
    for a, b in zip(fused, (logp, lse, ent)):
        assert np.array_equal(f32_bits(a), f32_bits(b))


def test_temperature():
    n, h, v = 130, 256, 1100
    x, w, t = make_case(n, h, v, seed=8)
    xd, wd, td = to_dev(x, w, t, "bfloat16")
    for temp in (0.6, 1.7):
        logp, lse, ent = bil.linear_logp(xd, wd, td, temperature=temp, return_entropy=True)
        torch.cuda.synchronize()
        rl, rs, _, rh = oracle.linear_logp_fwd(x, w, "bfloat16", t, temperature=temp, entropy=True)
        assert_close_abs(logp.cpu().numpy(), rl, LOGP_ATOL, "logp")
        assert_close_abs(lse.cpu().numpy(), rs, LOGP_ATOL, "lse")
        assert_close_abs(ent.cpu().numpy(), rh, ENTROPY_ATOL, "entropy")
    a = bil.linear_logp(xd, wd, td, temperature=1.0)
    b = bil.linear_logp(xd, wd, td)
    torch.cuda.synchronize()
    assert np.array_equal(f32_bits(a[0]), f32_bits(b[0]))


def test_partials_vs_oracle():
    """Per-tile (m_t, s_t) and the target logit against the oracle's partials of the
    float64 projection (tile width 256)."""
    n, h, v = 150, 320, 1234
    x, w, t = make_case(n, h, v, seed=9)
    xd, wd, td = to_dev(x, w, t, "bfloat16")
    nt = -(-v // TILE)
    pm = torch.zeros((n, nt), device="cuda")
    ps = torch.zeros((n, nt), device="cuda")
    tl = torch.full((n,), float("nan"), device="cuda")
    bil.linear_logp_partials(xd, wd, td, v, 0, nt, pm, ps, tl)
    torch.cuda.synchronize()
    z = oracle.linear_logits(x, w, "bfloat16")
    rm, rsum, rtl = oracle.tile_partials(z, "float64", v, TILE, 0, nt, t)
    act = t != wl.IGNORE_INDEX
    zb = z_bound(x, w, "bfloat16").max(axis=1)
    assert np.all(np.abs(pm.cpu().numpy()[act] - rm[act]) <= zb[act, None])
    assert np.all(np.abs(ps.cpu().numpy()[act] / rsum[act] - 1) <= 1e-4)
    assert np.all(np.abs(tl.cpu().numpy()[act] - rtl[act]) <= zb[act])
    assert np.all(pm.cpu().numpy()[~act] == -np.inf) and np.all(ps.cpu().numpy()[~act] == 0)


def test_full_size_sampled_rows():
    """Qwen3-8B-shaped LM head (H = 4096, V = 151936) over 16384 rows, in the launch
    configuration the benchmark times; 24 sampled rows against the oracle, and the
    sampled rows alone give the same bits."""
    lw = wl.linear(16384)
    xd = device_logits(lw.hidden, lw.dtype)
    wd = device_logits(lw.weight, lw.dtype)
    td = torch.from_numpy(lw.target_ids).cuda()
    logp, lse, ent = bil.linear_logp(xd, wd, td, return_entropy=True)
    torch.cuda.synchronize()
    idx = np.sort(wl.rng(5, 20).choice(16384, 24, replace=False))
    rl, rs, bad, rh = oracle.linear_logp_fwd(np.ascontiguousarray(lw.hidden[idx]), lw.weight, lw.dtype,
                                             lw.target_ids[idx], entropy=True)
    assert bad == 0
    assert_close_abs(logp.cpu().numpy()[idx], rl, LOGP_ATOL, "logp")
    assert_close_abs(lse.cpu().numpy()[idx], rs, LOGP_ATOL, "lse")
    assert_close_abs(ent.cpu().numpy()[idx], rh, ENTROPY_ATOL, "entropy")
    sel = torch.from_numpy(idx).cuda()
    alone = bil.linear_logp(xd.index_select(0, sel), wd, td.index_select(0, sel), return_entropy=True)
    torch.cuda.synchronize()
    for a, b in zip(alone, (logp, lse, ent)):
        assert np.array_equal(f32_bits(a), f32_bits(b)[idx])


def test_argument_errors_queue_nothing():
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((300, 64), dtype=torch.bfloat16, device="cuda")
    t = torch.zeros(4, dtype=torch.int64, device="cuda")
    with pytest.raises(TypeError):
        bil.linear_logp(x.float(), w.float(), t)
    with pytest.raises(TypeError):
        bil.linear_logp(x, w.half(), t)
    nt = -(-300 // TILE)
    pm = torch.zeros((4, nt), device="cuda")
    with pytest.raises(bil.BilError) as e:
        bil.linear_logp_partials(x, w, t, 300, 1, 1, pm, pm.clone(), torch.zeros(4, device="cuda"))
    assert e.value.status == 1
    with pytest.raises(bil.BilError) as e:  # target out of range with validate
        bil.linear_logp(x, w, torch.full((4,), 300, dtype=torch.int64, device="cuda"), validate=True)
    assert e.value.status == 4


@pytest.mark.parametrize("n,h,v", [(1, 64, 300), (5, 8, 100), (130, 24, 256), (3, 4096, 40)])
def test_small_and_ragged_shapes(n, h, v):
    """A vocabulary inside one tile, a hidden size below one K block (the TMA
    box reads zeros past it), a single row."""
    x, w, t = make_case(n, h, v, seed=n * 7 + v, ignore_every=0)
    xd, wd, td = to_dev(x, w, t, "bfloat16")
    logp, lse, ent = bil.linear_logp(xd, wd, td, return_entropy=True)
    torch.cuda.synchronize()
    rl, rs, _, rh = oracle.linear_logp_fwd(x, w, "bfloat16", t, entropy=True)
    assert_close_abs(logp.cpu().numpy(), rl, LOGP_ATOL, "logp")
    assert_close_abs(lse.cpu().numpy(), rs, LOGP_ATOL, "lse")
    assert_close_abs(ent.cpu().numpy(), rh, ENTROPY_ATOL, "entropy")


def test_empty_batch_and_invalid_targets():
    x, w, t = make_case(6, 64, 500, seed=3, ignore_every=0)
    xd, wd, td = to_dev(x, w, t, "bfloat16")
    lp, ls = bil.linear_logp(xd[:0], wd, td[:0])
    assert lp.numel() == 0 and ls.numel() == 0
    bad = td.clone()
    bad[2] = 500        # one past the vocabulary
    bad[4] = -1         # negative, not the ignore index
    lp, ls = bil.linear_logp(xd, wd, bad)
    ref, rls = bil.linear_logp(xd, wd, td)
    torch.cuda.synchronize()
    lpn = lp.cpu().numpy()
    assert np.isnan(lpn[2]) and np.isnan(lpn[4])
    keep = [0, 1, 3, 5]
    assert np.array_equal(f32_bits(lp)[keep], f32_bits(ref)[keep])
    assert np.array_equal(f32_bits(ls), f32_bits(rls))  # lse never depends on the target
