"""Rows whose tiles do not start on a 16-byte boundary, through the C ABI.

The forward copies such a tile from the 16-byte boundary below it and the
reducing warp shifts the words back into place as it reads them.  The
results are a function of the values alone ("Batch-Invariant LogP" operator
page, section "Batch-Invariance"), so every start offset must give the bits
of a 16-byte aligned copy of the same rows.  A row pitch of 50257 elements
moves the start offset from row to row through every value the element size
allows (every even byte offset for 16-bit types, every multiple of 4 for
float32); base shifts of whole elements move it further.  Tile sizes cover
the register path (up to 4096 16-bit or 2048 float32 elements, whole and
ragged) and the two-pass shared-memory path (larger tiles).
"""
import numpy as np
import pytest
import torch

import invariant_token_log_gb300 as bil
import oracle
import workloads as wl
from gpu_helpers import LOGP_ATOL, assert_close_abs, check_watchdog, device_logits, f32_bits

pytestmark = pytest.mark.gpu

VOCAB = 50257  # an odd row length: the row pitch is not a multiple of 16 bytes


@pytest.fixture(autouse=True)
def _watchdog():
    yield
    check_watchdog()


def _place(x: torch.Tensor, shift: int) -> torch.Tensor:
    """x's rows at the same pitch, starting `shift` elements past an aligned address."""
    flat = x.reshape(-1)
    big = torch.empty(flat.numel() + 16, dtype=flat.dtype, device=flat.device)
    big[shift:shift + flat.numel()] = flat
    return big[shift:shift + flat.numel()].view(x.shape)


def _aligned_copy(x: torch.Tensor) -> torch.Tensor:
    """The same rows at a pitch that is a multiple of 16 bytes (pad columns NaN)."""
    n, v = x.shape
    ld = -(-v * x.element_size() // 16) * 16 // x.element_size()
    out = torch.full((n, ld), float("nan"), dtype=x.dtype, device=x.device)
    out[:, :v] = x
    return out


@pytest.mark.parametrize("dtype", ["bfloat16", "float16", "float32"])
@pytest.mark.parametrize("tile_v", [1024, 4096, 8192])
@pytest.mark.parametrize("shift", [0, 1, 3])
def test_every_start_offset_gives_the_aligned_bits(dtype, tile_v, shift):
    n = 37
    w = wl.random_rows(seed=61, n_rows=n, vocab=VOCAB, dtype=dtype, tile_v=tile_v, ignore_every=5)
    x = _place(device_logits(w.logits, dtype), shift)
    eb = x.element_size()
    assert (x.stride(0) * eb) % 16 != 0
    offsets = {(x.data_ptr() + r * x.stride(0) * eb) % 16 for r in range(n)}
    assert offsets == set(range(0, 16, eb))  # every start offset occurs
    xa = _aligned_copy(x)
    t = torch.from_numpy(w.target_ids).cuda()
    for temperature, ent in ((1.0, False), (0.7, True)):
        a = bil.logp_fwd(xa, t, w.ignore_index, tile_v, vocab=VOCAB, temperature=temperature, return_entropy=ent)
        b = bil.logp_fwd(x, t, w.ignore_index, tile_v, vocab=VOCAB, temperature=temperature, return_entropy=ent)
        torch.cuda.synchronize()
        for p, q in zip(a, b):
            assert np.array_equal(f32_bits(p), f32_bits(q)), (temperature, ent)


@pytest.mark.parametrize("dtype", ["bfloat16", "float32"])
@pytest.mark.parametrize("tile_v", [2048, 8192])
def test_unaligned_tile_partials_give_the_aligned_bits(dtype, tile_v):
    """The partials kernel over a shard that starts mid-row (its column 0 is
    global column tile_begin * tile_v) on rows with an odd pitch."""
    n = 19
    w = wl.random_rows(seed=62, n_rows=n, vocab=VOCAB, dtype=dtype, tile_v=tile_v, ignore_every=4)
    x = _place(device_logits(w.logits, dtype), 1)
    xa = _aligned_copy(x)
    t = torch.from_numpy(w.target_ids).cuda()
    num_tiles = -(-VOCAB // tile_v)
    begin, end = 2, num_tiles
    outs = []
    for rows in (xa, x):
        pm = torch.full((n, num_tiles), 7.0, dtype=torch.float32, device="cuda")
        ps = torch.full_like(pm, 7.0)
        pe = torch.full_like(pm, 7.0)
        tl = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
        bil.logp_tile_partials(rows[:, begin * tile_v:], t, VOCAB, tile_v, begin, end, pm, ps, tl, w.ignore_index,
                               temperature=0.7, part_ent=pe)
        outs.append((pm, ps, pe, tl))
    torch.cuda.synchronize()
    for p, q in zip(*outs):
        assert np.array_equal(f32_bits(p), f32_bits(q))


def test_unaligned_rows_match_the_oracle():
    """The shifted read agrees with the oracle as well as with the aligned path."""
    n, tile_v = 23, 4096
    w = wl.random_rows(seed=63, n_rows=n, vocab=VOCAB, dtype="bfloat16", tile_v=tile_v, ignore_every=6)
    x = _place(device_logits(w.logits, "bfloat16"), 5)
    t = torch.from_numpy(w.target_ids).cuda()
    logp, lse = bil.logp_fwd(x, t, w.ignore_index, tile_v, vocab=VOCAB)
    ref_logp, ref_lse, _ = oracle.logp_fwd(w.logits, "bfloat16", VOCAB, w.target_ids, w.ignore_index)
    torch.cuda.synchronize()
    assert_close_abs(logp.cpu().numpy(), ref_logp, LOGP_ATOL, "logp")
    assert_close_abs(lse.cpu().numpy(), ref_lse, LOGP_ATOL, "lse")


@pytest.mark.parametrize("dtype", ["bfloat16", "float32"])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("shift", [0, 3])
def test_unaligned_backward_gives_the_aligned_bits(dtype, out_dtype, shift):
    """The backward on rows with an odd pitch and a shifted base, writing
    output rows at another odd pitch and offset than the input's (so the two
    start at different offsets), two pad columns past the vocabulary, with a
    temperature and the entropy term."""
    n = 29
    w = wl.random_rows(seed=64, n_rows=n, vocab=VOCAB, ld=VOCAB + 2, dtype=dtype, tile_v=4096, ignore_every=5)
    x = _place(device_logits(w.logits, dtype), shift)
    width = x.shape[1]
    xa = _aligned_copy(x)[:, :width]
    t = torch.from_numpy(w.target_ids).cuda()
    g = torch.from_numpy(w.grad_logp).cuda()
    gh = torch.from_numpy(wl.rng(64, 7).standard_normal(n).astype(np.float32)).cuda()
    _, lse, ent = bil.logp_fwd(xa, t, w.ignore_index, 4096, vocab=VOCAB, temperature=0.7, return_entropy=True)
    ob = torch.empty((), dtype=out_dtype).element_size()
    pitch_a = -(-width * ob // 16) * 16 // ob + 8
    buf_a = torch.full((n, pitch_a), 9.0, dtype=out_dtype, device="cuda")
    pitch_u = width + 2
    assert (pitch_u * ob) % 16 != 0
    buf_u = torch.full((n * pitch_u + 8,), 9.0, dtype=out_dtype, device="cuda")
    out_u = buf_u[1:1 + n * pitch_u].view(n, pitch_u)
    for rows, out in ((xa, buf_a[:, :width]), (x, out_u[:, :width])):
        bil.logp_bwd(rows, t, lse, g, w.ignore_index, vocab=VOCAB, out=out, temperature=0.7, entropy=ent,
                     grad_entropy=gh)
    torch.cuda.synchronize()
    view = torch.int16 if out_dtype == torch.bfloat16 else torch.int32
    assert torch.equal(buf_a[:, :width].view(view), out_u[:, :width].view(view))
    assert torch.all(buf_a[:, width:] == 9.0) and torch.all(out_u[:, width:] == 9.0)
    assert buf_u[0] == 9.0 and torch.all(buf_u[1 + n * pitch_u:] == 9.0)


@pytest.mark.parametrize("dtype", ["bfloat16", "float16"])
@pytest.mark.parametrize("vocab", [50257, 50263, 151935])
@pytest.mark.parametrize("n", [1, 5, 16, 17, 128, 129])
@pytest.mark.parametrize("tile_v", [1024, 4096])
def test_small_unaligned_batches_give_the_aligned_bits(dtype, vocab, n, tile_v):
    """Up to 16 rows of a 16-bit type off 16-byte boundaries (128 aligned)
    take the cluster path, which reads its tiles straight from global memory:
    such rows are read as the 16-byte units that hold them and shifted, and a
    partial last group reads only the units that hold its elements.  With
    vocab 50257 the last group holds one element, with 50263 seven.  A single
    row counts as aligned whenever its base is (its stride is never used).
    The other sizes cross the path boundaries on either side."""
    w = wl.random_rows(seed=65, n_rows=n, vocab=vocab, dtype=dtype, tile_v=tile_v, ignore_every=3)
    t = torch.from_numpy(w.target_ids).cuda()
    for shift in (0, 1, 7):
        x = _place(device_logits(w.logits, dtype), shift)
        xa = _aligned_copy(x)
        for temperature, ent in ((1.0, False), (0.7, True)):
            a = bil.logp_fwd(xa, t, w.ignore_index, tile_v, vocab=vocab, temperature=temperature,
                             return_entropy=ent)
            b = bil.logp_fwd(x, t, w.ignore_index, tile_v, vocab=vocab, temperature=temperature,
                             return_entropy=ent)
            torch.cuda.synchronize()
            for p, q in zip(a, b):
                assert np.array_equal(f32_bits(p), f32_bits(q)), (shift, temperature, ent)


@pytest.mark.parametrize("dtype", ["bfloat16", "float16", "float32"])
@pytest.mark.parametrize("shift", [0, 3])
@pytest.mark.parametrize("pad", [0, 5])
def test_backward_with_shared_offsets_gives_the_aligned_bits(dtype, shift, pad):
    """Contiguous [N, V + pad] logits and an output of the same layout at an
    odd pitch: input and output rows share their offsets from a 16-byte
    boundary (every offset occurs), so the backward's groups start at the first
    column where both are aligned and the few columns around them go one by
    one.  Bits must equal those of an aligned copy, with and without a
    temperature and the entropy term; the pad columns get +0.0."""
    n = 33
    w = wl.random_rows(seed=66, n_rows=n, vocab=VOCAB, ld=VOCAB + pad, dtype=dtype, tile_v=4096, ignore_every=5)
    x = _place(device_logits(w.logits, dtype), shift)
    out = _place(torch.full_like(x, 9.0), shift)
    assert (x.data_ptr() - out.data_ptr()) % 16 == 0 and (x.stride(0) * x.element_size()) % 16 != 0
    xa = _aligned_copy(x)
    t = torch.from_numpy(w.target_ids).cuda()
    g = torch.from_numpy(w.grad_logp).cuda()
    gh = torch.from_numpy(wl.rng(66, 7).standard_normal(n).astype(np.float32)).cuda()
    view = torch.int16 if x.element_size() == 2 else torch.int32
    for temperature, ent in ((1.0, False), (0.7, True)):
        _, lse, h = bil.logp_fwd(xa, t, w.ignore_index, 4096, vocab=VOCAB, temperature=temperature,
                                 return_entropy=True)
        kw = dict(temperature=temperature, entropy=h, grad_entropy=gh) if ent else dict(temperature=temperature)
        da = bil.logp_bwd(xa, t, lse, g, w.ignore_index, vocab=VOCAB, **kw)
        bil.logp_bwd(x, t, lse, g, w.ignore_index, vocab=VOCAB, out=out, **kw)
        torch.cuda.synchronize()
        assert torch.equal(da[:, :VOCAB].view(view), out[:, :VOCAB].view(view)), (temperature, ent)
        assert torch.all(out[:, VOCAB:].view(view) == 0)
