"""The seeded input generators (workloads.py), which both the oracle's tests
and the CUDA path's tests and benchmark read: bf16 storage is round-to-nearest-
even, chunks regenerate byte for byte on their own, and each workload keeps the
recipe it states (targets, ignored rows, pad columns, packing)."""
import numpy as np
import torch

import workloads as wl


def test_bf16_storage_is_round_to_nearest_even():
    r = np.random.default_rng(7)
    x = np.concatenate([
        (r.standard_normal(100000) * 3.0).astype(np.float32),
        r.standard_normal(1000).astype(np.float32) * np.float32(1e-38),            # subnormals
        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, -3.3895314e38, 1e-45], np.float32),
    ])
    # exact midpoints between neighbouring bf16 values, both tie directions
    mids = (np.arange(0x3F80, 0x3FA0, dtype=np.uint32) << 16) | 0x8000
    x = np.concatenate([x, mids.view(np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(wl.f32_to_bf16_bits(x), want)
    nan = wl.f32_to_bf16_bits(np.array([np.nan], np.float32))
    assert np.isnan(wl.bf16_bits_to_f32(nan)).all()
    assert np.array_equal(wl.bf16_bits_to_f32(want), torch.from_numpy(want.view(np.int16)).view(
        torch.bfloat16).float().numpy())


def test_chunks_regenerate_on_their_own():
    full = wl.training(n_rows=2 * wl.CHUNK_ROWS)
    part = wl.training(n_rows=2 * wl.CHUNK_ROWS, chunks=[1])
    rows = slice(wl.CHUNK_ROWS, 2 * wl.CHUNK_ROWS)
    assert np.array_equal(full.logits[rows], part.logits[rows])
    assert np.array_equal(full.target_ids[rows], part.target_ids[rows])
    again = wl.training(n_rows=2 * wl.CHUNK_ROWS)
    assert np.array_equal(full.logits, again.logits) and np.array_equal(full.grad_logp, again.grad_logp)


def test_training_targets_follow_the_recipe():
    w = wl.training(n_rows=2 * wl.CHUNK_ROWS)
    v = w.vocab
    assert w.logits.shape == (2 * wl.CHUNK_ROWS, v) and w.logits.dtype == np.uint16
    t = w.target_ids
    assert ((t >= 0) & (t < v)).all()                     # no ignored rows in this workload
    vals = wl.bf16_bits_to_f32(w.logits)
    fifth = np.partition(vals, v - 5, axis=1)[:, v - 5]
    in_top5 = vals[np.arange(len(t)), t] >= fifth
    # 70% drawn from the top five, plus the uniform draws that land there (5/V)
    assert 0.6 < in_top5.mean() < 0.8
    assert abs(float(vals.std()) - 3.0) < 0.01
    assert w.grad_logp.dtype == np.float32 and abs(float(w.grad_logp.std()) - 1.0) < 0.15


def test_prefill_pads_and_ignored_rows():
    w = wl.prefill(chunks=[0])
    assert w.logits.shape == (4096, wl.PADDED_VOCAB)
    assert (w.logits[: wl.CHUNK_ROWS, wl.VOCAB:] == wl.BF16_NEG_INF).all()
    ignored = w.target_ids == wl.IGNORE_INDEX
    assert ignored.sum() == round(0.05 * 4096) == 205
    active = w.target_ids[~ignored]
    assert ((active >= 0) & (active < wl.VOCAB)).all()


def test_packed_layout_is_greedy_and_in_bounds():
    B, T = 2, 8192
    seqs = wl.packed_layout(B, T)
    for b in range(B):
        mine = [(s, n) for bb, s, n in seqs if bb == b]
        assert mine and mine[0][0] == 0
        for (s0, n0), (s1, _) in zip(mine, mine[1:]):
            assert s1 == s0 + n0                          # packed back to back
        assert all(256 <= n <= 4096 for _, n in mine)
        end = mine[-1][0] + mine[-1][1]
        assert end <= T and T - end < 4096                # the next draw did not fit
