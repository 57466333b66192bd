"""The full-size workloads, in the launch configuration the benchmark times.

prefill  N=4096 (B=4 x T=1024), V=151936 bf16 with one +12 spike per row, row
         stride 155648 with -inf pad columns, 5% ignored rows, tile 4096.
         Forward on every row against the oracle; the padded and the unpadded
         layouts give identical bits.
training N=16384 (B=8 x T=2048), V=151936 bf16, targets 70% from the row's
         top-5, g ~ N(0, 1), bf16 gradient, tile 4096.  Forward on every row
         against the oracle; the bf16 backward (and a float32-output run of
         the same kernel) on sampled rows against the oracle.
"""
import numpy as np
import pytest
import torch

import invariant_token_log_gb300 as bil
import oracle
import workloads as wl
from gpu_helpers import (LOGP_ATOL, assert_close_abs, assert_rounded, check_dlogits_split, check_watchdog,
                         device_logits, dlogits_tol, f32_bits, host_bits)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _watchdog():
    yield
    check_watchdog()


@pytest.fixture(scope="module")
def prefill():
    return wl.prefill()


@pytest.fixture(scope="module")
def training():
    return wl.training()


@pytest.fixture(scope="module")
def training_ref(training):
    """The oracle's forward over every row, and each row's maximum (from its tile partials)."""
    w = training
    ref_logp, ref_lse, bad = oracle.logp_fwd(w.logits, w.dtype, w.vocab, w.target_ids, w.ignore_index)
    assert bad == 0
    num_tiles = -(-w.vocab // w.tile_v)
    pm, _, _ = oracle.tile_partials(w.logits, w.dtype, w.vocab, w.tile_v, 0, num_tiles, w.target_ids,
                                    w.ignore_index)
    return ref_logp, ref_lse, pm.max(axis=1)


def test_prefill_every_row(prefill):
    w = prefill
    x_pad = device_logits(w.logits, w.dtype)                 # [4096, 155648], pad = -inf
    t = torch.from_numpy(w.target_ids).cuda()
    logp, lse = bil.logp_fwd(x_pad, t, w.ignore_index, w.tile_v, vocab=w.vocab)
    x = x_pad[:, :w.vocab].contiguous()                       # the same rows at stride 151936
    logp2, lse2 = bil.logp_fwd(x, t, w.ignore_index, w.tile_v)
    torch.cuda.synchronize()
    assert np.array_equal(f32_bits(logp), f32_bits(logp2))
    assert np.array_equal(f32_bits(lse), f32_bits(lse2))
    ref_logp, ref_lse, bad = oracle.logp_fwd(w.logits, w.dtype, w.vocab, w.target_ids, w.ignore_index)
    assert bad == 0
    assert_close_abs(logp.cpu().numpy(), ref_logp, LOGP_ATOL, "logp")
    assert_close_abs(lse.cpu().numpy(), ref_lse, LOGP_ATOL, "lse")
    ign = w.target_ids == w.ignore_index
    assert ign.sum() == w.meta["n_ignored"]
    assert np.all(f32_bits(logp)[ign] == 0)


def test_training_forward_every_row(training, training_ref):
    w = training
    x = device_logits(w.logits, w.dtype)
    t = torch.from_numpy(w.target_ids).cuda()
    logp, lse = bil.logp_fwd(x, t, w.ignore_index, w.tile_v)
    torch.cuda.synchronize()
    ref_logp, ref_lse, _ = training_ref
    assert_close_abs(logp.cpu().numpy(), ref_logp, LOGP_ATOL, "logp")
    assert_close_abs(lse.cpu().numpy(), ref_lse, LOGP_ATOL, "lse")


def backward_rows(w, ref_logp, ref_lse, row_max, count=512):
    """Rows of the training batch to check the backward on: the 192 rows with the
    largest |g| p over the row (p at the row's maximum) and the 192 with the
    largest |g| p at the target, where the float32 error of p weighs most; the
    first and last rows and both sides of every 2048-row boundary; seeded
    uniform rows up to `count`."""
    n = w.n_rows
    g = np.abs(w.grad_logp.astype(np.float64))
    gp_row = g * np.exp(row_max - ref_lse)
    gp_tgt = g * np.exp(ref_logp)
    rows = set(np.argsort(-gp_row)[:192].tolist()) | set(np.argsort(-gp_tgt)[:192].tolist())
    rows |= {0, n - 1}
    for b in range(2048, n, 2048):
        rows |= {b - 1, b}
    rng = wl.rng(77, 0)
    while len(rows) < count:
        rows.add(int(rng.integers(0, n)))
    return np.array(sorted(rows))


def test_training_backward_sampled_rows(training, training_ref):
    """The benchmarked backward (bf16 dlogits), and the same kernel with a float32
    output (the value before the final rounding), against the oracle on 512 rows
    chosen by backward_rows, in chunks of 64 rows.  Float32: the flat 1e-6 where
    |g| p <= 1/2, the derived bound beyond (gpu_helpers.dlogits_tol); bf16:
    correctly rounded up to the same bound."""
    w = training
    ref_logp, ref_lse, row_max = training_ref
    rows = backward_rows(w, ref_logp, ref_lse, row_max)
    assert len(rows) >= 512
    x = device_logits(w.logits, w.dtype)
    t = torch.from_numpy(w.target_ids).cuda()
    g = torch.from_numpy(w.grad_logp).cuda()
    _, lse = bil.logp_fwd(x, t, w.ignore_index, w.tile_v)
    rows_d = torch.from_numpy(rows).cuda()
    d = bil.logp_bwd(x, t, lse, g, w.ignore_index)            # bf16, the benchmarked configuration
    got16 = host_bits(d[rows_d])
    del d
    d32 = bil.logp_bwd(x, t, lse, g, w.ignore_index, dlogits_dtype=torch.float32)
    got32 = d32[rows_d].cpu().numpy()
    del d32
    torch.cuda.synchronize()
    flipped, records = [], []
    for c0 in range(0, len(rows), 64):
        r = rows[c0:c0 + 64]
        sub = np.ascontiguousarray(w.logits[r])
        ref_d, bad = oracle.logp_bwd(sub, w.dtype, w.vocab, w.target_ids[r], w.grad_logp[r].astype(np.float64))
        assert bad == 0
        p = np.exp(oracle.widen(sub, w.dtype)[:, :w.vocab] - ref_lse[r][:, None])
        tol, gp = dlogits_tol(p, w.grad_logp[r], ref_lse[r])
        records.append(check_dlogits_split(got32[c0:c0 + 64], ref_d, gp, f"training rows {r[0]}..{r[-1]}"))
        flipped.append(assert_rounded(got16[c0:c0 + 64], ref_d, "bfloat16", tol, "dlogits"))
    worst_flat = max(rec["worst_flat"] for rec in records)
    worst_beyond = max(rec.get("worst_beyond_ratio", 0.0) for rec in records)
    print(f"DLOGITS-BOUND training {len(rows)} rows: worst flat-region error {worst_flat:.3g}, "
          f"worst beyond |g|p>1/2 {worst_beyond:.3g} x its bound, "
          f"elements beyond {sum(rec['n_beyond'] for rec in records)}")
    assert float(np.mean(flipped)) < 1e-3
