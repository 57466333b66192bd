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
from gpu_helpers import (DLOGITS_ATOL, LOGP_ATOL, assert_close_abs, assert_rounded, check_watchdog,
                         device_logits, f32_bits, host_bits)

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


def test_training_forward_every_row(training):
    w = training
    x = device_logits(w.logits, w.dtype)
    t = torch.from_numpy(w.target_ids).cuda()
    logp, lse = bil.logp_fwd(x, t, w.ignore_index, w.tile_v)
    torch.cuda.synchronize()
    ref_logp, ref_lse, bad = oracle.logp_fwd(w.logits, w.dtype, w.vocab, w.target_ids, w.ignore_index)
    assert bad == 0
    assert_close_abs(logp.cpu().numpy(), ref_logp, LOGP_ATOL, "logp")
    assert_close_abs(lse.cpu().numpy(), ref_lse, LOGP_ATOL, "lse")


SAMPLE_ROWS = np.array([0, 1, 255, 4096, 8191, 10000, 16382, 16383])


def test_training_backward_sampled_rows(training):
    w = training
    x = device_logits(w.logits, w.dtype)
    t = torch.from_numpy(w.target_ids).cuda()
    g = torch.from_numpy(w.grad_logp).cuda()
    _, lse = bil.logp_fwd(x, t, w.ignore_index, w.tile_v)
    d = bil.logp_bwd(x, t, lse, g, w.ignore_index)            # bf16, the benchmarked configuration
    torch.cuda.synchronize()
    rows = SAMPLE_ROWS
    sub = np.ascontiguousarray(w.logits[rows])
    ref_d, _ = oracle.logp_bwd(sub, w.dtype, w.vocab, w.target_ids[rows], w.grad_logp[rows].astype(np.float64))
    got = host_bits(d[torch.from_numpy(rows).cuda()])
    frac = assert_rounded(got, ref_d, "bfloat16", DLOGITS_ATOL, "dlogits")
    assert frac < 1e-3
    # the same kernel with a float32 output: the value before the final rounding
    d32 = bil.logp_bwd(x, t, lse, g, w.ignore_index, dlogits_dtype=torch.float32)
    torch.cuda.synchronize()
    got32 = d32[torch.from_numpy(rows).cuda()].cpu().numpy()
    assert_close_abs(got32, ref_d, DLOGITS_ATOL, "dlogits (float32 output)")
    del d32
