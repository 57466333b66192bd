"""A seeded random sweep of configurations against the oracle: rows, widths
(odd ones included), tile sizes, dtypes, temperatures, the entropy output,
shifted base pointers and padded row pitches.  For each configuration the
forward and the backward agree with the oracle within the bounds of
tests/gpu_helpers.py, and the split path (tile partials, then the merge)
gives the fused forward's bits.
"""
import numpy as np
import pytest
import torch

import invariant_token_log_gb300 as bil
import oracle
import workloads as wl
from gpu_helpers import (ENTROPY_ATOL, LOGP_ATOL, assert_close_abs, assert_close_elementwise, check_watchdog,
                         device_logits, entropy_grad_tol, f32_bits)

pytestmark = pytest.mark.gpu

DTYPES = ["float32", "bfloat16", "float16"]


@pytest.fixture(autouse=True)
def _watchdog():
    yield
    check_watchdog()


def _config(k):
    r = np.random.default_rng(900 + k)
    dtype = DTYPES[k % 3]
    n = int(r.integers(1, 201))
    v = int(r.integers(1, 20001))
    eb = 4 if dtype == "float32" else 2
    tiles = [t for t in (64, 256, 1024, 2048, 4096, 8192) if t * eb <= 64 * 1024]
    tile = int(r.choice(tiles))
    temperature = float(r.choice([1.0, 0.7, 1.5]))
    ent = bool(r.integers(0, 2))
    shift = int(r.integers(0, 4))
    pad = int(r.choice([0, 1, 5, 8]))
    return dtype, n, v, tile, temperature, ent, shift, pad


@pytest.mark.parametrize("k", range(40))
def test_random_configuration(k):
    dtype, n, v, tile, temperature, ent, shift, pad = _config(k)
    w = wl.random_rows(seed=1000 + k, n_rows=n, vocab=v, ld=v + pad, dtype=dtype, scale=3.0, tile_v=tile,
                       ignore_every=int(np.random.default_rng(k).integers(0, 6)))
    flat = device_logits(w.logits, dtype).reshape(-1)
    big = torch.empty(flat.numel() + 8, dtype=flat.dtype, device="cuda")
    big[shift:shift + flat.numel()] = flat
    x = big[shift:shift + flat.numel()].view(n, v + pad)
    t = torch.from_numpy(w.target_ids).cuda()
    g = torch.from_numpy(w.grad_logp).cuda()
    gh = torch.from_numpy(wl.rng(1000 + k, 9).standard_normal(n).astype(np.float32)).cuda()

    res = bil.logp_fwd(x, t, w.ignore_index, tile, vocab=v, temperature=temperature, return_entropy=ent)
    logp, lse = res[0], res[1]
    kw = dict(entropy=res[2], grad_entropy=gh) if ent else {}
    d = bil.logp_bwd(x, t, lse, g, w.ignore_index, vocab=v, temperature=temperature,
                     dlogits_dtype=torch.float32, **kw)
    # the split path: partials of every tile, then the fixed-order merge
    nt = -(-v // tile)
    pm = torch.empty((n, nt), device="cuda")
    ps = torch.empty_like(pm)
    pe = torch.empty_like(pm) if ent else None
    tl = torch.full((n,), float("nan"), device="cuda")
    bil.logp_tile_partials(x, t, v, tile, 0, nt, pm, ps, tl, w.ignore_index, temperature=temperature, part_ent=pe)
    split = bil.logp_merge(pm, ps, nt, tl, t, v, w.ignore_index, part_ent=pe)
    torch.cuda.synchronize()
    for a, b in zip(res, split):
        assert np.array_equal(f32_bits(a), f32_bits(b)), (dtype, n, v, tile, temperature, ent, shift, pad)

    o = oracle.logp_fwd(w.logits, dtype, v, w.target_ids, w.ignore_index, temperature=temperature, entropy=ent)
    assert o[2] == 0
    assert_close_abs(logp.cpu().numpy(), o[0], LOGP_ATOL, "logp")
    assert_close_abs(lse.cpu().numpy(), o[1], LOGP_ATOL, "lse")
    if ent:
        assert_close_abs(res[2].cpu().numpy(), o[3], ENTROPY_ATOL, "entropy")
    ref_d, _ = oracle.logp_bwd(w.logits, dtype, v, w.target_ids, w.grad_logp.astype(np.float64), w.ignore_index,
                               out_cols=v + pad, temperature=temperature,
                               grad_entropy=gh.cpu().numpy().astype(np.float64) if ent else None)
    active = (w.target_ids != w.ignore_index)[:, None]
    z = oracle.widen(w.logits, dtype)[:, :v] / temperature
    with np.errstate(over="ignore", invalid="ignore"):
        a = z - o[1][:, None]
        p = np.where(active, np.exp(a), 0.0)
        a_plus_h = a + (o[3][:, None] if ent else 0.0)
    ghn = gh.cpu().numpy() if ent else np.zeros(n)
    tol = np.zeros((n, v + pad)) + 1e-6
    tol[:, :v] = entropy_grad_tol(p, np.where(active, a_plus_h, 0.0), w.grad_logp.astype(np.float64), ghn,
                                  1.0 / temperature)
    assert_close_elementwise(d.cpu().numpy(), ref_d, tol, "dlogits")
