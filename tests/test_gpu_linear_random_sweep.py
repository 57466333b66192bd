"""A seeded random sweep of fused LM-head configurations against the oracle:
rows (one row tile or several, small batches included), hidden sizes (ragged
K blocks included), vocabularies (ragged last tile included), dtypes,
temperatures and the entropy.  logp, lse and entropy within their bounds; the
projection within the derived per-element bound; the rows of a sub-batch
carry the full batch's bits.
"""
import numpy as np
import pytest
import torch

import invariant_token_log_gb300 as bil
import oracle
import workloads as wl
from gpu_helpers import ENTROPY_ATOL, LOGP_ATOL, assert_close_abs, check_watchdog, device_logits, f32_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _watchdog():
    yield
    check_watchdog()


def _config(k):
    r = np.random.default_rng(1700 + k)
    dtype = ("bfloat16", "float16")[k % 2]
    n = int(r.choice([1, 3, 16, 127, 128, 129, int(r.integers(1, 400))]))
    h = int(r.choice([64, 200, 256, 520, 1024]))
    v = int(r.integers(1, 3001))
    temperature = float(r.choice([1.0, 0.7, 1.3]))
    return dtype, n, h, v, temperature


@pytest.mark.parametrize("k", range(20))
def test_random_linear_configuration(k):
    dtype, n, h, v, temperature = _config(k)
    seed = 1800 + k
    x = wl.linear_hidden(n, h, seed=seed, dtype=dtype)
    w = wl.linear_weight(v, h, seed=seed, dtype=dtype)
    t = wl.rng(seed, 1, n, v).integers(0, v, n, dtype=np.int64)
    t[::4] = wl.IGNORE_INDEX
    xd, wd, td = device_logits(x, dtype), device_logits(w, dtype), torch.from_numpy(t).cuda()
    logp, lse, ent, z = bil.linear_logp(xd, wd, td, temperature=temperature, return_entropy=True, return_logits=True)
    torch.cuda.synchronize()
    rl, rs, bad, rh = oracle.linear_logp_fwd(x, w, dtype, t, temperature=temperature, entropy=True)
    assert bad == 0
    assert_close_abs(logp.cpu().numpy(), rl, LOGP_ATOL, "logp")
    assert_close_abs(lse.cpu().numpy(), rs, LOGP_ATOL, "lse")
    assert_close_abs(ent.cpu().numpy(), rh, ENTROPY_ATOL, "entropy")
    zr = oracle.linear_logits(x, w, dtype)
    bound = (np.abs(oracle.widen(x, dtype)) @ np.abs(oracle.widen(w, dtype)).T) * 2.0 ** -20 + 1e-6
    assert np.all(np.abs(z.cpu().numpy().astype(np.float64) - zr) <= bound)
    # a sub-batch of rows (fewer than one row tile when possible) carries the same bits
    idx = np.sort(wl.rng(seed, 3).permutation(n)[:max(1, n // 3)])
    sel = torch.from_numpy(idx).cuda()
    sub = bil.linear_logp(xd.index_select(0, sel), wd, td.index_select(0, sel), temperature=temperature,
                          return_entropy=True)
    torch.cuda.synchronize()
    for a, b in zip(sub, (logp, lse, ent)):
        assert np.array_equal(f32_bits(a), f32_bits(b)[idx])
