"""Properties the oracle must have on random small inputs (widths, tile sizes,
dtypes, temperatures, ignored rows), beyond the fixed pins:

- normalisation: sum_c exp(z_c - lse) = 1, z = x / T (the "Reference
  Semantics" log-softmax);
- the tile method ("Tensor Parallel", steps 1-6): partials of any tile width,
  filled by ranges in any split, merged, give the whole-row result;
- the backward's rows sum to g * (1 - sum p) = 0 (the gradient of a log-softmax).
"""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

import oracle  # noqa: E402
import workloads as wl  # noqa: E402

TOL = 1e-12


@st.composite
def cases(draw):
    n = draw(st.integers(min_value=1, max_value=4))
    v = draw(st.integers(min_value=1, max_value=700))
    dtype = draw(st.sampled_from(["float32", "bfloat16", "float16"]))
    tile = draw(st.sampled_from([8, 16, 64, 512]))
    temperature = draw(st.sampled_from([1.0, 0.7, 2.0]))
    seed = draw(st.integers(min_value=0, max_value=2**31 - 1))
    r = np.random.default_rng(seed)
    x = (r.standard_normal((n, v)) * draw(st.sampled_from([0.5, 3.0, 8.0]))).astype(np.float32)
    t = r.integers(0, v, n).astype(np.int64)
    if n > 1:
        t[r.integers(0, n)] = -100
    return wl.store(x, dtype), dtype, v, tile, temperature, t


@settings(max_examples=60, deadline=None)
@given(cases())
def test_softmax_normalises(case):
    x, dtype, v, _, temperature, t = case
    logp, lse, bad = oracle.logp_fwd(x, dtype, v, t, temperature=temperature)
    assert bad == 0
    z = oracle.widen(x, dtype)[:, :v] / temperature
    for i in range(x.shape[0]):
        if t[i] == -100:
            assert logp[i] == 0.0 and lse[i] == 0.0
        else:
            assert abs(np.exp(z[i] - lse[i]).sum() - 1.0) <= TOL
            assert abs(logp[i] - (z[i, t[i]] - lse[i])) <= TOL * max(1.0, abs(lse[i]))


@settings(max_examples=60, deadline=None)
@given(cases(), st.data())
def test_tile_partials_in_any_split_merge_to_the_whole_row(case, data):
    x, dtype, v, tile, temperature, t = case
    ref_logp, ref_lse, _ = oracle.logp_fwd(x, dtype, v, t, temperature=temperature)
    num_tiles = -(-v // tile)
    k = data.draw(st.integers(min_value=1, max_value=min(num_tiles, 4)))
    cuts = sorted(data.draw(st.sets(st.integers(min_value=1, max_value=max(1, num_tiles - 1)),
                                    min_size=k - 1, max_size=k - 1))) if k > 1 and num_tiles > 1 else []
    bounds = [0] + cuts + [num_tiles]
    pm = ps = tl = None
    for b, e in reversed(list(zip(bounds[:-1], bounds[1:]))):  # ranges finishing in any order
        pm, ps, tl = oracle.tile_partials(x, dtype, v, tile, b, e, t, part_max=pm, part_sum=ps, target_logit=tl,
                                          temperature=temperature)
    logp, lse, bad = oracle.merge(pm, ps, tl, t, v)
    assert bad == 0
    np.testing.assert_allclose(lse, ref_lse, rtol=TOL, atol=TOL)
    np.testing.assert_allclose(logp, ref_logp, rtol=TOL, atol=TOL)


@settings(max_examples=60, deadline=None)
@given(cases())
def test_backward_rows_sum_to_zero(case):
    x, dtype, v, _, temperature, t = case
    n = x.shape[0]
    g = np.linspace(-2.0, 3.0, n)
    d, bad = oracle.logp_bwd(x, dtype, v, t, g, temperature=temperature)
    assert bad == 0
    for i in range(n):
        if t[i] == -100:
            assert np.all(d[i] == 0.0)
        else:
            assert abs(d[i].sum()) <= 1e-10 * max(1.0, abs(g[i])) / temperature
