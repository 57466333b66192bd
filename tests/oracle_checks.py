"""Pins of the CPU oracle to things other than itself.

Each check takes the oracle build flags (``defines``) and raises AssertionError
when the oracle disagrees with what the pages or the mathematics fix:

  * brute force in 40-digit arithmetic on tiny inputs (no max shift, no tiles);
  * the pages' own reference semantics as a library routine
    (``torch.log_softmax(x.double()).gather`` and its autograd gradient);
  * closed forms (uniform logits, a one-hot spike, two classes, V = 1);
  * invariants (sum of probabilities, shift and permutation invariance, the
    gradient's row sum, central finite differences of the forward);
  * the tile construction: merged partials equal the whole-row value for any
    tile size and any split of the tiles between calls.
  * the ignore / invalid-target rules of the operator page;
  * the LM-head projection of the fused linear logp: 40-digit dot products,
    the library's float64 matmul, and unit-vector weights that select columns.

The same checks run against deliberately broken oracle builds in
``test_oracle_mutants.py``; every planted mistake must fail at least one.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(seed, n, v, scale=2.0, dtype="float32", grid=None, ld=None):
    """Random rows; columns past v (when ld > v) hold NaN so that reading them shows."""
    x = wl.rng(seed, 100, v).standard_normal((n, v), dtype=np.float32) * np.float32(scale)
    if grid is not None:  # coarse grid: shifts and +-h perturbations stay exact in float32
        x = np.round(x * grid) / grid
        x = x.astype(np.float32)
    if ld is not None and ld > v:
        x = np.concatenate([x, np.full((n, ld - v), np.nan, np.float32)], axis=1)
    return wl.store(x, dtype)


def _targets(seed, n, v, ignore_rows=()):
    t = wl.rng(seed, 101, v).integers(0, v, n, dtype=np.int64)
    for r in ignore_rows:
        t[r] = wl.IGNORE_INDEX
    return t


# ----------------------------------------------------------------------------
def check_widening(defines=()):
    """Stored -> float64 widening equals the library conversions, for all 2^16 patterns."""
    import torch
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.widen(bits, "bfloat16", defines=defines)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok]), "bf16 widening"
    got = oracle.widen(bits, "float16", defines=defines)
    ref = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok]), "fp16 widening"
    f = wl.rng(7, 1).standard_normal(1000).astype(np.float32)
    assert np.array_equal(oracle.widen(f, "float32", defines=defines), f.astype(np.float64))


def check_brute_force(defines=()):
    """Forward and backward against 40-digit arithmetic: log(sum exp) with no shift."""
    import mpmath
    mpmath.mp.dps = 40
    for seed, (n, v, dtype) in enumerate([(3, 1, "float32"), (4, 7, "bfloat16"), (4, 300, "float16"),
                                          (3, 513, "float32"), (2, 4096, "bfloat16")]):
        x = _rows(seed, n, v, dtype=dtype)
        t = _targets(seed, n, v, ignore_rows=(1,) if n > 2 else ())
        g = wl.rng(seed, 102).standard_normal(n)
        logp, lse, bad = oracle.logp_fwd(x, dtype, v, t, defines=defines)
        d, bad_b = oracle.logp_bwd(x, dtype, v, t, g, defines=defines)
        assert bad == 0 and bad_b == 0
        xv = oracle.widen(x, dtype)  # exact values (widening pinned separately)
        for r in range(n):
            if t[r] == wl.IGNORE_INDEX:
                assert logp[r] == 0.0 and lse[r] == 0.0
                assert np.all(d[r] == 0.0)
                continue
            total = mpmath.fsum(mpmath.exp(mpmath.mpf(float(c))) for c in xv[r])
            ref_lse = mpmath.log(total)
            ref = mpmath.mpf(float(xv[r, t[r]])) - ref_lse
            assert abs(float(ref) - logp[r]) <= 1e-12, (seed, r, float(ref), logp[r])
            assert abs(float(ref_lse) - lse[r]) <= 1e-12
            for c in range(0, v, max(1, v // 64)):
                p = mpmath.exp(mpmath.mpf(float(xv[r, c]))) / total
                ref_d = g[r] * ((1 if c == t[r] else 0) - p)
                assert abs(float(ref_d) - d[r, c]) <= 1e-12, (seed, r, c)
            c = int(t[r])
            p = mpmath.exp(mpmath.mpf(float(xv[r, c]))) / total
            assert abs(float(g[r] * (1 - p)) - d[r, c]) <= 1e-12


def check_library_log_softmax(defines=()):
    """The pages' reference semantics as a library routine, in float64 on the CPU."""
    import torch
    for seed, (n, v, dtype) in enumerate([(16, 4096, "float32"), (8, 1000, "bfloat16"),
                                          (8, 333, "float16"), (5, 8, "bfloat16")]):
        x = _rows(seed + 10, n, v, scale=3.0, dtype=dtype)
        t = _targets(seed + 10, n, v, ignore_rows=(0, n - 1))
        g = wl.rng(seed, 103).standard_normal(n)
        logp, lse, bad = oracle.logp_fwd(x, dtype, v, t, defines=defines)
        d, _ = oracle.logp_bwd(x, dtype, v, t, g, defines=defines)
        xt = torch.from_numpy(oracle.widen(x, dtype)).requires_grad_(True)
        tt = torch.from_numpy(t)
        active = tt != wl.IGNORE_INDEX
        safe = torch.where(active, tt, torch.zeros_like(tt))
        sel = torch.log_softmax(xt, dim=-1).gather(-1, safe.unsqueeze(-1)).squeeze(-1)
        out = torch.where(active, sel, torch.zeros_like(sel))
        (out * torch.from_numpy(g)).sum().backward()
        assert np.abs(out.detach().numpy() - logp).max() <= 1e-12, "forward vs log_softmax"
        assert np.abs(xt.grad.numpy() - d).max() <= 1e-12, "backward vs autograd"
        ref_lse = torch.logsumexp(xt.detach(), dim=-1).numpy()
        a = active.numpy()
        assert np.abs(ref_lse[a] - lse[a]).max() <= 1e-12


def check_closed_forms(defines=()):
    # uniform logits: every class has probability 1/V
    for v in (1, 300, 4096, 151936):
        for c in (0.0, 3.5, -7.0):
            x = np.full((1, v), c, np.float32)
            t = np.array([v // 3], np.int64)
            logp, lse, _ = oracle.logp_fwd(x, "float32", v, t, defines=defines)
            assert abs(logp[0] + math.log(v)) <= 1e-12, (v, c)
            assert abs(lse[0] - (c + math.log(v))) <= 1e-12
    # V = 1: the only class has probability 1
    x = np.array([[12.25], [-3.0]], np.float32)
    logp, _, _ = oracle.logp_fwd(x, "float32", 1, np.zeros(2, np.int64), defines=defines)
    assert np.all(logp == 0.0)
    # one-hot spike of height h over zeros
    v = 4096
    for h in (0.5, 4.0, 12.0, 40.0):
        x = np.zeros((2, v), np.float32)
        x[:, 1234] = h
        t = np.array([1234, 77], np.int64)
        logp, _, _ = oracle.logp_fwd(x, "float32", v, t, defines=defines)
        z = math.log1p((v - 1) * math.exp(-h))
        assert abs(logp[0] + z) <= 1e-12, h
        assert abs(logp[1] - (-h - z)) <= 1e-12, h
    # two classes: the logistic function
    for a, b in ((0.25, -1.5), (3.0, 3.0), (-20.0, 5.0)):
        x = np.array([[a, b], [a, b]], np.float32)
        logp, _, _ = oracle.logp_fwd(x, "float32", 2, np.array([0, 1], np.int64), defines=defines)
        assert abs(logp[0] + math.log1p(math.exp(-(a - b)))) <= 1e-12
        assert abs(logp[1] + math.log1p(math.exp(-(b - a)))) <= 1e-12


def check_invariants(defines=()):
    v = 513
    x = _rows(3, 1, v, scale=3.0, grid=64)
    # probabilities over all targets sum to one
    xs = np.repeat(x, v, axis=0)
    logp, _, _ = oracle.logp_fwd(xs, "float32", v, np.arange(v, dtype=np.int64), defines=defines)
    assert abs(np.exp(logp).sum() - 1.0) <= 1e-12
    # shift invariance (the grid keeps x + k exact in float32)
    t = np.array([17], np.int64)
    base, _, _ = oracle.logp_fwd(x, "float32", v, t, defines=defines)
    for k in (-50.0, 3.5, 1e3):
        y = (x + np.float32(k)).astype(np.float32)
        assert np.array_equal(y - np.float32(k), x)
        lp, _, _ = oracle.logp_fwd(y, "float32", v, t, defines=defines)
        assert abs(lp[0] - base[0]) <= 1e-9, k
    # permutation of the columns, with the target following its column
    perm = wl.rng(3, 9).permutation(v)
    lp, _, _ = oracle.logp_fwd(np.ascontiguousarray(x[:, perm]), "float32", v,
                               np.array([int(np.flatnonzero(perm == 17)[0])], np.int64), defines=defines)
    assert abs(lp[0] - base[0]) <= 1e-12
    # the gradient of a row sums to g * (1 - sum p) = 0
    g = np.array([-1.75])
    d, _ = oracle.logp_bwd(x, "float32", v, t, g, defines=defines)
    assert abs(d.sum()) <= 1e-12
    # the target column follows g, every other column moves against it
    assert d[0, 17] * g[0] > 0
    assert np.all(np.delete(d[0], 17) * g[0] <= 0)


def check_finite_differences(defines=()):
    """d(g*logp)/dx_c by central differences; the grid keeps x +- h exact."""
    v, h = 64, 2.0 ** -12
    x = _rows(4, 1, v, scale=2.0, grid=256)
    t = np.array([5], np.int64)
    g = np.array([0.8125])
    d, _ = oracle.logp_bwd(x, "float32", v, t, g, defines=defines)
    for c in (0, 5, 31, 63):
        xp = x.copy()
        xm = x.copy()
        xp[0, c] += np.float32(h)
        xm[0, c] -= np.float32(h)
        fp, _, _ = oracle.logp_fwd(xp, "float32", v, t, defines=defines)
        fm, _, _ = oracle.logp_fwd(xm, "float32", v, t, defines=defines)
        fd = g[0] * (fp[0] - fm[0]) / (2 * h)
        assert abs(fd - d[0, c]) <= 1e-6, (c, fd, d[0, c])


def check_tiles(defines=()):
    """Merged tile partials equal the whole-row LSE for any tile size and split."""
    for dtype, v, n in (("float32", 4096, 6), ("bfloat16", 1000, 5), ("float16", 777, 4)):
        x = _rows(5, n, v, scale=3.0, dtype=dtype, ld=-(-v // 4096) * 4096 + 8)
        t = _targets(5, n, v, ignore_rows=(2,))
        ref_logp, ref_lse, _ = oracle.logp_fwd(x, dtype, v, t, defines=defines)
        vals = oracle.widen(x, dtype)
        for tile in (8, 64, 512, 4096):
            nt = -(-v // tile)
            for split in (1, 2, 4):
                pm = np.full((n, nt), -np.inf)
                ps = np.zeros((n, nt))
                tl = np.full(n, np.nan)
                bounds = [(k * nt) // split for k in range(split + 1)]
                for k in reversed(range(split)):  # ranks may finish in any order
                    oracle.tile_partials(x, dtype, v, tile, bounds[k], bounds[k + 1], t,
                                         part_max=pm, part_sum=ps, target_logit=tl, defines=defines)
                logp, lse, _ = oracle.merge(pm, ps, tl, t, v, defines=defines)
                assert np.abs(logp - ref_logp).max() <= 1e-12, (dtype, tile, split)
                assert np.abs(lse - ref_lse).max() <= 1e-12
                for r in range(n):
                    if t[r] == wl.IGNORE_INDEX:
                        assert np.all(pm[r] == -np.inf) and np.all(ps[r] == 0.0)
                        continue
                    assert tl[r] == vals[r, t[r]]  # copied, never summed
                    for k in range(nt):
                        seg = vals[r, k * tile: min(v, (k + 1) * tile)]
                        assert pm[r, k] == seg.max()
                        assert 1.0 <= ps[r, k] <= len(seg)
    check_tiles_with_temperature(defines)


def check_tiles_with_temperature(defines=()):
    """Tile partials at a temperature T, split and merged, against the library
    log-softmax of x / T ("Reference Semantics" with the logits divided by T
    before the softmax); the copied target logit is x_t / T, and the tile
    maxima are the stored maxima divided by T."""
    import torch
    v, n, tile = 1000, 5, 64
    x = _rows(6, n, v, scale=3.0, dtype="bfloat16")
    t = _targets(6, n, v, ignore_rows=(1,))
    vals = oracle.widen(x, "bfloat16")
    active = t != wl.IGNORE_INDEX
    nt = -(-v // tile)
    for temp in (0.7, 2.0):
        ref_all = torch.log_softmax(torch.from_numpy(vals) / temp, -1)
        ref_lse = torch.logsumexp(torch.from_numpy(vals) / temp, -1).numpy()
        for split in (1, 3):
            pm = np.full((n, nt), -np.inf)
            ps = np.zeros((n, nt))
            tl = np.full(n, np.nan)
            bounds = [(k * nt) // split for k in range(split + 1)]
            for k in reversed(range(split)):
                oracle.tile_partials(x, "bfloat16", v, tile, bounds[k], bounds[k + 1], t, part_max=pm, part_sum=ps,
                                     target_logit=tl, temperature=temp, defines=defines)
            logp, lse, _ = oracle.merge(pm, ps, tl, t, v, defines=defines)
            for r in range(n):
                if not active[r]:
                    assert logp[r] == 0.0 and lse[r] == 0.0
                    continue
                assert abs(logp[r] - float(ref_all[r, t[r]])) <= 1e-12, (temp, split, r)
                assert abs(lse[r] - ref_lse[r]) <= 1e-12 * max(1.0, abs(ref_lse[r]))
                assert tl[r] == vals[r, t[r]] / temp
                for k in range(nt):
                    assert pm[r, k] == vals[r, k * tile: min(v, (k + 1) * tile)].max() / temp


def check_contract_rules(defines=()):
    rules = json.load(open(os.path.join(GOLDEN, "contract_rules.json")))
    assert rules["ignore_index_default"] == wl.IGNORE_INDEX
    v = 300
    x = _rows(6, 4, v, scale=2.0, dtype="bfloat16")
    # default ignore_index: -1 and V are invalid, V-1 is valid, -100 is ignored
    t = np.array([-1, v, v - 1, -100], np.int64)
    logp, lse, bad = oracle.logp_fwd(x, "bfloat16", v, t, defines=defines)
    assert bad == 2 and np.isnan(logp[0]) and np.isnan(logp[1])
    assert np.isfinite(logp[2]) and logp[2] < 0
    assert logp[3] == 0.0 and not np.signbit(logp[3]) and lse[3] == 0.0
    # ignore_index = -1 makes -1 an ignored row and -100 invalid
    logp, _, bad = oracle.logp_fwd(x, "bfloat16", v, t, ignore_index=-1, defines=defines)
    assert bad == 2 and logp[0] == 0.0 and np.isnan(logp[3])
    # ignored rows receive an all-zero gradient, padded output columns are zero
    d, bad = oracle.logp_bwd(x, "bfloat16", v, np.array([-100, 3, -100, 7], np.int64),
                             np.ones(4), out_cols=v + 12, defines=defines)
    assert bad == 0
    assert np.all(d[0] == 0.0) and np.all(d[2] == 0.0) and np.all(d[:, v:] == 0.0)
    assert not np.signbit(d[0]).any()
    check_nan_and_infinite_rows(defines)


def check_nan_and_infinite_rows(defines=()):
    """NaN and all -inf rows (a reading: the pages are silent) behave as the
    library's logsumexp and log-softmax do: a NaN anywhere in the row, even
    among -inf logits, gives NaN; an all -inf row gives lse = -inf and a NaN
    logp.  The whole-row forward and merged tile partials (the NaN in a tile of
    -inf) agree."""
    import torch
    v, tile = 64, 16
    x = np.tile(np.float32(0.5) * np.arange(v, dtype=np.float32), (4, 1))
    x[0, 10] = np.nan                       # NaN among finite logits
    x[1, :] = -np.inf                       # every logit -inf
    x[2, :] = -np.inf
    x[2, 40] = np.nan                       # NaN among -inf logits
    t = np.full(4, 3, np.int64)
    xt = torch.from_numpy(x.astype(np.float64))
    ref_lse = torch.logsumexp(xt, -1).numpy()
    ref_logp = torch.log_softmax(xt, -1)[:, 3].numpy()
    assert np.isnan(ref_lse[0]) and ref_lse[1] == -np.inf and np.isnan(ref_lse[2])
    logp, lse, bad = oracle.logp_fwd(x, "float32", v, t, defines=defines)
    nt = v // tile
    pm, ps, tl = oracle.tile_partials(x, "float32", v, tile, 0, nt, t, defines=defines)
    mlogp, mlse, mbad = oracle.merge(pm, ps, tl, t, v, defines=defines)
    assert bad == 0 and mbad == 0
    for got_logp, got_lse in ((logp, lse), (mlogp, mlse)):
        for r in range(3):
            assert np.isnan(got_logp[r]), r
            assert np.isnan(got_lse[r]) if np.isnan(ref_lse[r]) else got_lse[r] == ref_lse[r], r
        assert abs(got_logp[3] - ref_logp[3]) <= 1e-12 and abs(got_lse[3] - ref_lse[3]) <= 1e-12
    assert np.isnan(ps[2, 40 // tile]) and pm[2, 40 // tile] == -np.inf   # the tile holding the NaN


def check_minimal_example(defines=()):
    ex = json.load(open(os.path.join(GOLDEN, "minimal_example.json")))
    shape = ex["logits_shape"]
    n, v = int(np.prod(shape[:-1])), shape[-1]
    x = _rows(8, n, v, scale=1.0, dtype="bfloat16")
    t = _targets(8, n, v).reshape(shape[:-1])
    for pos in ex["ignored_positions"]:
        t[tuple(pos)] = ex["ignore_index"]
    logp, _, bad = oracle.logp_fwd(x, "bfloat16", v, t.reshape(-1), ex["ignore_index"], defines=defines)
    out = logp.astype(np.float32).reshape(t.shape)
    assert bad == 0
    assert list(out.shape) == ex["expect"]["out_shape"]
    assert out.dtype == np.float32 and str(out.dtype) == ex["expect"]["out_dtype"]
    assert out[0, 0] == ex["expect"]["out_at_ignored"]
    assert np.all(out.reshape(-1)[1:] < 0)


def check_special_values(defines=()):
    """A row of -inf has no distribution (NaN); NaN poisons its row only."""
    v = 40
    x = np.zeros((3, v), np.float32)
    x[0] = -np.inf
    x[1, 7] = np.nan
    x[2, :20] = -np.inf
    t = np.array([3, 3, 30], np.int64)
    logp, lse, _ = oracle.logp_fwd(x, "float32", v, t, defines=defines)
    assert lse[0] == -np.inf and np.isnan(logp[0])
    assert np.isnan(lse[1]) and np.isnan(logp[1])
    assert abs(logp[2] + math.log(20)) <= 1e-12


def check_entropy(defines=()):
    """Entropy: closed forms, the library's categorical entropy, 40-digit brute
    force, and the partials-merge identity."""
    import mpmath
    import torch
    # uniform logits: log V
    for v in (1, 7, 4096):
        x = np.full((1, v), 2.5, np.float32)
        _, _, _, h = oracle.logp_fwd(x, "float32", v, np.array([0], np.int64), entropy=True, defines=defines)
        assert abs(h[0] - math.log(v)) <= 1e-12, v
    # one spike of height hgt over zeros
    v, hgt = 1000, 6.0
    x = np.zeros((1, v), np.float32)
    x[0, 3] = hgt
    _, _, _, h = oracle.logp_fwd(x, "float32", v, np.array([3], np.int64), entropy=True, defines=defines)
    z = math.exp(hgt) + v - 1
    pt, po = math.exp(hgt) / z, 1 / z
    assert abs(h[0] + (pt * math.log(pt) + (v - 1) * po * math.log(po))) <= 1e-12
    # two classes: the binary entropy
    a, b = 1.25, -0.5
    x = np.array([[a, b]], np.float32)
    _, _, _, h = oracle.logp_fwd(x, "float32", 2, np.array([1], np.int64), entropy=True, defines=defines)
    q = 1 / (1 + math.exp(-(a - b)))
    assert abs(h[0] + q * math.log(q) + (1 - q) * math.log(1 - q)) <= 1e-12
    # the library routine, all element types, ignored rows 0
    for seed, (n, v, dtype) in enumerate([(6, 777, "float32"), (5, 1000, "bfloat16"), (4, 333, "float16")]):
        x = _rows(seed + 30, n, v, scale=3.0, dtype=dtype)
        t = _targets(seed + 30, n, v, ignore_rows=(1,))
        _, _, _, h = oracle.logp_fwd(x, dtype, v, t, entropy=True, defines=defines)
        ref = torch.distributions.Categorical(logits=torch.from_numpy(oracle.widen(x, dtype))).entropy().numpy()
        act = t != wl.IGNORE_INDEX
        assert np.abs(h[act] - ref[act]).max() <= 1e-12
        assert np.all(h[~act] == 0.0)
    # 40-digit brute force: -sum p log p with p = exp(x) / sum exp(x)
    mpmath.mp.dps = 40
    x = _rows(40, 2, 60, scale=2.0)
    _, _, _, h = oracle.logp_fwd(x, "float32", 60, np.array([0, 1], np.int64), entropy=True, defines=defines)
    for r in range(2):
        tot = mpmath.fsum(mpmath.exp(mpmath.mpf(float(c))) for c in x[r])
        ref = -mpmath.fsum((mpmath.exp(mpmath.mpf(float(c))) / tot) * (mpmath.mpf(float(c)) - mpmath.log(tot))
                           for c in x[r])
        assert abs(float(ref) - h[r]) <= 1e-12
    # -inf logits (a masked vocabulary slice, and one whole -inf tile) carry no
    # probability and add nothing to the entropy or its gradient
    v = 1024
    x = _rows(42, 2, v, scale=2.0)
    x[:, 100:140] = -np.inf
    x[:, 512:768] = -np.inf
    t2 = np.array([5, 900], np.int64)
    _, _, _, h = oracle.logp_fwd(x, "float32", v, t2, entropy=True, defines=defines)
    keep = np.isfinite(x[0])
    ref = torch.distributions.Categorical(logits=torch.from_numpy(x[0][keep].astype(np.float64))).entropy().item()
    assert np.all(np.isfinite(h)) and abs(h[0] - ref) <= 1e-12
    pm, ps, pe = np.full((2, 4), -np.inf), np.zeros((2, 4)), np.zeros((2, 4))
    tl = np.full(2, np.nan)
    oracle.tile_partials(x, "float32", v, 256, 0, 4, t2, part_max=pm, part_sum=ps, target_logit=tl, part_ent=pe,
                         defines=defines)
    assert np.all(pm[:, 2] == -np.inf)
    _, _, _, hm = oracle.merge(pm, ps, tl, t2, v, part_ent=pe, defines=defines)
    assert np.abs(hm - h).max() <= 1e-12
    d, _ = oracle.logp_bwd(x, "float32", v, t2, np.ones(2), grad_entropy=np.ones(2), defines=defines)
    assert np.all(np.isfinite(d)) and np.all(d[:, 512:768] == 0.0)
    # merged entropy partials equal the whole-row entropy for any tile size and split
    for dtype, v, n in (("float32", 3000, 4), ("bfloat16", 1000, 3)):
        x = _rows(41, n, v, scale=3.0, dtype=dtype)
        t = _targets(41, n, v, ignore_rows=(0,))
        _, _, _, ref = oracle.logp_fwd(x, dtype, v, t, entropy=True, defines=defines)
        for tile in (8, 512, 4096):
            nt = -(-v // tile)
            for split in (1, 3):
                pm, ps, pe = np.full((n, nt), -np.inf), np.zeros((n, nt)), np.zeros((n, nt))
                tl = np.full(n, np.nan)
                bnd = [(k * nt) // split for k in range(split + 1)]
                for k in range(split):
                    oracle.tile_partials(x, dtype, v, tile, bnd[k], bnd[k + 1], t, part_max=pm, part_sum=ps,
                                         target_logit=tl, part_ent=pe, defines=defines)
                _, _, _, h = oracle.merge(pm, ps, tl, t, v, part_ent=pe, defines=defines)
                assert np.abs(h - ref).max() <= 1e-12, (dtype, tile, split)


def check_temperature(defines=()):
    """Temperature: dividing by a power of two is exact, so logp(x, T) must equal
    logp(x / T, 1); arbitrary T against the library log-softmax of x / T; the
    backward against finite differences."""
    import torch
    v = 513
    x = _rows(50, 3, v, scale=3.0, grid=64)
    t = np.array([5, 100, 512], np.int64)
    for temp in (2.0, 0.5, 4.0):
        y = (x / np.float32(temp)).astype(np.float32)
        assert np.array_equal(y * np.float32(temp), x)
        a, la, _, ha = oracle.logp_fwd(x, "float32", v, t, temperature=temp, entropy=True, defines=defines)
        b, lb, _, hb = oracle.logp_fwd(y, "float32", v, t, entropy=True, defines=defines)
        assert np.abs(a - b).max() <= 1e-12 and np.abs(la - lb).max() <= 1e-12 and np.abs(ha - hb).max() <= 1e-12
    temp = 0.7
    xt = torch.from_numpy(oracle.widen(x, "float32")) / temp
    ref = torch.log_softmax(xt, -1).gather(-1, torch.from_numpy(t)[:, None])[:, 0].numpy()
    got, _, _ = oracle.logp_fwd(x, "float32", v, t, temperature=temp, defines=defines)
    assert np.abs(got - ref).max() <= 1e-12
    # d(g logp + gh H)/dx by central differences, with a temperature
    v, hstep = 48, 2.0 ** -12
    x = _rows(51, 1, v, scale=2.0, grid=256)
    t1 = np.array([7], np.int64)
    g, gh = np.array([0.75]), np.array([-1.5])
    d, _ = oracle.logp_bwd(x, "float32", v, t1, g, temperature=temp, grad_entropy=gh, defines=defines)

    def f(xx):
        lp, _, _, hh = oracle.logp_fwd(xx, "float32", v, t1, temperature=temp, entropy=True, defines=defines)
        return g[0] * lp[0] + gh[0] * hh[0]
    for c in (0, 7, 20, 47):
        xp, xm = x.copy(), x.copy()
        xp[0, c] += np.float32(hstep)
        xm[0, c] -= np.float32(hstep)
        fd = (f(xp) - f(xm)) / (2 * hstep)
        assert abs(fd - d[0, c]) <= 1e-6, (c, fd, d[0, c])


def check_entropy_gradient_library(defines=()):
    """The backward with an entropy term against autograd of the library's
    log-softmax and categorical entropy, in float64."""
    import torch
    for seed, (n, v, dtype, temp) in enumerate([(5, 300, "bfloat16", 1.0), (4, 1000, "float32", 0.8)]):
        x = _rows(seed + 60, n, v, scale=3.0, dtype=dtype)
        t = _targets(seed + 60, n, v, ignore_rows=(2,))
        g = wl.rng(seed, 61).standard_normal(n)
        gh = wl.rng(seed, 62).standard_normal(n)
        d, _ = oracle.logp_bwd(x, dtype, v, t, g, temperature=temp, grad_entropy=gh, defines=defines)
        xt = torch.from_numpy(oracle.widen(x, dtype)).requires_grad_(True)
        z = xt / temp
        tt = torch.from_numpy(t)
        act = tt != wl.IGNORE_INDEX
        sel = torch.log_softmax(z, -1).gather(-1, torch.where(act, tt, 0)[:, None])[:, 0]
        ent = torch.distributions.Categorical(logits=z).entropy()
        loss = (torch.where(act, sel, 0) * torch.from_numpy(g)).sum() + \
               (torch.where(act, ent, 0) * torch.from_numpy(gh)).sum()
        loss.backward()
        assert np.abs(xt.grad.numpy() - d).max() <= 1e-12





def check_linear(defines=()):
    """The fused LM-head + logp ("[RFC][ROCm] End-to-end optimization of bitwise
    VIME R/R beyond native P/P", "Workstream 3"): z = hidden . weight^T, then the
    operator on z."""
    import mpmath
    import torch
    # 40-digit brute force: dot products, log-sum-exp without a shift, entropy
    mpmath.mp.dps = 40
    n, h, v = 2, 24, 9
    x = _rows(70, n, h, scale=1.0, dtype="bfloat16")
    w = _rows(71, v, h, scale=0.5, dtype="bfloat16")
    t = np.array([4, 8], np.int64)
    lp, ls, bad, ent = oracle.linear_logp_fwd(x, w, "bfloat16", t, entropy=True, defines=defines)
    xf, wf = oracle.widen(x, "bfloat16"), oracle.widen(w, "bfloat16")
    assert bad == 0
    for r in range(n):
        z = [mpmath.fsum(mpmath.mpf(float(xf[r, k])) * mpmath.mpf(float(wf[c, k])) for k in range(h))
             for c in range(v)]
        lse = mpmath.log(mpmath.fsum(mpmath.exp(zc) for zc in z))
        assert abs(float(z[t[r]] - lse) - lp[r]) <= 1e-12
        assert abs(float(lse) - ls[r]) <= 1e-12
        hh = -mpmath.fsum(mpmath.exp(zc - lse) * (zc - lse) for zc in z)
        assert abs(float(hh) - ent[r]) <= 1e-12
    # the library routine in float64, with a temperature, ragged sizes, ignored rows
    for seed, (n, h, v, dtype, temp) in enumerate([(5, 64, 300, "bfloat16", 1.0), (4, 40, 257, "float16", 0.7),
                                                    (3, 33, 129, "float32", 1.3)]):
        x = _rows(seed + 72, n, h, scale=1.0, dtype=dtype)
        w = _rows(seed + 73, v, h, scale=3.0 / math.sqrt(h), dtype=dtype)
        t = _targets(seed + 72, n, v, ignore_rows=(1,))
        lp, ls, _, ent = oracle.linear_logp_fwd(x, w, dtype, t, temperature=temp, entropy=True, defines=defines)
        z = torch.from_numpy(oracle.widen(x, dtype)) @ torch.from_numpy(oracle.widen(w, dtype)).T / temp
        tt = torch.from_numpy(t)
        act = (tt != wl.IGNORE_INDEX).numpy()
        ref = torch.log_softmax(z, -1).gather(-1, torch.where(tt == wl.IGNORE_INDEX, 0, tt)[:, None])[:, 0].numpy()
        href = torch.distributions.Categorical(logits=z).entropy().numpy()
        assert np.abs(lp[act] - ref[act]).max() <= 1e-12, (dtype, "logp")
        assert np.abs(ent[act] - href[act]).max() <= 1e-12, (dtype, "entropy")
        assert np.all(lp[~act] == 0.0)
    # weight rows that are unit vectors select hidden columns: z = hidden[:, cols]
    n, h = 6, 48
    x = _rows(76, n, h, scale=3.0, dtype="bfloat16")
    cols = wl.rng(76, 1).permutation(h)[:20]
    w = np.zeros((20, h), np.float32)
    w[np.arange(20), cols] = 1.0
    z = oracle.linear_logits(x, wl.store(w, "bfloat16"), "bfloat16", defines=defines)
    assert np.array_equal(z, oracle.widen(x, "bfloat16")[:, cols])


def check_linear_backward(defines=()):
    """The fused LM-head's backward ("Workstream 3", the autograd actor path):
    autograd of the library's float64 matmul + log-softmax + entropy, central
    differences on float64 inputs, and the bilinear identity
    <dX, X> = <dZ, z> = <dW, W> (z is bilinear in X and W)."""
    import torch
    for seed, (n, h, v, dtype, temp, ent) in enumerate([(5, 40, 300, "bfloat16", 1.0, False),
                                                         (4, 24, 257, "float16", 0.8, True),
                                                         (6, 16, 100, "float32", 1.3, True)]):
        x = _rows(seed + 80, n, h, scale=1.0, dtype=dtype)
        w = _rows(seed + 81, v, h, scale=3.0 / math.sqrt(h), dtype=dtype)
        t = _targets(seed + 80, n, v, ignore_rows=(1,))
        g = wl.rng(seed, 82).standard_normal(n)
        gh = wl.rng(seed, 83).standard_normal(n) if ent else None
        dx, dw, dz, bad = oracle.linear_logp_bwd(x, w, dtype, t, g, temperature=temp, grad_entropy=gh,
                                                  defines=defines)
        assert bad == 0
        xt = torch.from_numpy(oracle.widen(x, dtype)).requires_grad_(True)
        wt = torch.from_numpy(oracle.widen(w, dtype)).requires_grad_(True)
        z = xt @ wt.T / temp
        tt = torch.from_numpy(t)
        act = tt != wl.IGNORE_INDEX
        sel = torch.log_softmax(z, -1).gather(-1, torch.where(act, tt, 0)[:, None])[:, 0]
        loss = (torch.where(act, sel, 0) * torch.from_numpy(g)).sum()
        if ent:
            hh = torch.distributions.Categorical(logits=z).entropy()
            loss = loss + (torch.where(act, hh, 0) * torch.from_numpy(gh)).sum()
        loss.backward()
        assert np.abs(xt.grad.numpy() - dx).max() <= 1e-12 * max(1.0, np.abs(dx).max()), (dtype, "dhidden")
        assert np.abs(wt.grad.numpy() - dw).max() <= 1e-12 * max(1.0, np.abs(dw).max()), (dtype, "dweight")
        zz = oracle.linear_logits(x, w, dtype)
        ip_x = float((dx * oracle.widen(x, dtype)).sum())
        ip_w = float((dw * oracle.widen(w, dtype)).sum())
        ip_z = float((dz * zz).sum())
        assert abs(ip_x - ip_z) <= 1e-9 * max(1.0, abs(ip_z)) and abs(ip_w - ip_z) <= 1e-9 * max(1.0, abs(ip_z))
    # central differences on float64 inputs (every x +- h is exact on this grid)
    n, h, v, hs = 2, 8, 30, 2.0 ** -20
    x = np.round(wl.rng(90, 1).standard_normal((n, h)) * 64) / 64
    w = np.round(wl.rng(90, 2).standard_normal((v, h)) * 64) / 64
    t = np.array([3, 17], np.int64)
    g, gh = np.array([0.75, -1.25]), np.array([0.5, 2.0])
    dx, dw, _, _ = oracle.linear_logp_bwd(x, w, "float64", t, g, temperature=0.9, grad_entropy=gh, defines=defines)

    def f(xx, ww):
        lp, _, _, hh = oracle.linear_logp_fwd(xx, ww, "float64", t, temperature=0.9, entropy=True, defines=defines)
        return float((g * lp + gh * hh).sum())
    for (r, k) in ((0, 0), (1, 5), (0, 7)):
        xp, xm = x.copy(), x.copy()
        xp[r, k] += hs
        xm[r, k] -= hs
        assert abs((f(xp, w) - f(xm, w)) / (2 * hs) - dx[r, k]) <= 1e-6, ("dhidden", r, k)
    for (c, k) in ((3, 1), (17, 6), (29, 0)):
        wp, wm = w.copy(), w.copy()
        wp[c, k] += hs
        wm[c, k] -= hs
        assert abs((f(x, wp) - f(x, wm)) / (2 * hs) - dw[c, k]) <= 1e-6, ("dweight", c, k)


def check_rounding_helpers():
    """float64 -> bf16 rounding: ties to even at exact midpoints, nearest elsewhere,
    and equal to the library float32 -> bf16 conversion on float32 values."""
    import torch
    r = wl.rng(11, 1)
    b = r.integers(0, 0x7F7F, 20000).astype(np.uint16)  # finite positive bf16 values
    b = np.concatenate([b, b | 0x8000]).astype(np.uint16)
    lo = oracle.bf16_bits_to_float64(b)
    hi = oracle.bf16_bits_to_float64(b + 1)            # next value away from zero
    mid = (lo + hi) / 2                                 # exact in float64
    got = oracle.round_to_bf16_bits(mid)
    even = np.where((b & 1) == 0, b, b + 1).astype(np.uint16)
    assert np.array_equal(got, even), "ties to even"
    eps = np.abs(hi - lo) * 2.0 ** -20
    assert np.array_equal(oracle.round_to_bf16_bits(mid - np.sign(mid) * eps), b)
    assert np.array_equal(oracle.round_to_bf16_bits(mid + np.sign(mid) * eps), (b + 1).astype(np.uint16))
    f = (r.standard_normal(100000) * np.exp(r.uniform(-80, 80, 100000))).astype(np.float32)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.round_to_bf16_bits(f.astype(np.float64)), ref)
    tiny = np.array([2.0 ** -140, -(2.0 ** -133) * 1.5, 0.0, -0.0, 1e39, -1e39])
    assert list(oracle.round_to_bf16_bits(tiny)) == [0x0000, 0x8002, 0x0000, 0x8000, 0x7F80, 0xFF80]


ALL_CHECKS = [check_widening, check_brute_force, check_library_log_softmax, check_closed_forms,
              check_invariants, check_finite_differences, check_tiles, check_contract_rules,
              check_minimal_example, check_special_values, check_entropy, check_temperature,
              check_entropy_gradient_library, check_linear, check_linear_backward]
