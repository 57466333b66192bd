"""Entropy output and temperature, against the CPU oracle and for bit-invariance.

The linear-logp operator of "[RFC][ROCm] End-to-end optimization of bitwise
VIME R/R beyond native P/P" (section "Workstream 3: fused ROCm LM-head and
linear logp") optionally returns the full-vocabulary entropy and applies a
temperature at one fixed point; both must keep the row's bits independent of
its batch and of how the vocabulary tiles are split.
"""
import numpy as np
import pytest
import torch

import invariant_token_log_gb300 as bil
import oracle
import workloads as wl
from gpu_helpers import (ENTROPY_ATOL, LOGP_ATOL, assert_close_abs, assert_close_elementwise,
                         check_watchdog, device_logits, entropy_grad_tol, f32_bits)


def oracle_grad_bound(w, temperature, g, gh):
    """entropy_grad_tol from the oracle's own p, a + H for workload w."""
    _, lse, _, H = oracle.logp_fwd(w.logits, w.dtype, w.vocab, w.target_ids, w.ignore_index,
                                   temperature=temperature, entropy=True)
    z = oracle.widen(np.ascontiguousarray(w.logits[:, :w.vocab]), w.dtype) / temperature
    a = z - lse[:, None]
    p = np.exp(a)
    rcp = float(np.float32(1.0 / temperature))
    with np.errstate(invalid="ignore"):
        tol = entropy_grad_tol(p, a + H[:, None], np.asarray(g, np.float64), np.asarray(gh, np.float64), rcp)
    tol[w.target_ids == w.ignore_index] = 1e-6  # ignored rows are exactly zero
    return tol

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _watchdog():
    yield
    check_watchdog()


CASES = [("float32", 4096, 512), ("bfloat16", 12345, 1024), ("float16", 300, 512), ("bfloat16", 151936, 4096)]


@pytest.mark.parametrize("temperature", [1.0, 0.7, 2.0])
@pytest.mark.parametrize("dtype,v,tile", CASES)
def test_forward_entropy_vs_oracle(dtype, v, tile, temperature):
    n = 9 if v < 100000 else 6
    w = wl.random_rows(seed=v + 3, n_rows=n, vocab=v, dtype=dtype, tile_v=tile, ignore_every=4)
    x = device_logits(w.logits, dtype)
    t = torch.from_numpy(w.target_ids).cuda()
    logp, lse, ent = bil.logp_fwd(x, t, w.ignore_index, tile, temperature=temperature, return_entropy=True)
    torch.cuda.synchronize()
    rl, rs, bad, rh = oracle.logp_fwd(w.logits, dtype, v, w.target_ids, w.ignore_index,
                                      temperature=temperature, entropy=True)
    assert bad == 0
    assert_close_abs(logp.cpu().numpy(), rl, LOGP_ATOL, "logp")
    assert_close_abs(lse.cpu().numpy(), rs, LOGP_ATOL, "lse")
    assert_close_abs(ent.cpu().numpy(), rh, ENTROPY_ATOL, "entropy")
    ign = w.target_ids == w.ignore_index
    assert np.all(f32_bits(ent)[ign] == 0)


def test_entropy_leaves_logp_bits_alone_and_temperature_one_is_identity():
    w = wl.random_rows(seed=8, n_rows=40, vocab=151936, dtype="bfloat16", tile_v=4096, ignore_every=5)
    x = device_logits(w.logits, "bfloat16")
    t = torch.from_numpy(w.target_ids).cuda()
    a = bil.logp_fwd(x, t, w.ignore_index, 4096)
    b = bil.logp_fwd(x, t, w.ignore_index, 4096, temperature=1.0, return_entropy=True)
    torch.cuda.synchronize()
    assert np.array_equal(f32_bits(a[0]), f32_bits(b[0]))
    assert np.array_equal(f32_bits(a[1]), f32_bits(b[1]))


@pytest.mark.parametrize("temperature", [1.0, 0.8])
def test_split_entropy_is_bitwise_fused(temperature):
    n, v, tile = 33, 151936, 4096
    w = wl.random_rows(seed=13, n_rows=n, vocab=v, dtype="bfloat16", tile_v=tile, ignore_every=6)
    x = device_logits(w.logits, "bfloat16")
    t = torch.from_numpy(w.target_ids).cuda()
    fused = bil.logp_fwd(x, t, w.ignore_index, tile, temperature=temperature, return_entropy=True)
    nt = -(-v // tile)
    for k in (1, 2, 4):
        pm = torch.full((n, nt), float("nan"), device="cuda")
        ps = torch.full_like(pm, float("nan"))
        pe = torch.full_like(pm, float("nan"))
        tl = torch.full((n,), float("nan"), device="cuda")
        b = [(r * nt) // k for r in range(k + 1)]
        for r in range(k):
            bil.logp_tile_partials(x[:, b[r] * tile:], t, v, tile, b[r], b[r + 1], pm, ps, tl, w.ignore_index,
                                   temperature=temperature, part_ent=pe)
        split = bil.logp_merge(pm, ps, nt, tl, t, v, w.ignore_index, part_ent=pe)
        torch.cuda.synchronize()
        for got, ref in zip(split, fused):
            assert np.array_equal(f32_bits(got), f32_bits(ref)), k
    # and the oracle's entropy partials agree
    rm, rs, rtl = oracle.tile_partials(w.logits, "bfloat16", v, tile, 0, nt, w.target_ids, w.ignore_index,
                                       temperature=temperature, part_ent=(rpe := np.zeros((n, nt))))
    act = w.target_ids != w.ignore_index
    got_pe = pe.cpu().numpy()
    assert np.abs(got_pe[act] - rpe[act]).max() <= 1e-5 * np.abs(rpe[act]).max()


def test_entropy_rows_are_batch_invariant():
    bank = wl.decode_bank()
    x = device_logits(bank.logits, "bfloat16")
    t = torch.from_numpy(bank.target_ids).cuda()
    ref = bil.logp_fwd(x, t, -100, 4096, temperature=0.9, return_entropy=True)
    torch.cuda.synchronize()
    for n in (1, 3, 64):
        for draw in wl.decode_draws(n, draws=3):
            idx = torch.from_numpy(draw).cuda()
            got = bil.logp_fwd(x.index_select(0, idx), t.index_select(0, idx), -100, 4096, temperature=0.9,
                               return_entropy=True)
            for g, r in zip(got, ref):
                assert np.array_equal(f32_bits(g), f32_bits(r)[draw])


@pytest.mark.parametrize("temperature", [1.0, 0.7])
@pytest.mark.parametrize("dtype,v", [("float32", 4096), ("bfloat16", 9999)])
def test_backward_with_entropy_and_temperature_vs_oracle(dtype, v, temperature):
    n = 7
    w = wl.random_rows(seed=v + 17, n_rows=n, vocab=v, dtype=dtype, scale=2.0, tile_v=512, ignore_every=3)
    gh = wl.rng(5, 77).standard_normal(n).astype(np.float32)
    x = device_logits(w.logits, dtype)
    t = torch.from_numpy(w.target_ids).cuda()
    logp, lse, ent = bil.logp_fwd(x, t, w.ignore_index, 512, temperature=temperature, return_entropy=True)
    d = bil.logp_bwd(x, t, lse, torch.from_numpy(w.grad_logp).cuda(), w.ignore_index, dlogits_dtype=torch.float32,
                     temperature=temperature, entropy=ent, grad_entropy=torch.from_numpy(gh).cuda())
    torch.cuda.synchronize()
    ref, _ = oracle.logp_bwd(w.logits, dtype, v, w.target_ids, w.grad_logp.astype(np.float64), w.ignore_index,
                             temperature=temperature, grad_entropy=gh.astype(np.float64))
    tol = oracle_grad_bound(w, temperature, w.grad_logp, gh)
    assert_close_elementwise(d.cpu().numpy(), ref, tol, "dlogits")


def test_autograd_logp_and_entropy():
    n, v = 6, 2000
    w = wl.random_rows(seed=99, n_rows=n, vocab=v, dtype="float32", scale=2.0, tile_v=512, ignore_every=4)
    x = device_logits(w.logits, "float32").requires_grad_(True)
    t = torch.from_numpy(w.target_ids).cuda()
    logp, ent = bil.batch_invariant_logp(x, t, return_entropy=True, tile_v=512, temperature=1.25)
    g = torch.from_numpy(w.grad_logp).cuda()
    gh = torch.linspace(-1, 1, n, device="cuda")
    ((logp * g).sum() + (ent * gh).sum()).backward()
    ghn = gh.cpu().numpy().astype(np.float64)
    ref, _ = oracle.logp_bwd(w.logits, "float32", v, w.target_ids, w.grad_logp.astype(np.float64), w.ignore_index,
                             temperature=1.25, grad_entropy=ghn)
    tol = oracle_grad_bound(w, 1.25, w.grad_logp, ghn)
    assert_close_elementwise(x.grad.cpu().numpy(), ref, tol, "dlogits via autograd")


def test_entropy_with_negative_infinite_logits():
    """-inf logits carry no probability: entropy and its gradient stay finite and
    match the oracle, fused and split alike (a whole -inf tile included)."""
    n, v, tile = 4, 4096, 512
    x = (wl.rng(7, 1).standard_normal((n, v)) * 2).astype(np.float32)
    x[:, 100:140] = -np.inf
    x[:, 1024:1536] = -np.inf        # tile 2 entirely -inf
    x[1, 4000:] = -np.inf            # a ragged masked tail
    t = np.array([5, 900, 3000, -100], np.int64)
    xd = torch.from_numpy(x).cuda()
    td = torch.from_numpy(t).cuda()
    logp, lse, ent = bil.logp_fwd(xd, td, -100, tile, return_entropy=True)
    rl, rs, _, rh = oracle.logp_fwd(x, "float32", v, t, entropy=True)
    assert_close_abs(logp.cpu().numpy(), rl, LOGP_ATOL, "logp")
    assert_close_abs(ent.cpu().numpy(), rh, ENTROPY_ATOL, "entropy")
    nt = v // tile
    pm = torch.empty(n, nt, device="cuda")
    ps, pe = torch.empty_like(pm), torch.empty_like(pm)
    tl = torch.empty(n, device="cuda")
    bil.logp_tile_partials(xd, td, v, tile, 0, nt, pm, ps, tl, -100, part_ent=pe)
    split = bil.logp_merge(pm, ps, nt, tl, td, v, -100, part_ent=pe)
    assert np.array_equal(f32_bits(split[2]), f32_bits(ent))
    g = torch.ones(n, device="cuda")
    d = bil.logp_bwd(xd, td, lse, g, -100, dlogits_dtype=torch.float32, entropy=ent, grad_entropy=g)
    ref, _ = oracle.logp_bwd(x, "float32", v, t, np.ones(n), grad_entropy=np.ones(n))
    ww = wl.Workload("neginf", x, "float32", v, tile, t)
    tol = oracle_grad_bound(ww, 1.0, np.ones(n), np.ones(n))
    assert_close_elementwise(d.cpu().numpy(), ref, tol, "dlogits")


@pytest.mark.parametrize("dtype", ["bfloat16", "float32"])
@pytest.mark.parametrize("temperature", [1.0, 0.7])
def test_unaligned_rows_same_bits_with_temperature_and_entropy(dtype, temperature):
    """Rows one element past a 16-byte boundary take the forward's shifted
    reads and the scalar backward; aligned rows the plain reads and the packed
    vector backward.  With a temperature and the entropy term, every output
    bit must still agree: the packed and scalar forms perform the same rounded
    and fused operations."""
    n, v = 9, 9000
    w = wl.random_rows(seed=44, n_rows=n, vocab=v, ld=v + 8, dtype=dtype, tile_v=1024, ignore_every=4)
    flat = device_logits(w.logits, dtype).reshape(-1)
    big = torch.empty(flat.numel() + 8, dtype=flat.dtype, device="cuda")
    big[1:1 + flat.numel()] = flat
    x_odd = big[1:1 + flat.numel()].view(n, v + 8)
    x = flat.view(n, v + 8)
    assert x_odd.data_ptr() % 16 != 0 and x.data_ptr() % 16 == 0
    t = torch.from_numpy(w.target_ids).cuda()
    g = torch.from_numpy(w.grad_logp).cuda()
    gh = torch.from_numpy(wl.rng(44, 7).standard_normal(n).astype(np.float32)).cuda()
    a = bil.logp_fwd(x, t, w.ignore_index, 1024, vocab=v, temperature=temperature, return_entropy=True)
    b = bil.logp_fwd(x_odd, t, w.ignore_index, 1024, vocab=v, temperature=temperature, return_entropy=True)
    for p, q in zip(a, b):
        assert np.array_equal(f32_bits(p), f32_bits(q))
    for od in (torch.float32, torch.bfloat16):
        da = bil.logp_bwd(x, t, a[1], g, w.ignore_index, vocab=v, temperature=temperature, entropy=a[2],
                          grad_entropy=gh, dlogits_dtype=od)
        db = bil.logp_bwd(x_odd, t, a[1], g, w.ignore_index, vocab=v, temperature=temperature, entropy=a[2],
                          grad_entropy=gh, dlogits_dtype=od)
        torch.cuda.synchronize()
        assert torch.equal(da.view(torch.int16 if od == torch.bfloat16 else torch.int32),
                           db.view(torch.int16 if od == torch.bfloat16 else torch.int32)), od
