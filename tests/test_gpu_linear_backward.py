"""Backward of the fused LM-head + logp on the GPU: against the CPU oracle, against
the logits path's backward, for batch-invariance of dhidden, and through autograd.

"[RFC][ROCm] End-to-end optimization of bitwise VIME R/R beyond native P/P",
section "Workstream 3": the autograd actor path, recomputing the projection's
tiles from the saved LSE.

Tolerances, derived per element from the arithmetic (all from oracle values):
  z       |dz| <= 2^-20 * sum_k |x_k w_k| + 1e-6 (the forward's bound).
  lse, H  the forward's float32 errors plus what |dz| moves them:
          eL = 2e-6 + rcp * max_c dz_c,   eH = 2e-5 + rcp * max_c dz_c * sum_c p_c |a_c + H|.
  a = z*rcp - lse:  da <= rcp * dz_c + eL + 2^-24 |a|;   p: dp <= p (3e-7 + da).
  dZ before rounding:
          rcp * (|g| dp + |gh| (dp |a + H| + p (da + eH))) + 2^-22 |dZ|
  dZ stored: plus u |dZ| + s with u = 2^-8 (bf16) or 2^-11 (fp16), the relative storage
          rounding, and s = half the subnormal spacing (2^-134 bf16, 2^-25 fp16), where
          the storage's spacing is absolute.
  dhidden = dZ . W and dweight = dZ^T . X accumulate in float32 over K terms:
          tol(dZ) . |W| + gamma_K * (|dZ| + tol(dZ)) . |W|,  gamma_K = max(2^-20, K/4 * 2^-24)
          (at most one float32 rounding per 4 products), plus u |result| for 16-bit outputs.
"""
import numpy as np
import pytest
import torch

import invariant_token_log_gb300 as bil
import oracle
import workloads as wl
from gpu_helpers import check_watchdog, device_logits, f32_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _watchdog():
    yield
    check_watchdog()


U16 = {"bfloat16": 2.0 ** -8, "float16": 2.0 ** -11}
SUB16 = {"bfloat16": 2.0 ** -134, "float16": 2.0 ** -25}


def make_case(n, h, v, dtype="bfloat16", seed=21, ignore_every=5, entropy=False):
    x = wl.linear_hidden(n, h, seed=seed, dtype=dtype)
    w = wl.linear_weight(v, h, seed=seed, dtype=dtype)
    t = wl.rng(seed, 1, n, v).integers(0, v, n, dtype=np.int64)
    if ignore_every:
        t[::ignore_every] = wl.IGNORE_INDEX
    g = wl.rng(seed, 2).standard_normal(n).astype(np.float32)
    gh = wl.rng(seed, 3).standard_normal(n).astype(np.float32) if entropy else None
    return x, w, t, g, gh


def tolerances(x, w, dtype, t, g, gh, temp):
    """Per-element bounds on dZ, dhidden and dweight (see the module docstring)."""
    rcp = float(np.float32(1.0 / temp))
    xf, wf = oracle.widen(x, dtype), oracle.widen(w, dtype)
    z = xf @ wf.T
    dz_bound = (np.abs(xf) @ np.abs(wf).T) * 2.0 ** -20 + 1e-6
    _, lse, _, H = oracle.logp_fwd(z, "float64", z.shape[1], t, temperature=temp, entropy=True)
    a = z / temp - lse[:, None]
    p = np.exp(a)
    act = (t != wl.IGNORE_INDEX)[:, None]
    mz = dz_bound.max(axis=1, keepdims=True)
    eL = 2e-6 + rcp * mz
    eH = 2e-5 + rcp * mz * (p * np.abs(a + H[:, None])).sum(axis=1, keepdims=True)
    da = rcp * dz_bound + eL + 2.0 ** -24 * np.abs(a)
    dp = p * (3e-7 + da)
    ag = np.abs(g.astype(np.float64))[:, None]
    agh = np.abs(gh.astype(np.float64))[:, None] if gh is not None else 0.0
    dx_, dw_, dZ, _ = oracle.linear_logp_bwd(x, w, dtype, t, g, temperature=temp, grad_entropy=gh)
    pre = rcp * (ag * dp + agh * (dp * np.abs(a + H[:, None]) + p * (da + eH))) + 2.0 ** -22 * np.abs(dZ)
    tol_dz = np.where(act, pre * (1 + U16[dtype]) + U16[dtype] * np.abs(dZ) + SUB16[dtype], 0.0)
    aw, ax = np.abs(wf), np.abs(xf)

    def gamma(k):
        return max(2.0 ** -20, k / 4 * 2.0 ** -24)
    tol_dx = tol_dz @ aw + gamma(w.shape[0]) * ((np.abs(dZ) + tol_dz) @ aw) + 1e-30
    tol_dw = tol_dz.T @ ax + gamma(x.shape[0]) * ((np.abs(dZ) + tol_dz).T @ ax) + 1e-30
    return dx_, dw_, dZ, tol_dz, tol_dx, tol_dw


def within(got, ref, tol, what):
    err = np.abs(np.asarray(got, np.float64) - ref)
    ratio = err / tol
    worst = float(ratio.max())
    assert worst <= 1.0, f"{what}: error {worst:.3g} x its bound (max |err| {err.max():.3g})"
    return worst


def run_bwd(x, w, t, g, gh, dtype, temp, out_dtype=torch.float32):
    xd, wd, td = device_logits(x, dtype), device_logits(w, dtype), torch.from_numpy(t).cuda()
    res = bil.linear_logp(xd, wd, td, temperature=temp, return_entropy=gh is not None)
    lse = res[1]
    ent = res[2] if gh is not None else None
    gd = torch.from_numpy(g).cuda()
    ghd = torch.from_numpy(gh).cuda() if gh is not None else None
    dh, dw, dz = bil.linear_logp_bwd(xd, wd, td, lse, gd, temperature=temp, entropy=ent, grad_entropy=ghd,
                                     out_dtype=out_dtype, return_dz=True)
    torch.cuda.synchronize()
    return dh, dw, dz, (xd, wd, td, lse, ent, gd, ghd)


CASES = [
    (128, 64, 256, "bfloat16", 1.0, False),
    (300, 200, 1000, "bfloat16", 1.0, True),    # ragged rows, K and last tile; entropy
    (257, 320, 777, "float16", 0.8, False),
    (200, 256, 1500, "bfloat16", 1.3, True),
]


@pytest.mark.parametrize("n,h,v,dtype,temp,ent", CASES)
def test_backward_vs_oracle(n, h, v, dtype, temp, ent):
    x, w, t, g, gh = make_case(n, h, v, dtype, seed=n + v, entropy=ent)
    dh, dw, dz, _ = run_bwd(x, w, t, g, gh, dtype, temp)
    rdx, rdw, rdz, tdz, tdx, tdw = tolerances(x, w, dtype, t, g, gh, temp)
    within(oracle.widen(dz.cpu().contiguous().view(torch.int16).numpy().view(np.uint16), dtype), rdz, tdz + 1e-30,
           "dZ")
    within(dh.cpu().numpy(), rdx, tdx, "dhidden")
    within(dw.cpu().numpy(), rdw, tdw, "dweight")
    ign = t == wl.IGNORE_INDEX
    assert np.all(dz.cpu().float().numpy()[ign] == 0)


def test_16bit_outputs_are_the_rounded_float32_outputs():
    x, w, t, g, gh = make_case(300, 200, 1000, seed=3, entropy=True)
    dh32, dw32, _, _ = run_bwd(x, w, t, g, gh, "bfloat16", 1.0)
    dh16, dw16, _, _ = run_bwd(x, w, t, g, gh, "bfloat16", 1.0, out_dtype=torch.bfloat16)
    assert torch.equal(dh16.contiguous().view(torch.int16), dh32.to(torch.bfloat16).contiguous().view(torch.int16))
    assert torch.equal(dw16.contiguous().view(torch.int16), dw32.to(torch.bfloat16).contiguous().view(torch.int16))


def test_dz_is_the_logits_backward_of_the_projection():
    """dZ equals, bit for bit, what bil_logp_bwd writes for the float32 logits the
    forward stores: one recomputation, one formula."""
    x, w, t, g, gh = make_case(300, 256, 1000, seed=4, entropy=True)
    for temp in (1.0, 0.7):
        dh, dw, dz, (xd, wd, td, lse, ent, gd, ghd) = run_bwd(x, w, t, g, gh, "bfloat16", temp)
        _, _, _, z = bil.linear_logp(xd, wd, td, temperature=temp, return_entropy=True, return_logits=True)
        d = bil.logp_bwd(z, td, lse, gd, -100, temperature=temp, entropy=ent, grad_entropy=ghd,
                         out=torch.empty(z.shape, dtype=torch.bfloat16, device="cuda"))
        torch.cuda.synchronize()
        assert torch.equal(d.view(torch.int16), dz.contiguous().view(torch.int16)), temp


def test_dhidden_rows_are_batch_invariant_and_dweight_is_deterministic():
    n, h, v = 256, 256, 1200
    x, w, t, g, gh = make_case(n, h, v, seed=5, ignore_every=0)
    dh, dw, _, (xd, wd, td, lse, _, gd, _) = run_bwd(x, w, t, g, None, "bfloat16", 1.0)
    _, dw2, _, _ = run_bwd(x, w, t, g, None, "bfloat16", 1.0)
    assert np.array_equal(f32_bits(dw), f32_bits(dw2))
    ref = f32_bits(dh)
    r = wl.rng(5, 9)
    for size in (1, 3, 7, 64, 200):
        idx = r.permutation(n)[:size]
        sel = torch.from_numpy(idx).cuda()
        dhs, _ = bil.linear_logp_bwd(xd.index_select(0, sel), wd, td.index_select(0, sel), lse.index_select(0, sel),
                                     gd.index_select(0, sel), out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert np.array_equal(f32_bits(dhs), ref[idx]), size


def test_autograd_matches_the_c_abi():
    n, h, v = 200, 192, 900
    x, w, t, g, gh = make_case(n, h, v, seed=6, entropy=True)
    xd = device_logits(x, "bfloat16").requires_grad_(True)
    wd = device_logits(w, "bfloat16").requires_grad_(True)
    td = torch.from_numpy(t).cuda()
    gd, ghd = torch.from_numpy(g).cuda(), torch.from_numpy(gh).cuda()
    logp, ent = bil.batch_invariant_linear_logp(xd, wd, td, temperature=0.9, return_entropy=True)
    ((logp * gd).sum() + (ent * ghd).sum()).backward()
    lp2, lse2, ent2 = bil.linear_logp(xd.detach(), wd.detach(), td, temperature=0.9, return_entropy=True)
    dh, dw = bil.linear_logp_bwd(xd.detach(), wd.detach(), td, lse2, gd, temperature=0.9, entropy=ent2,
                                 grad_entropy=ghd)
    torch.cuda.synchronize()
    assert np.array_equal(f32_bits(logp), f32_bits(lp2))
    assert torch.equal(xd.grad.view(torch.int16), dh.contiguous().view(torch.int16))
    assert torch.equal(wd.grad.view(torch.int16), dw.contiguous().view(torch.int16))


@pytest.mark.parametrize("dtype,temp,entropy,lead", [("bfloat16", 0.9, True, (200,)), ("float16", 1.0, False, (4, 50)),
                                                   ("bfloat16", 1.0, False, (300,))])
def test_keeping_the_logits_gives_the_recomputing_backwards_bits(dtype, temp, entropy, lead):
    """keep_logits: the forward keeps its float32 logits and the backward starts from them
    (the logits path's backward for dZ, then the two products) instead of recomputing the
    projection; the gradients have the same bits, through autograd and through the call."""
    n = int(np.prod(lead))
    h, v = 192, 900
    x, w, t, g, gh = make_case(n, h, v, seed=8, entropy=True, dtype=dtype)
    grads = []
    for keep in (False, True):
        xd = device_logits(x, dtype).reshape(*lead, h).requires_grad_(True)
        wd = device_logits(w, dtype).requires_grad_(True)
        td = torch.from_numpy(t).cuda().reshape(lead)
        gd, ghd = torch.from_numpy(g).cuda().reshape(lead), torch.from_numpy(gh).cuda().reshape(lead)
        if entropy:
            logp, ent = bil.batch_invariant_linear_logp(xd, wd, td, temperature=temp, return_entropy=True,
                                                        keep_logits=keep)
            ((logp * gd).sum() + (ent * ghd).sum()).backward()
        else:
            logp = bil.batch_invariant_linear_logp(xd, wd, td, temperature=temp, keep_logits=keep)
            (logp * gd).sum().backward()
        grads.append((f32_bits(logp), xd.grad.contiguous().view(torch.int16).clone(),
                      wd.grad.contiguous().view(torch.int16).clone()))
    torch.cuda.synchronize()
    assert np.array_equal(grads[0][0], grads[1][0])
    assert torch.equal(grads[0][1], grads[1][1])
    assert torch.equal(grads[0][2], grads[1][2])
    xd, wd = device_logits(x, dtype), device_logits(w, dtype)
    td, gd = torch.from_numpy(t).cuda(), torch.from_numpy(g).cuda()
    lp, lse, logits = bil.linear_logp(xd, wd, td, temperature=temp, return_logits=True, logits_dtype=torch.float32)
    dh, dw = bil.linear.linear_logp_bwd_from_logits(xd, wd, td, logits, lse, gd, temperature=temp)
    dh2, dw2 = bil.linear_logp_bwd(xd, wd, td, lse, gd, temperature=temp)
    torch.cuda.synchronize()
    assert torch.equal(dh.contiguous().view(torch.int16), dh2.contiguous().view(torch.int16))
    assert torch.equal(dw.contiguous().view(torch.int16), dw2.contiguous().view(torch.int16))


def test_full_size_sampled_rows_and_the_bilinear_identity():
    """Qwen3-8B-shaped LM head over 16384 rows: four sampled dhidden rows against the
    oracle (a row's dhidden depends on that row only), and <dX, X> = <dW, W> for the
    whole batch (both equal <dZ, z>; z is bilinear in X and W)."""
    lw = wl.linear(16384)
    xd = device_logits(lw.hidden, lw.dtype)
    wd = device_logits(lw.weight, lw.dtype)
    td = torch.from_numpy(lw.target_ids).cuda()
    gd = torch.from_numpy(lw.grad_logp).cuda()
    logp, lse = bil.linear_logp(xd, wd, td)
    dh, dw = bil.linear_logp_bwd(xd, wd, td, lse, gd, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ip_x = float((dh.double() * xd.double()).sum())
    ip_w = float((dw.double() * wd.double()).sum())
    scale = float((dh.double().abs() * xd.double().abs()).sum())
    assert abs(ip_x - ip_w) <= 2.0 ** -7 * scale, (ip_x, ip_w, scale)
    idx = np.array([3, 4100, 9999, 16383])
    xs = np.ascontiguousarray(lw.hidden[idx])
    rdx, _, _, _ = oracle.linear_logp_bwd(xs, lw.weight, lw.dtype, lw.target_ids[idx], lw.grad_logp[idx])
    got = dh.cpu().numpy()[idx].astype(np.float64)
    # the dominant term of the bound: the bf16 storage of dZ, 2^-8 |dZ| . |W|, is
    # bounded by 2^-8 * sum_c |dZ_c| * max |W| <= 2^-8 * 2 |g| * max|W| per element
    # (bf16 bit patterns without the sign bit order like the magnitudes they hold)
    wmax = float(wl.bf16_bits_to_f32(np.array([(lw.weight & np.uint16(0x7FFF)).max()], np.uint16))[0])
    bound = (2.0 ** -8 + 151936 / 4 * 2.0 ** -24) * 2 * np.abs(lw.grad_logp[idx])[:, None] * wmax * 2 + 1e-6
    assert np.all(np.abs(got - rdx) <= bound)


def test_full_size_keeping_the_logits_gives_the_recomputing_bits():
    """The Qwen3-8B-shaped LM head over 16384 rows: the backward from the forward's kept
    float32 logits (9.96 GB) and the recomputing backward give the same dhidden and dweight
    bits (the dZ bits equal, and the same two products)."""
    lw = wl.linear(16384)
    xd = device_logits(lw.hidden, lw.dtype)
    wd = device_logits(lw.weight, lw.dtype)
    td = torch.from_numpy(lw.target_ids).cuda()
    gd = torch.from_numpy(lw.grad_logp).cuda()
    lp, lse, logits = bil.linear_logp(xd, wd, td, return_logits=True, logits_dtype=torch.float32)
    dh, dw = bil.linear.linear_logp_bwd_from_logits(xd, wd, td, logits, lse, gd)
    del logits
    dh2, dw2 = bil.linear_logp_bwd(xd, wd, td, lse, gd)
    torch.cuda.synchronize()
    assert torch.equal(dh.contiguous().view(torch.int16), dh2.contiguous().view(torch.int16))
    assert torch.equal(dw.contiguous().view(torch.int16), dw2.contiguous().view(torch.int16))


def test_backward_edges():
    """No rows: dweight is zero.  An active row with an out-of-range target makes
    its dZ row NaN (and so its dhidden row); ignored rows are exactly zero."""
    n, h, v = 6, 64, 300
    x, w, t, g, _ = make_case(n, h, v, seed=8, ignore_every=0)
    xd, wd, td = device_logits(x, "bfloat16"), device_logits(w, "bfloat16"), torch.from_numpy(t).cuda()
    gd = torch.from_numpy(g).cuda()
    lse = bil.linear_logp(xd, wd, td)[1]
    dh0, dw0 = bil.linear_logp_bwd(xd[:0], wd, td[:0], lse[:0], gd[:0], out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert dh0.numel() == 0 and torch.count_nonzero(dw0).item() == 0
    bad = td.clone()
    bad[1] = v + 5
    bad[3] = -100
    dh, dw, dz = bil.linear_logp_bwd(xd, wd, bad, lse, gd, out_dtype=torch.float32, return_dz=True)
    torch.cuda.synchronize()
    dzf = dz.float().cpu().numpy()
    assert np.all(np.isnan(dzf[1])) and np.all(np.isnan(dh.cpu().numpy()[1]))
    assert np.all(dzf[3] == 0) and not np.isnan(dzf[[0, 2, 4, 5]]).any()
    assert np.all(np.isnan(dw.cpu().numpy()))  # every dweight entry sums over row 1
