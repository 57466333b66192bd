"""The fused LM-head backward's steps as separate calls, and its store GEMM.

bil_linear_logp_bwd is the gradient pass (dZ from the recomputed projection)
and two store GEMMs C = A . B^T that read dZ, the weight and the hidden states
where they lie (K-major or MN-major).  Queued one by one through
bil_linear_logp_grad and bil_linear_gemm they must give the same bits; the
store GEMM alone must match the oracle's float64 product, and a row's bits must
depend neither on the operands' layouts nor on the shape of the work unit that
computed it; and store GEMMs running at once on two streams (whose copy threads
keep in step through one shared position table) must give the bits they give
one at a time.

"[RFC][ROCm] End-to-end optimization of bitwise VIME R/R beyond native P/P",
section "Workstream 3" (the autograd actor path: fixed-order contractions).
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


def _dev(stored, dtype):
    return device_logits(stored, dtype)


@pytest.mark.parametrize("dtype,temp,entropy", [("bfloat16", 1.0, False), ("float16", 0.7, True)])
def test_backward_steps_one_by_one_give_the_backwards_bits(dtype, temp, entropy):
    n, h, v = 300, 256, 1000
    x = wl.linear_hidden(n, h, seed=41, dtype=dtype)
    w = wl.linear_weight(v, h, seed=41, dtype=dtype)
    t = wl.rng(41, 1, n, v).integers(0, v, n, dtype=np.int64)
    t[::6] = wl.IGNORE_INDEX
    xd, wd, td = _dev(x, dtype), _dev(w, dtype), torch.from_numpy(t).cuda()
    res = bil.linear_logp(xd, wd, td, temperature=temp, return_entropy=entropy)
    lse = res[1]
    ent = res[2] if entropy else None
    g = torch.from_numpy(wl.rng(41, 2).standard_normal(n).astype(np.float32)).cuda()
    gh = torch.from_numpy(wl.rng(41, 3).standard_normal(n).astype(np.float32)).cuda() if entropy else None
    dh, dw, dz = bil.linear_logp_bwd(xd, wd, td, lse, g, temperature=temp, entropy=ent, grad_entropy=gh,
                                     out_dtype=torch.float32, return_dz=True)
    dz2 = bil.linear_logp_grad(xd, wd, td, lse, g, temperature=temp, entropy=ent, grad_entropy=gh)
    dh2 = bil.matmul(dz2, wd)
    dw2 = bil.matmul(dz2.t(), xd)
    torch.cuda.synchronize()
    assert torch.equal(dz.contiguous().view(torch.int16), dz2.contiguous().view(torch.int16))
    assert np.array_equal(f32_bits(dh), f32_bits(dh2))
    assert np.array_equal(f32_bits(dw), f32_bits(dw2))


def _row_major(x):
    """A row-major copy of x whose rows are padded to 8 elements (16 bytes)."""
    rows, cols = x.shape
    return torch.empty((rows, -(-cols // 8) * 8), dtype=x.dtype, device=x.device)[:, :cols].copy_(x)


def _layouts(a, b):
    """The operands of a . b^T (a [m, k], b [n, k]) as matmul takes them, each in both
    layouts: K-major (K the unit-stride dimension) and MN-major (a transposed view of
    a row-major [k, rows] copy)."""
    return {"a": {"K": a, "MN": _row_major(a.t()).t()}, "b": {"K": b.t(), "MN": _row_major(b.t())}}


@pytest.mark.parametrize("m,n,k,dtype", [(520, 264, 1000, "bfloat16"), (136, 72, 200, "bfloat16"),
                                         (8, 8, 8, "bfloat16"), (1, 520, 64, "bfloat16"), (3, 24, 40, "float16"),
                                         (300, 136, 130, "float16")])
def test_matmul_gives_the_same_bits_for_every_operand_layout(m, n, k, dtype):
    """C[i, j] sums A(i, k) B(j, k) over its K blocks in the same order whichever way
    each operand is stored, so the four layout pairs give one set of bits (ragged K,
    rows fewer than a 64-row box, one-half and two-half work units)."""
    a = _dev(wl.linear_hidden(m, k, seed=71, dtype=dtype), dtype)
    b = _dev(wl.linear_weight(n, k, seed=72, dtype=dtype), dtype)
    ops = _layouts(a, b)
    assert ops["a"]["MN"].stride(0) == 1 and ops["b"]["MN"].stride(1) == 1
    ref = bil.gemm_nt(a, b)
    outs = {(la, lb): bil.matmul(ops["a"][la], ops["b"][lb]) for la in ("K", "MN") for lb in ("K", "MN")}
    torch.cuda.synchronize()
    for key, c in outs.items():
        assert np.array_equal(f32_bits(c), f32_bits(ref)), key


@pytest.mark.parametrize("m,n,k", [(333, 520, 1000), (300, 260, 66000)])
def test_matmul_of_mn_major_operands_against_the_oracle(m, n, k):
    """Both operands MN-major, against the oracle's float64 product, with the
    accumulation bound for K terms; K = 66000 (1032 blocks) keeps the copy threads in step."""
    a = wl.linear_hidden(m, k, seed=73)
    b = wl.linear_weight(n, k, seed=74)
    ref = oracle.linear_logits(a, b, "bfloat16")
    bound = (np.abs(oracle.widen(a, "bfloat16")) @ np.abs(oracle.widen(b, "bfloat16")).T) * (k / 4 * 2.0 ** -24) + 1e-6
    ops = _layouts(_dev(a, "bfloat16"), _dev(b, "bfloat16"))
    c = bil.matmul(ops["a"]["MN"], ops["b"]["MN"])
    torch.cuda.synchronize()
    err = np.abs(c.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= bound), float((err / bound).max())


@pytest.mark.parametrize("m,n,k,dtype", [(333, 520, 1000, "bfloat16"), (128, 256, 64, "float16"),
                                         (1, 8, 8, "bfloat16")])
def test_gemm_nt_against_the_oracle(m, n, k, dtype):
    """C = A . B^T against the oracle's float64 product of the same stored
    elements: |dC| <= 2^-20 * sum_k |a b| + 1e-6 (products of two 16-bit values
    are exact in float32; only the accumulation rounds), and a 16-bit C is the
    float32 value rounded (2^-8 or 2^-11 relative more)."""
    a = wl.linear_hidden(m, k, seed=43, dtype=dtype)
    b = wl.linear_weight(n, k, seed=44, dtype=dtype)
    ref = oracle.linear_logits(a, b, dtype)
    bound = (np.abs(oracle.widen(a, dtype)) @ np.abs(oracle.widen(b, dtype)).T) * 2.0 ** -20 + 1e-6
    ad, bd = _dev(a, dtype), _dev(b, dtype)
    c = bil.gemm_nt(ad, bd)
    c16 = bil.gemm_nt(ad, bd, out_dtype=ad.dtype)
    torch.cuda.synchronize()
    err = np.abs(c.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= bound), float((err / bound).max())
    u = 2.0 ** -8 if dtype == "bfloat16" else 2.0 ** -11
    err16 = np.abs(c16.float().cpu().numpy().astype(np.float64) - ref)
    assert np.all(err16 <= bound * (1 + u) + u * np.abs(ref) + 2.0 ** -24), float((err16 / (bound + u * np.abs(ref))).max())


def test_gemm_nt_of_a_long_k_against_the_oracle():
    """A K long enough (66000, ragged: 1032 blocks of 64) that the copy threads keep in step,
    against the oracle's float64 product; the float32 accumulation's bound for K terms,
    gamma_K * sum_k |a b| with gamma_K = K/4 * 2^-24 (one rounding per four products)."""
    m, n, k = 130, 260, 66000
    a = wl.linear_hidden(m, k, seed=51)
    b = wl.linear_weight(n, k, seed=52)
    ref = oracle.linear_logits(a, b, "bfloat16")
    bound = (np.abs(oracle.widen(a, "bfloat16")) @ np.abs(oracle.widen(b, "bfloat16")).T) * (k / 4 * 2.0 ** -24) + 1e-6
    c = bil.gemm_nt(_dev(a, "bfloat16"), _dev(b, "bfloat16"))
    torch.cuda.synchronize()
    err = np.abs(c.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= bound), float((err / bound).max())


def test_gemm_nt_of_a_long_k_in_two_half_units_against_the_oracle():
    """The same bound with 300 rows (work units of two 128-row halves, the second unit's
    second half past the last row) and a K of 66000, where the copy threads keep in step."""
    m, n, k = 300, 260, 66000
    a = wl.linear_hidden(m, k, seed=53)
    b = wl.linear_weight(n, k, seed=54)
    ref = oracle.linear_logits(a, b, "bfloat16")
    bound = (np.abs(oracle.widen(a, "bfloat16")) @ np.abs(oracle.widen(b, "bfloat16")).T) * (k / 4 * 2.0 ** -24) + 1e-6
    c = bil.gemm_nt(_dev(a, "bfloat16"), _dev(b, "bfloat16"))
    torch.cuda.synchronize()
    err = np.abs(c.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= bound), float((err / bound).max())


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_store_gemm_rows_agree_across_work_unit_shapes(out_dtype):
    """From 256 rows on the store GEMM's work unit is two 128-row A tiles sharing one B
    tile, below that one 128-row tile.  Each element sums its K blocks in the same order
    either way, so a row has the same bits whichever unit computed it, wherever the batch
    starts: a 600-row A against slices of it of 200 and 100 rows (one-half units) and of
    500 and 257 rows (two-half units at other offsets)."""
    m, n, k = 600, 520, 5000
    a = _dev(wl.linear_hidden(m, k, seed=61), "bfloat16")
    b = _dev(wl.linear_weight(n, k, seed=62), "bfloat16")
    c = bil.gemm_nt(a, b, out_dtype=out_dtype)
    parts = {(256, 456): None, (333, 433): None, (100, 600): None, (343, 600): None}
    for lo, hi in parts:
        parts[(lo, hi)] = bil.gemm_nt(a[lo:hi], b, out_dtype=out_dtype)
    torch.cuda.synchronize()
    full = c.contiguous().view(torch.int32 if out_dtype == torch.float32 else torch.int16)
    for (lo, hi), cp in parts.items():
        got = cp.contiguous().view(full.dtype)
        assert torch.equal(got, full[lo:hi]), (lo, hi)


def test_store_gemms_at_once_on_two_streams_keep_their_bits():
    """Two store GEMMs of several waves each (512 work units for 152 SMs) run at
    the same time on two streams; each must give the bits it gives alone."""
    m, n, k = 4096, 4096, 4096
    a1 = _dev(wl.linear_hidden(m, k, seed=45), "bfloat16")
    b1 = _dev(wl.linear_weight(n, k, seed=46), "bfloat16")
    a2 = _dev(wl.linear_hidden(m, k, seed=47), "bfloat16")
    b2 = _dev(wl.linear_weight(n, k, seed=48), "bfloat16")
    _two_streams_same_bits(a1, b1, a2, b2)


def test_store_gemms_of_long_k_at_once_on_two_streams_keep_their_bits():
    """The same with a K of 65600 (1025 blocks of 64), where the copy threads of each GEMM keep
    in step through the one position table the two launches share: each still gives its bits."""
    m, n, k = 2048, 1024, 65600
    a1 = _dev(wl.linear_hidden(m, k, seed=55), "bfloat16")
    b1 = _dev(wl.linear_weight(n, k, seed=56), "bfloat16")
    a2 = _dev(wl.linear_hidden(m, k, seed=57), "bfloat16")
    b2 = _dev(wl.linear_weight(n, k, seed=58), "bfloat16")
    _two_streams_same_bits(a1, b1, a2, b2)


def _two_streams_same_bits(a1, b1, a2, b2):
    ref1, ref2 = bil.gemm_nt(a1, b1), bil.gemm_nt(a2, b2)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(3):
        with torch.cuda.stream(s1):
            c1 = bil.gemm_nt(a1, b1)
        with torch.cuda.stream(s2):
            c2 = bil.gemm_nt(a2, b2)
        outs.append((c1, c2))
    torch.cuda.synchronize()
    for c1, c2 in outs:
        assert np.array_equal(f32_bits(c1), f32_bits(ref1))
        assert np.array_equal(f32_bits(c2), f32_bits(ref2))
