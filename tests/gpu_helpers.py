"""Shared helpers of the GPU tests: move seeded workloads to the device and
compare CUDA results with the CPU oracle.

Tolerances (written here once, used by every GPU test):
  LOGP_ATOL   1e-4 absolute on float32 logp and lse against the float64 oracle.
  DLOGITS_ATOL 1e-6 absolute per element on float32 dlogits against the
              float64 oracle.
  bf16/fp16 dlogits: the stored value must equal the correctly rounded
              oracle value, or be the other neighbour of the oracle value when
              that value lies within DLOGITS_ATOL of the rounding midpoint
              (no 1e-6 bound can hold on a 2^-8-relative storage format, so the
              bound applies to the value before the final rounding).
  Partials:   m_t and the target logit exactly (both are copies or exact maxima
              of exactly widened values); s_t within 1e-5 relative.
  ENTROPY_ATOL 1e-4 absolute on the float32 entropy: H = log S - U / S from
              float32 sums whose relative error is ~1e-6, with |U / S| at most
              about log V (12 at V = 151936), i.e. ~1e-5 worst case.
  Gradient with an entropy term (entropy_grad_tol): the backward consumes the
              forward's float32 lse and H, whose errors eps_L <= 2e-6 and
              eps_H <= 2e-5 reach the element through p and through H:
                d = rcp * (g (onehot - p) - gh p (a + H)),  a = z - lse
                |err| <= 1e-6 + rcp p (|g| rho + |gh| (rho |a + H| + eps_L + eps_H))
              with rho = eps_L + 3e-7 the relative error of p (2-ulp exp and
              the rounding of a).  Without an entropy term and at rcp = 1 this
              is the 1e-6 bound up to p |g| rho, and those tests use 1e-6.
  float32 dlogits where |g| p is not small (dlogits_tol): the element's error
              is about |g| p times the relative error of p, and that relative
              error is rho_row = half an ulp of the row's float32 lse (4.8e-7
              for 8 <= lse < 16, 9.5e-7 for 16 <= lse < 32) + the forward's own
              error (about 4e-7: a 2-ulp exp in every sum term and the log) +
              the backward's 2-ulp exp (2.4e-7): at most 1.7e-6 for lse < 32.
              So the flat 1e-6 holds where |g| p <= 1/2 (FLAT_GP); beyond it
              the bound is 1e-6 + |g| p rho with rho = 2.3e-6 (as above).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

LOGP_ATOL = 1e-4
DLOGITS_ATOL = 1e-6
ENTROPY_ATOL = 1e-4
PART_SUM_RTOL = 1e-5

TORCH_DTYPE = {"float32": torch.float32, "bfloat16": torch.bfloat16, "float16": torch.float16}


def device_logits(stored: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """Stored elements (float32, or uint16 bit patterns) -> a device tensor of `dtype`."""
    if dtype == "float32":
        return torch.from_numpy(np.ascontiguousarray(stored)).to(device)
    t = torch.from_numpy(np.ascontiguousarray(stored).view(np.int16)).to(device)
    return t.view(TORCH_DTYPE[dtype])


def host_bits(t: torch.Tensor) -> np.ndarray:
    """A device tensor's stored elements back on the host (uint16 bits for 16-bit types)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.float32:
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def f32_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int32).numpy()


def assert_close_abs(got: np.ndarray, ref: np.ndarray, atol: float, what: str):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    nan_ok = np.array_equal(np.isnan(got), np.isnan(ref))
    assert nan_ok, f"{what}: NaN pattern differs"
    fin = ~np.isnan(ref)
    inf_ok = np.array_equal(got[fin & np.isinf(ref)], ref[fin & np.isinf(ref)])
    assert inf_ok, f"{what}: infinities differ"
    m = fin & np.isfinite(ref)
    err = np.abs(got[m] - ref[m])
    worst = float(err.max()) if err.size else 0.0
    assert worst <= atol, f"{what}: max |err| {worst:.3g} > {atol:g} (at {np.argmax(err)})"
    return worst


EPS_LSE = 2e-6
EPS_ENTROPY = 2e-5


def entropy_grad_tol(p: np.ndarray, a_plus_h: np.ndarray, g: np.ndarray, gh: np.ndarray, rcp: float) -> np.ndarray:
    """Per-element bound for gradients with an entropy term (see the module docstring);
    p, a_plus_h are [N, V] float64 from the oracle, g, gh are [N]."""
    rho = EPS_LSE + 3e-7
    with np.errstate(invalid="ignore"):
        p_ah = np.where(p > 0, p * np.abs(a_plus_h), 0.0)  # p -> 0 at a = -inf
    return 1e-6 + rcp * (np.abs(g)[:, None] * rho * p +
                         np.abs(gh)[:, None] * (rho * p_ah + (EPS_LSE + EPS_ENTROPY) * p))


FLAT_GP = 0.5
RHO_P = EPS_LSE + 3e-7


def dlogits_tol(p: np.ndarray, g: np.ndarray, lse: np.ndarray):
    """(per-element bound, |g| p) for float32 dlogits without an entropy term: the
    flat DLOGITS_ATOL where |g| p <= FLAT_GP, DLOGITS_ATOL + |g| p RHO_P beyond
    (see the module docstring; derived for rows whose lse is below 32)."""
    assert np.all(np.abs(lse[np.isfinite(lse)]) < 32.0), "the bound is derived for |lse| < 32"
    gp = np.abs(np.asarray(g, np.float64))[:, None] * p
    return np.where(gp <= FLAT_GP, DLOGITS_ATOL, DLOGITS_ATOL + gp * RHO_P), gp


def check_dlogits_split(got: np.ndarray, ref: np.ndarray, gp: np.ndarray, what: str) -> dict:
    """Assert the flat 1e-6 where |g| p <= FLAT_GP and the derived bound beyond;
    return the worst error found in each region (printed for the record)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref)), f"{what}: NaN pattern differs"
    fin = np.isfinite(ref)
    err = np.where(fin, np.abs(got - ref), 0.0)
    flat = fin & (gp <= FLAT_GP)
    beyond = fin & (gp > FLAT_GP)
    out = {"n_flat": int(flat.sum()), "worst_flat": float(err[flat].max()) if flat.any() else 0.0,
           "n_beyond": int(beyond.sum()), "worst_beyond": float(err[beyond].max()) if beyond.any() else 0.0,
           "max_gp": float(gp[fin].max()) if fin.any() else 0.0}
    if beyond.any():
        ratio = err[beyond] / (DLOGITS_ATOL + gp[beyond] * RHO_P)
        out["worst_beyond_ratio"] = float(ratio.max())
        out["gp_at_worst_beyond"] = float(gp[beyond][np.argmax(err[beyond])])
    print(f"DLOGITS-BOUND {what}: {out}")
    assert out["worst_flat"] <= DLOGITS_ATOL, f"{what}: {out}"
    assert out.get("worst_beyond_ratio", 0.0) <= 1.0, f"{what}: {out}"
    return out


def assert_close_elementwise(got: np.ndarray, ref: np.ndarray, tol: np.ndarray, what: str):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref)), f"{what}: NaN pattern differs"
    m = np.isfinite(ref)
    ratio = np.abs(got[m] - ref[m]) / tol[m]
    worst = float(ratio.max()) if ratio.size else 0.0
    assert worst <= 1.0, f"{what}: error {worst:.3g} x its bound (at {np.argmax(ratio)})"
    return worst


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.ldexp(1.0, (np.maximum(e, -126) - 7).astype(np.int64))


def f16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.ldexp(1.0, (np.maximum(e, -14) - 10).astype(np.int64))


def assert_rounded(got_bits: np.ndarray, exact: np.ndarray, dtype: str, atol: float, what: str):
    """Low-precision gradient check: correct rounding of the exact value, up to
    a flip between the two neighbours when the exact value is within `atol`
    of their midpoint.  Returns the fraction of elements that were flipped."""
    exact = np.asarray(exact, np.float64)
    if dtype == "bfloat16":
        rne = oracle.round_to_bf16_bits(exact)
        gv = oracle.bf16_bits_to_float64(got_bits)
        ulp = bf16_ulp(exact)
    else:
        rne = oracle.round_to_f16(exact).view(np.uint16)
        gv = got_bits.view(np.float16).astype(np.float64)
        ulp = f16_ulp(exact)
    same = got_bits == rne
    flip_ok = np.abs(gv - exact) <= ulp / 2 + atol
    bad = ~(same | flip_ok)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements off by more than a rounding flip, " \
                          f"e.g. got {gv[bad][:4]} exact {exact[bad][:4]}"
    return float((~same).mean())


def check_watchdog():
    import invariant_token_log_gb300 as bil
    assert bil.watchdog_status(clear=True) == 0, "a kernel wait ran out"
