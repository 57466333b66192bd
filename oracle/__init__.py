"""CPU oracle for the batch-invariant selected-token log-probability.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
package.  The CUDA library never calls it and it never calls the CUDA library.

The arithmetic lives in ``bil_oracle.c`` (plain C, float64, OpenMP over rows);
this module compiles it with gcc on first use (once per machine architecture)
and wraps it for numpy arrays.  It also holds the exact float64 -> bfloat16 /
float16 round-to-nearest-even used to turn the oracle's float64 gradients into
the value a correctly rounded low-precision store would hold.

Page citations ("Batch-Invariant LogP" operator page):
  * "Reference Semantics": logp = log_softmax(float(x))[target]; ignored rows
    give 0 and a zero gradient row; other targets outside [0, V) are invalid.
  * "Tensor Parallel", steps 1-6: fixed vocab tiles, per-tile (max, sumexp),
    a fixed-order merge, the target logit copied from its owning tile.
  * "Batch-Invariance": the backward recomputes softmax from the saved LSE.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bil_oracle.c")

# element-type codes of the C oracle (its own; not shared with the CUDA library)
F32, BF16, F16, F64 = 0, 1, 2, 3
DTYPE_CODES = {"float32": F32, "bfloat16": BF16, "float16": F16, "float64": F64}

_lock = threading.Lock()
_libs: dict[tuple, ctypes.CDLL] = {}


def library_path(defines: tuple[str, ...] = ()) -> str:
    """Where the compiled oracle for this machine (and these -D flags) lives."""
    tag = "libbil_oracle" + "".join("_" + d.lower() for d in defines) + ".so"
    return os.path.join(_HERE, "_build", platform.machine(), tag)


def build(defines: tuple[str, ...] = (), force: bool = False) -> str:
    """Compile bil_oracle.c with gcc (-O2, OpenMP, no fast-math).

    ``defines`` adds ``-D<name>`` flags; the oracle's mutation tests use them to
    plant one deliberate mistake per build and check that the pins catch it.
    """
    out = library_path(defines)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
           "-Wall", "-Wextra", _SRC, "-o", tmp, "-lm"]
    # planted mistakes may leave a variable unused; the real build stays warning-free
    cmd[1:1] = [f"-D{d}" for d in defines] if defines else ["-Werror"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(defines: tuple[str, ...] = ()) -> ctypes.CDLL:
    with _lock:
        lib = _libs.get(defines)
        if lib is not None:
            return lib
        lib = ctypes.CDLL(build(defines))
        i64, i32, vp, dp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p
        lib.bil_oracle_num_threads.restype = i32
        lib.bil_oracle_num_threads.argtypes = []
        lib.bil_oracle_logp_fwd.restype = i64
        f64 = ctypes.c_double
        lib.bil_oracle_logp_fwd.argtypes = [vp, i32, i64, i64, i64, vp, i64, f64, dp, dp, dp]
        lib.bil_oracle_tile_partials.restype = None
        lib.bil_oracle_tile_partials.argtypes = [vp, i32, i64, i64, i64, i64, i64, i64, vp,
                                                 i64, f64, dp, dp, dp, i64, dp]
        lib.bil_oracle_merge.restype = i64
        lib.bil_oracle_merge.argtypes = [dp, dp, dp, i64, i64, i64, dp, vp, i64, i64, dp, dp, dp]
        lib.bil_oracle_logp_bwd.restype = i64
        lib.bil_oracle_logp_bwd.argtypes = [vp, i32, i64, i64, i64, vp, i64, f64, dp, dp, dp, i64, i64]
        lib.bil_oracle_linear_logits.restype = None
        lib.bil_oracle_linear_logits.argtypes = [vp, vp, i32, i64, i64, i64, i64, i64, dp, i64]
        lib.bil_oracle_linear_bwd.restype = i64
        lib.bil_oracle_linear_bwd.argtypes = [vp, vp, i32, i64, i64, i64, i64, i64, vp, i64, f64, dp, dp, dp, dp,
                                              dp]
        lib.bil_oracle_widen.restype = None
        lib.bil_oracle_widen.argtypes = [vp, i32, i64, dp]
        _libs[defines] = lib
        return lib


def num_threads() -> int:
    return int(load().bil_oracle_num_threads())


# --------------------------------------------------------------------------
# numpy front end.  Logits arrive as the raw stored bytes: float32 arrays for
# fp32, uint16 arrays holding the bit patterns for bf16 / fp16.
# --------------------------------------------------------------------------

def _code(dtype: str) -> int:
    try:
        return DTYPE_CODES[dtype]
    except KeyError:
        raise ValueError(f"oracle: unsupported element type {dtype!r}") from None


def _check_logits(logits: np.ndarray, dtype: str) -> tuple[int, int]:
    want = {"float32": np.float32, "float64": np.float64}.get(dtype, np.uint16)
    if logits.dtype != want or logits.ndim != 2 or logits.strides[1] != logits.itemsize:
        raise ValueError("oracle: logits must be a 2-D row-major array of the stored element type")
    return logits.shape[0], logits.strides[0] // logits.itemsize


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _optr(a):
    return None if a is None else _ptr(a)


def logp_fwd(logits: np.ndarray, dtype: str, vocab: int, target_ids: np.ndarray,
             ignore_index: int = -100, defines: tuple[str, ...] = (), temperature: float = 1.0,
             entropy: bool = False):
    """float64 (logp[N], lse[N], n_invalid_targets), plus entropy[N] when asked,
    for the first ``vocab`` columns divided by ``temperature``."""
    n, ld = _check_logits(logits, dtype)
    tgt = np.ascontiguousarray(target_ids, dtype=np.int64)
    assert tgt.shape == (n,)
    logp = np.empty(n, np.float64)
    lse = np.empty(n, np.float64)
    ent = np.empty(n, np.float64) if entropy else None
    bad = load(defines).bil_oracle_logp_fwd(_ptr(logits), _code(dtype), n, vocab, ld, _ptr(tgt),
                                            ignore_index, float(temperature), _ptr(logp), _ptr(lse),
                                            _optr(ent))
    return (logp, lse, int(bad), ent) if entropy else (logp, lse, int(bad))


def tile_partials(logits: np.ndarray, dtype: str, vocab: int, tile_v: int, tile_begin: int,
                  tile_end: int, target_ids: np.ndarray, ignore_index: int = -100,
                  part_max: np.ndarray | None = None, part_sum: np.ndarray | None = None,
                  target_logit: np.ndarray | None = None, defines: tuple[str, ...] = (),
                  temperature: float = 1.0, part_ent: np.ndarray | None = None):
    """Fill float64 [N, T] (max, sumexp) partials for tiles [tile_begin, tile_end).

    Arrays passed in are updated in place (so that several calls can fill one
    buffer, as the tensor-parallel ranks do); missing ones are created
    (partials -inf / 0, target_logit NaN).  ``part_ent``, when given, receives
    the entropy partials sum exp(z - m) * (z - m).
    """
    n, ld = _check_logits(logits, dtype)
    num_tiles = -(-vocab // tile_v)
    tgt = np.ascontiguousarray(target_ids, dtype=np.int64)
    if part_max is None:
        part_max = np.full((n, num_tiles), -np.inf)
    if part_sum is None:
        part_sum = np.zeros((n, num_tiles))
    if target_logit is None:
        target_logit = np.full(n, np.nan)
    for a in (part_max, part_sum) + ((part_ent,) if part_ent is not None else ()):
        assert a.dtype == np.float64 and a.flags.c_contiguous and a.shape[0] == n
    assert part_ent is None or part_ent.shape == part_max.shape
    load(defines).bil_oracle_tile_partials(_ptr(logits), _code(dtype), n, vocab, ld, tile_v,
                                           tile_begin, tile_end, _ptr(tgt), ignore_index,
                                           float(temperature), _ptr(part_max), _ptr(part_sum),
                                           _optr(part_ent), part_max.shape[1], _ptr(target_logit))
    return part_max, part_sum, target_logit


def merge(part_max: np.ndarray, part_sum: np.ndarray, target_logit: np.ndarray,
          target_ids: np.ndarray, vocab: int, ignore_index: int = -100,
          defines: tuple[str, ...] = (), part_ent: np.ndarray | None = None):
    """Fixed-order merge of float64 partials: (logp[N], lse[N], n_invalid_targets),
    plus entropy[N] when ``part_ent`` is given."""
    n, num_tiles = part_max.shape
    tgt = np.ascontiguousarray(target_ids, dtype=np.int64)
    tl = np.ascontiguousarray(target_logit, dtype=np.float64)
    logp = np.empty(n, np.float64)
    lse = np.empty(n, np.float64)
    ent = np.empty(n, np.float64) if part_ent is not None else None
    bad = load(defines).bil_oracle_merge(_ptr(part_max), _ptr(part_sum), _optr(part_ent), n, num_tiles,
                                         part_max.shape[1], _ptr(tl), _ptr(tgt), ignore_index,
                                         vocab, _ptr(logp), _ptr(lse), _optr(ent))
    return (logp, lse, int(bad), ent) if part_ent is not None else (logp, lse, int(bad))


def logp_bwd(logits: np.ndarray, dtype: str, vocab: int, target_ids: np.ndarray,
             grad_logp: np.ndarray, ignore_index: int = -100, out_cols: int | None = None,
             defines: tuple[str, ...] = (), temperature: float = 1.0,
             grad_entropy: np.ndarray | None = None):
    """float64 dlogits [N, out_cols] of g * logp (+ gH * entropy) and the number
    of invalid targets."""
    n, ld = _check_logits(logits, dtype)
    out_cols = vocab if out_cols is None else out_cols
    tgt = np.ascontiguousarray(target_ids, dtype=np.int64)
    g = np.ascontiguousarray(grad_logp, dtype=np.float64)
    gh = None if grad_entropy is None else np.ascontiguousarray(grad_entropy, dtype=np.float64)
    d = np.empty((n, out_cols), np.float64)
    bad = load(defines).bil_oracle_logp_bwd(_ptr(logits), _code(dtype), n, vocab, ld, _ptr(tgt),
                                            ignore_index, float(temperature), _ptr(g), _optr(gh),
                                            _ptr(d), out_cols, out_cols)
    return d, int(bad)


def linear_logits(hidden: np.ndarray, weight: np.ndarray, dtype: str,
                  defines: tuple[str, ...] = ()) -> np.ndarray:
    """float64 logits z [N, V] = hidden [N, H] . weight [V, H]^T, summed over k in order.

    "[RFC][ROCm] End-to-end optimization of bitwise VIME R/R beyond native P/P",
    section "Workstream 3: fused ROCm LM-head and linear logp": the LM-head
    projection whose output the fused operator reduces without storing."""
    n, ld_h = _check_logits(hidden, dtype)
    v, ld_w = _check_logits(weight, dtype)
    h = hidden.shape[1]
    assert weight.shape[1] == h
    z = np.empty((n, v), np.float64)
    load(defines).bil_oracle_linear_logits(_ptr(hidden), _ptr(weight), _code(dtype), n, h, ld_h, v, ld_w,
                                           _ptr(z), v)
    return z


def linear_logp_fwd(hidden: np.ndarray, weight: np.ndarray, dtype: str, target_ids: np.ndarray,
                    ignore_index: int = -100, temperature: float = 1.0, entropy: bool = False,
                    defines: tuple[str, ...] = ()):
    """The fused LM-head + logp: the operator applied to the float64 projection.
    Returns (logp, lse, n_invalid_targets[, entropy])."""
    z = linear_logits(hidden, weight, dtype, defines)
    return logp_fwd(z, "float64", z.shape[1], target_ids, ignore_index, defines, temperature, entropy)


def linear_logp_bwd(hidden: np.ndarray, weight: np.ndarray, dtype: str, target_ids: np.ndarray,
                    grad_logp: np.ndarray, ignore_index: int = -100, temperature: float = 1.0,
                    grad_entropy: np.ndarray | None = None, defines: tuple[str, ...] = ()):
    """float64 (dhidden [N, H], dweight [V, H], dZ [N, V], n_invalid_targets): the
    gradient of g * logp (+ gH * entropy) of the fused LM-head + logp."""
    n, ld_h = _check_logits(hidden, dtype)
    v, ld_w = _check_logits(weight, dtype)
    h = hidden.shape[1]
    tgt = np.ascontiguousarray(target_ids, dtype=np.int64)
    g = np.ascontiguousarray(grad_logp, dtype=np.float64)
    gh = None if grad_entropy is None else np.ascontiguousarray(grad_entropy, dtype=np.float64)
    dx = np.empty((n, h), np.float64)
    dw = np.empty((v, h), np.float64)
    dz = np.empty((n, v), np.float64)
    bad = load(defines).bil_oracle_linear_bwd(_ptr(hidden), _ptr(weight), _code(dtype), n, h, ld_h, v, ld_w,
                                              _ptr(tgt), ignore_index, float(temperature), _ptr(g), _optr(gh),
                                              _ptr(dx), _ptr(dw), _ptr(dz))
    if bad < 0:
        raise MemoryError("oracle: out of memory in linear_logp_bwd")
    return dx, dw, dz, int(bad)


def widen(stored: np.ndarray, dtype: str, defines: tuple[str, ...] = ()) -> np.ndarray:
    """Exact float64 value of stored elements (raw uint16 bits for bf16 / fp16)."""
    src = np.ascontiguousarray(stored)
    out = np.empty(src.size, np.float64)
    load(defines).bil_oracle_widen(_ptr(src), _code(dtype), src.size, _ptr(out))
    return out.reshape(src.shape)


# --------------------------------------------------------------------------
# Correct rounding of float64 values to the stored output types.  A single
# round-to-nearest-even step straight from float64 (no detour through
# float32, which could round twice).
# --------------------------------------------------------------------------

def round_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """float64 -> bfloat16 bit patterns, round to nearest, ties to even."""
    v = np.asarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    a = np.abs(v)
    sign = np.signbit(v)
    # bfloat16 keeps 8 significant bits for |v| >= 2^-126 and has a fixed
    # spacing of 2^-133 below that (its subnormals).
    e = np.floor(np.log2(np.where((a > 0) & np.isfinite(a), a, 1.0)))
    e = np.maximum(e, -126.0)
    # np.log2 can be off by one near powers of two: correct e so that
    # 2^e <= a < 2^(e+1) holds exactly for normal values.
    e = np.where((a >= 2.0 ** -126) & (np.ldexp(1.0, (e + 1).astype(np.int64)) <= a), e + 1, e)
    e = np.where((a >= 2.0 ** -126) & (np.ldexp(1.0, e.astype(np.int64)) > a), e - 1, e)
    e = np.maximum(e, -126.0)
    quantum = np.ldexp(1.0, (e - 7).astype(np.int64))  # spacing of bf16 values near a
    r = np.rint(a / quantum) * quantum  # a / quantum is exact; rint ties to even
    r = np.where(np.isfinite(a), r, a)
    with np.errstate(over="ignore"):  # values past the largest bf16 are set to inf below
        f32 = np.where(sign, -r, r).astype(np.float32)  # r has <= 8 significant bits: exact
    bits = f32.view(np.uint32)
    out[...] = (bits >> 16).astype(np.uint16)
    over = np.isfinite(a) & (r >= 2.0 ** 128)  # rounded past the largest finite bf16
    out[over] = np.where(sign[over], 0xFF80, 0x7F80)
    nan = np.isnan(v)
    out[nan] = 0x7FC0
    return out


def bf16_bits_to_float64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def round_to_f16(v: np.ndarray) -> np.ndarray:
    """float64 -> float16, numpy's direct (single) round-to-nearest-even."""
    return np.asarray(v, dtype=np.float64).astype(np.float16)
