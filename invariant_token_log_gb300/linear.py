"""PyTorch front end of the fused LM-head + logp: argument marshalling only.

"[RFC][ROCm] End-to-end optimization of bitwise VIME R/R beyond native P/P",
section "Workstream 3: fused ROCm LM-head and linear logp": the projection
z = hidden . weight^T and the selected-token log-probability (with the
optional lse, entropy and unscaled logits) are one operation; the logits are
stored only when asked for, and logp / lse / entropy are the same bits either
way.  The projection runs on the tensor cores (tcgen05) inside the CUDA
library, followed by the operator's fixed-order merge over tiles of
``LINEAR_TILE_V`` (256) vocabulary columns.

Layouts: hidden [*lead, H] and weight [V, H] (one row per vocabulary entry,
as an LM-head ``Linear`` stores it), both bfloat16 or both float16, rows
16-byte aligned.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from .logp import IGNORE_INDEX, _need_cuda, _ptr, _stream, logp_bwd

LINEAR_TILE_V = _lib.LINEAR_TILE_V
_IN_DTYPES = {torch.bfloat16: _lib.BF16, torch.float16: _lib.F16}
_OUT_DTYPES = {torch.float32: _lib.F32, torch.bfloat16: _lib.BF16}


def _in_code(dtype: torch.dtype) -> int:
    try:
        return _IN_DTYPES[dtype]
    except KeyError:
        raise TypeError(f"hidden and weight must be bfloat16 or float16, not {dtype}") from None


def _matrix(x: torch.Tensor, what: str) -> torch.Tensor:
    """[*lead, H] -> [N, H] with unit column stride and a row stride the C ABI accepts."""
    x2 = x.reshape(-1, x.shape[-1])
    if x2.shape[0] and (x2.stride(-1) != 1 or (x2.stride(0) * 2) % 16 or x2.data_ptr() % 16):
        x2 = x2.contiguous()
        if (x2.stride(0) * 2) % 16:
            raise ValueError(f"{what}: the last dimension must be a multiple of 8 elements (16-byte rows)")
    return x2


def _ld(x2: torch.Tensor) -> int:
    return x2.stride(0) if x2.shape[0] > 1 else max(x2.stride(0), x2.shape[1])


def num_tiles(vocab: int) -> int:
    """Vocabulary tiles of the fused LM-head: ceil(vocab / 256), the GEMM's N tile."""
    return -(-vocab // LINEAR_TILE_V)


def workspace_bytes(n_rows: int, vocab: int, entropy: bool = False) -> int:
    """Device scratch bytes bil_linear_logp_fwd needs for n_rows rows: the [n_rows, num_tiles]
    float32 partials (max, sum-exp and, with the entropy, its sums) and the target logits."""
    out = ctypes.c_int64(0)
    _lib.check("bil_linear_logp_workspace_bytes",
               _lib.load().bil_linear_logp_workspace_bytes(n_rows, vocab, int(entropy), ctypes.byref(out)))
    return out.value


def linear_logp_partials(hidden: torch.Tensor, weight_shard: torch.Tensor, target_ids: torch.Tensor, vocab: int,
                         tile_begin: int, tile_end: int, part_max: torch.Tensor, part_sum: torch.Tensor,
                         target_logit: torch.Tensor, ignore_index: int = IGNORE_INDEX, temperature: float = 1.0,
                         part_ent: torch.Tensor | None = None, logits_out: torch.Tensor | None = None) -> None:
    """Tile partials of tiles [tile_begin, tile_end) into [N, ld_part] float32 buffers.

    ``weight_shard`` row j is the LM-head row of global vocabulary column
    ``tile_begin * LINEAR_TILE_V + j``; ``logits_out`` (optional, float32 or
    bfloat16, [N, >= shard columns]) receives the shard's unscaled logits."""
    _need_cuda(hidden, weight_shard, target_ids, part_max, part_sum, target_logit, part_ent, logits_out)
    h2, w2 = _matrix(hidden, "hidden"), _matrix(weight_shard, "weight")
    if h2.dtype != w2.dtype:
        raise TypeError("hidden and weight must have the same element type")
    if h2.shape[1] != w2.shape[1]:
        raise ValueError(f"hidden size {h2.shape[1]} != weight's {w2.shape[1]}")
    t = target_ids.reshape(-1).to(torch.int64).contiguous()
    n = h2.shape[0]
    if t.shape[0] != n:
        raise ValueError("target_ids must have one entry per hidden row")
    for buf in (part_max, part_sum) + ((part_ent,) if part_ent is not None else ()):
        if buf.dtype != torch.float32 or buf.dim() != 2 or buf.shape[0] != n or buf.stride(1) != 1:
            raise ValueError("partials must be [N, >= num_tiles] float32 with unit column stride")
    if part_ent is not None and part_ent.stride(0) != part_max.stride(0):
        raise ValueError("part_ent must have part_max's row stride")
    ld_out, out_code = 0, _lib.F32
    if logits_out is not None:
        if logits_out.dtype not in _OUT_DTYPES or logits_out.dim() != 2 or logits_out.stride(1) != 1:
            raise ValueError("logits_out must be [N, >= shard columns] float32 or bfloat16, unit column stride")
        ld_out, out_code = logits_out.stride(0), _OUT_DTYPES[logits_out.dtype]
    _lib.check("bil_linear_logp_partials", _lib.load().bil_linear_logp_partials(
        _ptr(h2), _ptr(w2), _in_code(h2.dtype), n, h2.shape[1], _ld(h2), vocab, _ld(w2), tile_begin, tile_end,
        float(temperature), _ptr(t), ignore_index, _ptr(part_max), _ptr(part_sum), _ptr(part_ent),
        part_max.stride(0), _ptr(target_logit), _ptr(logits_out), out_code, ld_out, _stream(h2.device)))


def linear_logp(hidden: torch.Tensor, weight: torch.Tensor, target_ids: torch.Tensor,
                ignore_index: int = IGNORE_INDEX, temperature: float = 1.0, return_entropy: bool = False,
                return_logits: bool = False, logits_dtype: torch.dtype = torch.float32, validate: bool = False,
                workspace: torch.Tensor | None = None):
    """Fused LM-head + logp: (logp, lse[, entropy][, logits]) for hidden [*lead, H] and
    weight [V, H]; logp/lse/entropy are float32 with the targets' shape, logits
    [*lead, V] of ``logits_dtype`` (the projection before the temperature)."""
    _need_cuda(hidden, weight, target_ids, workspace)
    lead = hidden.shape[:-1]
    if tuple(target_ids.shape) != tuple(lead):
        raise ValueError(f"target_ids shape {tuple(target_ids.shape)} != hidden's leading shape {tuple(lead)}")
    h2, w2 = _matrix(hidden, "hidden"), _matrix(weight, "weight")
    if h2.dtype != w2.dtype:
        raise TypeError("hidden and weight must have the same element type")
    if h2.shape[1] != w2.shape[1]:
        raise ValueError(f"hidden size {h2.shape[1]} != weight's {w2.shape[1]}")
    n, vocab = h2.shape[0], w2.shape[0]
    t = target_ids.reshape(-1).to(torch.int64).contiguous()
    dev = h2.device
    logp = torch.empty(n, dtype=torch.float32, device=dev)
    lse = torch.empty(n, dtype=torch.float32, device=dev)
    ent = torch.empty(n, dtype=torch.float32, device=dev) if return_entropy else None
    logits = None
    if return_logits:
        if logits_dtype not in _OUT_DTYPES:
            raise TypeError("logits_dtype must be float32 or bfloat16")
        cols = -(-vocab // 8) * 8  # 16-byte rows for either output type
        logits = torch.empty((n, cols), dtype=logits_dtype, device=dev)[:, :vocab]
    need = workspace_bytes(n, vocab, return_entropy)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    elif workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace holds {workspace.numel() * workspace.element_size()} bytes, needs {need}")
    _lib.check("bil_linear_logp_fwd", _lib.load().bil_linear_logp_fwd(
        _ptr(h2), _ptr(w2), _in_code(h2.dtype), n, h2.shape[1], _ld(h2), vocab, _ld(w2), float(temperature),
        _ptr(t), ignore_index, _ptr(logp), _ptr(lse), _ptr(ent), _ptr(logits),
        _OUT_DTYPES.get(logits_dtype, _lib.F32), logits.stride(0) if logits is not None else 0, _ptr(workspace),
        workspace.numel() * workspace.element_size(), int(validate), _stream(dev)))
    out = [logp.reshape(lead), lse.reshape(lead)]
    if return_entropy:
        out.append(ent.reshape(lead))
    if return_logits:
        out.append(logits.reshape(*lead, vocab))
    return tuple(out)


def _pad8(n: int) -> int:
    return -(-n // 8) * 8


def linear_logp_bwd(hidden: torch.Tensor, weight: torch.Tensor, target_ids: torch.Tensor, lse: torch.Tensor,
                    grad_logp: torch.Tensor, ignore_index: int = IGNORE_INDEX, temperature: float = 1.0,
                    entropy: torch.Tensor | None = None, grad_entropy: torch.Tensor | None = None,
                    out_dtype: torch.dtype | None = None, return_dz: bool = False, vocab: int | None = None,
                    tile_begin: int = 0, tile_end: int | None = None):
    """(dhidden [*lead, H], dweight [cols, H][, dZ [N, cols]]) of g * logp (+ gh * entropy).

    ``weight`` holds the LM-head rows of global vocabulary columns
    [tile_begin * 256, min(tile_end * 256, vocab)) ("cols"; by default the
    whole vocabulary, vocab = weight rows).  With a shard, dhidden is the
    shard's part of the sum over the vocabulary.  ``out_dtype`` is float32 or
    the inputs' type (the default)."""
    _need_cuda(hidden, weight, target_ids, lse, grad_logp, entropy, grad_entropy)
    lead = hidden.shape[:-1]
    h2, w2 = _matrix(hidden, "hidden"), _matrix(weight, "weight")
    if h2.dtype != w2.dtype or h2.shape[1] != w2.shape[1]:
        raise ValueError("hidden and weight must share the element type and the hidden size")
    n, hs = h2.shape
    vocab = w2.shape[0] if vocab is None else vocab
    tile_end = num_tiles(vocab) if tile_end is None else tile_end
    v = min(tile_end * LINEAR_TILE_V, vocab) - tile_begin * LINEAR_TILE_V  # the shard's columns
    if v <= 0 or w2.shape[0] < v:
        raise ValueError(f"the weight holds {w2.shape[0]} rows; tiles [{tile_begin}, {tile_end}) need {v}")
    w2 = w2[:v]
    dev = h2.device
    t = target_ids.reshape(-1).to(torch.int64).contiguous()
    if (entropy is None) != (grad_entropy is None):
        raise ValueError("entropy and grad_entropy come together")
    f32 = [x.reshape(-1).float().contiguous() if x is not None else None
           for x in (lse, grad_logp, entropy, grad_entropy)]
    out_dtype = h2.dtype if out_dtype is None else out_dtype
    if out_dtype not in (torch.float32, h2.dtype):
        raise TypeError("out_dtype must be float32 or the inputs' type")
    dz = torch.empty((n, _pad8(v)), dtype=h2.dtype, device=dev)[:, :v]
    dh = torch.empty((n, _pad8(hs)), dtype=out_dtype, device=dev)[:, :hs]
    dw = torch.empty((v, _pad8(hs)), dtype=out_dtype, device=dev)[:, :hs]
    oc = _lib.F32 if out_dtype == torch.float32 else _in_code(out_dtype)
    _lib.check("bil_linear_logp_bwd", _lib.load().bil_linear_logp_bwd(
        _ptr(h2), _ptr(w2), _in_code(h2.dtype), n, hs, _ld(h2), vocab, _ld(w2), tile_begin, tile_end,
        float(temperature), _ptr(t), ignore_index, _ptr(f32[0]), _ptr(f32[1]), _ptr(f32[2]), _ptr(f32[3]),
        _ptr(dz), dz.stride(0), _ptr(dh), oc, dh.stride(0), _ptr(dw), oc, dw.stride(0), _stream(dev)))
    out = (dh.reshape(*lead, hs), dw)
    return out + (dz,) if return_dz else out


def linear_logp_grad(hidden: torch.Tensor, weight: torch.Tensor, target_ids: torch.Tensor, lse: torch.Tensor,
                     grad_logp: torch.Tensor, ignore_index: int = IGNORE_INDEX, temperature: float = 1.0,
                     entropy: torch.Tensor | None = None, grad_entropy: torch.Tensor | None = None) -> torch.Tensor:
    """dZ [N, V] of g * logp (+ gh * entropy) over the whole vocabulary (V =
    weight rows): the first step of ``linear_logp_bwd`` alone, the same bits.
    The other two are ``matmul(dz, weight)`` and ``matmul(dz.t(), hidden)``."""
    _need_cuda(hidden, weight, target_ids, lse, grad_logp, entropy, grad_entropy)
    h2, w2 = _matrix(hidden, "hidden"), _matrix(weight, "weight")
    if h2.dtype != w2.dtype or h2.shape[1] != w2.shape[1]:
        raise ValueError("hidden and weight must share the element type and the hidden size")
    if (entropy is None) != (grad_entropy is None):
        raise ValueError("entropy and grad_entropy come together")
    n, hs = h2.shape
    v = w2.shape[0]
    dev = h2.device
    t = target_ids.reshape(-1).to(torch.int64).contiguous()
    f32 = [x.reshape(-1).float().contiguous() if x is not None else None
           for x in (lse, grad_logp, entropy, grad_entropy)]
    dz = torch.empty((n, _pad8(v)), dtype=h2.dtype, device=dev)[:, :v]
    _lib.check("bil_linear_logp_grad", _lib.load().bil_linear_logp_grad(
        _ptr(h2), _ptr(w2), _in_code(h2.dtype), n, hs, _ld(h2), v, _ld(w2), 0, num_tiles(v), float(temperature),
        _ptr(t), ignore_index, _ptr(f32[0]), _ptr(f32[1]), _ptr(f32[2]), _ptr(f32[3]), _ptr(dz), dz.stride(0),
        _stream(dev)))
    return dz


def _rows_over_k(x: torch.Tensor, k_dim: int) -> tuple[torch.Tensor, int, int]:
    """(tensor, layout, row stride) of a 2-D operand whose dimension ``k_dim`` is K, as
    bil_linear_gemm finds it: K-major when K is the unit-stride dimension, MN-major
    when the other one is (a transposed view of a row-major matrix), else a
    contiguous copy with the rows over K."""
    r_dim = 1 - k_dim
    rows, k = x.shape[r_dim], x.shape[k_dim]
    for layout, unit, ld_dim, run in ((_lib.LAYOUT_K_MAJOR, k_dim, r_dim, k), (_lib.LAYOUT_MN_MAJOR, r_dim, k_dim, rows)):
        outer = x.shape[ld_dim]
        ld = x.stride(ld_dim) if outer > 1 else max(x.stride(ld_dim), run)
        if (x.stride(unit) == 1 or x.shape[unit] == 1) and ld >= run and (ld * 2) % 16 == 0 and x.data_ptr() % 16 == 0:
            return x, layout, ld
    y = x.transpose(0, 1) if k_dim == 0 else x
    y = torch.empty((rows, _pad8(k)), dtype=x.dtype, device=x.device)[:, :k].copy_(y)
    return y, _lib.LAYOUT_K_MAJOR, y.stride(0)


def matmul(a: torch.Tensor, b: torch.Tensor, out_dtype: torch.dtype = torch.float32) -> torch.Tensor:
    """C = a @ b for a [m, k] and b [k, n] (both bfloat16 or both float16) on the
    tensor cores, float32 accumulation over K blocks of 64 in order: the
    backward's dhidden (``matmul(dz, weight)``) and dweight (``matmul(dz.t(),
    hidden)``) contraction.  Each operand is read where it lies when one of
    its dimensions has unit stride (a row-major matrix or a transposed view of
    one, 16-byte aligned rows), else from a copy.  C is float32 or the inputs'
    type."""
    _need_cuda(a, b)
    if a.dim() != 2 or b.dim() != 2 or a.shape[1] != b.shape[0] or a.dtype != b.dtype:
        raise ValueError("matmul takes a [m, k] and b [k, n] of one 16-bit type")
    if out_dtype not in (torch.float32, a.dtype):
        raise TypeError("out_dtype must be float32 or the inputs' type")
    m, k = a.shape
    n = b.shape[1]
    c = torch.empty((m, _pad8(n)), dtype=out_dtype, device=a.device)[:, :n]
    if m == 0 or n == 0:
        return c
    if k == 0:
        raise ValueError("matmul needs k >= 1 (the library computes no empty sums)")
    a2, la, lda = _rows_over_k(a, 1)
    b2, lb, ldb = _rows_over_k(b, 0)
    oc = _lib.F32 if out_dtype == torch.float32 else _in_code(out_dtype)
    _lib.check("bil_linear_gemm", _lib.load().bil_linear_gemm(
        _ptr(a2), la, _ptr(b2), lb, _in_code(a2.dtype), m, n, k, lda, ldb, _ptr(c), oc, c.stride(0),
        _stream(a2.device)))
    return c


def gemm_nt(a: torch.Tensor, b: torch.Tensor, out_dtype: torch.dtype = torch.float32) -> torch.Tensor:
    """C = a . b^T for a [m, k] and b [n, k]: ``matmul(a, b.t())``."""
    return matmul(a, b.t(), out_dtype)


def linear_logp_bwd_from_logits(hidden: torch.Tensor, weight: torch.Tensor, target_ids: torch.Tensor,
                                logits: torch.Tensor, lse: torch.Tensor, grad_logp: torch.Tensor,
                                ignore_index: int = IGNORE_INDEX, temperature: float = 1.0,
                                entropy: torch.Tensor | None = None, grad_entropy: torch.Tensor | None = None,
                                out_dtype: torch.dtype | None = None):
    """(dhidden [N, H], dweight [V, H]) like ``linear_logp_bwd``, from the forward's float32
    logits [N, V] (``linear_logp(..., return_logits=True, logits_dtype=torch.float32)``)
    instead of recomputing the projection: dZ by the logits path's backward on the stored
    logits, then the two products.  The same bits as ``linear_logp_bwd``; the logits cost
    4 bytes per row and vocabulary column while they are kept."""
    _need_cuda(hidden, weight, target_ids, logits, lse, grad_logp, entropy, grad_entropy)
    h2, w2 = _matrix(hidden, "hidden"), _matrix(weight, "weight")
    if logits.dtype != torch.float32 or logits.dim() != 2 or logits.shape != (h2.shape[0], w2.shape[0]):
        raise ValueError("logits must be the forward's float32 [N, V] projection")
    n, v = logits.shape
    dz = torch.empty((n, _pad8(v)), dtype=h2.dtype, device=h2.device)[:, :v]
    logp_bwd(logits, target_ids.reshape(-1), lse.reshape(-1), grad_logp.reshape(-1), ignore_index, out=dz,
             temperature=temperature, entropy=None if entropy is None else entropy.reshape(-1),
             grad_entropy=None if grad_entropy is None else grad_entropy.reshape(-1))
    out_dtype = h2.dtype if out_dtype is None else out_dtype
    return matmul(dz, w2, out_dtype), matmul(dz.t(), h2, out_dtype)


class LinearLogp(torch.autograd.Function):
    """Fused LM-head + logp with the autograd actor path: the forward keeps only
    lse (and the entropy), and the backward recomputes the projection tiles; or,
    with ``keep_logits``, the forward also keeps its float32 logits and the
    backward starts from them (the same bits, one GEMM fewer, 4 bytes per row and
    vocabulary column kept until the backward)."""

    @staticmethod
    def forward(ctx, hidden, weight, target_ids, ignore_index, temperature, return_entropy, keep_logits=False):
        lead = hidden.shape[:-1]
        if keep_logits:
            res = linear_logp(hidden.reshape(-1, hidden.shape[-1]), weight, target_ids.reshape(-1), ignore_index,
                              temperature, return_entropy, return_logits=True, logits_dtype=torch.float32)
            logits = res[-1]
            res = tuple(r.reshape(lead) for r in res[:-1])
            ctx.save_for_backward(hidden, weight, target_ids, logits, *res[1:])
        else:
            res = linear_logp(hidden, weight, target_ids, ignore_index, temperature, return_entropy)
            ctx.save_for_backward(hidden, weight, target_ids, *res[1:])
        ctx.ignore_index, ctx.temperature, ctx.return_entropy = ignore_index, temperature, return_entropy
        ctx.keep_logits = keep_logits
        ctx.mark_non_differentiable(res[1])
        return res

    @staticmethod
    def backward(ctx, grad_logp, grad_lse, *rest):
        saved = list(ctx.saved_tensors)
        hidden, weight, target_ids = saved[:3]
        logits = saved[3] if ctx.keep_logits else None
        lse, *ent = saved[4:] if ctx.keep_logits else saved[3:]
        g = torch.zeros_like(lse) if grad_logp is None else grad_logp
        entropy = grad_entropy = None
        if ctx.return_entropy and rest and rest[0] is not None:
            entropy, grad_entropy = ent[0], rest[0]
        need_h, need_w = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        nones = (None,) * 5
        if not (need_h or need_w):
            return (None, None) + nones
        if logits is not None:
            dh, dw = linear_logp_bwd_from_logits(hidden, weight, target_ids, logits, lse, g, ctx.ignore_index,
                                                 ctx.temperature, entropy, grad_entropy)
            dh = dh.reshape(hidden.shape)
        else:
            dh, dw = linear_logp_bwd(hidden, weight, target_ids, lse, g, ctx.ignore_index, ctx.temperature,
                                     entropy, grad_entropy)
        return (dh if need_h else None, dw if need_w else None) + nones


def batch_invariant_linear_logp(hidden: torch.Tensor, weight: torch.Tensor, target_ids: torch.Tensor,
                                ignore_index: int = IGNORE_INDEX, temperature: float = 1.0,
                                return_entropy: bool = False, keep_logits: bool = False):
    """Differentiable fused LM-head + logp: logp (and the entropy when asked) with
    gradients for hidden and weight.  ``keep_logits`` trades 4 bytes per row and
    vocabulary column, kept from the forward to the backward, for the backward's
    recomputation of the projection (the same bits)."""
    res = LinearLogp.apply(hidden, weight, target_ids, ignore_index, temperature, return_entropy, keep_logits)
    return (res[0], res[2]) if return_entropy else res[0]


def sum_f32(parts: list[torch.Tensor], out: torch.Tensor | None = None) -> torch.Tensor:
    """((parts[0] + parts[1]) + parts[2]) + ... elementwise in float32, in list order."""
    _need_cuda(*parts)
    ps = [p.contiguous() for p in parts]
    if any(p.dtype != torch.float32 or p.shape != ps[0].shape for p in ps):
        raise ValueError("sum_f32 takes float32 tensors of one shape")
    out = torch.empty_like(ps[0]) if out is None else out
    arr = (ctypes.c_void_p * len(ps))(*[p.data_ptr() for p in ps])
    _lib.check("bil_sum_f32", _lib.load().bil_sum_f32(arr, len(ps), ps[0].numel(), _ptr(out), _stream(ps[0].device)))
    return out
