"""PyTorch front end of the C ABI: argument marshalling only.

PyTorch supplies device memory and the current stream; every step of the
operator runs in the CUDA library (``libbil.so``).  Functions here check
shapes and devices, flatten ``[*lead, V]`` logits to ``[N, V]`` row-major
views (copying only when no such view exists), pass raw device pointers and
the current stream, and turn status codes into exceptions.

Operator: "Batch-Invariant LogP" operator page -- "Entry Point" (call shape:
logits, target_ids, ignore_index, validate), "Tensor Contract" (shapes and
dtypes), "Reference Semantics" (what is computed), "Tensor Parallel" (the
tile partials and fixed-order merge), "Batch-Invariance" (backward from the
saved per-row LSE).
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib

DEFAULT_TILE_V = 4096
IGNORE_INDEX = -100

_DTYPES = {torch.float32: _lib.F32, torch.bfloat16: _lib.BF16, torch.float16: _lib.F16}


def _code(dtype: torch.dtype) -> int:
    try:
        return _DTYPES[dtype]
    except KeyError:
        raise TypeError(f"unsupported element type {dtype}; expected float32, bfloat16 or float16") from None


def _rows2d(x: torch.Tensor) -> torch.Tensor:
    """[*lead, V] -> [N, V] with unit column stride (a view when one exists)."""
    if x.dim() == 2 and x.stride(-1) == 1:
        return x
    v = x.shape[-1]
    x2 = x.reshape(-1, v)
    if x2.stride(-1) != 1 and x2.numel() > 0:
        x2 = x2.contiguous()
    return x2


def _row_stride(x2: torch.Tensor) -> int:
    return x2.stride(0) if x2.shape[0] > 1 else max(x2.stride(0), x2.shape[1])


# The current stream's raw handle of a device, by index.  The private accessor
# skips building a torch.cuda.Stream object on every call; the public route is
# the fallback should a PyTorch build lack it.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(index: int) -> int:
    if _raw_stream is not None:
        return _raw_stream(index)
    return torch.cuda.current_stream(index).cuda_stream


def _stream(device: torch.device) -> ctypes.c_void_p:
    return ctypes.c_void_p(_stream_handle(device.index))


def _ptr(t: torch.Tensor | None):
    return None if t is None else t.data_ptr()


_get_device = getattr(torch._C, "_cuda_getDevice", None) or torch.cuda.current_device


def _on_device(index: int, fn, *args):
    """fn(*args) with device `index` current (switching only when it is not)."""
    if _get_device() == index:
        return fn(*args)
    with torch.cuda.device(index):
        return fn(*args)


_NARROW_INTS = (torch.int32, torch.int16, torch.int8, torch.uint8)


def _targets1d(target_ids: torch.Tensor, lead_shape, device) -> torch.Tensor:
    if target_ids.shape != lead_shape:
        if tuple(target_ids.shape) != tuple(lead_shape):
            raise ValueError(f"target_ids shape {tuple(target_ids.shape)} != logits leading shape {tuple(lead_shape)}")
    if target_ids.device != device:
        raise ValueError("target_ids must be on the logits' device")
    if target_ids.dtype is torch.int64:
        if target_ids.dim() == 1 and target_ids.is_contiguous():
            return target_ids
        return target_ids.reshape(-1).contiguous()
    if target_ids.dtype not in _NARROW_INTS:
        raise TypeError("target_ids must be an integer tensor")
    # the C ABI reads int64 targets; narrower integer types are widened here
    return target_ids.reshape(-1).to(torch.int64).contiguous()


def _f32_1d(t: torch.Tensor) -> torch.Tensor:
    """A contiguous float32 [N] view of a per-row tensor (converted only when it is not one)."""
    if t.dtype is torch.float32 and t.dim() == 1 and t.is_contiguous():
        return t
    return t.reshape(-1).to(torch.float32).contiguous()


def _check_out(t: torch.Tensor, n: int, index: int, what: str) -> None:
    """A caller-supplied per-row output: contiguous float32 with n elements on the device."""
    if t.dtype is not torch.float32 or t.numel() != n or not t.is_contiguous() or t.get_device() != index:
        raise ValueError(f"{what} must be a contiguous float32 tensor of {n} elements on the logits' device")


# torch.device objects by CUDA index: allocating with a device object skips
# parsing an integer into one on every call.
_DEVICE_OBJECTS: dict = {}


def _device_object(index: int) -> torch.device:
    dev = _DEVICE_OBJECTS[index] = torch.device("cuda", index)
    return dev


def _need_cuda(*ts: torch.Tensor) -> None:
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("the CUDA library needs CUDA tensors (there is no CPU path)")


def logp_fwd(logits: torch.Tensor, target_ids: torch.Tensor, ignore_index: int = IGNORE_INDEX,
             tile_v: int = DEFAULT_TILE_V, validate: bool = False, vocab: int | None = None,
             out: torch.Tensor | None = None, lse: torch.Tensor | None = None, temperature: float = 1.0,
             return_entropy: bool = False, entropy: torch.Tensor | None = None, with_lse: bool = True):
    """Selected-token log-probabilities: (logp, lse), both float32 with the targets' shape,
    and the row entropy as a third result when ``return_entropy`` (or ``entropy``) is given.

    ``with_lse=False`` (inference, no backward to come) returns ``(logp, None)``: the
    LSE is neither allocated nor written, and logp has the same bits.

    ``vocab`` (default: the last dimension) lets the row carry padding columns
    that are never read (e.g. a vocabulary padded to a multiple of the tile).
    ``temperature`` divides the logits before the softmax (applied as a
    multiplication by the float32 reciprocal).
    """
    index = logits.get_device()  # -1 for a CPU tensor
    tindex = target_ids.get_device()
    if index < 0 or tindex < 0:
        _need_cuda(logits, target_ids)
    shape = logits.shape
    tshape = target_ids.shape
    if (len(shape) == 2 and len(tshape) == 1 and tshape[0] == shape[0] and vocab is None
            and not (return_entropy or entropy is not None) and logits.is_contiguous()
            and target_ids.dtype is torch.int64 and target_ids.is_contiguous()):
        # The common call, [N, V] row-major logits and int64 [N] targets, without
        # the general path's reshaping: the per-call host time is what bounds
        # small (decode-sized) batches.
        n, width = shape
        if tindex != index:
            raise ValueError("target_ids must be on the logits' device")
        if out is None or (lse is None and with_lse):
            dev = _DEVICE_OBJECTS.get(index) or _device_object(index)
        if out is None:
            out = torch.empty(n, dtype=torch.float32, device=dev)
        else:
            _check_out(out, n, index, "out")
        if not with_lse:
            lse = None
        elif lse is None:
            lse = torch.empty(n, dtype=torch.float32, device=dev)
        else:
            _check_out(lse, n, index, "lse")
        fn = _lib.load().bil_logp_fwd
        args = (logits.data_ptr(), _code(logits.dtype), n, width, width, target_ids.data_ptr(), int(ignore_index),
                int(tile_v), float(temperature), out.data_ptr(), None if lse is None else lse.data_ptr(), None,
                1 if validate else 0, _stream_handle(index))
        st = fn(*args) if _get_device() == index else _on_device(index, fn, *args)
        if st:
            _lib.check("bil_logp_fwd", st)
        return out, lse
    if len(shape) == 2 and logits.is_contiguous():
        x2, lead = logits, shape[:1]
        n, width = shape
        ld = width
    else:
        lead = shape[:-1]
        x2 = _rows2d(logits)
        n, width = x2.shape
        ld = _row_stride(x2)
    v = width if vocab is None else int(vocab)
    if not 1 <= v <= width:
        raise ValueError(f"vocab {v} outside [1, {width}]")
    device = logits.device
    index = device.index
    t1 = _targets1d(target_ids, lead, device)
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=device)
    else:
        _check_out(out, n, index, "out")
    if not with_lse:
        lse = None
    elif lse is None:
        lse = torch.empty(n, dtype=torch.float32, device=device)
    else:
        _check_out(lse, n, index, "lse")
    want_ent = return_entropy or entropy is not None
    if want_ent and entropy is None:
        entropy = torch.empty(n, dtype=torch.float32, device=device)
    elif want_ent:
        _check_out(entropy, n, index, "entropy")
    st = _on_device(index, _lib.load().bil_logp_fwd, x2.data_ptr(), _code(x2.dtype), n, v, ld,
                    t1.data_ptr(), int(ignore_index), int(tile_v), float(temperature), out.data_ptr(),
                    None if lse is None else lse.data_ptr(), entropy.data_ptr() if want_ent else None,
                    1 if validate else 0, _stream_handle(index))
    if st:
        _lib.check("bil_logp_fwd", st)
    if len(lead) != 1:
        out = out.reshape(lead)
        lse = None if lse is None else lse.reshape(lead)
        if want_ent:
            entropy = entropy.reshape(lead)
    return (out, lse, entropy) if want_ent else (out, lse)


def logp_tile_partials(logits_shard: torch.Tensor, target_ids: torch.Tensor, vocab: int, tile_v: int,
                       tile_begin: int, tile_end: int, part_max: torch.Tensor, part_sum: torch.Tensor,
                       target_logit: torch.Tensor, ignore_index: int = IGNORE_INDEX, temperature: float = 1.0,
                       part_ent: torch.Tensor | None = None) -> None:
    """Fill columns [tile_begin, tile_end) of the [N, T] partial buffers
    (and of ``part_ent``, the entropy partials, when given).

    ``logits_shard`` is [N, >= shard columns]; its column 0 is global column
    ``tile_begin * tile_v`` (a rank's own vocabulary shard, or a column slice
    of the full logits)."""
    _need_cuda(logits_shard, target_ids, part_max, part_sum, target_logit)
    x2 = _rows2d(logits_shard)
    n = x2.shape[0]
    t1 = _targets1d(target_ids, (n,), logits_shard.device)
    bufs = (("part_max", part_max), ("part_sum", part_sum)) + ((("part_ent", part_ent),) if part_ent is not None else ())
    for name, b in bufs:
        if b.dtype != torch.float32 or b.dim() != 2 or b.shape[0] != n or b.stride(1) != 1:
            raise ValueError(f"{name} must be a row-major float32 [N, >= num_tiles] tensor")
        if b.stride(0) != part_max.stride(0):
            raise ValueError("the partial buffers must share a row stride")
    if target_logit.dtype != torch.float32 or target_logit.numel() != n or not target_logit.is_contiguous():
        raise ValueError("target_logit must be a contiguous float32 [N] tensor")
    index = logits_shard.device.index
    st = _on_device(index, _lib.load().bil_logp_tile_partials, x2.data_ptr(), _code(x2.dtype), n, int(vocab),
                    _row_stride(x2), int(tile_v), int(tile_begin), int(tile_end), float(temperature),
                    t1.data_ptr(), int(ignore_index), part_max.data_ptr(), part_sum.data_ptr(), _ptr(part_ent),
                    part_max.stride(0), target_logit.data_ptr(), _stream_handle(index))
    if st:
        _lib.check("bil_logp_tile_partials", st)


def logp_merge(part_max: torch.Tensor, part_sum: torch.Tensor, num_tiles: int, target_logit: torch.Tensor,
               target_ids: torch.Tensor, vocab: int, ignore_index: int = IGNORE_INDEX, validate: bool = False,
               part_ent: torch.Tensor | None = None, out: torch.Tensor | None = None,
               lse: torch.Tensor | None = None, entropy: torch.Tensor | None = None):
    """Fixed-order merge of [N, T] partials: (logp, lse) float32 [N], and the
    entropy as a third result when ``part_ent`` is given (``out``, ``lse``,
    ``entropy``: optional preallocated float32 [N] outputs)."""
    _need_cuda(part_max, part_sum, target_logit, target_ids)
    n = part_max.shape[0]
    t1 = _targets1d(target_ids, (n,), part_max.device)
    for b in (part_sum,) + ((part_ent,) if part_ent is not None else ()):
        if b.stride(0) != part_max.stride(0) or b.stride(1) != 1:
            raise ValueError("the partial buffers must be row-major with one row stride")
    if part_max.stride(1) != 1:
        raise ValueError("part_max must be row-major")
    for o in (out, lse, entropy):
        if o is not None and (o.dtype != torch.float32 or o.numel() != n or not o.is_contiguous()):
            raise ValueError("merge outputs must be contiguous float32 [N]")
    out = torch.empty(n, dtype=torch.float32, device=part_max.device) if out is None else out
    lse = torch.empty(n, dtype=torch.float32, device=part_max.device) if lse is None else lse
    ent = None
    if part_ent is not None:
        ent = torch.empty(n, dtype=torch.float32, device=part_max.device) if entropy is None else entropy
    index = part_max.device.index
    st = _on_device(index, _lib.load().bil_logp_merge, part_max.data_ptr(), part_sum.data_ptr(), _ptr(part_ent), n,
                    int(num_tiles), part_max.stride(0), target_logit.data_ptr(), t1.data_ptr(), int(ignore_index),
                    int(vocab), out.data_ptr(), lse.data_ptr(), _ptr(ent), 1 if validate else 0,
                    _stream_handle(index))
    if st:
        _lib.check("bil_logp_merge", st)
    return (out, lse, ent) if ent is not None else (out, lse)


def logp_bwd(logits: torch.Tensor, target_ids: torch.Tensor, lse: torch.Tensor, grad_logp: torch.Tensor,
             ignore_index: int = IGNORE_INDEX, dlogits_dtype: torch.dtype | None = None,
             vocab: int | None = None, out: torch.Tensor | None = None, temperature: float = 1.0,
             entropy: torch.Tensor | None = None, grad_entropy: torch.Tensor | None = None) -> torch.Tensor:
    """dlogits of g * logp (+ gh * entropy) from the saved LSE (and entropy).

    Returns a tensor of the logits' shape (columns past ``vocab`` are zero) in
    ``dlogits_dtype`` (default: the logits' dtype)."""
    _need_cuda(logits, target_ids, lse, grad_logp)
    if (entropy is None) != (grad_entropy is None):
        raise ValueError("entropy and grad_entropy go together")
    lead = logits.shape[:-1]
    x2 = _rows2d(logits)
    n, width = x2.shape
    v = width if vocab is None else int(vocab)
    t1 = _targets1d(target_ids, lead, logits.device)
    lse1 = _f32_1d(lse)
    g1 = _f32_1d(grad_logp)
    h1 = gh1 = None
    if entropy is not None:
        h1 = _f32_1d(entropy)
        gh1 = _f32_1d(grad_entropy)
        if h1.numel() != n or gh1.numel() != n:
            raise ValueError("entropy and grad_entropy must have the targets' shape")
    if lse1.numel() != n or g1.numel() != n:
        raise ValueError("lse and grad_logp must have the targets' shape")
    odt = logits.dtype if dlogits_dtype is None else dlogits_dtype
    if out is None:
        out = torch.empty((n, width), dtype=odt, device=logits.device)
    if n == 0:
        return out.reshape(logits.shape) if out.numel() == 0 else out
    o2 = out if out.dim() == 2 else out.reshape(n, -1)
    if o2.shape[0] != n or o2.stride(-1) != 1 or o2.shape[1] < width:
        raise ValueError("out must be row-major with at least the logits' columns")
    index = logits.device.index
    st = _on_device(index, _lib.load().bil_logp_bwd, x2.data_ptr(), _code(x2.dtype), n, v, _row_stride(x2),
                    t1.data_ptr(), int(ignore_index), float(temperature), lse1.data_ptr(), g1.data_ptr(), _ptr(h1),
                    _ptr(gh1), o2.data_ptr(), _code(o2.dtype), _row_stride(o2), width, _stream_handle(index))
    if st:
        _lib.check("bil_logp_bwd", st)
    return out.reshape(logits.shape) if out.numel() == logits.numel() else out


class BatchInvariantLogp(torch.autograd.Function):
    """logp = BatchInvariantLogp.apply(logits, target_ids, ignore_index, tile_v, validate, temperature)

    The forward saves the per-row LSE; the backward recomputes the softmax
    from it.  target_ids receives no gradient."""

    @staticmethod
    def forward(ctx, logits, target_ids, ignore_index=IGNORE_INDEX, tile_v=DEFAULT_TILE_V, validate=False,
                temperature=1.0):
        logp, lse = logp_fwd(logits, target_ids, ignore_index, tile_v, validate, temperature=temperature)
        ctx.save_for_backward(logits, target_ids, lse)
        ctx.ignore_index, ctx.temperature = ignore_index, temperature
        return logp

    @staticmethod
    def backward(ctx, grad_logp):
        logits, target_ids, lse = ctx.saved_tensors
        d = logp_bwd(logits, target_ids, lse, grad_logp.contiguous(), ctx.ignore_index, temperature=ctx.temperature)
        return d, None, None, None, None, None


class BatchInvariantLogpEntropy(torch.autograd.Function):
    """(logp, entropy) = BatchInvariantLogpEntropy.apply(logits, target_ids, ignore_index, tile_v,
    validate, temperature): both outputs differentiable with respect to the logits."""

    @staticmethod
    def forward(ctx, logits, target_ids, ignore_index=IGNORE_INDEX, tile_v=DEFAULT_TILE_V, validate=False,
                temperature=1.0):
        logp, lse, ent = logp_fwd(logits, target_ids, ignore_index, tile_v, validate, temperature=temperature,
                                  return_entropy=True)
        ctx.save_for_backward(logits, target_ids, lse, ent)
        ctx.ignore_index, ctx.temperature = ignore_index, temperature
        return logp, ent

    @staticmethod
    def backward(ctx, grad_logp, grad_ent):
        logits, target_ids, lse, ent = ctx.saved_tensors
        if grad_logp is None:
            grad_logp = torch.zeros_like(lse)
        if grad_ent is None:
            grad_ent = torch.zeros_like(ent)
        d = logp_bwd(logits, target_ids, lse, grad_logp.contiguous(), ctx.ignore_index, temperature=ctx.temperature,
                     entropy=ent, grad_entropy=grad_ent.contiguous())
        return d, None, None, None, None, None


def batch_invariant_logp(logits: torch.Tensor, target_ids: torch.Tensor, ignore_index: int = IGNORE_INDEX,
                         validate: bool = False, tile_v: int = DEFAULT_TILE_V, temperature: float = 1.0,
                         return_entropy: bool = False):
    """Differentiable selected-token log-probability, float32 with the targets' shape;
    with ``return_entropy``, (logp, entropy)."""
    if return_entropy:
        return BatchInvariantLogpEntropy.apply(logits, target_ids, ignore_index, tile_v, validate, temperature)
    return BatchInvariantLogp.apply(logits, target_ids, ignore_index, tile_v, validate, temperature)


def watchdog_status(clear: bool = True) -> int:
    """Bits set by kernel waits that ran out on the current device (0 = none)."""
    flags = ctypes.c_uint(0)
    _lib.check("bil_watchdog_status", _lib.load().bil_watchdog_status(ctypes.byref(flags), int(clear)))
    return int(flags.value)
