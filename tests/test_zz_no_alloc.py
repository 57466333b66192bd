"""bil_linear_logp_fwd_static: the fused LM-head + logp with its scratch in a
static device array of BIL_LINEAR_STATIC_SCRATCH_BYTES (no workspace argument,
no allocation).  It must give the same bits as bil_linear_logp_fwd with a
caller workspace, call after call, and refuse sizes whose scratch would not
fit before queueing anything.

The file name puts it last in collection order, so that in a full run it also
executes after every other test has used the library; it passes alone too.
Calls go straight through the C ABI (ctypes), not through the Python binding.
"""
import ctypes

import numpy as np
import pytest
import torch

import invariant_token_log_gb300 as bil
from invariant_token_log_gb300 import _lib
import workloads as wl

V = wl.VOCAB  # the static array's limits are stated for this vocabulary
H = 256
MAX_ROWS = 1763          # without the entropy
MAX_ROWS_ENTROPY = 1176  # with it


def _p(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def workspace_bytes(n, entropy):
    out = ctypes.c_int64(0)
    assert _lib.load().bil_linear_logp_workspace_bytes(n, V, int(entropy), ctypes.byref(out)) == _lib.OK
    return out.value


def test_row_limits_follow_the_array_size():
    """Host arithmetic only: the largest row counts that fit are the stated ones."""
    cap = _lib.LINEAR_STATIC_SCRATCH_BYTES
    assert workspace_bytes(MAX_ROWS, False) <= cap < workspace_bytes(MAX_ROWS + 1, False)
    assert workspace_bytes(MAX_ROWS_ENTROPY, True) <= cap < workspace_bytes(MAX_ROWS_ENTROPY + 1, True)


def test_oversize_is_refused_before_anything_is_queued():
    """The size check comes first: no pointer is touched, so null pointers are fine here."""
    lib = _lib.load()
    for n, ent in ((MAX_ROWS + 1, None), (MAX_ROWS_ENTROPY + 1, ctypes.c_void_p(8))):
        st = lib.bil_linear_logp_fwd_static(None, None, _lib.BF16, n, H, H, V, H, 1.0, None, -100, None, None, ent, 0,
                                            None)
        assert st == _lib.E_UNSUPPORTED


def _inputs(n, seed):
    x = wl.linear_hidden(n, H, seed=seed)
    t = wl.rng(seed, 1).integers(0, V, n, dtype=np.int64)
    t[::7] = wl.IGNORE_INDEX
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    return xd, torch.from_numpy(t).cuda()


def _outputs(n, entropy):
    return [torch.full((n,), float("nan"), device="cuda") for _ in range(3 if entropy else 2)]


def _static(lib, xd, wd, td, outs):
    ent = outs[2] if len(outs) == 3 else None
    st = lib.bil_linear_logp_fwd_static(_p(xd), _p(wd), _lib.BF16, xd.shape[0], H, H, V, H, 1.0, _p(td), -100,
                                        _p(outs[0]), _p(outs[1]), _p(ent), 0, _stream())
    assert st == _lib.OK, _lib.status_string(st)


def _with_workspace(lib, xd, wd, td, outs):
    ent = outs[2] if len(outs) == 3 else None
    need = workspace_bytes(xd.shape[0], ent is not None)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = lib.bil_linear_logp_fwd(_p(xd), _p(wd), _lib.BF16, xd.shape[0], H, H, V, H, 1.0, _p(td), -100,
                                 _p(outs[0]), _p(outs[1]), _p(ent), None, _lib.F32, 0, _p(ws), need, 0, _stream())
    assert st == _lib.OK, _lib.status_string(st)


def _bits(t):
    return t.cpu().view(torch.int32).numpy()


@pytest.mark.gpu
def test_static_scratch_matches_the_workspace_entry_point():
    lib = _lib.load()
    wd = torch.from_numpy(wl.linear_weight(V, H, seed=31).view(np.int16)).cuda().view(torch.bfloat16)
    cases = [(_inputs(MAX_ROWS, 32), False), (_inputs(MAX_ROWS_ENTROPY, 33), True), (_inputs(5, 34), True)]
    # the workspace entry point's results first
    refs = []
    for (xd, td), ent in cases:
        outs = _outputs(xd.shape[0], ent)
        _with_workspace(lib, xd, wd, td, outs)
        refs.append(outs)
    torch.cuda.synchronize()
    # then the static entry point, several calls in a row on one stream: each
    # call reuses the scratch the previous one left behind
    for rep in range(2):
        for ((xd, td), ent), ref in zip(cases, refs):
            outs = _outputs(xd.shape[0], ent)
            _static(lib, xd, wd, td, outs)
            torch.cuda.synchronize()
            for a, b in zip(outs, ref):
                assert np.array_equal(_bits(a), _bits(b)), (rep, xd.shape[0], ent)
    assert bil.watchdog_status() == 0


@pytest.mark.gpu
def test_static_calls_allocate_nothing():
    """After a first call (which looks up the array's address), further calls
    leave both the CUDA allocator's and the device's free memory unchanged."""
    lib = _lib.load()
    wd = torch.from_numpy(wl.linear_weight(V, H, seed=35).view(np.int16)).cuda().view(torch.bfloat16)
    xd, td = _inputs(300, 36)
    outs = _outputs(300, True)
    _static(lib, xd, wd, td, outs)
    torch.cuda.synchronize()
    torch_before = torch.cuda.memory_allocated()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        _static(lib, xd, wd, td, outs)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == torch_before
    assert free_after == free_before, (free_before, free_after)
    assert bil.watchdog_status() == 0


@pytest.mark.gpu
def test_static_validate_reports_an_out_of_range_target():
    """validate=1 checks the targets on the host before anything is queued: an
    active target at the vocabulary size gives BIL_E_TARGET_RANGE and leaves
    the outputs untouched."""
    lib = _lib.load()
    wd = torch.from_numpy(wl.linear_weight(V, H, seed=37).view(np.int16)).cuda().view(torch.bfloat16)
    xd, td = _inputs(40, 38)
    td[11] = V
    outs = _outputs(40, False)
    st = lib.bil_linear_logp_fwd_static(_p(xd), _p(wd), _lib.BF16, 40, H, H, V, H, 1.0, _p(td), -100,
                                        _p(outs[0]), _p(outs[1]), None, 1, _stream())
    assert st == _lib.E_TARGET_RANGE
    torch.cuda.synchronize()
    assert all(torch.isnan(o).all() for o in outs)
    td[11] = 3
    _static(lib, xd, wd, td, outs)
    torch.cuda.synchronize()
    assert not any(torch.isnan(o).any() for o in outs)
    assert bil.watchdog_status() == 0
