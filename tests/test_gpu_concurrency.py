"""Several host threads, each on its own CUDA stream, call the library at once.

The library keeps no per-call state (its only caches are per-device
attributes, published atomically), and ctypes releases the GIL during the
calls, so the host threads really overlap in it.  Every thread's results must
equal the serial results bit for bit.
"""
import threading

import numpy as np
import pytest
import torch

import invariant_token_log_gb300 as bil
import workloads as wl
from gpu_helpers import check_watchdog, device_logits, f32_bits, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _watchdog():
    yield
    check_watchdog()


def _batches():
    out = []
    for k, (n, v) in enumerate(((64, 32000), (7, 50257), (300, 8192), (1, 151936))):
        w = wl.random_rows(seed=80 + k, n_rows=n, vocab=v, dtype="bfloat16", tile_v=4096, ignore_every=5)
        out.append((device_logits(w.logits, "bfloat16"), torch.from_numpy(w.target_ids).cuda(),
                    torch.from_numpy(w.grad_logp).cuda(), w.ignore_index))
    return out


def _run(x, t, g, ignore):
    logp, lse, ent = bil.logp_fwd(x, t, ignore, 4096, temperature=0.9, return_entropy=True)
    d = bil.logp_bwd(x, t, lse, g, ignore, temperature=0.9)
    return logp, lse, ent, d


def test_threads_on_their_own_streams_get_the_serial_bits():
    batches = _batches()
    ref = [_run(*b) for b in batches]
    torch.cuda.synchronize()
    ref_bits = [(f32_bits(a), f32_bits(b), f32_bits(c), host_bits(d)) for a, b, c, d in ref]

    results = [[None] * 6 for _ in batches]
    errors = []
    start = threading.Barrier(len(batches))

    def worker(i):
        try:
            s = torch.cuda.Stream()
            start.wait()
            with torch.cuda.stream(s):
                for r in range(6):
                    results[i][r] = _run(*batches[i])
            s.synchronize()
        except Exception as e:  # reported below, in the main thread
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(batches))]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=120)
    assert not errors, errors
    assert not any(th.is_alive() for th in threads)
    torch.cuda.synchronize()
    for i, rb in enumerate(ref_bits):
        for r in range(6):
            a, b, c, d = results[i][r]
            got = (f32_bits(a), f32_bits(b), f32_bits(c), host_bits(d))
            for gbits, want in zip(got, rb):
                assert np.array_equal(gbits, want), (i, r)
