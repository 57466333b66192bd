"""Host-resident batches streamed in row chunks give the one-shot bits.

Every row's result is independent of the batch it is computed in, so
cutting the batch into chunks that overlap copies and kernels
(HostStreamedLogp) must reproduce logp and dlogits exactly, including a
ragged last chunk and ignored rows.
"""
import numpy as np
import pytest
import torch

import invariant_token_log_gb300 as bil
import workloads as wl
from gpu_helpers import check_watchdog, device_logits, f32_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("chunk_rows", [1000, 4096])
def test_streamed_host_batch_matches_one_shot(chunk_rows):
    w = wl.random_rows(seed=21, n_rows=2500, vocab=151936, dtype="bfloat16", tile_v=4096, ignore_every=9)
    x = device_logits(w.logits, "bfloat16")
    t = torch.from_numpy(w.target_ids).cuda()
    g = torch.from_numpy(w.grad_logp).cuda()
    logp, lse = bil.logp_fwd(x, t, w.ignore_index, 4096)
    d = bil.logp_bwd(x, t, lse, g, w.ignore_index)
    torch.cuda.synchronize()

    n, v = w.n_rows, w.vocab
    x_h = x.cpu().pin_memory()
    t_h = t.cpu().pin_memory()
    g_h = g.cpu().pin_memory()
    lp_h = torch.full((n,), float("nan")).pin_memory()
    d_h = torch.zeros((n, v), dtype=torch.bfloat16).pin_memory()
    pipe = bil.HostStreamedLogp(n, v, torch.bfloat16, torch.bfloat16, chunk_rows=chunk_rows)
    launches = pipe.run(x_h, t_h, g_h, lp_h, d_h, w.ignore_index, 4096)
    torch.cuda.synchronize()
    assert launches == 2 * (-(-n // min(chunk_rows, n)))
    assert np.array_equal(lp_h.view(torch.int32).numpy(), f32_bits(logp))
    assert torch.equal(d_h.view(torch.int16), d.cpu().view(torch.int16))
    check_watchdog()


def test_back_to_back_batches_without_input_ordering_keep_their_bits():
    """order_inputs=False lets each batch's copies in start while the batch before is still
    copying out; the chunk buffers are guarded by the pipeline's events across calls.  Three
    different batches queued back to back (3 chunks each, so the buffers' turns cross the call
    boundary) must each give their one-shot bits."""
    n, v, chunk = 2500, 50257, 1000
    batches = [wl.random_rows(seed=s, n_rows=n, vocab=v, dtype="bfloat16", tile_v=4096, ignore_every=7)
               for s in (31, 32, 33)]
    pipe = bil.HostStreamedLogp(n, v, torch.bfloat16, torch.bfloat16, chunk_rows=chunk)
    ref, host = [], []
    for w in batches:
        x = device_logits(w.logits, "bfloat16")
        t = torch.from_numpy(w.target_ids).cuda()
        g = torch.from_numpy(w.grad_logp).cuda()
        logp, lse = bil.logp_fwd(x, t, w.ignore_index, 4096)
        ref.append((f32_bits(logp), bil.logp_bwd(x, t, lse, g, w.ignore_index).cpu().view(torch.int16)))
        host.append((x.cpu().pin_memory(), t.cpu().pin_memory(), g.cpu().pin_memory(),
                     torch.full((n,), float("nan")).pin_memory(),
                     torch.zeros((n, v), dtype=torch.bfloat16).pin_memory()))
    torch.cuda.synchronize()
    for _ in range(2):
        for x_h, t_h, g_h, lp_h, d_h in host:
            pipe.run(x_h, t_h, g_h, lp_h, d_h, batches[0].ignore_index, 4096, order_inputs=False)
    torch.cuda.synchronize()
    for (lp_ref, d_ref), (_, _, _, lp_h, d_h) in zip(ref, host):
        assert np.array_equal(lp_h.view(torch.int32).numpy(), lp_ref)
        assert torch.equal(d_h.view(torch.int16), d_ref)
    check_watchdog()
