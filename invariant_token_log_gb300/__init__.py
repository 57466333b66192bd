"""Batch-invariant selected-token log-probability for GB300 (sm_103a).

    logp = log_softmax(logits)[target]        (ignore_index rows give 0)

computed from fixed vocabulary tiles merged in one fixed order, so that a
row's bits never depend on the batch it is in.  The arithmetic runs in the
CUDA library ``libbil.so`` (C ABI in ``include/bil.h``); this package is its
PyTorch front end.  Build the library with
``python -m invariant_token_log_gb300.build``.
"""
from ._lib import BilError, contract_id, library_path, load  # noqa: F401
from .host_pipeline import HostStreamedLogp  # noqa: F401
from .linear import (  # noqa: F401
    LINEAR_TILE_V,
    LinearLogp,
    batch_invariant_linear_logp,
    gemm_nt,
    linear_logp,
    linear_logp_bwd,
    linear_logp_grad,
    linear_logp_partials,
    matmul,
)
from .logp import (  # noqa: F401
    DEFAULT_TILE_V,
    IGNORE_INDEX,
    BatchInvariantLogp,
    BatchInvariantLogpEntropy,
    batch_invariant_logp,
    logp_bwd,
    logp_fwd,
    logp_merge,
    logp_tile_partials,
    watchdog_status,
)
