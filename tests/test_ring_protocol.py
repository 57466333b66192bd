"""The forward kernels' shared-memory ring protocol, checked on the CPU.

The producer warp fills stages in unit order with bulk copies that may
complete in any order; consumer warp c takes units c, c+W, c+2W, ... and
waits on a stage's "full" barrier by the parity of that stage's fill count
(that is all an mbarrier wait can tell).  The simulation below models those
barriers exactly and runs random schedules; every consumer must read the unit
it expects.  It is driven by the pipeline shapes the library itself reports
(bil_stream_shape), and it must catch the unsound shape it was written to
rule out (a stage count that is not a multiple of the consumer count).
"""
import random

import pytest

from invariant_token_log_gb300 import _lib
from invariant_token_log_gb300 import build as lib_build


def simulate(stages, consumers, units, seed):
    """None if every consumer read the unit it expected, else a description."""
    S, W = stages, consumers
    rnd = random.Random(seed)
    full_phase = [0] * S          # completed phases (fills) per stage
    empty_phase = [0] * S         # completed phases (releases) per stage
    landed = {}                   # stage -> unit whose copy completed last
    inflight = []                 # issued copies not yet complete
    k = 0
    total = units + W             # W end markers follow the real units
    cons = [{"k": c, "stage": c, "phase": 0, "done": False} for c in range(W)]
    for _ in range(10 ** 6):
        if all(c["done"] for c in cons):
            return None
        r = rnd.random()
        if r < 0.3 and k < total:
            st, fill = k % S, k // S
            if (empty_phase[st] & 1) != ((fill & 1) ^ 1):    # producer's wait for a free stage
                if k >= units:                                # end marker: completes at once
                    full_phase[st] += 1
                    landed[st] = k
                else:
                    inflight.append((st, k))
                k += 1
        elif r < 0.6 and inflight:
            st, u = inflight.pop(rnd.randrange(len(inflight)))  # any completion order
            full_phase[st] += 1
            landed[st] = u
        else:
            c = rnd.choice([c for c in cons if not c["done"]])
            if (full_phase[c["stage"]] & 1) != c["phase"]:      # consumer's wait succeeds
                if landed.get(c["stage"]) != c["k"]:
                    return f"stage {c['stage']}: read unit {landed.get(c['stage'])}, expected {c['k']}"
                if c["k"] >= units:
                    c["done"] = True
                    continue
                empty_phase[c["stage"]] += 1
                c["k"] += W
                c["stage"] += W
                if c["stage"] >= S:
                    c["stage"] -= S
                    c["phase"] ^= 1
    return "did not finish"


def test_simulator_catches_an_unsound_shape():
    failures = [simulate(12, 7, 300, seed) for seed in range(50)]
    assert any(f is not None and f.startswith("stage") for f in failures)


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return _lib.load()


@pytest.mark.parametrize("dtype,tile_v", [(_lib.BF16, 4096), (_lib.BF16, 512), (_lib.F16, 1024),
                                          (_lib.F32, 512), (_lib.F32, 4096), (_lib.F32, 8192),
                                          (_lib.BF16, 32768), (_lib.F32, 16384), (_lib.BF16, 8)])
@pytest.mark.parametrize("fused,entropy", [(True, False), (False, False), (True, True)])
def test_library_shapes_are_sound(lib, dtype, tile_v, fused, entropy):
    num_tiles = -(-151936 // tile_v) if tile_v >= 64 else 2048
    stages, consumers, smem = _lib.stream_shape(dtype, tile_v, num_tiles, fused, entropy)
    assert 1 <= consumers <= 7 and stages >= 2 and stages % consumers == 0
    assert smem <= 227 * 1024
    for seed in range(25):
        assert simulate(stages, consumers, 4 * stages + 3, seed) is None
