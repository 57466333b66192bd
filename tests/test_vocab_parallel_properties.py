"""Properties of the vocabulary-parallel host logic ("Tensor Parallel", steps
3-5: every rank's block goes to its own tile columns, the target logit comes
from the rank that owns the target's tile), over random partitions of the
tiles into contiguous ranges owned by ranks in any order."""
import pytest
import torch

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

from invariant_token_log_gb300 import vocab_parallel as vp  # noqa: E402


@st.composite
def partitions(draw):
    """(num_tiles, ranges in rank order): contiguous ranges covering [0, T) once."""
    t = draw(st.integers(min_value=1, max_value=40))
    k = draw(st.integers(min_value=1, max_value=min(t, 6)))
    cuts = sorted(draw(st.sets(st.integers(min_value=1, max_value=t - 1), min_size=k - 1, max_size=k - 1))) \
        if k > 1 else []
    bounds = [0] + cuts + [t]
    ranges = [(bounds[i], bounds[i + 1]) for i in range(k)]
    order = draw(st.permutations(list(range(k))))
    return t, [ranges[i] for i in order]


def _blocks(ranges, n):
    """Each rank's block: value 1000 * row + global tile, padded to the longest range."""
    pad = max(e - b for b, e in ranges)
    return [torch.tensor([[1000.0 * r + t for t in range(b, e)] + [-1.0] * (pad - (e - b)) for r in range(n)])
            for b, e in ranges]


@settings(max_examples=150, deadline=None)
@given(partitions(), st.integers(min_value=1, max_value=5))
def test_assembly_places_every_block_at_its_tiles(part, n):
    t, ranges = part
    full = vp.assemble(_blocks(ranges, n), ranges, t)
    assert full.tolist() == [[1000.0 * r + c for c in range(t)] for r in range(n)]


@settings(max_examples=150, deadline=None)
@given(partitions(), st.integers(min_value=1, max_value=16), st.data())
def test_target_logit_comes_from_its_owner(part, tile_v, data):
    t, ranges = part
    n = 12
    targets = torch.tensor(data.draw(st.lists(st.integers(min_value=-3, max_value=t * tile_v + 2), min_size=n,
                                              max_size=n)))
    targets[0] = -100  # an ignored row
    per_rank = [torch.full((n,), float(rank)) for rank in range(len(ranges))]
    owner = vp.owner_target_logit(per_rank, ranges, targets, tile_v)
    for i, tg in enumerate(targets.tolist()):
        if tg == -100 or tg < 0 or tg >= t * tile_v:
            assert owner[i] != owner[i]  # no owner: NaN
        else:
            rank = next(k for k, (b, e) in enumerate(ranges) if b <= tg // tile_v < e)
            assert owner[i] == float(rank)


@settings(max_examples=100, deadline=None)
@given(partitions(), st.data())
def test_a_gap_or_an_overlap_is_rejected(part, data):
    t, ranges = part
    k = data.draw(st.integers(min_value=0, max_value=len(ranges) - 1))
    b, e = ranges[k]
    broken = list(ranges)
    if data.draw(st.booleans()) and e - b > 1:
        broken[k] = (b, e - 1)  # a gap
    else:
        broken[k] = (max(0, b - 1), e) if b > 0 else (b, min(t, e + 1))  # an overlap
        if broken[k] == ranges[k]:
            broken.append((0, 1))  # a single tile: overlap it again
    if broken == ranges:
        return
    with pytest.raises(ValueError):
        vp.assemble(_blocks(broken, 2), broken, t)
