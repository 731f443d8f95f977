"""The attention kernels' CTA launch order (host-side query through the C
ABI, no GPU): every (sequence·head pair, tile) item launched exactly once, and
the causal load balance of longest-processing-time-first scheduling ("LLM
Systems 22: Flash Attention", section 4.1.5).  The page's worked example
(two batches on three SMs, makespan 9 -> 7) gives no task sizes, so what is
pinned is the property it illustrates: on a greedy list scheduler (each
freed SM takes the next CTA), the kernels' order finishes no later than the
sequential order, and within a few percent of sorting every item by cost.
"""
import heapq

import numpy as np
import pytest

from io_aware_attention_flash_gb300 import _binding as b

SMS = 152
# (name, pairs, tiles per pair, resident CTAs): the launch configurations of
# the forward (256 query rows per tile at d = 128, one CTA per SM; 128 rows
# at d = 64, two per SM) and the backward (128 keys, one CTA per SM).
CONFIGS = [
    ("fwd mid  B2 H16 N4096 d128", 32, 16, SMS), ("bwd mid  B2 H16 N4096 d128", 32, 32, SMS),
    ("fwd long B1 H8 N32768 d128", 8, 128, SMS), ("bwd long B1 H8 N32768 d128", 8, 256, SMS),
    ("fwd small B4 H16 N1024 d64", 64, 8, 2 * SMS), ("bwd small B4 H16 N1024 d64", 64, 8, SMS),
    ("fwd packed 16x32 N<=4096", 512, 16, SMS), ("bwd packed 16x32 N<=4096", 512, 32, SMS),
    ("bwd B6 H16 N2048", 96, 16, SMS), ("fwd B3 H7 N640", 21, 3, SMS), ("bwd one head", 1, 5, SMS),
]


def _makespan(costs, slots, overhead=1.0):
    free = [0.0] * slots
    for c in costs:
        heapq.heappush(free, heapq.heappop(free) + c + overhead)
    return max(free)


@pytest.mark.parametrize("name,npairs,ntiles,slots", CONFIGS)
def test_every_item_launched_once(name, npairs, ntiles, slots):
    group, pair, tile = b.fa_cta_order(npairs, ntiles, slots)
    assert npairs % group == 0
    assert group == npairs or group * ntiles >= slots
    assert len(pair) == npairs * ntiles
    seen = np.zeros((npairs, ntiles), dtype=np.int64)
    np.add.at(seen, (pair, tile), 1)
    assert (seen == 1).all()
    # within a group, tiles in heaviest-first order (tile 0 first) and pairs in order
    first = pair[:group * ntiles].reshape(ntiles, group)
    assert (first == np.arange(group)[None, :]).all()
    assert (tile[:group * ntiles].reshape(ntiles, group) == np.arange(ntiles)[:, None]).all()


@pytest.mark.parametrize("name,npairs,ntiles,slots", CONFIGS)
def test_causal_balance_of_the_launch_order(name, npairs, ntiles, slots):
    """Causal cost of tile t in the kernels' index (heaviest first): ntiles - t
    (query-tile groups from the last in the forward, key tiles from the first
    in the backward), plus a fixed per-CTA cost."""
    _, pair, tile = b.fa_cta_order(npairs, ntiles, slots)
    cost = lambda t: float(ntiles - t)  # noqa: E731
    ours = _makespan([cost(t) for t in tile], slots)
    # sequential: pair by pair, tiles from the lightest (a plain loop over the
    # causal triangle)
    sequential = _makespan([cost(t) for p in range(npairs) for t in reversed(range(ntiles))], slots)
    lpt = _makespan(sorted((cost(t) for t in tile), reverse=True), slots)
    assert ours <= sequential
    assert ours <= 1.05 * lpt + 1.0


def test_order_query_rejects_bad_sizes():
    for args in ((0, 4, 152), (4, 0, 152), (4, 4, 0), (1 << 20, 1 << 12, 152)):
        with pytest.raises(b.FaError):
            b.fa_cta_order(*args)
