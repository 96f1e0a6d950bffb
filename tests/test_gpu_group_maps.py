"""Per-group tensor maps of the K-grouped weight-gradient GEMMs: copies of a
host-encoded map written on the device with each group's row extent (the group's
end) must equal, byte for byte, the driver's own encoding of that extent.  The
self test runs no copy through the maps."""
import numpy as np
import pytest

import situ_glu_activation_gb300 as situ
from situ_glu_activation_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("offsets,rows,cols", [
    ([0, 1, 63, 64, 65, 65, 200, 333], 333, 2048),   # ragged ends, an empty group
    ([0, 333], 333, 3072),                            # one group ending at the last row
    ([0, 0, 0, 5], 64, 256),                          # leading empty groups
])
def test_group_maps_match_driver_encoding(cuda_dev, offsets, rows, cols):
    bad = situ.selftest_group_maps(offsets, rows, cols)
    ends = np.asarray(offsets[1:])
    assert not bad.any(), f"maps differing for group ends {ends[bad.any(axis=1)].tolist()}: {bad.tolist()}"


def test_group_maps_small_and_large_extents(cuda_dev):
    """Every group end from 1 to 130 (one-row groups; an end before row 32 moves the
    map's base), and ends around powers of two up to 2^24 + 1."""
    bad = situ.selftest_group_maps(list(range(131)), 130, 2048)
    assert not bad.any(), f"group ends {np.nonzero(bad.any(axis=1))[0] + 1}"
    ends = [65535, 65536, 65537, 131071, 131072, 262143, 262144, 1 << 20, (1 << 24) + 1]
    bad = situ.selftest_group_maps([0] + ends, ends[-1], 2048)
    assert not bad.any(), f"group ends {np.asarray(ends)[bad.any(axis=1)].tolist()}"


def test_group_maps_zipf_routes(cuda_dev):
    """The 64-expert Zipf routes' expert offsets, at the grouped backward's operand
    widths (dW_gate_up reads d(g, u) [R, 2I], dW_down reads dy [R, M])."""
    w = wl.WORKLOADS["grouped"]
    ids = wl.routes(w, seed=0).numpy().reshape(-1)
    counts = np.bincount(ids, minlength=w.num_experts)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(off[-1])
    for cols in (w.M, 2 * w.I):
        bad = situ.selftest_group_maps(off, R, cols)
        assert not bad.any(), f"group ends {off[1:][bad.any(axis=1)].tolist()}"


def test_group_maps_many_groups(cuda_dev):
    g = np.random.default_rng(3)
    counts = g.integers(0, 700, size=898)
    counts[g.integers(0, 898, size=40)] = 0
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    bad = situ.selftest_group_maps(off, int(off[-1]), 2048)
    assert not bad.any(), f"group ends {off[1:][bad.any(axis=1)].tolist()[:20]}"
