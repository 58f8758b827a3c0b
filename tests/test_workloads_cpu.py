"""The seeded workload generator reproduces its documented packings: the
document lengths drawn for the 128K and 512K packs (seeds 1003 and 1005), the
fixed packings of the other three workloads, totals equal to T, and the
recipe's ranges (log-uniform in [512, 32768] for the 128K pack; for the 512K
pack, each length from [1024, 8192] or [32768, 131072]; in both, the last
document is cut to the remainder)."""
import numpy as np

from sequence_blockwise_gb300 import workloads as wl

DOCUMENTED = {
    "fp32-tiny-T256-2docs-ring-P4": [100, 156],
    "llama-gqa32x8-d128-T32K-causal-zigzag-P8": [32768],
    "hybrid-pack-T128K-loguniform-gqa32x8-tasp-P8": [1118, 1489, 4006, 7994, 11687, 10359, 2109, 6145, 28994,
                                                     9676, 1263, 919, 9696, 18527, 2587, 825, 4749, 4602, 4327],
    "noncausal-T64K-mha16-ring-P16": [65536],
    "ultralong-pack-T512K-mixture-gqa64x8-tasp-P32": [7892, 7695, 116876, 114832, 6580, 81606, 3345, 7795,
                                                      126534, 4581, 45918, 634],
}


def test_documented_packings():
    assert sorted(w.name for w in wl.WORKLOADS) == sorted(DOCUMENTED)
    for w in wl.WORKLOADS:
        lens = wl.doc_lengths(w)
        assert lens == DOCUMENTED[w.name], w.name
        assert sum(lens) == w.T
        cu = wl.cu_seqlens(w)
        assert cu[0] == 0 and cu[-1] == w.T and np.all(np.diff(cu) > 0)


def test_recipe_ranges():
    pack128 = wl.doc_lengths(wl.BY_NAME["hybrid-pack-T128K-loguniform-gqa32x8-tasp-P8"])
    assert all(512 <= x <= 32768 for x in pack128[:-1])
    pack512 = wl.doc_lengths(wl.BY_NAME["ultralong-pack-T512K-mixture-gqa64x8-tasp-P32"])
    assert all(1024 <= x <= 8192 or 32768 <= x <= 131072 for x in pack512[:-1])
    assert pack512[-1] < 1024  # the remainder (documented: 634)
