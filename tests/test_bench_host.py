"""Host-side logic of bench.py that needs no GPU: the prefill segmentation of the
end-to-end step.  The segments must cover the sequence exactly and, where there
is more than one, be multiples of the 64-token chunk, so that resumed calls see
the chunk grid of one call (the GPU test test_prefill_in_segments_is_bit_identical
checks that such calls give one call's results bit for bit)."""
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    return bench


@pytest.mark.parametrize("T", [8192, 65536, 6144, 4096, 3136, 2048, 1536, 1088, 1024, 1000, 960, 64, 1])
def test_e2e_segments_cover_the_sequence_on_the_chunk_grid(T):
    segs = _bench().Workload.e2e_segments(T)
    assert sum(segs) == T and all(L > 0 for L in segs)
    if len(segs) > 1:
        assert all(L % 64 == 0 for L in segs)
        assert segs[-1] <= min(segs[:-1])   # the tail is short: little left once the last inputs land


def test_e2e_segments_of_the_workload():
    assert _bench().Workload.e2e_segments(8192) == (2048, 2048, 2048, 1024, 768, 256)
