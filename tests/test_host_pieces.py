"""Host logic of the end-to-end path (CPU): the pieces a host call is cut
into cover every (batch, head) exactly once, keep each kv head's query heads
together, are contiguous slices of the head-major arrays, and number at most
64."""
import pytest

from tiled_online_softmax_02_gb300 import _binding


@pytest.mark.parametrize("B,Hq,Hkv,layout", [(2, 32, 8, 0), (1, 24, 24, 1), (8, 32, 4, 0), (3, 6, 3, 0),
                                             (4, 16, 8, 1), (1, 4, 1, 0), (7, 8, 8, 0), (70, 4, 2, 0),
                                             (200, 8, 8, 1), (64, 2, 1, 0)])
def test_pieces_cover_the_problem(B, Hq, Hkv, layout):
    pieces = _binding._host_pieces(B, Hq, Hkv, layout)
    assert 1 <= len(pieces) <= 64
    covered = sorted((b, h) for b0, b1, h0, h1, _, _ in pieces for b in range(b0, b1) for h in range(h0, h1))
    assert covered == [(b, h) for b in range(B) for h in range(Hq)]
    g = Hq // Hkv
    for b0, b1, h0, h1, kv0, kv1 in pieces:
        assert h0 == kv0 * g and h1 == kv1 * g
        # a run of several batches takes every head, so its slices are contiguous
        assert b1 - b0 == 1 or (h0, h1) == (0, Hq)
        if layout == 1:  # token-major output rows hold every head of a token
            assert (h0, h1) == (0, Hq)
    if layout == 0 and B < 8:
        assert len(pieces) >= min(8, B * Hkv)
