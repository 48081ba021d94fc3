"""Host-side arithmetic of bench.py that sets reported rates: the count of visible
(query, key) pairs under a window and a key count, which the score-modification,
padded and split-KV sweep lines divide by their times."""
import itertools

import bench
import synth


def _brute(Sq, Sk, wl, wr):
    n = 0
    for i, j in itertools.product(range(Sq), range(Sk)):
        if (wl < 0 or j >= i - wl) and (wr < 0 or j <= i + wr):
            n += 1
    return n


def test_visible_pairs_brute_force():
    for Sq, Sk in ((1, 1), (7, 5), (5, 9), (33, 33), (40, 17)):
        for wl in (-1, 0, 1, 6, 50):
            for wr in (-1, 0, 2, 7, 60):
                assert bench.visible_pairs(Sq, Sk, wl, wr) == _brute(Sq, Sk, wl, wr), (Sq, Sk, wl, wr)


def test_visible_pairs_special_cases():
    # no window: every pair; causal (-1, 0) with Sq = Sk: the lower triangle;
    # a key count of 0 leaves no pair; a count is a cut of the key axis
    assert bench.visible_pairs(100, 70, -1, -1) == 100 * 70
    assert bench.visible_pairs(64, 64, -1, 0) == 64 * 65 // 2
    assert bench.visible_pairs(10, 0, -1, -1) == 0
    assert bench.visible_pairs(10, 0, -1, 0) == 0
    # causal over a batch padded to 3/4 of S: the rows below the count see
    # their triangle, the rest see all the count's keys
    S, L = 128, 96
    assert bench.visible_pairs(S, L, -1, 0) == L * (L + 1) // 2 + (S - L) * L


def test_flop_convention_matches_pairs():
    """The workload FLOP count (4 D per visible pair forward, x2.5 backward,
    causal counted as exactly half) against the pair count."""
    B, H, S, D = 2, 3, 256, 64
    full = 4.0 * B * H * D * bench.visible_pairs(S, S, -1, -1)
    assert synth.flop_count(B, H, S, S, D, causal=False) == full
    assert synth.flop_count(B, H, S, S, D, causal=True) == full / 2
    assert synth.flop_count(B, H, S, S, D, causal=False, backward=True) == 2.5 * full
