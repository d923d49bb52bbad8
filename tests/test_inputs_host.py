"""Host logic of the seeded input generators (no GPU): the packed-sequence length draw that the
benchmark's packed leg and its full-size parity test share, and the packed segment positions."""
import numpy as np

from linear_recurrent_rnn_gb300.inputs import packed_lengths, segment_positions


def test_packed_lengths_fill_the_row():
    for seed, T, lo, hi in ((5, 8192, 1, 2048), (1, 100, 1, 7), (2, 4096, 256, 4096), (3, 1, 1, 2048)):
        lengths = packed_lengths(seed, T, lo, hi)
        assert sum(lengths) == T
        assert all(lo <= n <= hi for n in lengths[:-1])
        assert 1 <= lengths[-1] <= hi
        assert packed_lengths(seed, T, lo, hi) == lengths  # seeded: the same draw again


def test_packed_lengths_of_the_benchmark():
    """The packed leg's eight sequences (B1 T8192, lengths U[1, 2048], seed 5): the parity test
    and the bench read the same draw."""
    lengths = packed_lengths(5, 8192, 1, 2048)
    assert len(lengths) == 8
    assert min(lengths) < 64  # a sequence shorter than one 64-token chunk


def test_segment_positions_restart_at_each_segment():
    rng = np.random.default_rng(0)
    pos = segment_positions(rng, 300, 1, 40, continuation=False)
    assert pos[0] == 0
    steps = np.diff(pos)
    assert np.all((steps == 1) | (pos[1:] == 0))  # +1 inside a segment, 0 at a new one
    rng = np.random.default_rng(0)
    cont = segment_positions(rng, 300, 1, 40, continuation=True)
    assert cont[0] >= 1  # the first segment continues an earlier one
