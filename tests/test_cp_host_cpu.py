"""Host logic of the context-parallel prefill (no GPU): the segment table."""
import pytest

from kimi_delta_attention_13_gb300.context_parallel import segments


def test_segments_cover_every_token_in_order():
    lengths = [300, 0, 5, 128, 129]
    bounds, seq_seg = segments(lengths, 128)
    assert bounds[0] == (0, 128) and bounds[2] == (256, 300)
    assert seq_seg == [0, 3, 4, 5, 6, 8]
    assert bounds[3] == (300, 300)             # the empty sequence keeps one empty segment
    flat = [t for b, e in bounds for t in range(b, e)]
    assert flat == list(range(sum(lengths)))
    for n in range(len(lengths)):
        lo, hi = seq_seg[n], seq_seg[n + 1]
        assert hi - lo == max(1, -(-lengths[n] // 128))
        assert all(e - b <= 128 for b, e in bounds[lo:hi])


def test_bad_arguments():
    with pytest.raises(ValueError):
        segments([10], 0)
    with pytest.raises(ValueError):
        segments([-1], 8)


def test_auto_seg_len_is_one_wave():
    from kimi_delta_attention_13_gb300.context_parallel import auto_seg_len

    L = auto_seg_len(262144, 8, 152)
    assert L % 32 == 0
    n_seg = -(-262144 // L)
    assert n_seg == 16                            # 16 x 8 = 128 CTAs: 7/8 of 152 SMs
    assert auto_seg_len(100, 200, 152) >= 100     # more heads than SMs: no split
