"""Benefit condition (KVServe §3.1, §6.1 Eq. (5)) from measured throughputs."""
import pytest

from kv_cache_compression_encode_gb300.benefit import break_even_bandwidth, effective_throughput, segment_time


def test_effective_throughput_is_the_harmonic_combination():
    # encode + decode of V bytes take V / s_p
    enc, dec, v = 1377.0, 2110.0, 537.0
    s = effective_throughput(enc, dec)
    assert v / s == pytest.approx(v / enc + v / dec)
    assert s < min(enc, dec)
    assert effective_throughput(100.0, 100.0) == pytest.approx(50.0)


def test_break_even_bandwidth_is_where_both_segment_times_meet():
    cr, s = 3.7347, effective_throughput(1377.0, 2110.0)
    b_star = break_even_bandwidth(cr, s)
    v = 1.0
    assert segment_time(v, b_star, cr, s) == pytest.approx(segment_time(v, b_star))
    # slower links gain from compression, faster ones do not
    assert segment_time(v, 0.5 * b_star, cr, s) < segment_time(v, 0.5 * b_star)
    assert segment_time(v, 2.0 * b_star, cr, s) > segment_time(v, 2.0 * b_star)


def test_no_compression_never_pays():
    assert break_even_bandwidth(1.0, 500.0) == 0.0
    with pytest.raises(ValueError):
        effective_throughput(0.0, 1.0)
    with pytest.raises(ValueError):
        break_even_bandwidth(0.0, 1.0)
