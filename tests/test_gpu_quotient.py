"""The encoders' quotient steps against the correctly rounded division.

The min-max rule ("Beyond Compression Ratio" §4.1; "KVServe" §5.1) divides twice:
the group scale fp16_up(RN((max - z) / (2^b - 1))) and the code
rint(RN(RN(y - z) / s)).  The key and value encoders form both quotients as
RN(t RN(1/d)) corrected once by the exact residual (Markstein's correction step)
instead of dividing; this checks, through the C ABI and against CUDA's __fdiv_rn,
every positive finite binary16 divisor with dividends packed around the code
decision points (k s and (k + 1/2) s), uniform ones and arbitrary normal ones, and
every non-negative binary32 range for the four widths.
"""
import pytest

pytestmark = pytest.mark.gpu


def test_corrected_quotients_equal_division():
    from kv_cache_compression_encode_gb300 import kvc

    bad_q, bad_code, tested, bad_rq, bad_scale, patterns = kvc.kvc_debug_quotient_check(seed=0x5EED, rounds=2)
    per_round = 0x7BFF * 256 * 256
    assert tested > 0.9 * 2 * per_round  # a few near-zero dividends step below 0 and are skipped
    assert bad_q == 0, f"{bad_q} code quotients differ from the correctly rounded division"
    assert bad_code == 0, f"{bad_code} codes differ from rint of the correctly rounded quotient"
    # the group scale: every non-negative binary32 range, four widths
    assert patterns == 1 << 31
    assert bad_rq == 0, f"{bad_rq} scale quotients differ from the correctly rounded division"
    assert bad_scale == 0, f"{bad_scale} binary16 scales differ"
