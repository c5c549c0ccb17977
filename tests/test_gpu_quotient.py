"""The encoders' quotient step against the correctly rounded division.

The min-max rule codes rint(RN(RN(y - z) / s)) ("Beyond Compression Ratio" §4.1;
"KVServe" §5.1).  The key and value encoders form the quotient as q = RN(t RN(1/s))
corrected once by the exact residual (Markstein's correction step) instead of
dividing; this checks, through the C ABI, every positive finite binary16 divisor
against dividends packed around the code decision points (k s and (k + 1/2) s),
uniform ones and arbitrary normal ones, comparing with CUDA's __fdiv_rn.
"""
import pytest

pytestmark = pytest.mark.gpu


def test_corrected_quotient_equals_division_for_every_binary16_divisor():
    from kv_cache_compression_encode_gb300 import kvc

    bad_q, bad_code, tested = kvc.kvc_debug_quotient_check(seed=0x5EED, rounds=2)
    per_round = 0x7BFF * 256 * 256
    assert tested > 0.9 * 2 * per_round  # a few near-zero dividends step below 0 and are skipped
    assert bad_q == 0, f"{bad_q} quotients differ from the correctly rounded division"
    assert bad_code == 0, f"{bad_code} codes differ from rint of the correctly rounded quotient"
