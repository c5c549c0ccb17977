"""The allocation-free lossless encode (kvc_lossless_encode_noalloc) against the
workspace-based kvc_lossless_encode, through the C ABI.

Callers that cannot allocate device memory (for example a transport plugin that
only receives the payload and output buffers) use the variant whose scratch is a
device array inside the library.  Two calls in a row, with different payloads,
must each produce exactly the stream of the existing entry point: the second
call also shows that what the first call left in the shared array does not leak
into the next stream."""
import numpy as np
import pytest
import torch

from kv_cache_compression_encode_gb300 import kvc
from kv_cache_compression_encode_gb300.codec import Codec

pytestmark = pytest.mark.gpu


def _payload(n, seed):
    rng = np.random.default_rng(seed)
    out = rng.integers(0, 256, n, dtype=np.uint8)
    blk = 5000
    for s in range(0, n, 2 * blk):  # compressible and incompressible regions
        out[s:s + blk] = np.where(rng.random(min(blk, n - s)) < 0.05, 3, 0)
    return out


def test_noalloc_matches_workspace_encode_twice():
    prof = kvc.make_profile(smooth_keys=True, hadamard=True, bits_k=4, bits_v=4, group_k=128, group_v=128,
                            stages=((1, 8), (2, 8), (3, 1), (4, 2)), chunk_bytes=16384)
    codec = Codec(prof, kvc.make_shape(4, 1000, 8, 128, kvc.BF16))
    plan = codec.plan
    n = plan.payload_bytes
    out = torch.empty(plan.max_stream_bytes, dtype=torch.uint8, device="cuda")
    d_size = torch.zeros(1, dtype=torch.int64, device="cuda")
    d_status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for call, seed in enumerate((11, 12)):
        Q = torch.from_numpy(_payload(n, seed)).cuda()
        ref = codec.lossless_encode(Q)
        st, ref_bytes, flags = codec.query()
        assert st == kvc.KVC_OK and flags == 0
        out.fill_(0xA5)
        kvc.kvc_lossless_encode_noalloc(plan, Q.data_ptr(), out.data_ptr(), out.numel(), d_size.data_ptr(),
                                        d_status.data_ptr(), stream)
        torch.cuda.synchronize()
        nbytes = int(d_size.item())
        assert int(d_status.item()) == 0, call
        assert nbytes == ref_bytes, (call, nbytes, ref_bytes)
        assert torch.equal(out[:nbytes], ref[:ref_bytes]), call
        # the stream decodes back to the payload
        back = codec.lossless_decode(out, nbytes)
        st, _, flags = codec.query()
        assert st == kvc.KVC_OK and flags == 0
        assert torch.equal(back[:n], Q), call


def test_noalloc_without_stages_and_without_status_word():
    """No lossless stages: the stream is the header plus the payload, its size set
    by the prologue; d_status may be NULL."""
    prof = kvc.make_profile(bits_k=4, bits_v=4, group_k=64, group_v=64, stages=())
    codec = Codec(prof, kvc.make_shape(2, 300, 4, 128, kvc.BF16))
    plan = codec.plan
    n = plan.payload_bytes
    Q = torch.from_numpy(_payload(n, 21)).cuda()
    ref = codec.lossless_encode(Q)
    st, ref_bytes, flags = codec.query()
    assert st == kvc.KVC_OK and flags == 0 and ref_bytes == 64 + n
    out = torch.full((plan.max_stream_bytes,), 0xA5, dtype=torch.uint8, device="cuda")
    d_size = torch.zeros(1, dtype=torch.int64, device="cuda")
    kvc.kvc_lossless_encode_noalloc(plan, Q.data_ptr(), out.data_ptr(), out.numel(), d_size.data_ptr(), 0,
                                    torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert int(d_size.item()) == ref_bytes
    assert torch.equal(out[:ref_bytes], ref[:ref_bytes])


def test_noalloc_reports_a_device_timeout_then_recovers():
    """A device-side error reaches d_status through the shared array: the test hook
    makes one chunk skip its publication, so its successor's bounded wait runs out
    (TIMEOUT).  The next call resets the array's words and is clean again."""
    prof = kvc.make_profile(bits_k=4, bits_v=4, group_k=64, group_v=64, stages=((1, 8), (2, 8), (4, 2)),
                            chunk_bytes=4096)
    codec = Codec(prof, kvc.make_shape(1, 512, 2, 128, kvc.BF16))
    plan = codec.plan
    n = plan.payload_bytes
    Q = torch.from_numpy(_payload(n, 31)).cuda()
    out = torch.empty(plan.max_stream_bytes, dtype=torch.uint8, device="cuda")
    d_size = torch.zeros(1, dtype=torch.int64, device="cuda")
    d_status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    kvc.kvc_debug_lookback(plan, 3, 2000)
    kvc.kvc_lossless_encode_noalloc(plan, Q.data_ptr(), out.data_ptr(), out.numel(), d_size.data_ptr(),
                                    d_status.data_ptr(), stream)
    torch.cuda.synchronize()
    assert int(d_status.item()) & kvc.FLAG_TIMEOUT
    kvc.kvc_debug_lookback(plan, -1, 0)
    ref = codec.lossless_encode(Q)
    st, ref_bytes, flags = codec.query()
    assert st == kvc.KVC_OK and flags == 0
    kvc.kvc_lossless_encode_noalloc(plan, Q.data_ptr(), out.data_ptr(), out.numel(), d_size.data_ptr(),
                                    d_status.data_ptr(), stream)
    torch.cuda.synchronize()
    assert int(d_status.item()) == 0
    assert int(d_size.item()) == ref_bytes and torch.equal(out[:ref_bytes], ref[:ref_bytes])


def test_noalloc_rejects_plans_beyond_the_array():
    # 256 + 8 * chunks > 1 MiB: more than 131040 chunks of 256 bytes
    prof = kvc.make_profile(bits_k=8, bits_v=8, group_k=32, group_v=32, stages=((1, 8), (4, 1)), chunk_bytes=256)
    plan = kvc.Plan(prof, kvc.make_shape(8, 8192, 8, 128, kvc.BF16))
    assert 256 + 8 * plan.n_chunks > (1 << 20)
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_lossless_encode_noalloc(plan, 256, 512, plan.max_stream_bytes, 1024, 0, 0)
    assert e.value.status == kvc.KVC_ERR_CAPACITY
