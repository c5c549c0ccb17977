"""Stage-list search (the pages' offline pipeline search, "Beyond Compression
Ratio" §4.2): candidate rules and the Pareto marking on the CPU; the search itself
through the library on the GPU."""
import numpy as np
import pytest
import torch

from kv_cache_compression_encode_gb300 import kvc, synth
from kv_cache_compression_encode_gb300.codec import Codec
from kv_cache_compression_encode_gb300.stage_search import (BIT, DELTA, RZE, TUPL, Candidate, candidate_stage_lists,
                                                            pareto_front, search)


def test_candidates_follow_the_format_rules():
    c = candidate_stage_lists()
    assert len(c) == 96 and len(set(c)) == 96
    order = {TUPL: 0, BIT: 1, DELTA: 2, RZE: 3}
    for st in c:
        assert st[-1][0] == RZE and st[-1][1] in (1, 2, 4)
        assert [order[k] for k, _ in st] == sorted(order[k] for k, _ in st)  # pages' stage order
        for k, p in st:
            assert (k, p) in {(TUPL, 2), (TUPL, 4), (TUPL, 8), (BIT, 8), (DELTA, 1), (DELTA, 2), (DELTA, 4),
                              (RZE, 1), (RZE, 2), (RZE, 4)}
    assert ((TUPL, 8), (BIT, 8), (RZE, 2)) in c  # the pages' chosen pipeline is a candidate


def test_pareto_marks_exactly_the_undominated():
    a = Candidate((), 100, 0, 1.0, 1.0)   # smallest
    b = Candidate((), 120, 0, 0.5, 1.0)   # fastest encode
    c = Candidate((), 130, 0, 0.6, 1.2)   # worse than b everywhere
    d = Candidate((), 100, 0, 1.0, 1.0)   # ties with a: neither dominates
    e = Candidate((), 90, 0, 2.0, 0.4)    # smallest and fastest decode
    front = pareto_front([a, b, c, d, e])
    assert [x.pareto for x in (a, b, c, d, e)] == [True, True, False, True, True]
    assert len(front) == 4


@pytest.mark.gpu
def test_search_on_a_quantized_payload():
    prof = dict(smooth_keys=True, hadamard=True, bits_k=4, bits_v=4, group_k=128, group_v=128, chunk_bytes=4096)
    L, T, H = 2, 512, 4
    kv = [synth.layer_kv("llama", l, T, H, 128, "bf16", 21, "cuda") for l in range(L)]
    k = [a.contiguous() for a, _ in kv]
    v = [b.contiguous() for _, b in kv]
    shape = kvc.make_shape(L, T, H, 128, kvc.BF16)
    q = Codec(kvc.make_profile(**prof), shape)
    payload = q.quantize(k, v)
    assert q.query()[0] == kvc.KVC_OK
    lists = candidate_stage_lists()[::8] + [((TUPL, 8), (BIT, 8), (RZE, 2))]
    cands = search(payload, prof, shape, lists, reps=2)
    assert len(cands) == len(lists)
    n = q.plan.payload_bytes
    for c in cands:
        assert c.ratio == pytest.approx(n / c.stream_bytes)
        assert c.enc_ms > 0 and c.dec_ms > 0
        # the stream size is what a plain encode of the same pipeline reports
        codec = Codec(kvc.make_profile(**{**prof, "stages": c.stages}), shape)
        codec.lossless_encode(payload)
        assert codec.query()[1] == c.stream_bytes
    front = [c for c in cands if c.pareto]
    assert front and min(c.stream_bytes for c in cands) == min(c.stream_bytes for c in front)
    assert any(c.pareto_generic for c in cands)
    # kernels named per candidate: the pages' pipeline at 4 KiB chunks has the fast pair, RZE_4 lists do not
    lc = [c for c in cands if c.stages == ((TUPL, 8), (BIT, 8), (RZE, 2))][0]
    assert (lc.enc_kernel, lc.dec_kernel) == ("kvc_lossless_enc_fast", "kvc_lossless_dec_fast")
    assert lc.enc_ms_generic > 0 and lc.dec_ms_generic > 0
    for c in cands:
        if c.stages[-1] == (RZE, 4):
            assert (c.enc_kernel, c.dec_kernel) == ("kvc_lossless_enc", "kvc_lossless_dec")
    # every candidate's stream equals the oracle's lossless encode of the same payload
    from oracle import oracle as O
    Qh = payload[:n].cpu().numpy()
    ok_shape = O.make_shape(L, T, H, 128, 2)
    for c in cands:
        so = O.lossless_encode(O.make_profile(**{**prof, "stages": c.stages}), ok_shape, Qh)
        codec = Codec(kvc.make_profile(**{**prof, "stages": c.stages}), shape)
        kvc.kvc_debug_generic_stages(codec.plan, True)
        sg = codec.lossless_encode(payload)
        st, nb, _ = codec.query()
        assert st == kvc.KVC_OK and nb == so.size and np.array_equal(sg[:nb].cpu().numpy(), so), c.stages
