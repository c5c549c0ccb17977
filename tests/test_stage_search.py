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
