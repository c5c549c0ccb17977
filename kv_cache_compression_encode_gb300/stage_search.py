"""Stage-list search over a quantized payload: size, encode time and decode time of
every lossless pipeline in a candidate set, and the Pareto-optimal ones.

"Beyond Compression Ratio: High-Throughput KV Compression for Disaggregated LLM
Serving", §4.2: the LC backend's pipeline (TUPL8_1 -> BIT_8 -> RZE_2) was chosen
by searching stage combinations offline for compression ratio against throughput
on quantized KV.  This runs that search with this library's own stages (format
v1: TUPL_k, BIT_8, DELTA_w, RZE_w, RZE last) on a payload that is already in
device memory.  Orchestration only: every encode and decode is a call into
libkvc.so, timed with CUDA events on the current stream, and every candidate's
round trip is checked byte for byte.

Some stage lists have fast kernels (the worker/publisher encoder and the fast
chunk decoder: TUPL_8 [BIT_8] [DELTA_1] RZE_1/2 at 4-16 KiB chunks), the rest run
the generic stage kernels.  So that the front compares pipelines and not which
ones have a fast kernel, every candidate is also timed with the generic kernels
forced (kvc_debug_generic_stages; same stream bytes) and a second front is taken
over those times; each candidate names the kernels its default times came from.
"""
from __future__ import annotations

import itertools
from dataclasses import dataclass

import torch

from . import kvc
from .codec import Codec

TUPL, BIT, DELTA, RZE = kvc.ST_TUPL, kvc.ST_BIT, kvc.ST_DELTA, kvc.ST_RZE


def candidate_stage_lists():
    """Pipelines in the pages' stage order: [TUPL_k] [BIT_8] [DELTA_w] RZE_w, with
    k in {2, 4, 8} and w in {1, 2, 4}; RZE is the only stage that shrinks a chunk,
    so every candidate ends with it (96 lists)."""
    out = []
    for tupl, bit, delta, rze in itertools.product((None, 2, 4, 8), (False, True), (None, 1, 2, 4), (1, 2, 4)):
        st = []
        if tupl:
            st.append((TUPL, tupl))
        if bit:
            st.append((BIT, 8))
        if delta:
            st.append((DELTA, delta))
        st.append((RZE, rze))
        out.append(tuple(st))
    return out


@dataclass
class Candidate:
    stages: tuple
    stream_bytes: int
    ratio: float          # payload bytes / stream bytes
    enc_ms: float         # with the library's default kernels for this list
    dec_ms: float
    pareto: bool = False
    enc_kernel: str = ""  # launch names the default times came from
    dec_kernel: str = ""
    enc_ms_generic: float = 0.0  # with the generic stage kernels forced
    dec_ms_generic: float = 0.0
    pareto_generic: bool = False


def pareto_front(cands: list[Candidate], generic: bool = False) -> list[Candidate]:
    """Marks the candidates no other candidate beats on size, encode time and decode
    time at once (at least as good on all three, better on one); with generic=True
    on the times taken with the generic kernels forced (field pareto_generic)."""
    def key(c: Candidate):
        return (c.stream_bytes, c.enc_ms_generic, c.dec_ms_generic) if generic else \
               (c.stream_bytes, c.enc_ms, c.dec_ms)

    def dominates(a: Candidate, b: Candidate) -> bool:
        ka, kb = key(a), key(b)
        return all(x <= y for x, y in zip(ka, kb)) and any(x < y for x, y in zip(ka, kb))

    for c in cands:
        flag = not any(dominates(o, c) for o in cands if o is not c)
        if generic:
            c.pareto_generic = flag
        else:
            c.pareto = flag
    return [c for c in cands if (c.pareto_generic if generic else c.pareto)]


def search(payload: torch.Tensor, profile_kwargs: dict, shape: kvc.Shape, stage_lists=None, reps: int = 5,
           device="cuda") -> list[Candidate]:
    """Encodes and decodes `payload` (the quantized payload of `profile_kwargs` and
    `shape`, on the device) with each stage list; returns every candidate with the
    Pareto ones marked.  Raises if a round trip does not reproduce the payload."""
    stage_lists = candidate_stage_lists() if stage_lists is None else stage_lists
    cands = []
    for stages in stage_lists:
        codec = Codec(kvc.make_profile(**{**profile_kwargs, "stages": stages}), shape, device)
        n = codec.plan.payload_bytes
        if payload.numel() < n:
            raise ValueError("payload smaller than the plan's payload")
        s = codec.new_stream_buffer()
        back = codec.new_payload_buffer()
        codec.lossless_encode(payload, out=s)
        st, nbytes, flags = codec.query()
        if st != kvc.KVC_OK:
            raise RuntimeError(f"{stages}: encode failed ({kvc.status_str(st)}, flags {flags})")
        codec.lossless_decode(s, nbytes, out=back)
        st, _, flags = codec.query()
        if st != kvc.KVC_OK or not torch.equal(back[:n], payload[:n]):
            raise RuntimeError(f"{stages}: round trip failed ({kvc.status_str(st)}, flags {flags})")
        cs = torch.cuda.current_stream(codec.device)

        def timed(generic: bool):
            kvc.kvc_debug_generic_stages(codec.plan, generic)
            kvc.kvc_timing_enable(codec.plan, True, capacity=8)
            codec.lossless_encode(payload, out=s)
            codec.lossless_decode(s, nbytes, out=back)
            names = [nm for nm, _ in kvc.kvc_timing_read(codec.plan, 8)]
            kvc.kvc_timing_enable(codec.plan, False)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            ev[0].record(cs)
            for _ in range(reps):
                codec.lossless_encode(payload, out=s)
            ev[1].record(cs)
            for _ in range(reps):
                codec.lossless_decode(s, nbytes, out=back)
            ev[2].record(cs)
            ev[2].synchronize()
            if not torch.equal(back[:n], payload[:n]):
                raise RuntimeError(f"{stages}: round trip failed (generic kernels {generic})")
            enc = [nm for nm in names if nm.startswith("kvc_lossless_enc")]
            dec = [nm for nm in names if nm.startswith("kvc_lossless_dec")]
            return (ev[0].elapsed_time(ev[1]) / reps, ev[1].elapsed_time(ev[2]) / reps,
                    enc[0] if enc else "", dec[0] if dec else "")

        e, d, ek, dk = timed(False)
        eg, dg, _, _ = timed(True)
        kvc.kvc_debug_generic_stages(codec.plan, False)
        cands.append(Candidate(stages, nbytes, n / nbytes, e, d, enc_kernel=ek, dec_kernel=dk, enc_ms_generic=eg,
                               dec_ms_generic=dg))
        del codec, s, back
    pareto_front(cands)
    pareto_front(cands, generic=True)
    return cands


def main(argv=None):
    """python -m kv_cache_compression_encode_gb300.stage_search [--workload llama8b]:
    quantizes the workload's synthetic KV with its profile, searches every
    candidate pipeline on that payload and prints the Pareto-optimal ones (one JSON
    line each, smallest stream first) and a summary line."""
    import argparse
    import json

    from . import synth
    from .workloads import PROFILES, WORKLOADS

    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="llama8b")
    ap.add_argument("--reps", type=int, default=5)
    args = ap.parse_args(argv)
    w = WORKLOADS[args.workload]
    prof = dict(PROFILES[args.workload])
    current = tuple(tuple(s) for s in prof.pop("stages", ()))
    layers = [synth.layer_kv(w.dist, l, w.tokens, w.kv_heads, w.head_dim, w.dtype, w.seed, "cuda")
              for l in range(w.layers)]
    k = [a.contiguous() for a, _ in layers]
    v = [b.contiguous() for _, b in layers]
    shape = kvc.make_shape(w.layers, w.tokens, w.kv_heads, w.head_dim, kvc.BF16 if w.dtype == "bf16" else kvc.F16)
    q = Codec(kvc.make_profile(**prof), shape)
    payload = q.quantize(k, v)
    st, _, flags = q.query()
    if st != kvc.KVC_OK:
        raise RuntimeError(f"quantize failed ({kvc.status_str(st)}, flags {flags})")
    cands = sorted(search(payload, prof, shape, reps=args.reps), key=lambda c: c.stream_bytes)
    for c in cands:
        if c.pareto or c.pareto_generic:
            print(json.dumps({"stages": c.stages, "ratio": round(c.ratio, 4), "enc_ms": round(c.enc_ms, 4),
                              "dec_ms": round(c.dec_ms, 4), "kernels": [c.enc_kernel, c.dec_kernel],
                              "enc_ms_generic": round(c.enc_ms_generic, 4), "dec_ms_generic": round(c.dec_ms_generic, 4),
                              "front": "both" if c.pareto and c.pareto_generic else
                                       ("default kernels" if c.pareto else "generic kernels")}))
    cur = [c for c in cands if c.stages == current]
    print(json.dumps({"workload": w.name, "payload_bytes": q.plan.payload_bytes, "candidates": len(cands),
                      "pareto": sum(c.pareto for c in cands), "pareto_generic": sum(c.pareto_generic for c in cands),
                      "profile_pipeline": {"stages": current, "ratio": round(cur[0].ratio, 4),
                                           "enc_ms": round(cur[0].enc_ms, 4), "dec_ms": round(cur[0].dec_ms, 4),
                                           "pareto": cur[0].pareto, "pareto_generic": cur[0].pareto_generic}
                      if cur else None}))


if __name__ == "__main__":
    main()
