"""Benchmark of the KV-cache compression path on GB300.

One step = one full pass of the path over the workload's KV: kvc_encode (fused
smoothing + Hadamard + quantize + pack, then the lossless chunk stages) followed
by kvc_decode (lossless decode, then fused reconstruction), all layers.

Metric: KV encode/decode GB/s counted on uncompressed input bytes (K+V of all
layers), the convention of "Beyond Compression Ratio: High-Throughput KV
Compression for Disaggregated LLM Serving", Table 1 (GB/s x ms = the raw bytes for
both directions).  `value` = raw bytes per step / device time per step, i.e. the
combined encode+decode throughput s_p of "KVServe" §3.1 (1/s_p = 1/s_enc + 1/s_dec);
encode and decode are also reported apart.

  python bench.py [--workload llama8b] [--steps K] [--warmup W] [--gpus N] [--impl kvc|reference]

Multi-GPU (torchrun): every rank runs its own replica of the workload (the path
has no exchange step); the job value is all ranks' bytes over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV encode/decode GB/s (input bytes) on 1 GB300 and % of HBM roofline"
FALLBACK_HBM_GBS = 6800.0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def source_sha() -> str:
    csrc = os.path.join(ROOT, "kv_cache_compression_encode_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current sources."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if kernel in PAIRS:  # a pair's traffic: its two kernels' captures together
        parts = [d.get(workload, {}).get(k) for k, pair in PAIRED.items() if pair == kernel]
        parts = [r for r in parts if r]
        if len(parts) != 2 or any(r.get("source_sha") != source_sha() for r in parts):
            return None
        return sum(r["dram_bytes_per_launch"] for r in parts)
    rec = d.get(workload, {}).get(kernel)
    if not rec or rec.get("source_sha") != source_sha():
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"kvc_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if not self.proc or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------- workload
def workload_and_profile(name: str):
    """A workload name, or a format-v2 variant of the Llama-8B workload (V2_PROFILES)."""
    from kv_cache_compression_encode_gb300.workloads import PROFILES, V2_PROFILES, WORKLOADS

    if name in V2_PROFILES:
        return WORKLOADS["llama8b"], V2_PROFILES[name]
    if name.endswith(FUSED_SUFFIX):  # the same workload, encoded with kvc_fuse_value_chunks
        base = name[: -len(FUSED_SUFFIX)]
        return WORKLOADS[base], PROFILES[base]
    return WORKLOADS[name], PROFILES[name]


def json_profile(prof: dict) -> dict:
    out = {}
    for k_, v_ in prof.items():
        if k_ == "stages":
            out[k_] = [list(x) for x in v_]
        elif k_.startswith("bits_map"):
            rows = [list(map(int, r)) for r in v_]
            # one row repeated for every layer is written once
            out[k_] = f"{len(rows)} layers x {rows[0]}" if all(r == rows[0] for r in rows) else rows
        else:
            out[k_] = v_
    return out


def workload_setup(name: str, device):
    import torch

    from kv_cache_compression_encode_gb300 import kvc, synth

    w, prof = workload_and_profile(name)
    k, v = [], []
    for l in range(w.layers):
        a, b = synth.layer_kv(w.dist, l, w.tokens, w.kv_heads, w.head_dim, w.dtype, w.seed, device)
        k.append(a.contiguous())
        v.append(b.contiguous())
    torch.cuda.synchronize(device)
    shape = kvc.make_shape(w.layers, w.tokens, w.kv_heads, w.head_dim, kvc.BF16 if w.dtype == "bf16" else kvc.F16)
    return w, prof, shape, k, v


# the two kernels of a quantize / dequantize pair and the pair's timing name
PAIRED = {"kvc_enc_ktile": "kvc_quantize_kv", "kvc_enc_tile": "kvc_quantize_kv", "kvc_enc_rows": "kvc_quantize_kv",
          "kvc_dec_ktile": "kvc_dequantize_kv", "kvc_dec_tile": "kvc_dequantize_kv", "kvc_dec_rows": "kvc_dequantize_kv"}
PAIRS = {"kvc_quantize_kv", "kvc_dequantize_kv"}


def in_place_ranges(plan, tokens: int):
    """The chunk ranges of the code sections whose stored chunks kvc_decode's
    dequantizers read straight from the stream (the library's rule for
    kvc_decode_codes_in_place, restated for the byte counts)."""
    p = plan.profile
    cb = p.chunk_bytes
    if not p.n_stages or p.bits_map_k or p.bits_map_v or cb & (cb - 1):
        return []
    out = []
    for t in (0, 1):
        bits, G = (p.bits_v, p.group_v) if t else (p.bits_k, p.group_k)
        off, size = plan.section(2 * t)
        ok = bits in (2, 4, 8) and off % cb == 0 and (off + size) // cb > off // cb
        if (p.axis_v if t else p.axis_k) == 0:  # groups over tokens: the key-tile decoder
            ok = ok and (-(-tokens // G) * G) % 128 == 0 and cb % (2048 * bits) == 0
        else:  # the value-row decoder
            ok = ok and not (t == 0 and p.smooth_keys) and cb % (256 * bits) == 0
        if ok:
            out.append((off // cb, (off + size) // cb))
    return out


def raw_in_place_bytes(plan, tokens: int, stream_buf) -> int:
    """Bytes of the stored (raw) chunks that kvc_decode leaves in the stream: the
    lossless decoder neither reads nor writes them."""
    ranges = in_place_ranges(plan, tokens)
    if not ranges:
        return 0
    h = plan.header_bytes
    table = stream_buf[h:h + 4 * plan.n_chunks].cpu().numpy().view(np.uint32)
    return sum(int((table[lo:hi] >> 31).sum()) for lo, hi in ranges) * plan.profile.chunk_bytes


def kernel_bytes(plan, w, name: str, stream_bytes: int, in_place: int = 0) -> int:
    """Algorithmic bytes one launch of `name` must move (read + write); a pair moves
    both tensors' bytes.  `in_place`: bytes of the stored chunks the dequantizers
    read from the stream, which the lossless decoder skips."""
    raw_tensor = w.layers * w.tokens * w.kv_heads * w.head_dim * 2
    sec = [plan.section(i)[1] for i in range(8)]
    k_out = sec[0] + sec[1] + sec[4] + sec[5] + sec[6]
    v_out = sec[2] + sec[3] + sec[7]
    Q = plan.payload_bytes
    table = 4 * plan.n_chunks
    # the split encode (value-code chunks written by the value encoder): the lossless
    # launches before and after them read their chunks and write their stored form
    # (the stream's ratio to the payload assumed for each part)
    cb = plan.profile.chunk_bytes if hasattr(plan, "profile") else 0
    head = tail = 0
    if cb:
        off2, size2 = plan.section(2)
        c0, nfull = off2 // cb, size2 // cb
        head = min(c0 * cb, Q)
        tail = max(Q - (c0 + nfull) * cb, 0)
    ratio = stream_bytes / Q if Q else 0.0
    return {
        "kvc_enc_rows_lc": raw_tensor + v_out,
        "kvc_lossless_enc_fast_head": int(head * (1 + ratio)),
        "kvc_lossless_enc_fast_tail": int(tail * (1 + ratio)),
        "kvc_enc_tile": raw_tensor + k_out,
        "kvc_enc_ktile": raw_tensor + k_out,
        "kvc_enc_rows": raw_tensor + v_out,
        "kvc_dec_tile": raw_tensor + k_out,
        "kvc_dec_ktile": raw_tensor + k_out,
        "kvc_dec_rows": raw_tensor + v_out,
        "kvc_lossless_enc": Q + stream_bytes,
        "kvc_lossless_enc_fast": Q + stream_bytes,
        "kvc_lossless_dec": stream_bytes + Q,
        "kvc_lossless_dec_fast": stream_bytes + Q,
        "kvc_lossless_dec_inplace": stream_bytes + Q - 2 * in_place,
        "kvc_lossless_dec_fast_inplace": stream_bytes + Q - 2 * in_place,
        "kvc_decode_prepare": table + 8 * plan.n_chunks,
        "kvc_prologue": 64 + 8 * plan.n_chunks,
        "kvc_quantize_kv": 2 * raw_tensor + k_out + v_out,
        "kvc_dequantize_kv": 2 * raw_tensor + k_out + v_out,
    }.get(name, 0)


def max_over_ranks(ms: float, world: int, device=None) -> float:
    """Longest timed region over the ranks: the job is done when its slowest rank is."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(raw_bytes: int, world: int, steps: int, max_ms: float) -> float:
    """Whole-job GB/s: the input bytes of every rank's steps over the slowest rank's time."""
    return raw_bytes * world * steps / (max_ms * 1e-3) / 1e9


def benefit_report(enc_gbs: float, dec_gbs: float, cr: float) -> dict:
    """s_p and the break-even link bandwidth B*_p of the measured profile (KVServe
    §3.1 and §6.1 Eq. (5)): compressing pays off on links slower than B*_p."""
    from kv_cache_compression_encode_gb300.benefit import break_even_bandwidth, effective_throughput

    s_p = effective_throughput(enc_gbs, dec_gbs)
    return {"s_p_gbs": round(s_p, 2), "break_even_gbs": round(break_even_bandwidth(cr, s_p), 2),
            "compression_ratio": round(cr, 4)}


def run_kvc(args):
    import torch
    import torch.distributed as dist

    from kv_cache_compression_encode_gb300 import kvc
    from kv_cache_compression_encode_gb300.codec import Codec

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)

    w, prof, shape, k, v = workload_setup(args.workload, device)
    raw = w.raw_bytes
    codec = Codec(kvc.make_profile(**prof), shape, device)
    stream_buf = codec.new_stream_buffer()
    ok = [torch.empty_like(x) for x in k]
    ov = [torch.empty_like(x) for x in v]
    cs = torch.cuda.current_stream(device)

    def step():
        codec.encode(k, v, out=stream_buf)
        # the decode consumes the bytes the encode produced; its size is the
        # worst-case bound here (the stream is self-delimiting), so no host sync
        codec.decode(stream_buf, codec.plan.max_stream_bytes, ok, ov)

    # correctness of the timed configuration: one round trip, checked on the device
    codec.encode(k, v, out=stream_buf)
    st, nbytes, flags = codec.query()
    if st != kvc.KVC_OK:
        raise RuntimeError(f"encode failed: {kvc.status_str(st)} flags={flags}")
    codec.decode(stream_buf, nbytes, ok, ov)
    st, _, flags = codec.query()
    if st != kvc.KVC_OK:
        raise RuntimeError(f"decode failed: {kvc.status_str(st)} flags={flags}")
    in_place = raw_in_place_bytes(codec.plan, w.tokens, stream_buf)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)

    # encode-only and decode-only timings (untimed by the contract; reported apart)
    def time_loop(fn, n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cs)
        for _ in range(n):
            fn()
        b.record(cs)
        b.synchronize()
        return a.elapsed_time(b) / n

    n_side = max(3, min(50, args.steps // 10))
    enc_ms = time_loop(lambda: codec.encode(k, v, out=stream_buf), n_side)
    dec_ms = time_loop(lambda: codec.decode(stream_buf, nbytes, ok, ov), n_side)
    # the same decode with every code chunk restored into the payload first
    kvc.kvc_decode_codes_in_place(codec.plan, False)
    dec_payload_ms = time_loop(lambda: codec.decode(stream_buf, nbytes, ok, ov), n_side)
    kvc.kvc_decode_codes_in_place(codec.plan, True)

    # ---- timed region: K steps as a user runs them (no per-launch events)
    launches0 = codec.plan.launches
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(device)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(cs)
        for _ in range(args.steps):
            step()
        ev1.record(cs)
        ev1.synchronize()
    torch.cuda.synchronize(device)
    if world > 1:
        dist.barrier()
    total_ms = ev0.elapsed_time(ev1)
    launches = codec.plan.launches - launches0
    total_ms = max_over_ranks(total_ms, world, device)

    # ---- the same K steps again with an event pair around every launch (the
    # library's timing records, on the stream each kernel runs on): the per-kernel
    # durations of the `kernels` block and the roofline.  Kept out of the timed
    # region above: the events cost about 5% of the step.
    kvc.kvc_timing_enable(codec.plan, True, capacity=args.steps * 12 + 64)
    torch.cuda.synchronize(device)
    ek0, ek1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ek0.record(cs)
    for _ in range(args.steps):
        step()
    ek1.record(cs)
    ek1.synchronize()
    instrumented_ms = ek0.elapsed_time(ek1)
    recs = kvc.kvc_timing_read(codec.plan, args.steps * 12 + 64)
    kvc.kvc_timing_enable(codec.plan, False)
    st, _, flags = codec.query()
    if st != kvc.KVC_OK:
        raise RuntimeError(f"timed steps reported {kvc.status_str(st)} flags={flags}")

    if rank == 0:
        ms_step = total_ms / args.steps
        value = job_throughput(raw, world, args.steps, total_ms)
        # per-kernel live timings.  The K and V reconstruction kernels run side by
        # side (two streams); their pair is also timed as one unit
        # (kvc_dequantize_kv, from fork to join on the caller's stream), and the
        # units that partition the step -- not the overlapping kernels -- give the
        # shares and the roofline's dominant unit.
        per = {}
        for name, ms in recs:
            d = per.setdefault(name, [0.0, 0])
            d[0] += ms
            d[1] += 1
        inner = {n for n in per if PAIRED.get(n) in per}  # kernels timed inside an overlapped pair
        units = {n: d for n, d in per.items() if n not in inner}
        step_kernel_ms = sum(d[0] for d in units.values())
        kernels = {}
        for name, (ms_sum, n) in sorted(per.items(), key=lambda kv: -kv[1][0]):
            avg = ms_sum / n
            b = kernel_bytes(codec.plan, w, name, nbytes, in_place)
            rec = {"launches": n, "avg_ms": round(avg, 5), "alg_bytes": b,
                   "gbs": round(b / (avg * 1e-3) / 1e9, 1) if avg > 0 else None}
            if name in units:
                rec["share"] = round(ms_sum / step_kernel_ms, 4)
            else:
                rec["runs_beside"] = [o for o in PAIRED if o != name and o in per and PAIRED[o] == PAIRED[name]]
            kernels[name] = rec
        top = max(units.items(), key=lambda kv: kv[1][0])[0]
        peak, peak_src = peaks()
        top_avg = per[top][0] / per[top][1]
        achieved = kernel_bytes(codec.plan, w, top, nbytes, in_place) / (top_avg * 1e-3) / 1e9
        e2e = run_e2e(codec, k, v, ok, ov, w, args, device) if args.e2e else None
        # free this workload before the other configurations are set up
        del k, v, ok, ov, stream_buf
        torch.cuda.empty_cache()
        configs = other_configs(args, device) if args.configs else None
        cpu = cpu_baseline(w, prof, args) if not args.no_cpu_baseline else None
        clocks = clk.summary()
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "layers": w.layers, "tokens": w.tokens, "kv_heads": w.kv_heads,
                       "head_dim": w.head_dim, "elt": w.dtype, "distribution": w.dist,
                       "profile": json_profile(prof),
                       "raw_bytes": raw, "stream_bytes": nbytes, "compression_ratio": round(raw / nbytes, 4),
                       "step": "kvc_encode + kvc_decode", "l2": "inputs larger than L2 (no flush needed)",
                       "parallelism": f"replicas x{world}"},
            "encode_gbs": round(raw / (enc_ms * 1e-3) / 1e9, 2), "decode_gbs": round(raw / (dec_ms * 1e-3) / 1e9, 2),
            "decode_payload_path_gbs": round(raw / (dec_payload_ms * 1e-3) / 1e9, 2),
            "decode_in_place_bytes": in_place,
            "benefit": benefit_report(raw / (enc_ms * 1e-3) / 1e9, raw / (dec_ms * 1e-3) / 1e9, raw / nbytes),
            "roofline": {"bound": "hbm", "kernel": top, "achieved": round(achieved, 1), "peak": peak,
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                         else "fallback", "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": ncu_traffic(top, w.name),
                         **({"kernels": sorted(n for n in per if PAIRED.get(n) == top)} if top in PAIRS else {})},
            "kernels": kernels,
            "kernels_pass": {"ms_per_step": round(instrumented_ms / args.steps, 5),
                             "how": "the same steps again, an event pair around every launch"},
            "configs": configs,
            "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks, "gpu_launches": launches,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


FUSED_SUFFIX = "_fused_values"
OTHER_CONFIGS = ("llama70b", "llama8b_32k", "llama8b_mixhq", "llama8b_delta", "llama8b" + FUSED_SUFFIX)


def other_configs(args, device):
    """Encode and decode GB/s of the other workloads (the 70B one is quoted on its
    decode side) and of the format-v2 variants of Llama-8B: CUDA events on the
    launching stream, after a checked round trip and warm-up, inputs larger than L2.
    Reported beside `value`, which stays the metric's llama8b configuration."""
    import torch

    from kv_cache_compression_encode_gb300 import kvc
    from kv_cache_compression_encode_gb300.codec import Codec

    out = {}
    cs = torch.cuda.current_stream(device)
    for name in OTHER_CONFIGS:
        w, prof, shape, k, v = workload_setup(name, device)
        codec = Codec(kvc.make_profile(**prof), shape, device)
        sbuf = codec.new_stream_buffer()
        ok = [torch.empty_like(x) for x in k]
        ov = [torch.empty_like(x) for x in v]
        fused = name.endswith(FUSED_SUFFIX)
        if fused:  # the stream must not depend on the execution choice
            ref = codec.encode(k, v).clone()
            _, nref, _ = codec.query()
            kvc.kvc_fuse_value_chunks(codec.plan, True)
        codec.encode(k, v, out=sbuf)
        st, nbytes, _ = codec.query()
        codec.decode(sbuf, nbytes, ok, ov)
        st2, _, _ = codec.query()

        def loop(fn, n):
            for _ in range(3):
                fn()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(cs)
            for _ in range(n):
                fn()
            b.record(cs)
            b.synchronize()
            return a.elapsed_time(b) / n

        n = max(5, min(50, args.steps // 40))
        enc_ms = loop(lambda: codec.encode(k, v, out=sbuf), n)
        dec_ms = loop(lambda: codec.decode(sbuf, nbytes, ok, ov), n)
        kvc.kvc_decode_codes_in_place(codec.plan, False)
        dec_payload_ms = loop(lambda: codec.decode(sbuf, nbytes, ok, ov), n)
        kvc.kvc_decode_codes_in_place(codec.plan, True)
        out[name] = {"workload": w.name, "raw_bytes": w.raw_bytes, "stream_bytes": nbytes,
                     "compression_ratio": round(w.raw_bytes / nbytes, 4), "encode_ms": round(enc_ms, 4),
                     "decode_ms": round(dec_ms, 4), "encode_gbs": round(w.raw_bytes / (enc_ms * 1e-3) / 1e9, 1),
                     "decode_gbs": round(w.raw_bytes / (dec_ms * 1e-3) / 1e9, 1),
                     "decode_payload_path_gbs": round(w.raw_bytes / (dec_payload_ms * 1e-3) / 1e9, 1), "steps": n,
                     "status": kvc.status_str(st) if st != kvc.KVC_OK else kvc.status_str(st2)}
        if name == "llama70b":
            out[name]["headline"] = "decode"
        if fused:
            out[name]["execution"] = "value-code chunks written by the value encoder (kvc_fuse_value_chunks)"
            out[name]["stream_matches_unfused"] = bool(nref == nbytes and torch.equal(ref[:nref], sbuf[:nbytes]))
        if prof.get("bits_map_k") is not None or prof.get("token_delta"):
            out[name]["profile"] = json_profile(prof)
        del k, v, ok, ov, sbuf, codec
        torch.cuda.empty_cache()
    return out


def run_e2e(codec, k, v, ok, ov, w, args, device):
    """Same metric through the public API with host buffers: every step copies the
    KV from pinned host memory, encodes, reads the size and the stream back, then
    copies the stream in, decodes and copies the KV out.  Three requests (--e2e-requests) are in
    flight, each on its own CUDA stream with its own plan, workspace and buffers
    (a serving process overlaps one request's uploads with others' downloads);
    every step still moves all of its own bytes.  Each request's K (and V) for all
    layers sits in one contiguous buffer, host and device, whose per-layer views the
    API takes, so that a direction's KV moves in one copy (a serving KV pool is laid
    out so; many small copies run the link about 14% slower both ways).
    `host_link` holds the copy rates over the same buffers (each direction alone,
    both at once) and the bound they set on this figure.  Three timed windows of
    the same length; the median is the figure (all three are listed)."""
    import torch

    from kv_cache_compression_encode_gb300.codec import Codec

    hK, hV = torch.stack(k).cpu().pin_memory(), torch.stack(v).cpu().pin_memory()

    class Lane:
        def __init__(self, c):
            self.codec = c
            self.s = torch.cuda.Stream(device)
            self.rK, self.rV = torch.empty_like(hK).pin_memory(), torch.empty_like(hV).pin_memory()
            self.rk, self.rv = list(self.rK.unbind(0)), list(self.rV.unbind(0))
            self.hs = torch.empty(c.plan.max_stream_bytes, dtype=torch.uint8).pin_memory()
            self.dK, self.dV = torch.empty_like(hK, device=device), torch.empty_like(hV, device=device)
            self.dk, self.dv = list(self.dK.unbind(0)), list(self.dV.unbind(0))
            self.sbuf = c.new_stream_buffer()
            self.rbuf = c.new_stream_buffer()

    n_lanes = args.e2e_requests
    lanes = [Lane(codec)] + [Lane(Codec(codec.profile, codec.shape, device)) for _ in range(n_lanes - 1)]
    counts = {"h2d": 0, "d2h": 0}

    def front(L):  # inputs up, encode
        with torch.cuda.stream(L.s):
            L.dK.copy_(hK, non_blocking=True)
            L.dV.copy_(hV, non_blocking=True)
            L.codec.encode(L.dk, L.dv, out=L.sbuf)

    def back(L):  # size scalar to the host, stream down and up again, decode, KV down
        with torch.cuda.stream(L.s):
            _, n, _ = L.codec.query()  # synchronizes this lane's stream only
            L.hs[:n].copy_(L.sbuf[:n], non_blocking=True)
            L.rbuf[:n].copy_(L.hs[:n], non_blocking=True)  # the receiving side's upload
            L.codec.decode(L.rbuf, n, L.dk, L.dv)
            L.rK.copy_(L.dK, non_blocking=True)
            L.rV.copy_(L.dV, non_blocking=True)
        counts["h2d"] = w.raw_bytes + n
        counts["d2h"] = n + w.raw_bytes + 16

    def run(n):  # request i: front when i - (n_lanes - 1) has been taken back, then back in order
        for j in range(min(n_lanes - 1, n)):
            front(lanes[j])
        for i in range(n):
            if i + n_lanes - 1 < n:
                front(lanes[(i + n_lanes - 1) % n_lanes])
            back(lanes[i % n_lanes])
        for L in lanes:
            L.s.synchronize()

    run(4)
    n_steps = max(4, min(20, args.steps // 100))
    # the host side of the link is shared with other jobs on the machine, which
    # now and then halve its rate for a while: three windows, the median reported
    windows = []
    for _ in range(3):
        torch.cuda.synchronize(device)
        t0 = time.perf_counter()
        run(n_steps)
        windows.append((time.perf_counter() - t0) / n_steps)
    dt = sorted(windows)[1]
    ok_rt = all(torch.equal(a, b.to(a.device)) for L in lanes for a, b in zip(ok + ov, L.rk + L.rv))

    # the host link on its own, over the same pinned buffers with all lanes copying at
    # once: each direction alone, and both together (uploads on the lanes' streams,
    # downloads on a second stream per lane), each the best of three; the bound they
    # put on this figure
    down = [torch.cuda.Stream(device) for _ in lanes]
    srcK, srcV = torch.stack(k), torch.stack(v)  # downloads read these, which nothing writes meanwhile

    def link(up: bool, dn: bool):
        reps = 2
        torch.cuda.synchronize(device)
        t0 = time.perf_counter()
        for _ in range(reps):
            for L, sd in zip(lanes, down):
                for d, h, r, src in ((L.dK, hK, L.rK, srcK), (L.dV, hV, L.rV, srcV)):
                    if up:
                        with torch.cuda.stream(L.s):
                            d.copy_(h, non_blocking=True)
                    if dn:
                        with torch.cuda.stream(sd):
                            r.copy_(src, non_blocking=True)
        torch.cuda.synchronize(device)
        return reps * n_lanes * w.raw_bytes * (int(up) + int(dn)) / (time.perf_counter() - t0) / 1e9

    link(True, False)

    def best3(up, dn):  # the link's rate when nothing else on the host is using it
        return max(link(up, dn) for _ in range(3))

    h2d_gbs, d2h_gbs, both_gbs = best3(True, False), best3(False, True), best3(True, True)
    link_ms = max(counts["h2d"] / h2d_gbs, counts["d2h"] / d2h_gbs, (counts["h2d"] + counts["d2h"]) / both_gbs) / 1e6
    return {"value": round(w.raw_bytes / dt / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": counts["h2d"],
            "d2h_bytes_per_step": counts["d2h"], "ms_per_step": round(dt * 1e3, 3), "steps": n_steps,
            "requests_in_flight": n_lanes, "roundtrip_matches_device_path": bool(ok_rt),
            "windows_gbs": [round(w.raw_bytes / x / 1e9, 2) for x in windows],
            "host_link": {"h2d_gbs": round(h2d_gbs, 1), "d2h_gbs": round(d2h_gbs, 1),
                          "both_ways_gbs": round(both_gbs, 1), "bound_gbs": round(w.raw_bytes / link_ms / 1e6, 2)}}


# ---------------------------------------------------------------------------- oracle
def oracle_sample(w, prof, layers: int, device=None):
    """Host bits of the first `layers` layers of the workload (same generator as the GPU run)."""
    from kv_cache_compression_encode_gb300 import synth

    hk, hv = [], []
    for l in range(layers):
        a, b = synth.layer_kv(w.dist, l, w.tokens, w.kv_heads, w.head_dim, w.dtype, w.seed,
                              device if device is not None else "cpu")
        hk.append(synth.to_bits_numpy(a))
        hv.append(synth.to_bits_numpy(b))
    return hk, hv


def time_oracle_step(w, prof, hk, hv, layers):
    from oracle import oracle as O

    shape = O.make_shape(layers, w.tokens, w.kv_heads, w.head_dim, 2 if w.dtype == "bf16" else 1)
    oprof = O.make_profile(**prof)
    t0 = time.perf_counter()
    s, _ = O.encode(oprof, shape, hk, hv)
    rk = [np.empty_like(a) for a in hk]
    rv = [np.empty_like(a) for a in hv]
    O.decode(oprof, shape, s, rk, rv)
    return time.perf_counter() - t0


def oracle_layers(w, args) -> int:
    """Layers of the oracle sample: all of them (or --oracle-layers), at most ~1 GiB of host KV."""
    per_layer = 2 * w.tokens * w.kv_heads * w.head_dim * (2 if w.dtype in ("bf16", "f16") else 4)
    cap = max(1, (1 << 30) // per_layer)
    want = w.layers if args.oracle_layers <= 0 else args.oracle_layers
    return max(1, min(w.layers, want, cap))


def cpu_baseline(w, prof, args):
    """The oracle on the host cores: whole passes over the sample until --oracle-seconds have elapsed."""
    from oracle import oracle as O

    cores = len(os.sched_getaffinity(0))
    O.set_threads(cores)
    layers = oracle_layers(w, args)
    hk, hv = oracle_sample(w, prof, layers, device="cuda" if not args.cpu_inputs else "cpu")
    dt, passes = 0.0, 0
    while passes == 0 or (dt < args.oracle_seconds and dt + dt / passes <= 30.0):
        dt += time_oracle_step(w, prof, hk, hv, layers)
        passes += 1
    sample_bytes = 2 * layers * w.tokens * w.kv_heads * w.head_dim * 2
    return {"value": round(passes * sample_bytes / dt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{passes} encode+decode passes over {layers} of {w.layers} layers of {w.name} "
                      f"({sample_bytes} raw bytes each), {dt:.1f} s"}


def run_reference(args):
    """The reference arm for this build is the oracle itself, on the host cores."""
    from oracle import oracle as O

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w, prof = workload_and_profile(args.workload)
    cores = len(os.sched_getaffinity(0))
    O.set_threads(cores)
    layers = oracle_layers(w, args)
    hk, hv = oracle_sample(w, prof, layers, device="cpu")
    for _ in range(min(args.warmup, 1)):
        time_oracle_step(w, prof, hk, hv, layers)
    steps = max(1, min(args.steps, args.reference_steps))
    dts = [time_oracle_step(w, prof, hk, hv, layers) for _ in range(steps)]
    sample_bytes = 2 * layers * w.tokens * w.kv_heads * w.head_dim * 2
    dt = float(np.mean(dts))
    value = sample_bytes / dt / 1e9
    sample = f"{layers} of {w.layers} layers of {w.name} ({sample_bytes} raw bytes) per step, encode+decode"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "layers": w.layers, "tokens": w.tokens, "kv_heads": w.kv_heads,
                   "head_dim": w.head_dim, "elt": w.dtype, "sample_layers": layers},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="llama8b")
    ap.add_argument("--impl", default="kvc", choices=["kvc", "reference"])
    ap.add_argument("--oracle-layers", type=int, default=0)  # 0: all layers (host sample capped near 1 GiB)
    ap.add_argument("--oracle-seconds", type=float, default=10.0)
    ap.add_argument("--reference-steps", type=int, default=3)
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--e2e-requests", type=int, default=3, help="requests in flight in the end-to-end run")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-inputs", action="store_true")
    ap.add_argument("--no-configs", dest="configs", action="store_false")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus != world:
        # one process per GPU: N > 1 runs under torchrun, which sets WORLD_SIZE = N
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}: launch N > 1 with "
                         f"python -m torch.distributed.run --nproc-per-node {args.gpus} bench.py --gpus {args.gpus}")
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_kvc(args)


if __name__ == "__main__":
    main()
