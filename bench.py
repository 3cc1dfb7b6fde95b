#!/usr/bin/env python
"""Benchmark of the Engram layer forward (one GB300 per rank).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

A step is one engram_forward (gather + dequantise -> tcgen05 wkv projection ->
gate + residual add) over one batch of synthetic inputs resident in HBM.  The
default workload is the largest configuration of the layer's benchmark that
one GPU holds: the full-size table (384,016,682 rows, 98.3 GB of fp8 codes plus
3.1 GB of scales) with a prefill batch of B=2, T=8192.  The same JSON line
carries a `per_config` list with the benchmark's other configurations (tiny,
decode batch, Zipf prefill, skewed large decode), each measured the same way
(`--no-per-config` leaves them out; `--workload` picks another main one).

One JSON line is printed by rank 0 (see the keys below).  `value` is tokens/s
over all ranks, timed on the device with CUDA events around each step; the L2
is flushed between timed steps, outside the events (a 256 MB write, then a
256 MB read that leaves none of the write's dirty lines to the step).  `e2e`
times the same call with the inputs in pinned host memory: the host->device
copies of hash_ids, x and the mask and the device->host copy of the output are
inside its timed region.  `roofline` describes the dominant kernel (the wkv
projection) from its own CUDA-event durations; `cpu_baseline` is the CPU oracle
timed on a bounded sample of the same workload.  `--impl reference` times the
oracle alone as the reference arm.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Engram layer tokens/s (prefill, decode); gather HBM GB/s; % of roofline"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "full_2x8192"
# the benchmark's other configurations, measured after the main one and reported in `per_config`
PER_CONFIG = ["tiny_1x16", "decode_64x1", "prefill_1x4096_zipf", "decode_512x1_skew"]
PER_CONFIG_CPU_SECONDS = 4.0
ARGS = None
FLUSH_BYTES = 256 << 20


# ---------------------------------------------------------------- helpers
L2_NOTE = ("flushed between timed steps, outside the events: a 256 MB write, then a 256 MB read, so no dirty "
           "line of the write is written back inside the step")


class L2Flush:
    """Leaves the L2 cold for the next step: writes a buffer twice the L2's
    size, then reads another, so the step finds none of its own data in L2 and
    the write-back of the write's dirty lines happens here, not in the step."""

    def __init__(self, torch, dev):
        self._torch = torch
        self._w = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self._r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self._sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        self._w.zero_()
        self._torch.sum(self._r, dim=0, out=self._sink)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def algorithmic(w, M):
    """Bytes and FLOPs the layer must move / compute for M tokens: per token
    the ids (n_cols*8), codes (n_cols*head_dim), scales, x and out (hc*dim*2
    each) and the mask byte; per call the wkv weight and q/k weights."""
    nb = w.head_dim // w.scale_block
    sb = 1 if w.scale_fmt == 1 else 4
    per_tok = (w.n_cols * 8 + w.n_cols * w.head_dim + w.n_cols * nb * sb + 2 * w.hc_mult * w.dim * 2 + 1)
    per_call = weight_bytes(w) + 2 * w.hc_mult * w.dim * 2
    flops = 2.0 * w.N * w.K * M
    return per_tok * M + per_call, flops


def weight_bytes(w):
    """The projection weight as the layer reads it: bf16, or e4m3 codes plus
    one E8M0 byte per 32 inputs."""
    return w.N * w.K * 2 if w.wkv_fmt == 0 else w.N * w.K + w.N * w.K // 32


def projection_bytes(w, M, fused=False):
    """Algorithmic bytes of one projection launch: the weight once, the
    gathered rows read once, kv written once in bf16 -- or, with the gate in
    the epilogue, x read once and the output written once instead of kv."""
    a_bytes = w.K * 2 if w.wkv_fmt == 0 else w.K + w.K // 32   # bf16 rows, or codes + scales
    out_bytes = 2 * w.hc_mult * w.dim * 2 if fused else w.N * 2
    return weight_bytes(w) + M * a_bytes + M * out_bytes


def gather_bytes(w, M):
    nb = w.head_dim // w.scale_block
    sb = 1 if w.scale_fmt == 1 else 4
    written = w.K * 2 if w.wkv_fmt == 0 else w.K + w.K // 32
    return M * (w.n_cols * 8 + w.n_cols * w.head_dim + w.n_cols * nb * sb + written)


def _projection_part(text: bytes) -> bytes:
    """internal.cuh as far as the projection kernel sees it: the shared header
    and the projection's section, without the gather's and the gate's."""
    rows, proj, gate = b"// ---- rows", b"// ---- projection", b"// ---- gate"
    i, j, k = text.find(rows), text.find(proj), text.find(gate)
    if min(i, j, k) < 0 or not i < j < k:
        return text
    return text[:i] + text[j:k]


def _code_only(text: bytes) -> bytes:
    """The source without // comments, blank lines and indentation: a change
    of wording leaves the digest, and so the recorded traffic, as it was."""
    out = []
    for line in text.splitlines():
        code = line.split(b"//", 1)[0].strip()
        if code:
            out.append(code)
    return b"\n".join(out)


def source_digest(files):
    h = hashlib.sha256()
    for f in files:
        text = open(os.path.join(ROOT, f), "rb").read()
        h.update(_code_only(_projection_part(text) if f.endswith("internal.cuh") else text))
    return h.hexdigest()[:16]


# the projection kernel's source: its translation unit, the device helpers and
# the launch declarations it shares (a recorded ncu traffic figure is reported
# only while these are unchanged)
GEMM_SOURCES = ["engram_hashed_gram_gb300/csrc/gemm.cu", "engram_hashed_gram_gb300/csrc/common.cuh",
                "engram_hashed_gram_gb300/csrc/internal.cuh"]


def plan_key(info):
    """The plan as the traffic record names it: <split-K factor>x<CTAs>, with
    a trailing p for CTA pairs, r<tiles>x<ranges> for a remainder split and f
    for the gate in the projection's epilogue."""
    key = "%dx%d" % (info["splits"], info["ctas"])
    if info.get("cta_pairs"):
        key += "p"
    if info.get("rem_tiles"):
        key += "r%dx%d" % (info["rem_tiles"], info["rem_splits"])
    if info.get("fused_gate"):
        key += "f"
    return key


def recorded_traffic(workload, plan=None):
    """DRAM bytes per launch of the projection kernel from the committed ncu
    summary, if it was taken on the current kernel source (and, when the record
    names one, the same plan, plan_key); else None."""
    p = os.path.join(ROOT, "profiles", "wkv_gemm_traffic.txt")
    if not os.path.exists(p):
        return None
    digest = source_digest(GEMM_SOURCES)
    for line in open(p):
        kv = dict(tok.split("=", 1) for tok in line.split() if "=" in tok)
        if kv.get("workload") == workload and kv.get("source_sha256") == digest:
            if plan is not None and "plan" in kv and kv["plan"] != plan:
                continue
            return float(kv["dram_bytes_per_launch"])
    return None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.marks = []

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        busy = [r for r in rows if r["power"] > 1.3 * min(x["power"] for x in rows)] or rows
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(busy)}


# ---------------------------------------------------------------- CPU oracle
def cpu_oracle_run(w, inp, min_seconds=12.0, max_passes=50, tok=None):
    """Times the oracle as it stands on passes over a bounded token sample;
    returns (tokens/s, seconds, tokens, description).  Regenerating the table
    rows the sample references is input generation and is not timed."""
    import numpy as np
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from oracle import engram_oracle as O
    from parity import compact_rows
    M = w.M
    if tok is None:
        tok = np.arange(min(M, 64))
    ids = inp.hash_ids.reshape(M, w.n_cols)[tok]
    cids, codes, scales = compact_rows(w, ids)
    x = inp.x.reshape(M, w.hc_mult, w.dim)[tok]
    mask = None if inp.mask is None else inp.mask.reshape(M)[tok]
    t0 = time.perf_counter()
    passes = 0
    while True:
        O.forward(cids, x, codes, scales, inp.wkv, inp.q, inp.k, mask, scale_block=w.scale_block,
                  scale_fmt=w.scale_fmt, eps=w.eps, wkv_scale=inp.wkv_scale)
        passes += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or passes >= max_passes:
            break
    n = passes * len(tok)
    desc = f"{passes} pass(es) of the oracle over {len(tok)} of the workload's {M} tokens"
    return n / el, el, n, desc


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = max((d.get("num_threads", 0) for d in threadpool_info()), default=0)
        if n:
            return n
    except Exception:
        pass
    return os.cpu_count()


# ---------------------------------------------------------------- arms
def run_reference(args, w):
    """The oracle as the reference arm, on the host cores."""
    from engram_hashed_gram_gb300 import synth
    import numpy as np
    inp = synth.make_inputs(w)
    tok = np.arange(min(w.M, 64))
    for _ in range(args.warmup):
        cpu_oracle_run(w, inp, min_seconds=0.0, max_passes=1, tok=tok)
    times = []
    for _ in range(args.steps):
        v, el, n, desc = cpu_oracle_run(w, inp, min_seconds=0.0, max_passes=1, tok=tok)
        times.append(el)
    total = sum(times)
    value = len(tok) * args.steps / total
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                         "sample": f"each step: one oracle pass over {len(tok)} of the workload's {w.M} tokens"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def config_of(w):
    return {"workload": w.name, "B": w.B, "T": w.T, "tokens": w.M, "dim": w.dim, "hc_mult": w.hc_mult,
            "n_cols": w.n_cols, "head_dim": w.head_dim, "table_rows": w.num_rows(),
            "table_gb": round(w.num_rows() * w.head_dim / 1e9, 2), "hash_ids": w.ids, "mask": w.mask,
            "prime_base": w.prime_base,
            "wkv": "bf16 [25600, 6144]" if w.wkv_fmt == 0 else "mxfp8 [25600, 6144]: e4m3 + e8m0 per 32 inputs",
            "table_scales": "fp32 per 128" if w.scale_fmt == 0 else "e8m0 per 32", "fuse_gate": getattr(ARGS, "fuse_gate", "auto"),
            "table_placement": ("pinned host memory, read in place over the host link"
                                if getattr(ARGS, "table_host", False) else "device"),
            "l2": L2_NOTE}


def run_ours(args, w, rank, world, local_rank):
    import numpy as np
    import torch
    import torch.distributed as dist
    from engram_hashed_gram_gb300 import build as B
    from engram_hashed_gram_gb300 import synth
    from engram_hashed_gram_gb300 import synth_device as SD
    from engram_hashed_gram_gb300.layer import EngramLayer

    B.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    M = w.M
    inp = synth.make_inputs(w)
    table, scale = SD.make_table(w, device=dev, host=args.table_host)
    d = SD.upload_inputs(inp, device=dev)
    layer = EngramLayer(table, scale, d["wkv"], d["q"], d["k"], max_tokens=M, eps=w.eps,
                        fuse_gate={"auto": None, "on": True, "off": False}[args.fuse_gate],
                        device=dev,
                        scale_block=w.scale_block, scale_fmt=w.scale_fmt, wkv_scale=d["wkv_scale"])
    ids, x, mask = d["hash_ids"], d["x"], d["mask"]
    out = torch.empty_like(x)
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream(dev)

    sampler = ClockSampler(local_rank)
    sampler.start()
    # the first warm-up step on its own (its launches load the kernels); the
    # other warm-up steps are queued right before the timed ones, so the first
    # timed step follows warm steps as every later one does
    first = min(1, args.warmup)
    for _ in range(first):
        layer.forward(ids, x, mask, out=out)
    torch.cuda.synchronize()
    st, _ = layer.sync_status()
    if st != 0:
        raise RuntimeError(f"engram_forward reported status {st} in warm-up")

    # ---- device-timed steps (inputs resident in HBM); one event pair per step
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # lets the host queue ahead (~0.1 ms of Python per step at most): no step
    # waits on the Python call
    torch.cuda._sleep(int(2e7 + 2e5 * (args.steps + args.warmup)))
    for _ in range(args.warmup - first):
        flush()
        layer.forward(ids, x, mask, out=out)
    for i in range(args.steps):
        flush()
        ev[i][0].record(stream)
        layer.forward(ids, x, mask, out=out)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = sum(step_ms)

    # ---- per-kernel durations: the timed region's steps again, queued the same
    # way (flush + forward, the host ahead of the device), with an event
    # between the kernels.  Events between kernels also stop them from
    # overlapping, so these are each kernel's own duration; they are not used
    # for `value`.
    layer.enable_stage_timing(True, calls=args.steps)
    torch.cuda.synchronize()
    torch.cuda._sleep(int(2e7 + 2e5 * args.steps))
    for i in range(args.steps):
        flush()
        layer.forward(ids, x, mask, out=out)
    stages = layer.stage_times_n(args.steps)      # waits for the last step's last event
    layer.enable_stage_timing(False)

    # keep the GPU busy a little longer so the clock sampler sees the load
    t_end = time.perf_counter() + 1.0
    while time.perf_counter() < t_end:
        for _ in range(20):
            layer.forward(ids, x, mask, out=out)
        torch.cuda.synchronize()
    clocks = sampler.stop()
    st, _ = layer.sync_status()
    if st != 0:
        raise RuntimeError(f"engram_forward reported status {st}")

    # ---- end to end, through the public call with host buffers: every step
    # copies its inputs (x, ids and mask, packed in one pinned buffer) to the
    # device and its output back.  Two device buffer sets and two copy streams
    # let step i+1's upload and step i-1's download overlap step i's compute,
    # as a serving loop would.  No L2 flush here: each step streams the whole
    # weight (larger than L2) and its inputs arrive from the host.
    nb_x, nb_ids = inp.x.nbytes, inp.hash_ids.nbytes
    nb_m = 0 if inp.mask is None else inp.mask.nbytes
    nb_in = (nb_x + nb_ids + nb_m + 15) // 16 * 16
    h_in = torch.zeros(nb_in, dtype=torch.uint8).pin_memory()
    h_in[:nb_x].copy_(torch.from_numpy(inp.x.reshape(-1).view(np.uint8)))
    h_in[nb_x:nb_x + nb_ids].copy_(torch.from_numpy(inp.hash_ids.reshape(-1).view(np.uint8)))
    if nb_m:
        h_in[nb_x + nb_ids:nb_x + nb_ids + nb_m].copy_(torch.from_numpy(inp.mask.reshape(-1)))
    d_in = [torch.empty(nb_in, dtype=torch.uint8, device=dev) for _ in range(2)]
    views = []
    for buf in d_in:
        vx = buf[:nb_x].view(torch.bfloat16).view(x.shape)
        vi = buf[nb_x:nb_x + nb_ids].view(torch.int64).view(ids.shape)
        vm = buf[nb_x + nb_ids:nb_x + nb_ids + nb_m].view(mask.shape) if nb_m else None
        views.append((vi, vx, vm))
    d_out = [torch.empty_like(x) for _ in range(2)]
    h_out = [torch.empty(x.shape, dtype=torch.int16).pin_memory() for _ in range(2)]
    up_s, down_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_run(n):
        """n pipelined steps; returns the device milliseconds from the first
        upload to the last download.  Uploads and downloads run on their own
        streams (the two copy directions overlap each other and the steps)."""
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        uploaded = [torch.cuda.Event() for _ in range(n)]
        computed = [torch.cuda.Event() for _ in range(n)]
        downloaded = [torch.cuda.Event() for _ in range(n)]
        torch.cuda.synchronize()
        with torch.cuda.stream(up_s):
            torch.cuda._sleep(int(2e7))    # the host queues every step ahead of the device
        stream.wait_stream(up_s)
        down_s.wait_stream(up_s)
        t0.record(up_s)
        down_s.wait_event(t0)
        h0 = time.perf_counter()
        for i in range(n):
            b = i % 2
            if i >= 2:
                up_s.wait_event(computed[i - 2])           # step i-2 has read input buffer b
            with torch.cuda.stream(up_s):
                d_in[b].copy_(h_in, non_blocking=True)
                uploaded[i].record(up_s)
            stream.wait_event(uploaded[i])
            if i >= 2:
                stream.wait_event(downloaded[i - 2])       # output buffer b is back on the host
            vi, vx, vm = views[b]
            layer.forward(vi, vx, vm, out=d_out[b])
            computed[i].record(stream)
            down_s.wait_event(computed[i])
            with torch.cuda.stream(down_s):
                h_out[b].copy_(d_out[b].view(torch.int16), non_blocking=True)
                downloaded[i].record(down_s)
        t1.record(down_s)
        host_us[0] = (time.perf_counter() - h0) / n * 1e6
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    host_us = [0.0]
    e2e_run(max(3, args.warmup))
    e2e_ms = e2e_run(args.steps)
    last = (args.steps - 1) % 2
    if not np.array_equal(h_out[last].numpy().view(np.uint16), out.view(torch.int16).cpu().numpy().view(np.uint16)):
        raise RuntimeError("end-to-end output differs from the device-resident run")
    h2d = nb_in
    d2h = inp.x.nbytes

    # ---- aggregate over ranks
    value, e2e_value, total_ms, e2e_ms = aggregate_over_ranks(total_ms, e2e_ms, M, args.steps, world, dev)

    pk = peaks()
    if w.wkv_fmt == 1:
        # an FP8 contraction: the measured bf16 peaks times the nominal fp8 / bf16 ratio (4.5 / 2.25)
        sus = pk.get("bf16_tflops_sustained")
        pk = dict(pk, bf16_tflops=2.0 * pk["bf16_tflops"], bf16_tflops_sustained=None if sus is None else 2.0 * sus,
                  source=pk["source"] + " bf16 x 2 (nominal fp8/bf16)")
    splits, ctas = layer.plan(M)
    plan_info = layer.describe_plan(M)
    kernels_per_step = layer.forward_kernels(M)
    gather_ms = statistics.mean(s[0] for s in stages)
    proj_ms = statistics.mean(s[1] for s in stages)
    gate_ms = statistics.mean(s[2] for s in stages)
    pbytes = projection_bytes(w, M, fused=bool(plan_info["fused_gate"]))
    pflops = 2.0 * w.N * w.K * M
    t_mem = pbytes / (pk["hbm_gbs"] * 1e9)
    t_tc = pflops / (pk["bf16_tflops"] * 1e12)
    if t_mem >= t_tc:
        roof = {"bound": "hbm", "achieved": pbytes / (proj_ms * 1e-3) / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": pflops / (proj_ms * 1e-3) / 1e12, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s"}
        if pk.get("bf16_tflops_sustained"):
            # the peak a dense GEMM holds for seconds under the power cap
            roof["frac_of_sustained"] = roof["achieved"] / pk["bf16_tflops_sustained"]
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = recorded_traffic(w.name, plan_key(plan_info))
    roof["kernel"] = ("wkv_gemm_pair_kernel (tcgen05 cta_group::2 projection on CTA pairs)" if plan_info["cta_pairs"]
                      else "wkv_gemm_kernel (tcgen05 projection)")
    if plan_info["fused_gate"]:
        roof["kernel"] += ", gate and residual add in its epilogue"
    roof["peak_source"] = pk["source"]
    roof["algorithmic_bytes_per_launch"] = pbytes
    roof["algorithmic_flops_per_launch"] = pflops
    roof["avg_launch_ms"] = proj_ms

    lbytes, lflops = algorithmic(w, M)
    t_roof = max(lbytes / (pk["hbm_gbs"] * 1e9), lflops / (pk["bf16_tflops"] * 1e12))
    ms_per_step = total_ms / args.steps
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step,
        "step_ms_spread": {"median": statistics.median(step_ms), "min": min(step_ms), "max": max(step_ms)},
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.wkv_fmt == 0 else "mxfp8", "data": "synthetic",
        "config": config_of(w),
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "schedule": "each step uploads its inputs and downloads its output; upload and download streams "
                            "overlap the next upload and the previous download with the step (two buffer sets); "
                            "the host queues the steps ahead of the device",
                "host_enqueue_us_per_step": host_us[0]},
        "gpu_launches": kernels_per_step * args.steps,
        "roofline": roof,
        "layer_roofline": {"bytes": lbytes, "flops": lflops, "roofline_us": 1e6 * t_roof,
                           "achieved_us": 1e3 * ms_per_step, "frac": t_roof / (ms_per_step * 1e-3)},
        "stages_ms": {"gather": gather_ms, "projection": proj_ms, "gate": gate_ms},
        "gather_gbs": gather_bytes(w, M) / (gather_ms * 1e-3) / 1e9,
        "plan": plan_info,
        "clocks": clocks,
    }
    layer.close()
    del table, scale
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline:
        v, el, n, desc = cpu_oracle_run(w, inp, min_seconds=args.cpu_seconds)
        result["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                                  "sample": desc, "seconds": el}
    return result


def per_config_entry(r):
    """The keys of one configuration's measurement that the per_config list carries."""
    keys = ("value", "unit", "ms_per_step", "step_ms_spread", "dtype", "e2e", "gpu_launches", "roofline",
            "layer_roofline", "stages_ms", "gather_gbs", "plan", "clocks", "cpu_baseline")
    out = {"workload": r["config"]["workload"], "config": r["config"]}
    out.update({k: r[k] for k in keys if k in r})
    return out


def aggregate_over_ranks(total_ms, e2e_ms, tokens_per_rank, steps, world, device):
    """Whole-job throughput of a weak-scaling run: every rank processed
    tokens_per_rank tokens per step, and the job took as long as its slowest
    rank (max over ranks of the timed milliseconds).  Returns (tokens/s,
    e2e tokens/s, max timed ms, max e2e ms)."""
    import torch
    t = torch.tensor([total_ms, e2e_ms], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    total_ms, e2e_ms = float(t[0]), float(t[1])
    tokens = world * tokens_per_rank * steps
    return tokens / (total_ms / 1e3), tokens / (e2e_ms / 1e3), total_ms, e2e_ms


def inp_pinned(torch, a):
    return torch.from_numpy(a).pin_memory()


def run_hash(args, w):
    """Times engram_hash alone (two Engram layers, 3 orders x 8 heads, the 48
    primes above 16,000,000, synthetic token ids and map) on the workload's
    B x T; prints its own JSON line."""
    import numpy as np
    import torch
    from engram_hashed_gram_gb300 import build as B
    from engram_hashed_gram_gb300 import synth
    from engram_hashed_gram_gb300.layer import EngramHasher
    B.build()
    rng = np.random.default_rng(w.seed)
    vocab = 129_280
    primes = np.array(synth.consecutive_primes_above(16_000_000, 48), dtype=np.int64).reshape(2, 3, 8)
    offsets = np.stack([np.concatenate([[0], np.cumsum(primes[g].reshape(-1))[:-1]]) for g in range(2)])
    mult = (rng.integers(1, 1 << 62, size=(2, 4)) * 2 + 1).astype(np.int64)
    tmap = rng.integers(0, 99_092, size=vocab).astype(np.int32)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    hasher = EngramHasher(dev(tmap), dev(mult), dev(primes), dev(offsets), max_batch=w.B, max_len=w.T)
    ids = dev(rng.integers(0, vocab, size=(w.B, w.T)))
    out = torch.empty((2, w.B, w.T, 24), dtype=torch.int64, device="cuda")
    for _ in range(args.warmup):
        hasher(ids, 0, out=out)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    # a sleeping kernel holds the stream while the host queues every step, so
    # the events time the device work and not the Python call in front of it
    torch.cuda._sleep(int(2e7))
    t0 = time.perf_counter()
    for a, b in ev:
        a.record()
        hasher(ids, 0, out=out)
        b.record()
    host_us = (time.perf_counter() - t0) / args.steps * 1e6
    torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    per_tok = 8 + 4 + 2 * 24 * 8                     # ids read, cache write, ids of two layers written
    return {"component": "engram_hash", "metric": "hashed tokens/s", "value": w.M / (ms * 1e-3), "unit": "tokens/s",
            "ms_per_step": ms, "steps": args.steps, "warmup": args.warmup, "gbs": w.M * per_tok / (ms * 1e-3) / 1e9,
            "bytes_per_token": per_tok, "host_us_per_call": host_us, "config": {"workload": w.name, "B": w.B, "T": w.T, "n_layers": 2,
                                                   "orders": [2, 3, 4], "heads": 8}}


def _backbone(h, i, bw, w):
    return (h.view(-1, w.dim) @ bw[i]).view(h.shape)


def step_plain(layers, ids, x0, mask, bw, w):
    """One step with each Engram layer's forward inline (for the equality check)."""
    h = _backbone(x0, 0, bw, w)
    h = layers[0].forward(ids[0], h, mask)
    for i in range(1, 14):
        h = _backbone(h, i, bw, w)
    h = layers[1].forward(ids[1], h, mask)
    return _backbone(h, 14, bw, w)


def run_runahead(args, w):
    """Times the run-ahead schedule (EngramRunAhead) against the same step with
    each Engram layer's forward inline, around a backbone stand-in: two Engram
    layers at the V4.1 positions (layers 1 and 14), one bf16 [4M, 5120] x
    [5120, 5120] matmul (cuBLAS) for each of the 15 other layers up to layer
    15.  The stand-in only occupies the GPU the way dense layers would; it is
    not the model's backbone.  Both Engram layers share the workload's table
    (their gathers touch different rows); each has its own weight.  Prints
    one JSON line."""
    import numpy as np
    import torch
    from engram_hashed_gram_gb300 import build as B
    from engram_hashed_gram_gb300 import synth
    from engram_hashed_gram_gb300 import synth_device as SD
    from engram_hashed_gram_gb300.layer import EngramLayer, EngramRunAhead
    B.build()
    dev = torch.device("cuda", 0)
    M = w.M
    inp = synth.make_inputs(w)
    table, scale = SD.make_table(w, host=args.table_host)
    d = SD.upload_inputs(inp)
    w2 = dataclasses.replace(w, seed=w.seed + 100)
    wkv2 = SD.bits_to_device(synth.make_wkv(w2)) if w.wkv_fmt == 0 else None
    kw = dict(max_tokens=M, eps=w.eps, scale_block=w.scale_block, scale_fmt=w.scale_fmt, device=dev)
    if w.wkv_fmt == 0:
        layers = [EngramLayer(table, scale, d["wkv"], d["q"], d["k"], **kw),
                  EngramLayer(table, scale, wkv2, d["q"], d["k"], **kw)]
    else:
        c2, s2 = synth.make_wkv_mxfp8(w2)
        c2, s2 = torch.from_numpy(c2).to(dev), torch.from_numpy(s2).to(dev)
        layers = [EngramLayer(table, scale, d["wkv"], d["q"], d["k"], wkv_scale=d["wkv_scale"], **kw),
                  EngramLayer(table, scale, c2, d["q"], d["k"], wkv_scale=s2, **kw)]
    rng = np.random.default_rng([w.seed, 31])
    ids = [d["hash_ids"], torch.from_numpy(synth.make_hash_ids(w, rng=rng)).to(dev)]
    x0, mask = d["x"], d["mask"]
    g = torch.Generator(device=dev).manual_seed(5)
    bw = [torch.randn((w.dim, w.dim), device=dev, dtype=torch.bfloat16, generator=g) * (w.dim ** -0.5)
          for _ in range(15)]
    same = torch.equal(step_plain(layers, ids, x0, mask, bw, w).view(torch.int16),
                       step_plain(layers, ids, x0, mask, bw, w).view(torch.int16))
    budgets = [0, 0] if args.sm_budget is None else [int(v) for v in str(args.sm_budget).split(",")]
    if len(budgets) == 1:
        budgets = budgets * 2
    ra = EngramRunAhead(layers, max_tokens=M, sm_budget=budgets)
    flush = L2Flush(torch, dev)

    backbone = lambda h, i: _backbone(h, i, bw, w)

    def step_backbone():
        h = x0
        for i in range(15):
            h = backbone(h, i)
        return h

    def set_budget(per_layer):
        for lay, n in zip(layers, per_layer):
            lay.set_sm_budget(n)

    def step_serial():
        set_budget([0, 0])                 # inline: the projections take every SM
        h = backbone(x0, 0)
        h = layers[0].forward(ids[0], h, mask)
        for i in range(1, 14):
            h = backbone(h, i)
        h = layers[1].forward(ids[1], h, mask)
        return backbone(h, 14)

    def step_runahead():
        set_budget(budgets)
        ra.issue(ids)
        h = backbone(x0, 0)
        h = ra.apply(0, h, mask)
        for i in range(1, 14):
            h = backbone(h, i)
        h = ra.apply(1, h, mask)
        return backbone(h, 14)

    def timed(fns):
        """Median device ms of each step function, the three interleaved step
        by step so that clock and power drift hit them alike."""
        for _ in range(args.warmup):
            for fn in fns:
                fn()
        ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in fns]
              for _ in range(args.steps)]
        torch.cuda.synchronize()
        for row in ev:
            torch.cuda._sleep(int(2e6))         # the host queues the round ahead of the device
            for fn, (a, b) in zip(fns, row):
                flush()
                a.record()
                fn()
                b.record()
        torch.cuda.synchronize()
        return [statistics.median(row[j][0].elapsed_time(row[j][1]) for row in ev) for j in range(len(fns))]

    # the run-ahead result against the same step with each layer's forward inline
    # under the same projection plan (the budget fixes the split-K plan)
    ref = step_runahead()
    set_budget(budgets)
    same = same and torch.equal(step_plain(layers, ids, x0, mask, bw, w).view(torch.int16), ref.view(torch.int16))
    t_bb, t_serial, t_ra = timed([step_backbone, step_serial, step_runahead])
    set_budget(budgets)
    ra_plan = [list(lay.plan(M)) for lay in layers]
    for lay in layers:
        st, _ = lay.sync_status()
        if st != 0:
            raise RuntimeError(f"status {st}")
        lay.close()
    engram = t_serial - t_bb
    return {"component": "engram_runahead", "metric": "step ms with two Engram layers", "unit": "ms",
            "higher_is_better": False, "steps": args.steps, "warmup": args.warmup,
            "backbone_only_ms": t_bb, "serial_ms": t_serial, "runahead_ms": t_ra,
            "engram_inline_ms": engram, "engram_hidden_frac": (t_serial - t_ra) / engram if engram > 0 else None,
            "bitwise_equal": bool(same), "dtype": "bf16" if w.wkv_fmt == 0 else "mxfp8",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "engram_layers": [1, 14],
                       "engram_sm_budget": budgets, "engram_plan_runahead": ra_plan,
                       "backbone_stand_in": f"15 x bf16 [{4 * M}, {w.dim}] x [{w.dim}, {w.dim}] matmul",
                       "table_placement": "pinned host memory" if args.table_host else "device",
                       "l2": L2_NOTE}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-per-config", action="store_true",
                    help="measure the main workload only (no per_config list)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--component", choices=["layer", "hash", "runahead"], default="layer",
                    help="hash: time the n-gram hash (engram_hash) alone; runahead: two Engram layers run "
                         "ahead on a side stream vs inline, around a backbone stand-in; each prints its own "
                         "JSON line")
    ap.add_argument("--sm-budget", default=None,
                    help="runahead: cap the Engram projections at this many SMs (engram_set_sm_budget): one "
                         "count, or one per layer separated by commas (0 = all SMs)")
    ap.add_argument("--table-host", action="store_true",
                    help="keep the table and its scales in pinned host memory (the gather reads them over the "
                         "host link)")
    ap.add_argument("--fuse-gate", choices=["auto", "on", "off"], default="auto",
                    help="where the gate is formed (engram_config.fuse_gate): auto = the library's choice by batch "
                         "size, on = in the projection's epilogue, off = in a kernel of its own")
    ap.add_argument("--prime-base", type=int, default=None,
                    help="profiling only: build the table from the 24 primes above this base instead of the "
                         "workload's (the projection and gate kernels do the same work; the gather reads a "
                         "smaller table)")
    args = ap.parse_args()
    global ARGS
    ARGS = args
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    from engram_hashed_gram_gb300 import synth
    w = synth.workload(int(args.workload) if args.workload.isdigit() else args.workload)
    if args.prime_base is not None:
        w = dataclasses.replace(w, prime_base=args.prime_base, prime_skip=0)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.component == "hash":
        if rank == 0:
            print(json.dumps(run_hash(args, w)), flush=True)
        return
    if args.component == "runahead":
        if rank == 0:
            print(json.dumps(run_runahead(args, w)), flush=True)
        return

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, w)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    res = run_ours(args, w, rank, world, local_rank)
    if not args.no_per_config and args.workload == DEFAULT_WORKLOAD and args.prime_base is None:
        sub = argparse.Namespace(**dict(vars(args), cpu_seconds=min(args.cpu_seconds, PER_CONFIG_CPU_SECONDS)))
        res["per_config"] = [per_config_entry(run_ours(sub, synth.workload(name), rank, world, local_rank))
                             for name in PER_CONFIG]
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
