"""Benchmark of one paged-KV attention step on GB300.

A step is one pass of the hot path over one synthetic batch: the cache write
of this step's new K/V rows and the attention forward (split-KV decode +
combine, prefill, cascade as the batch needs), made through
paged_attn_forward_fused, which folds the cache write into the forward's
decode launch (the same bytes and results as reshape_and_cache followed by
paged_attn_forward; --two-call times that pair instead).  The headline workload is the decode-heavy batch: 128
decode requests, prior context ~ U[512, 8192], 32 query heads over 8 kv heads,
head_size 128, block_size 16, pages shuffled across the pool.  Its value is
KV bytes read per second (GB/s); its KV (about 2.3 GB) is far larger than L2,
so no flush is needed between steps.

Prints ONE JSON line (rank 0).  Flags:
  --gpus N --steps K --warmup W   (N > 1: launched by torchrun, one replica per GPU)
  --impl reference                the fp64 CPU oracle on a bounded sample, on the host cores
  --workload NAME                 another named workload (for profiling runs)
  --no-cpu-baseline               skip the oracle timing (profiling runs)
  --two-call                      write the cache with its own launch (reshape_and_cache)
  --no-fp8                        skip the fp8 e4m3 pool decode sub-measurement
  --no-workloads                  skip the other configurations' short timed runs
  --profile [--kv-dtype fp8]      short run for a profiler (optionally over an fp8 pool)
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_attention_33_gb300 import accounting as A  # noqa: E402
from paged_kv_attention_33_gb300 import workloads as W  # noqa: E402

METRIC = "paged-attn decode KV GB/s & prefill TFLOP/s, % of GB300 roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
SEED_OF = W.NAMED_SEEDS


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(PEAKS_FALLBACK), "fallback"


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(values, device):
    """Element-wise max of a list of floats over all ranks (identity at N=1).
    Each replica times its own work; the job's time is the slowest rank's."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock, power and throttle reasons."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str | None, interval_ms: int = 50):
        self.proc = None
        self.lines = []
        self.gpu_id = gpu_id
        self.interval_ms = interval_ms
        self.t_start = None

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=timestamp," + ",".join(self.FIELDS),
               "--format=csv,noheader,nounits", f"-lms={self.interval_ms}"]
        if self.gpu_id:
            cmd.append(f"--id={self.gpu_id}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
        self.t_start = time.time()

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        if self.proc is None or not self.lines:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        loaded = [x for x in sm if x > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_uuid(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# --------------------------------------------------------------------- workload
class Step:
    """Device-resident inputs of one workload and the call sequence of a step."""

    def __init__(self, name, dev, max_decodes=None):
        import dataclasses

        import torch

        import paged_kv_attention_33_gb300 as pka

        self.torch = torch
        self.pka = pka
        self.spec = W.named_spec(name)
        if max_decodes is not None:
            self.spec = dataclasses.replace(self.spec,
                                            decode_ctx=self.spec.decode_ctx[:max_decodes])
        self.name = name
        self.batch = W.make_batch(self.spec, seed=SEED_OF[name], device=dev)
        b = self.batch
        self.dev = dev
        self.slots = torch.from_numpy(b.slot_mapping).to(dev)
        self.meta = pka.Meta.from_host(b.query_start_loc, b.seq_lens, b.block_table,
                                       self.spec.num_decodes, dev,
                                       common_prefix_len=self.spec.common_prefix_len)
        T = b.num_tokens
        self.out = torch.empty((T, self.spec.num_heads, self.spec.head_size),
                               dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((T, self.spec.num_heads), dtype=torch.float32, device=dev)
        need = pka.workspace_size(self.meta, T, self.spec.num_heads, self.spec.num_kv_heads,
                                  self.spec.head_size, self.spec.block_size)
        self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)

    fused = True  # the cache write inside the forward (paged_attn_forward_fused)

    def run(self, q=None, k=None, v=None, slots=None, meta=None, out=None, lse=None):
        b = self.batch
        q = b.query if q is None else q
        k = b.key if k is None else k
        v = b.value if v is None else v
        slots = self.slots if slots is None else slots
        meta = self.meta if meta is None else meta
        out = self.out if out is None else out
        lse = self.lse if lse is None else lse
        if self.fused:
            self.pka.paged_attn_forward_fused(q, k, v, slots, b.cache, meta, out, lse,
                                              scale=self.spec.softmax_scale,
                                              causal=self.spec.causal, workspace=self.ws)
            return
        self.pka.reshape_and_cache(k, v, b.cache, slots)
        self.pka.paged_attn_forward(q, b.cache, meta, out, lse,
                                    scale=self.spec.softmax_scale, causal=self.spec.causal,
                                    workspace=self.ws)


def pack_buffers(torch, tensors, dev):
    """One pinned host byte buffer and one device byte buffer holding every
    tensor of `tensors` in 256-byte aligned regions (host contents copied in);
    returns (host, device, host views, device views) with the tensors' shapes."""
    offs, total = {}, 0
    for name, t in tensors.items():
        offs[name] = total
        total = (total + t.numel() * t.element_size() + 255) // 256 * 256
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    device = torch.empty(total, dtype=torch.uint8, device=dev)
    hv, dv = {}, {}
    for name, t in tensors.items():
        n = t.numel() * t.element_size()
        hv[name] = host[offs[name]:offs[name] + n].view(t.dtype).view(t.shape)
        dv[name] = device[offs[name]:offs[name] + n].view(t.dtype).view(t.shape)
        hv[name].copy_(t.detach().cpu())
    return host, device, hv, dv


def workload_config(name, spec):
    """The `config` keys that name the workload (shared by both arms)."""
    return {"workload": name, "num_decodes": spec.num_decodes,
            "num_prefills": len(spec.prefill), "num_heads": spec.num_heads,
            "num_kv_heads": spec.num_kv_heads, "head_size": spec.head_size,
            "block_size": spec.block_size,
            "kv_bytes_per_step": A.decode_kv_bytes(spec, spec.common_prefix_len)}


def units(spec):
    """(KV bytes, prefill flops) of one step."""
    return A.decode_kv_bytes(spec, spec.common_prefix_len), A.prefill_flops(spec)


# --------------------------------------------------------------------- reference arm
def oracle_sample_rows(batch, seqs):
    H = batch.spec.num_heads
    rows = []
    for s in seqs:
        t0, t1 = int(batch.query_start_loc[s]), int(batch.query_start_loc[s + 1])
        for t in range(t0, t1):
            rows.extend(range(t * H, (t + 1) * H))
    return np.asarray(rows, dtype=np.int64)


class OracleStep:
    """The workload's batch on the host, its new rows written by the oracle
    (set-up, untimed), for timing the oracle's attention."""

    def __init__(self, name):
        from oracle import Oracle

        self.name = name
        self.spec = W.named_spec(name)
        self.batch = W.make_batch(self.spec, seed=SEED_OF[name], device="cpu")
        self.oracle = Oracle()
        b = self.batch
        self.oracle.reshape_and_cache(b.key, b.value, b.cache, b.slot_mapping)


def time_oracle(name, seqs, threads, prepared=None):
    """Oracle on the whole heads of `seqs` of the workload; returns
    (seconds, KV bytes those sequences read, sample description)."""
    st = prepared or OracleStep(name)
    spec, b, orc, cache = st.spec, st.batch, st.oracle, st.batch.cache
    rows = oracle_sample_rows(b, seqs)
    t0 = time.perf_counter()
    orc.paged_attention(b.query, cache, b.query_start_loc, b.seq_lens, b.block_table,
                        spec.softmax_scale, spec.causal, rows=rows, threads=threads)
    dt = time.perf_counter() - t0
    row_bytes = spec.num_kv_heads * spec.head_size * 2 * 2
    nbytes = sum(int(b.seq_lens[s]) for s in seqs) * row_bytes
    return dt, nbytes, f"{name}: sequences {seqs[0]}..{seqs[-1]} ({len(seqs)} of " \
                       f"{len(b.seq_lens)}), all {spec.num_heads} heads, fp64"


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle

    threads = oracle.cpu_threads()
    name = args.workload
    spec = W.named_spec(name)
    # every sequence of the workload per step (decode_heavy: about 0.4 s on 16
    # host cores); the batch is drawn once, before the timed steps
    per_step = list(range(spec.num_decodes)) if spec.num_decodes else [0]
    prepared = OracleStep(name)
    times = []
    nbytes = 0
    for i in range(args.warmup + args.steps):
        dt, nb, desc = time_oracle(name, per_step, threads, prepared)
        if i >= args.warmup:
            times.append(dt)
            nbytes = nb
    sec = sum(times) / len(times)
    value = nbytes / sec / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {**workload_config(name, spec), "sample_per_step": desc,
                   "parallelism": f"fp64 oracle on {threads} host threads"},
        "impl": "reference",
        "cpu_baseline": {"kind": "oracle", "cores": threads, "sample": desc, "value": value,
                         "unit": "GB/s"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------- our arm
KERNEL_SOURCES = {"decode": ("decode.cu", "common.cuh"),
                  "prefill": ("prefill.cu", "common.cuh", "tcgen05.cuh")}


def code_only(text):
    """C/C++/CUDA source with comments removed and whitespace runs collapsed
    (string and character literals kept as written): what the compiler sees,
    so that editing a comment does not change a kernel's key."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(kernel="decode"):
    """Key of a kernel's code (its source files, comments and whitespace aside)."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "paged_kv_attention_33_gb300", "csrc", f)) as fh:
            h.update(code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def committed_traffic(workload, kv_dtype="bf16", kernel="decode"):
    """Per-launch DRAM bytes of the kernel from the committed ncu summary, or
    None when the kernel source changed since it was taken."""
    suffix = "" if kv_dtype == "bf16" else f"_{kv_dtype}"
    path = os.path.join(ROOT, "profiles", f"{kernel}_kernel_{workload}{suffix}_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("kernel_source_hash") != kernel_source_hash(kernel):
        return None
    return rec.get("traffic_bytes_per_launch")


def run_ours(args):
    import torch

    import paged_kv_attention_33_gb300 as pka

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device(dev))
    pka.load_library()
    peaks, peaks_kind = load_peaks()
    st = Step(args.workload, dev, args.max_decodes)
    spec = st.spec
    if args.profile:
        if args.kv_dtype == "fp8":
            to_fp8_pool(st)
        return run_profile(args, st)
    kv_bytes, pf_flops = units(spec)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    # warm-up (at least W steps, and at least ~1 s so that clocks settle)
    t_end = time.time() + 1.0
    n = 0
    while n < args.warmup or time.time() < t_end:
        st.run()
        n += 1
        if n % 50 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    pka.check_status()

    # timed region: K steps, per-step events around the decode kernel
    ev_k0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_k1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for e in ev_k0 + ev_k1:
        e.record(stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_uuid(torch, local))
    sampler.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    # the step time: K plain steps (no event records between the launches,
    # which would cost host time and break a dependent launch's overlap)
    launches0 = pka.kernel_launches()
    e0.record(stream)
    for i in range(args.steps):
        st.run()
    e1.record(stream)
    launches = pka.kernel_launches() - launches0
    torch.cuda.synchronize()
    barrier()
    ms = e0.elapsed_time(e1) / args.steps
    # the dominant kernel's time: K more steps, the library recording events
    # around the decode kernel on its stream
    for i in range(args.steps):
        pka.set_kernel_events(pka.KERNEL_DECODE, ev_k0[i], ev_k1[i])
        st.run()
    pka.set_kernel_events(pka.KERNEL_DECODE, None, None)
    torch.cuda.synchronize()
    k_ms = sum(a.elapsed_time(b) for a, b in zip(ev_k0, ev_k1)) / args.steps
    # clocks: keep loading the GPU for ~1 s more so that nvidia-smi sees it busy
    t_end = time.time() + 1.0
    while time.time() < t_end:
        for _ in range(20):
            st.run()
        torch.cuda.synchronize()
    sampler.stop()
    pka.check_status()
    ms, k_ms = max_over_ranks([ms, k_ms], dev)
    value = world * kv_bytes / (ms * 1e-3) / 1e9

    # end to end through the public API with host buffers: every step's inputs
    # (q, k, v, slot mapping, metadata) staged in one pinned buffer and copied in
    # one H2D copy, out and lse read back in one D2H copy; the library gets views.
    # As a serving loop runs it: two staging and two result buffers, the H2D and
    # the D2H copies each on a stream of their own, so that step i+1's inputs
    # arrive and step i-1's results leave while step i attends.
    b = st.batch
    parts = {
        "q": b.query.cpu(), "k": b.key.cpu(), "v": b.value.cpu(),
        "slots": torch.from_numpy(b.slot_mapping),
        "qsl": torch.from_numpy(b.query_start_loc),
        "sl": torch.from_numpy(b.seq_lens),
        "bt": torch.from_numpy(np.ascontiguousarray(b.block_table)),
    }
    bufs = []
    for _ in range(2):
        h_stage, d_stage, _, d_views = pack_buffers(torch, parts, dev)
        h_ret, d_ret, h_outs, d_outs = pack_buffers(torch, {"out": torch.zeros_like(st.out),
                                                       "lse": torch.zeros_like(st.lse)}, dev)
        meta_e2e = pka.Meta(d_views["qsl"], d_views["sl"], d_views["bt"], st.meta.num_decodes,
                            st.meta.max_query_len, st.meta.max_seq_len,
                            st.meta.common_prefix_len)
        bufs.append((h_stage, d_stage, d_views, h_ret, d_ret, d_outs, meta_e2e, h_outs))
    h2d = bufs[0][0].numel()
    d2h = bufs[0][3].numel()
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of buffer j copied in
    ev_done = [torch.cuda.Event() for _ in range(2)]  # step on buffer j finished
    ev_out = [torch.cuda.Event() for _ in range(2)]   # results of buffer j copied out

    def h2d_into(j):
        h_stage, d_stage = bufs[j][0], bufs[j][1]
        h2d_stream.wait_event(ev_done[j])  # the step that last read buffer j is done
        with torch.cuda.stream(h2d_stream):
            d_stage.copy_(h_stage, non_blocking=True)
        ev_in[j].record(h2d_stream)

    def e2e_steps(n, start):
        """n steps; `start` (an event on the compute stream) precedes the first copy."""
        h2d_stream.wait_event(start)
        h2d_into(0)
        for i in range(n):
            j = i & 1
            if i + 1 < n:
                h2d_into(1 - j)
            _, _, d_views, h_ret, d_ret, d_outs, meta_e2e, _ = bufs[j]
            stream.wait_event(ev_in[j])
            stream.wait_event(ev_out[j])  # buffer j's previous results have left
            st.run(q=d_views["q"], k=d_views["k"], v=d_views["v"], slots=d_views["slots"],
                   meta=meta_e2e, out=d_outs["out"], lse=d_outs["lse"])
            ev_done[j].record(stream)
            d2h_stream.wait_event(ev_done[j])
            with torch.cuda.stream(d2h_stream):
                h_ret.copy_(d_ret, non_blocking=True)
            ev_out[j].record(d2h_stream)
        stream.wait_stream(d2h_stream)  # the last results are back

    for e in ev_done + ev_out:
        e.record(stream)
    w0 = torch.cuda.Event()
    w0.record(stream)
    e2e_steps(max(3, args.warmup), w0)
    torch.cuda.synchronize()
    barrier()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    e2e_steps(args.steps, f0)
    f1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = max_over_ranks([f0.elapsed_time(f1) / args.steps], dev)[0]
    pka.check_status()
    # what came back to the host is the device-timed step's result, byte for byte
    want = {"out": st.out.cpu(), "lse": st.lse.cpu()}
    used = [0] if args.steps == 1 else [0, 1]
    e2e_same = all(torch.equal(bufs[j][7][n].view(torch.uint8), want[n].view(torch.uint8))
                   for j in used for n in want)

    # roofline of the dominant kernel (the split-KV decode kernel)
    achieved = kv_bytes / (k_ms * 1e-3) / 1e9
    peak = float(peaks["hbm_gbs"])
    roofline = {"bound": "hbm", "kernel": "paged_decode_kernel", "achieved": achieved,
                "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": f"{peaks_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                if peaks_kind == "measured" else "fallback 6.8 TB/s",
                "frac_of_nominal_8tbs": achieved / 8000.0,
                "kernel_ms": k_ms, "algorithmic_bytes_per_launch": kv_bytes,
                "traffic": committed_traffic(args.workload)}

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {**workload_config(args.workload, spec),
                   "l2": "inputs larger than L2 (KV per step >> 129 MB), no flush",
                   "step_calls": "paged_attn_forward_fused" if Step.fused
                   else "reshape_and_cache + paged_attn_forward",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "roofline": roofline,
        "e2e": {"value": world * kv_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": "every step: one H2D of its inputs from pinned memory and one D2H "
                          "of out and lse, on an H2D and a D2H stream with two buffers each "
                          "way, overlapping the neighbouring steps' attention",
                "results_equal_device_step": e2e_same},
        "gpu_launches": launches,
        "clocks": sampler.summary(),
        "timed_region": "CUDA events on the launching stream around K plain steps; the decode "
                        "kernel timed per launch in K more steps, with events recorded by the "
                        "library around it",
    }
    if pf_flops:
        line["prefill_tflops"] = pf_flops / (ms * 1e-3) / 1e12
    if args.workload == "decode_heavy" and not args.no_fp8:
        # the fp8 e4m3 pool: half the bytes of the same batch
        del st
        torch.cuda.empty_cache()
        line["fp8_decode"] = measure_fp8_decode(args, dev, peaks, peaks_kind)
        st = None
    if args.workload != "prefill" and not args.no_prefill:
        # the metric's second half: prefill TFLOP/s on the varlen prefill workload
        # (8 prompts, 1024..8192 tokens), timed in the same run
        del st
        torch.cuda.empty_cache()
        line["prefill"] = measure_prefill(args, dev, peaks, peaks_kind)
    if args.workload == "decode_heavy" and not args.no_workloads:
        line["workloads"] = measure_workloads(args, dev, peaks)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle

        threads = oracle.cpu_threads()
        seqs = list(range(spec.num_decodes)) if spec.num_decodes else [0]
        dt, nb, desc = time_oracle(args.workload, seqs, threads)
        line["cpu_baseline"] = {"value": nb / dt / 1e9, "unit": "GB/s", "cores": threads,
                                "kind": "oracle", "sample": desc, "seconds": dt}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def to_fp8_pool(st):
    """Replace the step's bf16 pool by its e4m3 quantisation (every slot written
    by the library's reshape_and_cache_fp8; per-tensor scales 4/448, i.e. |x| up
    to 4 sigma of the N(0, 1) rows is representable) and switch its metadata to
    the fp8 pool."""
    import torch

    pka, sp, b = st.pka, st.spec, st.batch
    k_scale = v_scale = 4.0 / 448
    pool8 = torch.zeros((b.cache.shape[0], 2, sp.block_size, sp.num_kv_heads, sp.head_size),
                        dtype=torch.uint8, device=b.cache.device)
    rows_k = b.cache[:, 0].reshape(-1, sp.num_kv_heads, sp.head_size).contiguous()
    rows_v = b.cache[:, 1].reshape(-1, sp.num_kv_heads, sp.head_size).contiguous()
    every_slot = torch.arange(rows_k.shape[0], dtype=torch.int64, device=b.cache.device)
    pka.reshape_and_cache_fp8(rows_k, rows_v, pool8, every_slot, k_scale, v_scale)
    del rows_k, rows_v, every_slot
    b.cache = pool8
    st.meta.kv_dtype, st.meta.k_scale, st.meta.v_scale = pka.KV_FP8_E4M3, k_scale, v_scale
    # prefills over an fp8 pool need the workspace for the bf16 copy of their blocks
    need = pka.workspace_size(st.meta, b.num_tokens, sp.num_heads, sp.num_kv_heads,
                              sp.head_size, sp.block_size)
    if need > st.ws.numel():
        st.ws = torch.empty(need, dtype=torch.uint8, device=b.cache.device)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def measure_fp8_decode(args, dev, peaks, peaks_kind):
    """The headline decode batch over an fp8 e4m3 pool (one byte per element,
    per-tensor scales): the same fused step (the new rows quantised into the
    pool inside the decode launch), its step and kernel time and the fp8 KV
    bytes per second against the copy roofline.  The pool is the bf16 pool's
    context quantised by the library's own reshape_and_cache_fp8 (setup, not
    timed)."""
    import torch

    import paged_kv_attention_33_gb300 as pka

    st = Step("decode_heavy", dev, args.max_decodes)
    to_fp8_pool(st)
    kv_bytes = A.decode_kv_bytes(st.spec, 0, elem_bytes=1)
    for _ in range(max(3, args.warmup)):
        st.run()
    torch.cuda.synchronize()
    steps = max(5, min(args.steps, 200))
    k0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    k1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for e in k0 + k1:
        e.record()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        pka.set_kernel_events(pka.KERNEL_DECODE, k0[i], k1[i])
        st.run()
    pka.set_kernel_events(pka.KERNEL_DECODE, None, None)
    e1.record()
    torch.cuda.synchronize()
    pka.check_status()
    ms, k_ms = max_over_ranks([e0.elapsed_time(e1) / steps,
                               sum(a.elapsed_time(c) for a, c in zip(k0, k1)) / steps], dev)
    peak = float(peaks["hbm_gbs"])
    achieved = kv_bytes / (k_ms * 1e-3) / 1e9
    return {"workload": "decode_heavy", "kv_dtype": "fp8_e4m3", "steps": steps,
            "kv_bytes_per_step": kv_bytes, "ms_per_step": ms,
            "GBps": kv_bytes / (ms * 1e-3) / 1e9,
            "roofline": {"bound": "hbm", "kernel": "paged_decode_kernel (fp8)",
                         "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "kernel_ms": k_ms,
                         "peak_source": f"{peaks_kind} copy bandwidth (hbm_gbs)",
                         "algorithmic_bytes_per_launch": kv_bytes,
                         "traffic": committed_traffic("decode_heavy", "fp8")}}


def timed_steps(torch, pka, st, steps, kernels=(0, 1), run=None):
    """Mean step time and mean per-launch kernel times (CUDA events; the library
    records the decode (0) and prefill (1) kernels' events on their stream).
    The step time comes from a loop without the per-kernel events (their
    records cost host time between launches); the kernel times from a second,
    instrumented loop."""
    run = st.run if run is None else run
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        run()
    e1.record()
    torch.cuda.synchronize()
    pka.check_status()
    ms = e0.elapsed_time(e1) / steps
    ev = {k: ([torch.cuda.Event(enable_timing=True) for _ in range(steps)],
              [torch.cuda.Event(enable_timing=True) for _ in range(steps)]) for k in kernels}
    for a, b in ev.values():
        for e in a + b:
            e.record()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        for k, (a, b) in ev.items():
            pka.set_kernel_events(k, a[i], b[i])
        run()
    for k in ev:
        pka.set_kernel_events(k, None, None)
    e1.record()
    torch.cuda.synchronize()
    pka.check_status()
    kms = {k: sum(x.elapsed_time(y) for x, y in zip(a, b)) / steps for k, (a, b) in ev.items()}
    return ms, kms


def graph_step_ms(torch, st, steps):
    """Mean step time when the step is captured once in a CUDA graph and
    replayed (how a serving loop removes the per-launch host overhead)."""
    st.run()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            st.run()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    st.pka.check_status()
    return e0.elapsed_time(e1) / steps


def measure_workloads(args, dev, peaks):
    """The other configurations of the method, one short timed run each (20 steps
    after 3 warm-ups, CUDA events): tiny_decode (latency), mixed (decode GB/s and
    prefill TFLOP/s against their peaks), cascade (suffix GB/s and the
    naive-equivalent GB/s), and decode_heavy's cache write and attention timed
    separately (two calls) beside the fused step."""
    import torch

    import paged_kv_attention_33_gb300 as pka

    hbm = float(peaks["hbm_gbs"])
    tf = float(peaks.get("bf16_tflops", PEAKS_FALLBACK["bf16_tflops"]))
    res = {}
    st = Step("tiny_decode", dev)
    ms, kms = timed_steps(torch, pka, st, 20)
    res["tiny_decode"] = {"ms_per_step": ms, "decode_kernel_ms": kms[0],
                          "bound": "latency (0.2 MB of KV)",
                          "graph_replay_ms_per_step": graph_step_ms(torch, st, 20)}
    del st
    st = Step("mixed", dev)
    kv, fl = units(st.spec)

    def mixed_entry(ms, kms, kv_bytes):
        # the step's roofline: the decode bytes at the copy bandwidth plus the
        # prefill flops at the bf16 peak (the two passes may run side by side)
        roof_ms = (kv_bytes / (hbm * 1e9) + fl / (tf * 1e12)) * 1e3
        e = {"ms_per_step": ms, "summed_roofline_ms": roof_ms,
             "frac_of_summed_roofline": roof_ms / ms,
             "kv_bytes_per_step": kv_bytes, "prefill_flops_per_step": fl}
        if abs(kms[0] - kms[1]) <= 0.05 * max(kms.values()):
            # side by side: the library's two timing brackets both span the pair
            e.update({"decode_and_prefill_passes_ms": kms[0],
                      "passes": "side by side (the decode on part of the SMs, the prefill "
                                "pass on the rest and then on all)"})
        else:
            e.update({"decode_kernel_ms": kms[0], "prefill_kernel_ms": kms[1],
                      "decode_GBps": kv_bytes / (kms[0] * 1e-3) / 1e9,
                      "decode_frac_of_hbm": kv_bytes / (kms[0] * 1e-3) / 1e9 / hbm,
                      "prefill_TFLOPs": fl / (kms[1] * 1e-3) / 1e12,
                      "prefill_frac_of_bf16": fl / (kms[1] * 1e-3) / 1e12 / tf})
        return e

    ms, kms = timed_steps(torch, pka, st, 20)
    res["mixed"] = mixed_entry(ms, kms, kv)
    del st
    torch.cuda.empty_cache()
    # the same batch over an fp8 pool (the prefills run on a bf16 copy of their blocks)
    st = Step("mixed", dev)
    to_fp8_pool(st)
    kv8 = A.decode_kv_bytes(st.spec, 0, elem_bytes=1)
    ms, kms = timed_steps(torch, pka, st, 20)
    res["mixed_fp8"] = mixed_entry(ms, kms, kv8)
    res["mixed_fp8"]["note"] = "step includes the copy of the prefill blocks to bf16"
    del st
    torch.cuda.empty_cache()
    st = Step("cascade", dev)
    kv, _ = units(st.spec)
    sp = st.spec
    naive, casc = A.cascade_prefix_token_reads(
        sp.num_decodes, sp.common_prefix_len,
        [L - sp.common_prefix_len for L in sp.seq_lens[: sp.num_decodes]])
    row = sp.num_kv_heads * sp.head_size * 2 * 2
    # the step's roofline: the suffix bytes at the copy bandwidth plus the
    # shared-prefix pass's flops (4*D per head and (token, prefix key) pair)
    # at the bf16 peak
    pre_flops = 4 * sp.head_size * sp.num_heads * st.batch.num_tokens * sp.common_prefix_len

    def cascade_entry(ms, kms, kv_bytes):
        roof_ms = (kv_bytes / (hbm * 1e9) + pre_flops / (tf * 1e12)) * 1e3
        # (side by side, both brackets span the pair of passes; one after the
        # other, they bracket a short prefix pass and a long decode)
        side_by_side = abs(kms[0] - kms[1]) <= 0.05 * max(kms.values())
        e = {"ms_per_step": ms, "summed_roofline_ms": roof_ms,
             "frac_of_summed_roofline": roof_ms / ms, "prefix_flops": pre_flops,
             "kv_bytes_suffix": kv_bytes}
        if side_by_side:
            # the prefix pass and the suffix decode run at the same time on
            # disjoint SMs: the library's two timing brackets span the pair
            e["prefix_and_suffix_passes_ms"] = kms[0]
            e["passes"] = "side by side (prefix pass on part of the SMs, suffix decode on the rest)"
        else:
            e["decode_kernel_ms"] = kms[0]
            e["prefix_pass_ms"] = kms[1]
            e["passes"] = "one after the other"
        return e

    def graph_ms():
        try:
            return graph_step_ms(torch, st, 20)
        except Exception as e:  # reported, not fatal: the eager step stands
            return f"capture failed: {e}"

    ms, kms = timed_steps(torch, pka, st, 20)
    res["cascade"] = {**cascade_entry(ms, kms, kv), "graph_replay_ms_per_step": graph_ms(),
                      "cascade_GBps_step": casc * row / (ms * 1e-3) / 1e9,
                      "naive_equivalent_GBps_step": naive * row / (ms * 1e-3) / 1e9,
                      "bytes_read_cascade": casc * row, "bytes_read_naive": naive * row}
    # the same over an fp8 pool (the prefix pass runs on a bf16 copy of its blocks)
    to_fp8_pool(st)
    ms, kms = timed_steps(torch, pka, st, 20)
    res["cascade_fp8"] = {**cascade_entry(ms, kms, kv // 2), "graph_replay_ms_per_step": graph_ms(),
                          "note": "step includes the copy of the prefix blocks to bf16"}
    del st
    torch.cuda.empty_cache()
    st = Step("decode_heavy", dev)
    kv, _ = units(st.spec)
    b = st.batch
    ms_w, _ = timed_steps(torch, pka, st, 20, kernels=(),
                          run=lambda: pka.reshape_and_cache(b.key, b.value, b.cache, st.slots))
    Step.fused = False
    try:
        ms2, kms2 = timed_steps(torch, pka, st, 20, kernels=(0,))
    finally:
        Step.fused = not args.two_call
    res["decode_heavy_two_call"] = {"reshape_and_cache_ms": ms_w, "step_ms": ms2,
                                    "decode_kernel_ms": kms2[0],
                                    "decode_frac_of_hbm": kv / (kms2[0] * 1e-3) / 1e9 / hbm}
    del st
    torch.cuda.empty_cache()
    return res


def measure_prefill(args, dev, peaks, peaks_kind):
    """Prefill workload: step and kernel time (CUDA events on the launching
    stream, the kernel bracketed by the library), TFLOP/s and the fraction of
    the measured dense bf16 peak (burst: the kernel is timed on its own)."""
    import torch

    import paged_kv_attention_33_gb300 as pka

    st = Step("prefill", dev)
    _, flops = units(st.spec)
    for _ in range(max(3, args.warmup)):
        st.run()
    torch.cuda.synchronize()
    steps = max(5, min(args.steps, 50))
    k0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    k1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for e in k0 + k1:
        e.record()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        pka.set_kernel_events(pka.KERNEL_PREFILL, k0[i], k1[i])
        st.run()
    pka.set_kernel_events(pka.KERNEL_PREFILL, None, None)
    e1.record()
    torch.cuda.synchronize()
    pka.check_status()
    ms, k_ms = max_over_ranks([e0.elapsed_time(e1) / steps,
                               sum(a.elapsed_time(b) for a, b in zip(k0, k1)) / steps], dev)
    peak = float(peaks.get("bf16_tflops", PEAKS_FALLBACK["bf16_tflops"]))
    achieved = flops / (k_ms * 1e-3) / 1e12
    return {"workload": "prefill", "steps": steps, "flops_per_step": flops,
            "ms_per_step": ms, "tflops": flops / (ms * 1e-3) / 1e12,
            "roofline": {"bound": "tensor", "kernel": "prefill_tc_kernel", "achieved": achieved,
                         "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                         "peak_source": f"{peaks_kind} dense bf16 burst (bf16_tflops)",
                         "kernel_ms": k_ms,
                         "traffic": committed_traffic("prefill", kernel="prefill")},
            "note": "the step includes the copy of the prompts' keys into 128-key blocks "
                    "(16-key pool pages) that the prefill kernel reads"}


def run_profile(args, st):
    """Short run for profilers: W warm-up steps and K steps, no clock sampler,
    no host-buffer leg, no oracle."""
    import torch

    for _ in range(args.warmup):
        st.run()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        st.run()
    e1.record()
    torch.cuda.synchronize()
    st.pka.check_status()
    ms = e0.elapsed_time(e1) / args.steps
    kv_bytes, flops = units(st.spec)
    if args.kv_dtype == "fp8":
        kv_bytes //= 2
    print(json.dumps({"profile_run": True, "workload": args.workload, "kv_dtype": args.kv_dtype,
                      "num_decodes": st.spec.num_decodes, "ms_per_step": ms,
                      "kv_bytes_per_step": kv_bytes, "prefill_flops_per_step": flops,
                      "GBps_step": kv_bytes / (ms * 1e-3) / 1e9,
                      "TFLOPs_step": flops / (ms * 1e-3) / 1e12}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="pka", choices=["pka", "reference"])
    ap.add_argument("--workload", default="decode_heavy", choices=list(W.NAMED))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the prefill sub-measurement")
    ap.add_argument("--no-fp8", action="store_true",
                    help="skip the fp8-pool decode sub-measurement")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other configurations' short timed runs")
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "fp8"],
                    help="pool element type of --profile runs (fp8: decode workloads)")
    ap.add_argument("--profile", action="store_true",
                    help="short run for a profiler: W + K steps only")
    ap.add_argument("--max-decodes", type=int, default=None,
                    help="keep only the first N decode requests (small profiling case)")
    ap.add_argument("--two-call", action="store_true",
                    help="reshape_and_cache and paged_attn_forward as two calls")
    args = ap.parse_args()
    if args.two_call:
        Step.fused = False
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
