"""Benchmark of unified paged attention on GB300 (one JSON line on rank 0).

Headline (`value`): decode KV GB/s of pa_forward on the Llama-3.1-8B-shaped
GQA decode at batch 64 (32 q heads, 8 KV heads, head_dim 128, block_size 16,
contexts uniform on [500, 8192], bf16): one step = one pa_forward call over
the whole batch (planner, row-streaming kernel, log-sum-exp merge); bytes =
the K and V bytes of every visible position, inputs resident in HBM and far
larger than L2 (~1.1 GB of KV per step, L2 is 129 MB).

The same run also measures, per step with an L2 flush between steps:
batch-1 decode at context 500, the Qwen3-235B-shaped mixed batch (TFLOPS),
the 128K chunked long-context batch and the absorbed MLA decode.  The flush
writes a 256 MB buffer and then reads another: the read evicts the written
lines, so their write-back happens before the timed call instead of inside
its first large kernel.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the fp64 CPU oracle on the same workload (a bounded
sample per step) as the reference arm.  Multi-GPU: N independent replicas
(weak scaling, no data-path collective); the timed region is bracketed by a
barrier and the max over ranks is reported.
"""
import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_attention_16_gb300 import inputs  # noqa: E402

# Measured DRAM traffic per launch (ncu dram__bytes_read.sum +
# dram__bytes_write.sum) is kept in a data file written by
# `bench.py --record-traffic`, keyed by kernel, workload and a hash of the
# kernel's source files: a kernel changed since its capture reads as null.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")
CSRC = os.path.join(ROOT, "paged_kv_attention_16_gb300", "csrc")
KERNEL_SOURCES = {
    "row_mma_kernel": ["pa_rows_mma.cu", "pa_common.cuh"],
    "tile_kernel": ["pa_tile.cu", "pa_common.cuh"],
    "mla_kernel": ["pa_mla.cu", "pa_common.cuh"],
    "upproj_kernel": ["pa_upproj.cu", "pa_common.cuh"],
}

METRIC = "decode KV GB/s (% of HBM peak); mixed-batch attention TFLOPS (% of peak)"
WORKLOAD = ("llama-3.1-8b-shaped GQA decode: batch 64, ctx uniform [500, 8192], 32 q heads, "
            "8 kv heads, head_dim 128, block_size 16, bf16, random page placement")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def source_sha(kernel):
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def read_traffic_file():
    rows = {}
    if os.path.exists(TRAFFIC_FILE):
        with open(TRAFFIC_FILE) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 5 and not line.startswith("#"):
                    rows[(parts[0], parts[1])] = (parts[2], int(parts[3]), int(parts[4]))
    return rows


def recorded_traffic(kernel, workload):
    """DRAM bytes read + written per launch from the last capture of this
    kernel on this workload, or None if the kernel changed since."""
    row = read_traffic_file().get((kernel, workload))
    if row is None or row[0] != source_sha(kernel):
        return None
    return row[1] + row[2]


def record_traffic(csv_path, kernel, workload):
    """Write the DRAM counters of an `ncu -i REP --page raw --csv` dump (the
    first launch of `kernel` in it) into the traffic file."""
    import csv
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12}
    with open(csv_path) as f:
        rows = list(csv.reader(f))
    hdr, units = rows[0], rows[1]
    ci = {n: i for i, n in enumerate(hdr)}
    data = [r for r in rows[2:] if kernel in r[ci["Kernel Name"]]]
    if not data:
        raise SystemExit(f"no launch of {kernel} in {csv_path}")
    vals = []
    for m in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
        vals.append(int(round(float(data[0][ci[m]].replace(",", "")) * scale[units[ci[m]]])))
    table = read_traffic_file()
    table[(kernel, workload)] = (source_sha(kernel), vals[0], vals[1])
    with open(TRAFFIC_FILE, "w") as f:
        f.write("# kernel workload source_sha16 dram_bytes_read dram_bytes_write "
                "(per launch, ncu; written by bench.py --record-traffic)\n")
        for (k, w), (sha, r, wr) in sorted(table.items()):
            f.write(f"{k} {w} {sha} {r} {wr}\n")
    print(f"{kernel} {workload}: read {vals[0]} write {vals[1]}")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def _plain(o):
    """JSON fallback for numpy scalars."""
    if isinstance(o, np.generic):
        return o.item()
    raise TypeError(f"not JSON serialisable: {type(o).__name__}")


def kv_bytes(b, window=0):
    """K and V bytes a step must read: every position some row of its request
    sees (with a sliding window, from the first row's window start on)."""
    es = b.k_cache.element_size()
    ctx = b.seq_lens.to(torch.int64)
    qsl = b.query_start_loc.to(torch.int64)
    q_len = qsl[1:] - qsl[:-1]
    if window:
        first = (ctx - q_len - window + 1).clamp(min=0)
        ctx = ctx - first
    ctx = torch.where(q_len > 0, ctx, torch.zeros_like(ctx))  # no rows, nothing read
    return int(ctx.sum()) * b.num_kv_heads * b.head_dim * es * 2


def io_bytes(b):
    return 2 * b.q.numel() * b.q.element_size()


def attn_flops(b, window=0):
    """4 * head_dim flops (QK and PV multiply-adds) per visible (row, key)
    pair; row i of a request sees pre + i + 1 keys, at most `window`."""
    qsl = b.query_start_loc.numpy().astype(np.int64)
    ctx = b.seq_lens.numpy().astype(np.int64)
    total = 0
    for s in range(b.num_seqs):
        ql = qsl[s + 1] - qsl[s]
        pre = ctx[s] - ql
        if window:
            seen = np.minimum(pre + np.arange(ql, dtype=np.int64) + 1, window)
            total += int(seen.sum())
        else:
            # sum over i < ql of (pre + i + 1)
            total += ql * pre + ql * (ql + 1) // 2
    return 4 * b.head_dim * b.num_heads * total


def mla_bytes(m):
    return int(m.seq_lens.to(torch.int64).sum()) * (m.kv_lora_rank + m.rope_dim) * 2


def mla_flops(m):
    return int(m.seq_lens.to(torch.int64).sum()) * m.num_heads * 2 * (
        2 * m.kv_lora_rank + m.rope_dim)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.samples = []
        self.proc = None
        self.sel = []
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            self.sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            self.sel = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", *self.sel, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()

    def summary(self, t0, t1):
        rows = [s for t, s in self.samples if t0 - 0.15 <= t <= t1 + 0.15] or \
               [s for _, s in self.samples]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [x.strip() for x in r.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:  # the multi-process path exercised on CPU: gloo
            dist.init_process_group("gloo")
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class L2Flush:
    """Between timed calls: write a buffer larger than L2 (129 MB), then read
    a second one.  After the write alone, L2 holds up to 129 MB of dirty lines
    that the next kernel's misses write back to HBM (measured: the long-context
    decode rows 64.1 us against 52.0 us after write + read, the mixed batch's
    rows 165 us against 156 us); the read leaves L2 clean and still cold for
    the call."""

    def __init__(self, nbytes=256 << 20):
        self.w = torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")
        self.r = torch.zeros(nbytes // 4, dtype=torch.float32, device="cuda")

    def __call__(self):
        self.w.zero_()
        self.r.sum()


def time_per_step(fn, steps, flush, settle=False):
    """Median device time of `steps` calls, each timed with events on the
    current stream, with an L2 flush (L2Flush, outside the events) between
    calls.
    settle: the device also spins for about 0.25 ms after the flush, so the
    host has enqueued the whole call before the device reaches it (per-kernel
    event brackets then hold device time only, not the host's launch work)."""
    st = torch.cuda.current_stream()
    times = []
    for _ in range(steps):
        flush()
        if settle:
            torch.cuda._sleep(500_000)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        fn()
        b.record(st)
        b.synchronize()
        times.append(a.elapsed_time(b))
    return statistics.median(times)


def plain_and_profiled(pa, fn, steps, flush):
    """(median ms per step without per-kernel events, {kernel: mean ms} from a
    second pass with CUDA events around every launch)."""
    ms = time_per_step(fn, steps, flush)
    pa.pa_profile_enable(True)
    pa.pa_profile_read()
    time_per_step(fn, steps, flush, settle=True)
    prof = pa.pa_profile_read()
    pa.pa_profile_enable(False)
    return ms, {k: v[0] / v[1] for k, v in prof.items()}


def graph_step_ms(pa, b, out, per_graph=20, reps=10):
    """Median device time of one pa_forward step when `per_graph` steps are
    captured in one CUDA graph and the graph is replayed (workspace reserved
    beforehand, as capture requires)."""
    dt = pa.PA_BF16 if b.q.dtype == torch.bfloat16 else pa.PA_F32
    pa.pa_reserve(pa.pa_forward_workspace_bytes(dt, b.num_seqs, b.num_tokens, b.num_heads,
                                                b.num_kv_heads, b.head_dim, b.max_seq_len,
                                                b.kv_split_tokens))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pa.forward(b, out=out, stream=s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(per_graph):
                pa.forward(b, out=out, stream=s)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        g.replay()
        e1.record(st)
        e1.synchronize()
        times.append(e0.elapsed_time(e1) / per_graph)
    return statistics.median(times)


def secondary_workloads(pa, flush, peaks):
    """Per-workload device times (median over steps, L2 flushed between)."""
    res = {}
    hbm = peaks["hbm_gbs"]
    tfl = peaks["bf16_tflops"]

    hb = inputs.llama_decode(1, poison=False)
    b = pa.to_device(hb)
    out = torch.empty_like(b.q)
    # declared decode-only (max_query_len = 1, as the headline): one launch
    fn1 = lambda: pa.forward(b, out=out, max_query_len=1)  # noqa: E731
    for _ in range(5):
        fn1()
    ms = time_per_step(fn1, 50, flush)
    gbs = kv_bytes(hb) / ms / 1e6
    res["llama_decode_b1"] = {"ms": ms, "kv_gbs": gbs, "hbm_frac": gbs / hbm,
                              "note": "2 MB of KV: latency bound; pa_forward_ex with "
                                      "max_query_len = 1, one kernel launch per call; "
                                      "L2 flushed before each call"}
    # the same calls back to back (the host enqueues while the device runs):
    # per-call time of a stream of single-step calls, caches warm
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(st)
    for _ in range(200):
        fn1()
    e1.record(st)
    e1.synchronize()
    res["llama_decode_b1"]["back_to_back_ms"] = e0.elapsed_time(e1) / 200
    # the same call without the declaration: planner, row and merge launches
    fn0 = lambda: pa.forward(b, out=out)  # noqa: E731
    for _ in range(5):
        fn0()
    ms0 = time_per_step(fn0, 50, flush)
    res["llama_decode_b1"]["undeclared"] = {"ms": ms0, "kv_gbs": kv_bytes(hb) / ms0 / 1e6,
                                            "note": "max_query_len = 0: planned path"}
    try:  # the undeclared step replayed from a CUDA graph (20 steps per graph)
        gms = graph_step_ms(pa, b, out)
        res["llama_decode_b1"]["graph_replay"] = {"ms": gms, "kv_gbs": kv_bytes(hb) / gms / 1e6}
    except Exception as e:  # report, never abort the benchmark
        res["llama_decode_b1"]["graph_replay"] = {"error": str(e)[:200]}
    del b, out

    # the headline decode batch with NHD and with head-major (HND) caches
    # (one (page, kv head) run of 16 slots is one contiguous 4 KB box), timed
    # the same way as the headline (back-to-back steps, KV >> L2, no flush),
    # alternating layouts over 5 rounds; median ms per step of each
    hn = inputs.llama_decode(64, poison=False)
    runs = {}
    for name, h in (("nhd", hn), ("hnd", inputs.as_hnd(hn))):
        d = pa.to_device(h)
        o = torch.empty_like(d.q)
        pa.forward(d, out=o, max_query_len=1)
        runs[name] = (d, o)
    per = {"nhd": [], "hnd": []}
    st = torch.cuda.current_stream()
    for _ in range(5):
        for name, (d, o) in runs.items():
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(st)
            for _ in range(100):
                pa.forward(d, out=o, max_query_len=1)
            e1.record(st)
            e1.synchronize()
            per[name].append(e0.elapsed_time(e1) / 100)
    lay = {}
    for name in ("nhd", "hnd"):
        ms = statistics.median(per[name])
        gbs = kv_bytes(hn) / ms / 1e6
        lay[name] = {"ms": ms, "kv_gbs": gbs, "hbm_frac": gbs / hbm}
    lay["hnd_over_nhd"] = lay["nhd"]["ms"] / lay["hnd"]["ms"]
    res["llama_decode_b64_layouts"] = lay
    del runs

    hb = inputs.mixed_qwen3(poison=False)
    b = pa.to_device(hb)
    out = torch.empty_like(b.q)
    pa.forward(b, out=out)
    ms, kms = plain_and_profiled(pa, lambda: pa.forward(b, out=out), 5, flush)
    tf = attn_flops(hb) / ms / 1e9
    res["mixed_qwen3"] = {"ms": ms, "tflops": tf, "tensor_frac": tf / tfl,
                          "kv_gbs": kv_bytes(hb) / ms / 1e6,
                          "tokens": hb.num_tokens, "requests": hb.num_seqs,
                          "kernel_ms": kms}
    del b, out

    # the model variants on the decode batch and the mixed batch: sinks, a
    # sliding window (GB/s and TFLOPS count only what the window leaves
    # visible), ALiBi and sqrt ALiBi; median of 5 rounds of 50 back-to-back
    # steps, inputs larger than L2
    var = {}
    st = torch.cuda.current_stream()
    for wl, maker in (("llama_decode_b64", lambda: inputs.llama_decode(64, poison=False)),
                      ("mixed_qwen3", lambda: inputs.mixed_qwen3(poison=False))):
        hb = maker()
        b = pa.to_device(hb)
        out = torch.empty_like(b.q)
        H = hb.num_heads
        g = torch.Generator().manual_seed(11)
        sk = torch.randn(H, generator=g).cuda()
        al = (2.0 ** (-8.0 * torch.arange(1, H + 1, dtype=torch.float32) / H)).cuda()
        cases = {"plain": {}, "sinks": dict(sinks=sk), "window_128": dict(sliding_window=128),
                 "window_1024": dict(sliding_window=1024), "alibi": dict(alibi_slopes=al),
                 "alibi_sqrt": dict(alibi_slopes=al, alibi_sqrt=True)}
        res_wl = {}
        for name, kw in cases.items():
            fn = lambda: pa.forward(b, out=out, **kw)  # noqa: E731
            fn()
            per = []
            for _ in range(5):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                e0.record(st)
                for _ in range(50):
                    fn()
                e1.record(st)
                e1.synchronize()
                per.append(e0.elapsed_time(e1) / 50)
            ms = statistics.median(per)
            w = kw.get("sliding_window", 0)
            gbs = kv_bytes(hb, w) / ms / 1e6
            tf = attn_flops(hb, w) / ms / 1e9
            res_wl[name] = {"ms": ms, "kv_gbs": gbs, "hbm_frac": gbs / hbm, "tflops": tf,
                            "tensor_frac": tf / tfl}
        var[wl] = res_wl
        del b, out
    res["variants"] = var

    hb = inputs.long_chunked(poison=False)
    b = pa.to_device(hb)
    out = torch.empty_like(b.q)
    pa.forward(b, out=out)
    ms, kms = plain_and_profiled(pa, lambda: pa.forward(b, out=out), 5, flush)
    tf = attn_flops(hb) / ms / 1e9
    res["long_chunked"] = {"ms": ms, "tflops": tf, "tensor_frac": tf / tfl,
                           "kv_split_tokens": 32768,
                           "kernel_ms": kms}
    del b, out

    hm = inputs.mla_decode_batch(poison=False)
    m = pa.to_device(hm)
    out = torch.empty((m.num_seqs, m.num_heads, m.kv_lora_rank), dtype=torch.bfloat16,
                      device="cuda")
    st = pa.pa_mla_decode(m.q, m.kv_cache, m.block_table, m.seq_lens, m.num_heads,
                          m.kv_lora_rank, m.rope_dim, m.block_size, m.scale, out,
                          max_seq_len=m.max_seq_len, check=False)
    if st == pa.PA_OK:
        ms = time_per_step(lambda: pa.mla_decode(m, out=out), 10, flush)
        gbs = mla_bytes(hm) / ms / 1e6
        tf = mla_flops(hm) / ms / 1e9
        # the roofline floor is the larger of the HBM time and the tensor time
        floor_ms = max(mla_bytes(hm) / hbm / 1e6, mla_flops(hm) / tfl / 1e9)
        res["mla_decode"] = {"ms": ms, "kv_gbs": gbs, "hbm_frac": gbs / hbm, "tflops": tf,
                             "tensor_frac": tf / tfl, "roofline_floor_ms": floor_ms,
                             "roofline_frac": floor_ms / ms}
    else:
        res["mla_decode"] = {"unavailable": pa.status_string(st)}
    del m, out

    # non-absorbed MLA prefill / extend: decompression (the up-projection
    # GEMM over every cached position) plus causal attention with 192-wide keys
    hp = inputs.mla_prefill_deepseek(poison=False)
    mp = pa.to_device(hp)
    outp = torch.empty((hp.num_tokens, hp.num_heads, hp.v_head_dim), dtype=torch.bfloat16,
                       device="cuda")
    st = pa.pa_mla_prefill(mp.q, mp.kv_cache, mp.w_kv, mp.block_table, mp.seq_lens,
                           mp.query_start_loc, hp.num_heads, hp.kv_lora_rank, hp.qk_nope_dim,
                           hp.rope_dim, hp.v_head_dim, hp.block_size, hp.scale, outp,
                           max_seq_len=hp.max_seq_len, max_total_kv=hp.max_total_kv,
                           check=False)
    if st == pa.PA_OK:
        ms, kms = plain_and_profiled(pa, lambda: pa.mla_prefill(mp, out=outp), 10, flush)
        ctx = hp.seq_lens.numpy().astype(np.int64)
        qsl = hp.query_start_loc.numpy().astype(np.int64)
        pairs = 0
        for s_ in range(hp.num_seqs):
            ql = qsl[s_ + 1] - qsl[s_]
            pairs += ql * (ctx[s_] - ql) + ql * (ql + 1) // 2
        att = int(pairs) * hp.num_heads * 2 * (hp.qk_nope_dim + hp.rope_dim + hp.v_head_dim)
        up = int(ctx.sum()) * hp.num_heads * 2 * hp.kv_lora_rank * (hp.qk_nope_dim + hp.v_head_dim)
        tf = (att + up) / ms / 1e9
        res["mla_prefill"] = {"ms": ms, "tflops": tf, "tensor_frac": tf / tfl,
                              "attention_flops": att, "up_projection_flops": up,
                              "tokens": hp.num_tokens, "kv_positions": int(ctx.sum()),
                              "kernel_ms": kms}
        if "tile" in kms:
            res["mla_prefill"]["tile_tflops"] = att / kms["tile"] / 1e9
        if "upproj" in kms:
            up_tf = up / kms["upproj"] / 1e9
            res["mla_prefill"]["upproj_tflops"] = up_tf
            res["mla_prefill"]["upproj_tensor_frac"] = up_tf / tfl
    else:
        res["mla_prefill"] = {"unavailable": pa.status_string(st)}
    del mp, outp

    # KV-cache write of a prefill-sized step: 16 requests x 512 new tokens
    # (Llama-3.1-8B shapes); bytes = K and V rows read and written
    hb = inputs.paged_batch([512] * 16, [1024 + 256 * i for i in range(16)], 32, 8, 128, 16,
                            dtype="bf16", seed=5, poison=False)
    b = pa.to_device(hb)
    g = torch.Generator().manual_seed(5)
    k_new = torch.randn((hb.num_tokens, 8, 128), generator=g).to(torch.bfloat16).cuda()
    v_new = torch.randn((hb.num_tokens, 8, 128), generator=g).to(torch.bfloat16).cuda()
    wr = lambda: pa.pa_cache_write(k_new, v_new, b.k_cache, b.v_cache, b.block_table,  # noqa: E731
                                   b.seq_lens, b.query_start_loc, hb.block_size)
    wr()
    ms = time_per_step(wr, 50, flush)
    nbytes = 2 * 2 * k_new.numel() * k_new.element_size()
    res["cache_write"] = {"ms": ms, "gbs": nbytes / ms / 1e6, "hbm_frac": nbytes / ms / 1e6 / hbm,
                          "tokens": hb.num_tokens, "bytes": nbytes}
    return res


def oracle_step_fn(host):
    """One CPU-baseline step: the fp64 oracle, as it stands, over every row
    of the whole decode batch (64 requests x 32 heads) in one call.  Returns
    (step function, KV bytes per step)."""
    from oracle import oracle as orc
    q = inputs.storage_array(host.q)
    kc = inputs.storage_array(host.k_cache)
    vc = inputs.storage_array(host.v_cache)
    bt, sl, qsl = host.block_table.numpy(), host.seq_lens.numpy(), host.query_start_loc.numpy()

    def step():
        orc.paged_attention(q, kc, vc, bt, sl, qsl, host.num_heads, host.num_kv_heads,
                            host.head_dim, host.block_size, host.scale)

    return step, kv_bytes(host)


CPU_SAMPLE = "each step: the whole batch (64 requests x 32 heads, one oracle call)"


def cpu_baseline_subprocess(steps=4, warmup=1):
    """The reference arm's own measurement, run as a fresh process (no CUDA
    context, no torch thread pools beside the oracle's), on the same sample:
    the repo arm's cpu_baseline.  Timing the oracle inside the GPU process
    measured several times slower than the same call in a fresh process."""
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", str(steps), "--warmup", str(warmup)],
                       capture_output=True, text=True, env=env, cwd=ROOT, timeout=900)
    line = [x for x in r.stdout.splitlines() if x.startswith("{")]
    if r.returncode != 0 or not line:
        return {"error": (r.stderr or r.stdout)[-300:]}
    ref = json.loads(line[-1])
    cb = dict(ref["cpu_baseline"])
    cb["sample"] += f"; {steps} timed steps in a fresh process"
    return cb


def run_ours(args):
    world, rank, local = dist_setup()
    from paged_kv_attention_16_gb300 import build as pbuild
    pbuild.build()
    from paged_kv_attention_16_gb300 import pa
    peaks, peak_src = load_peaks()
    dev = torch.cuda.current_device()

    host = inputs.llama_decode(64, poison=False)
    b = pa.to_device(host)
    out = torch.empty_like(b.q)
    step_kv = kv_bytes(b)
    step_io = io_bytes(b)

    for _ in range(max(args.warmup, 3)):
        pa.forward(b, out=out, max_query_len=1)
    torch.cuda.synchronize()

    clocks = ClockSampler(dev)
    clocks.start()
    time.sleep(0.3)
    stream = torch.cuda.current_stream()
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        pa.forward(b, out=out, max_query_len=1)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t_wall1 = time.time()
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), world)

    # Per-kernel device times: the same K steps again, with CUDA events
    # around every launch on the launching stream.  The events serialise the
    # launches (no programmatic overlap), so this pass is slower than the
    # one above; it gives the roofline kernel's own duration.
    pa.pa_profile_enable(True)
    pa.pa_profile_read()
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(args.steps):
        pa.forward(b, out=out, max_query_len=1)
    ev1.record(stream)
    torch.cuda.synchronize()
    pa.pa_profile_enable(False)
    prof = pa.pa_profile_read()
    ms_profiled = ev0.elapsed_time(ev1)
    time.sleep(0.2)
    clocks.stop()
    ms_step = ms_total / args.steps
    value = step_kv * args.steps * world / (ms_total / 1e3) / 1e9

    launches = sum(n for _, n in prof.values())  # same launches as the timed region
    row_ms, row_n = prof.get("row", (0.0, 1))
    row_avg = row_ms / max(row_n, 1)
    achieved = (step_kv + step_io) / (row_avg / 1e3) / 1e9
    hbm = peaks["hbm_gbs"]
    kernel_share = {k: round(v[0] / max(sum(x[0] for x in prof.values()), 1e-9), 4)
                    for k, v in prof.items()}

    # ---- end to end through the C ABI with host buffers ---------------------
    # The step's inputs (q and the three metadata arrays) live in one pinned
    # host buffer and one device buffer (256-byte aligned views), so each
    # step is one host-to-device copy, pa_forward, one device-to-host copy.
    parts = [host.q, host.block_table, host.seq_lens, host.query_start_loc]
    offs, off = [], 0
    for t in parts:
        offs.append(off)
        off = (off + t.numel() * t.element_size() + 255) // 256 * 256
    stage_h = torch.empty(off, dtype=torch.uint8).pin_memory()
    stage_d = torch.empty(off, dtype=torch.uint8, device="cuda")

    def view(buf, t, o):
        return buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)

    for t, o in zip(parts, offs):
        view(stage_h, t, o).copy_(t)
    be = dataclasses.replace(b, q=view(stage_d, host.q, offs[0]),
                             block_table=view(stage_d, host.block_table, offs[1]),
                             seq_lens=view(stage_d, host.seq_lens, offs[2]),
                             query_start_loc=view(stage_d, host.query_start_loc, offs[3]))
    out_h = torch.empty(host.q.shape, dtype=host.q.dtype).pin_memory()
    e2e_steps = min(args.steps, 200)

    def e2e_step():
        stage_d.copy_(stage_h, non_blocking=True)
        pa.forward(be, out=out, max_query_len=1)
        out_h.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    barrier(world)
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(ev0.elapsed_time(ev1), world) / e2e_steps
    h2d = stage_h.numel()
    d2h = out_h.numel() * out_h.element_size()

    secondary = {}
    if not args.skip_secondary:
        flush = L2Flush()
        secondary = secondary_workloads(pa, flush, peaks)
        del flush

    if rank != 0:
        return
    cpu = cpu_baseline_subprocess() if not args.skip_cpu else None
    clk = clocks.summary(t_wall0, t_wall1)
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) values, seeded page placement; no weights needed)",
        "config": workload_config(step_kv, world),
        "hbm_frac": value / hbm,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm,
                     "traffic": recorded_traffic("row_mma_kernel", "llama_decode_b64"),
                     "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)",
                     "kernel": "row_mma_kernel<128,4> (bf16 decode rows, warp MMAs)",
                     "kernel_ms": row_avg, "bytes_per_launch": step_kv + step_io,
                     "kernel_timing": "CUDA events around each launch, second pass of the "
                                      f"same {args.steps} steps ({ms_profiled / args.steps:.4f} "
                                      "ms per step with the events)",
                     "peak_source": f"{peak_src} hbm_gbs (copy read+write)"},
        "kernel_share": kernel_share,
        "gpu_launches": launches,
        "e2e": {"value": step_kv / (e2e_ms / 1e3) / 1e9 * world, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "note": "per step: q + block_table + seq_lens + query_start_loc copied from "
                        "one pinned host staging buffer in one copy, pa_forward, out copied "
                        "back; the KV cache is resident state"},
        "clocks": clk,
        "workloads": secondary,
        "cpu_baseline": cpu,
        "peaks": {"hbm_gbs": hbm, "bf16_tflops": peaks["bf16_tflops"], "source": peak_src},
    }
    print(json.dumps(line, default=_plain))


# ---------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores
# ---------------------------------------------------------------------------

def workload_config(step_kv, world=1):
    return {"workload": WORKLOAD, "batch": 64, "kv_bytes_per_step": step_kv,
            "call": "pa_forward_ex with max_query_len = 1 (a decode-only batch, as a "
                    "serving scheduler declares it)",
            "l2": "inputs larger than L2 (KV per step >> 129 MB); no flush",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import oracle as orc
    host = inputs.llama_decode(64, poison=False)
    step, nbytes = oracle_step_fn(host)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = nbytes * args.steps / dt / 1e9
    cores = orc.num_threads()
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) values, seeded page placement; no weights needed)",
        "config": workload_config(nbytes),
        "cpu_baseline": {"kind": "oracle", "cores": cores, "value": value, "unit": "GB/s",
                         "sample": CPU_SAMPLE,
                         "cores_source": "omp_get_max_threads() of the oracle library"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}))


def run_only(args):
    """A plain loop over one workload (for profiler captures): W warm-up
    calls then K timed calls; prints one JSON line with the mean time."""
    torch.cuda.set_device(0)
    from paged_kv_attention_16_gb300 import build as pbuild
    pbuild.build()
    from paged_kv_attention_16_gb300 import pa
    name = args.only
    if name == "mla_decode":
        host = inputs.mla_decode_batch(poison=False)
        m = pa.to_device(host)
        out = torch.empty((m.num_seqs, m.num_heads, m.kv_lora_rank), dtype=torch.bfloat16,
                          device="cuda")
        fn = lambda: pa.mla_decode(m, out=out)  # noqa: E731
    elif name == "mla_prefill":
        host = inputs.mla_prefill_deepseek(poison=False)
        m = pa.to_device(host)
        out = torch.empty((host.num_tokens, host.num_heads, host.v_head_dim),
                          dtype=torch.bfloat16, device="cuda")
        fn = lambda: pa.mla_prefill(m, out=out)  # noqa: E731
    else:
        host = inputs.WORKLOADS[name](poison=False)
        b = pa.to_device(host)
        out = torch.empty_like(b.q)
        # decode batches are declared decode-only, as the headline calls them
        mql = 1 if name.startswith("llama_decode") else 0
        fn = lambda: pa.forward(b, out=out, max_query_len=mql)  # noqa: E731
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for _ in range(args.steps):
        fn()
    ev1.record()
    torch.cuda.synchronize()
    print(json.dumps({"only": name, "steps": args.steps,
                      "ms_per_step": ev0.elapsed_time(ev1) / max(args.steps, 1)}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--skip-secondary", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--only", default=None,
                    choices=sorted(list(inputs.WORKLOADS) + ["mla_decode"]),
                    help="profile helper: loop over a single workload, no JSON contract")
    ap.add_argument("--record-traffic", nargs=3, metavar=("NCU_RAW_CSV", "KERNEL", "WORKLOAD"),
                    help="store a capture's DRAM bytes per launch for the roofline line")
    args = ap.parse_args()
    if args.record_traffic:
        record_traffic(*args.record_traffic)
    elif args.only:
        run_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
