"""Benchmark one decode step (append + paged decode attention) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                    [--impl native|reference]

A step is one layer's decode step over one batch: pkv_kv_append of each
sequence's newest K/V row, then pkv_paged_decode_attention over all cached
tokens.  Inputs are seeded synthetic tensors of the workload's shapes,
resident in HBM before the timed region.  The timed region is K steps
captured in one CUDA graph, bracketed by a barrier and a synchronize, timed
with CUDA events on the launching stream.  L2 hygiene: the steps rotate over
enough copies of the cache pool that each step reads pages no other step
touched within the last (R-1) steps (total footprint >= 4x the 129 MB L2).

Printed (rank 0, one JSON line): value = algorithmic bytes per step / step
time in GB/s; tokens/s per layer; the dominant kernel's roofline against the
measured HBM copy bandwidth; an end-to-end figure through the same C ABI with
the step's inputs copied from pinned host memory and the output read back
inside the timed region; the CPU oracle timed on a bounded sample; SM clocks
sampled during the timed region.

Multi-GPU: the decode path has no exchange step, so N ranks run N independent
replicas of the workload (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import itertools
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import paged_kv_cache_250_gb300 as pkv  # noqa: E402
from paged_kv_cache_250_gb300 import workloads as wl  # noqa: E402

DEFAULT_CONFIG = "llama3_8b_b32_ctx1-4096_bf16"
METRIC = "decode-attention achieved HBM GB/s (% of GB300 peak) and tokens/s per layer"
L2_BYTES = 129 * 1024 * 1024
PEAK_FALLBACK_GBS = 6800.0
_CODE = {"f16": pkv.PKV_F16, "bf16": pkv.PKV_BF16, "e4m3": pkv.PKV_FP8_E4M3,
         "e4m3tok": pkv.PKV_FP8_E4M3_TOKEN}
_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


# ---------------------------------------------------------------- helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time (replicas run in lockstep between barriers)."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbps(bytes_per_rank_step: int, ms_per_step: float, world: int) -> float:
    """Throughput of all ranks together: each moves its own step's bytes."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return PEAK_FALLBACK_GBS, "fallback"


def measured_tensor_peak():
    """Dense bf16 tensor peak: the burst figure (a kernel timed alone)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = [l for (t, l) in self.lines if t0 - 0.05 <= t <= t1 + 0.05] or \
            [l for (_, l) in self.lines]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def workload_config(cfg, ctx: torch.Tensor) -> dict:
    """The workload keys both arms report in `config`."""
    return {"workload": cfg.name, "batch": cfg.batch, "q_heads": cfg.q_heads,
            "kv_heads": cfg.kv_heads, "head_dim": cfg.head_dim, "page_size": wl.PAGE,
            "cache_dtype": cfg.cache, "total_context_tokens": int(ctx.sum())}


def algorithmic_bytes(cfg, ctx: torch.Tensor):
    """Bytes the step must move (read or write) at minimum.

    attention: every cached K and V element once, q, the output, the block-
    table entries used and the context lengths (+ the FP8 scales);
    append: the new K/V rows read and written, and the slot mapping."""
    B, Hq, Hkv, d = cfg.batch, cfg.q_heads, cfg.kv_heads, cfg.head_dim
    e_c = cfg.cache_elem_bytes
    e_q = 2
    e_out = 2
    ctx64 = ctx.to(torch.int64)
    pages = int(((ctx64 + wl.PAGE - 1) // wl.PAGE).sum())
    attn = int(ctx64.sum()) * Hkv * d * 2 * e_c + B * Hq * d * (e_q + e_out) + pages * 4 + 4 * B
    if cfg.cache == "e4m3":
        attn += 8 * Hkv
    append = B * Hkv * d * 2 * (2 + e_c) + 8 * B
    if cfg.cache == "e4m3tok":  # a K and a V scale per token and KV head, read and written
        attn += int(ctx64.sum()) * Hkv * 8
        append += B * Hkv * 8
    return attn, append


# ---------------------------------------------------------------- native arm
class Step:
    """Device state of one workload: R pool replicas, inputs, outputs."""

    def __init__(self, cfg, device, replicas: int, hint: int):
        self.cfg = cfg
        self.dev = device
        w = wl.generate(cfg, device=device)
        self.w = w
        self.hint = hint
        self.q = w.q.contiguous()
        self.k_new = w.k_new.contiguous()
        self.v_new = w.v_new.contiguous()
        self.slot = w.slot_mapping.to(device)
        self.tables = w.block_tables.to(device)
        self.ctx = w.ctx.to(device)
        self.k_scale = None if w.k_scale is None else w.k_scale.float().contiguous()
        self.v_scale = None if w.v_scale is None else w.v_scale.float().contiguous()
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.kc = [w.k_cache] + [w.k_cache.clone() for _ in range(replicas - 1)]
        self.vc = [w.v_cache] + [w.v_cache.clone() for _ in range(replicas - 1)]
        self.desc = pkv.make_desc(w.num_blocks, wl.PAGE, cfg.kv_heads, cfg.q_heads,
                                  cfg.head_dim, _CODE[cfg.cache], self.k_scale, self.v_scale,
                                  self.err)
        n = pkv.pkv_decode_workspace_bytes(self.desc, cfg.batch, w.max_blocks_per_seq, hint)
        self.ws = torch.zeros(n, dtype=torch.uint8, device=device)
        self.out = torch.empty(cfg.batch, cfg.q_heads, cfg.head_dim, dtype=torch.bfloat16
                               if cfg.cache != "f16" else torch.float16, device=device)
        # the K/V inputs of the per-head K/V projections are what drives the bytes
        self.R = replicas

    def append(self, r, stream):
        pkv.pkv_kv_append(self.desc, self.kc[r], self.vc[r], self.slot, self.k_new, self.v_new,
                          stream=stream)

    def decode(self, r, stream):
        pkv.pkv_paged_decode_attention(self.desc, self.q, self.kc[r], self.vc[r], self.tables,
                                       self.ctx, self.cfg.softmax_scale, self.out, self.ws,
                                       self.hint, stream=stream)

    def step_one(self, r, stream, overlap=True):
        """The whole step in one kernel: pkv_decode_step_fused.  With overlap
        (PKV_STEP_OVERLAP) it lays out its work while the previous step ends:
        lengths and tables are written by no kernel here."""
        pkv.pkv_decode_step_fused(self.desc, self.q, self.kc[r], self.vc[r], self.k_new,
                                  self.v_new, self.tables, self.ctx, self.cfg.softmax_scale,
                                  self.out, self.ws, self.hint, stream=stream, overlap=overlap)

    def step(self, r, stream):
        """The whole step as two kernels through pkv_decode_step."""
        pkv.pkv_decode_step(self.desc, self.q, self.kc[r], self.vc[r], self.slot, self.k_new,
                            self.v_new, self.tables, self.ctx, self.cfg.softmax_scale,
                            self.out, self.ws, self.hint, stream=stream)


class Staging:
    """A step's host inputs packed at 256-byte aligned offsets of one pinned
    buffer, with a device twin: one copy moves them all, and the step reads
    device views into the twin (the layout a caller staging its inputs would
    use)."""

    def __init__(self, tensors, device):
        offs, total = [], 0
        for t in tensors:
            offs.append(total)
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        self.host = torch.empty(total, dtype=torch.uint8).pin_memory()
        self.dev = torch.empty(total, dtype=torch.uint8, device=device)
        self.views = []
        self.payload_bytes = 0
        for t, o in zip(tensors, offs):
            n = t.numel() * t.element_size()
            self.payload_bytes += n
            self.host[o:o + n].copy_(t.detach().contiguous().view(-1).view(torch.uint8).cpu())
            self.views.append(self.dev[o:o + n].view(t.dtype).view(t.shape))


def capture(fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def run_native(args, cfg, rank, world, device):
    stream = torch.cuda.Stream(device)
    hint = {"llama3_8b_b32_ctx1-4096_bf16": 4096}.get(cfg.name, 0)
    # replicas: enough pool copies that the rotation spans >= 4x L2
    with torch.cuda.stream(stream):
        probe = Step(cfg, device, 1, hint)
    pool_bytes = probe.kc[0].numel() * probe.kc[0].element_size() * 2
    R = max(1, min(8, -(-4 * L2_BYTES // pool_bytes)))
    del probe
    torch.cuda.empty_cache()
    with torch.cuda.stream(stream):
        st = Step(cfg, device, R, hint)
    torch.cuda.synchronize(device)
    attn_bytes, append_bytes = algorithmic_bytes(cfg, st.w.ctx)
    step_bytes = attn_bytes + append_bytes
    K, W = args.steps, args.warmup

    # warm-up (also sets kernel attributes before capture)
    for i in range(W):
        st.step_one(i % R, stream)
        st.step_one(i % R, stream, overlap=False)
        st.step(i % R, stream)
        st.append(i % R, stream)
        st.decode(i % R, stream)
    stream.synchronize()

    # graph of K steps, events between the two calls of each step
    ev = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(3)]
          for _ in range(K)]

    def body_events():
        for i in range(K):
            ev[i][0].record(stream)
            st.append(i % R, stream)
            ev[i][1].record(stream)
            st.decode(i % R, stream)
            ev[i][2].record(stream)

    def body_plain():
        for i in range(K):
            st.step_one(i % R, stream)

    def body_two():
        for i in range(K):
            st.step(i % R, stream)

    def body_one_no_overlap():
        for i in range(K):
            st.step_one(i % R, stream, overlap=False)

    def body_warm():  # every step on replica 0: what the L2 kept of it is read again
        for i in range(K):
            st.step_one(0, stream)

    g_plain = capture(body_plain, stream)
    g_two = capture(body_two, stream)
    g_one_plain = capture(body_one_no_overlap, stream)
    g_warm = capture(body_warm, stream)
    g_events = capture(body_events, stream)

    # e2e: every step copies its inputs (q, new k/v, tables, lengths) in from
    # pinned host memory, packed in one staging buffer (one copy), runs the
    # step on views into it, and copies its output back.  Staging and outputs
    # are double-buffered and the copies run on their own streams, so step
    # i + 1's inputs and step i - 1's output move while step i computes.
    stages = [Staging([st.q, st.k_new, st.v_new, st.tables, st.ctx], device) for _ in range(2)]
    outs = [torch.empty_like(st.out) for _ in range(2)]
    h_outs = [torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory() for _ in range(2)]
    h2d = stages[0].host.numel()  # the bytes copied (inputs plus alignment padding)
    d2h = h_outs[0].numel() * h_outs[0].element_size()
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def body_e2e():
        ev_in = [torch.cuda.Event() for _ in range(K)]
        ev_k = [torch.cuda.Event() for _ in range(K)]
        ev_out = [torch.cuda.Event() for _ in range(K)]
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for i in range(K):
            bb = i % 2
            if i >= 2:
                s_in.wait_event(ev_k[i - 2])      # step i - 2 read this staging buffer
            with torch.cuda.stream(s_in):
                stages[bb].dev.copy_(stages[bb].host, non_blocking=True)
                ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])  # step i - 2's output has left
            sq, sk, sv, stab, sctx = stages[bb].views
            pkv.pkv_decode_step_fused(st.desc, sq, st.kc[i % R], st.vc[i % R], sk, sv, stab, sctx,
                                      cfg.softmax_scale, outs[bb], st.ws, st.hint, stream=stream,
                                      overlap=True)
            ev_k[i].record(stream)
            s_out.wait_event(ev_k[i])
            with torch.cuda.stream(s_out):
                h_outs[bb].copy_(outs[bb], non_blocking=True)
                ev_out[i].record(s_out)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    g_e2e = capture(body_e2e, stream)
    torch.cuda.synchronize(device)

    def timed(graph):
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            graph.replay()  # replays on the current stream, i.e. `stream`
            e1.record(stream)
        torch.cuda.synchronize(device)
        if world > 1:
            torch.distributed.barrier()
        return max_over_ranks(e0.elapsed_time(e1), world, device)

    with torch.cuda.stream(stream):
        g_plain.replay()  # graph warm-up
    torch.cuda.synchronize(device)
    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    t0 = time.time()
    ms_total = timed(g_plain)
    t1 = time.time()
    time.sleep(0.15)
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    ms_events = timed(g_events)
    ms_two = timed(g_two)
    ms_one_plain = timed(g_one_plain)
    with torch.cuda.stream(stream):
        g_warm.replay()  # leave replica 0's last-read pages in L2
    ms_warm = timed(g_warm)
    # host copies vary from replay to replay (one replay in several runs
    # 20-30% slower): the median of three replays
    ms_e2e = statistics.median(timed(g_e2e) for _ in range(3))
    err = int(st.err.item())
    if err != 0:
        raise RuntimeError(f"device error word {err} ({pkv.pkv_status_string(err)})")

    append_ms = statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for i in range(K))
    decode_ms = statistics.mean(ev[i][1].elapsed_time(ev[i][2]) for i in range(K))
    ms_step = ms_total / K
    value = whole_job_gbps(step_bytes, ms_step, world)
    peak, peak_kind = measured_peak()
    # the step is one kernel: its average launch time is the step time
    achieved = step_bytes / (ms_step * 1e-3) / 1e9
    traffic = committed_traffic(cfg.name)
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"bf16": "bf16", "f16": "f16", "e4m3": "e4m3", "e4m3tok": "e4m3"}[cfg.cache],
        "data": "synthetic (seeded N(0,1) q/k/v, uniform ragged context lengths, "
                "permuted block tables)",
        "config": {**workload_config(cfg, st.w.ctx),
                   "l2": f"rotating {R} cache-pool copies ({R * pool_bytes / 1e6:.0f} MB, "
                         f">= 4x L2); every step reads cold pages",
                   "timing": "K steps in one CUDA graph, CUDA events on the launch stream",
                   "step": "pkv_decode_step_fused, PKV_STEP_OVERLAP (lengths and tables "
                           "ready before the previous step ends)",
                   "parallelism": f"replicas x{world} (no data-path collective)"},
        "percent_of_peak": round(100 * value / world / peak, 1),
        "tokens_per_s_per_layer": round(world * cfg.batch / (ms_step * 1e-3), 1),
        "warm_l2": {"value": round(whole_job_gbps(step_bytes, ms_warm / K, world), 1),
                    "unit": "GB/s", "ms_per_step": round(ms_warm / K, 5),
                    "method": "the timed step, every step on the same cache-pool copy (the "
                              f"pool is {pool_bytes / 1e6:.0f} MB against a "
                              f"{L2_BYTES / 1e6:.0f} MB L2), so what the L2 kept of the "
                              "previous step is read again; not the headline"},
        "breakdown_us": {"one_kernel_step": round(ms_step * 1e3, 2),
                         "one_kernel_step_no_overlap": round(ms_one_plain / K * 1e3, 2),
                         "two_kernel_step": round(ms_two / K * 1e3, 2),
                         "append": round(append_ms * 1e3, 2),
                         "decode_attention": round(decode_ms * 1e3, 2),
                         "unfused_step_with_events": round(ms_events / K * 1e3, 2),
                         "note": "one_kernel_step is the timed step (pkv_decode_step_fused "
                                 "with PKV_STEP_OVERLAP; without it, every input is read "
                                 "after the previous step completes); "
                                 "two_kernel_step is pkv_decode_step (append, then attention "
                                 "overlapping its tail); append and decode_attention come "
                                 "from a third K-step graph of the two separate calls with "
                                 "CUDA events between them"},
        "bytes_per_step": {"attention": attn_bytes, "append": append_bytes},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic, "kernel": "decode_kernel (pkv_decode_step_fused: "
                     "append, attention and split combine in one launch)",
                     "peak_kind": peak_kind},
        "e2e": {"value": round(whole_job_gbps(step_bytes, ms_e2e / K, world), 1),
                "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(ms_e2e / K, 5),
                "method": "each step: one host-to-device copy of the step's inputs packed in a "
                          "pinned staging buffer, the step on views into its device twin, one "
                          "device-to-host copy of the output; double-buffered, the copies on their "
                          "own streams overlapping the neighbouring steps; all inside the timed "
                          "graph; median of three replays of the K-step graph"},
        # the one-kernel step is one launch for 16-bit caches; E4M3 steps
        # enqueue the append kernel, then the attention
        "gpu_launches": K * (2 if cfg.is_fp8 else 1),
        "clocks": clocks,
    }
    return res, st


def committed_traffic(workload):
    """DRAM traffic per decode launch from the committed ncu summary, if the
    kernel sources still hash to what was profiled; else null."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            j = json.load(f)
    except Exception:
        return None
    ent = j.get(workload)
    if not ent or ent.get("kernel_source_sha256") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


# the sources the decode and append kernels are built from (the prefill and
# block-copy kernels do not change them)
DECODE_SOURCES = ("pkv_decode_impl.cuh", "pkv_device.cuh", "pkv_internal.h", "pkv_api.cu",
                  "pkv_append.cu", "pkv_decode_bf16.cu", "pkv_decode_f16.cu", "pkv_decode_e4m3.cu",
                  "pkv_decode_e4m3_tok.cu")


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_250_gb300", "csrc")
    for fn in DECODE_SOURCES:
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode())
            h.update(f.read())
    return h.hexdigest()


# ---------------------------------------------------------------- oracle arm
def oracle_sample(cfg, w, max_seconds, whole_passes=True, threads=0):
    """Time the CPU oracle on whole sequences of the workload (all query
    heads), in order, until about `max_seconds` of work.  With
    `whole_passes` the pass over the batch repeats until the time is used.
    threads 0: every host core the oracle's OpenMP runtime offers."""
    import numpy as np

    import oracle
    threads = threads or oracle.max_threads()
    done_bytes = 0
    t_spent = 0.0
    seqs = 0
    prepared = {}
    while True:
        for b in range(cfg.batch):
            n = int(w.ctx[b])
            if n == 0:
                continue
            if b not in prepared:
                prepared[b] = (w.q[b].double().cpu().numpy()[None],
                               w.K_log[b, :n].double().cpu().numpy()[None],
                               w.V_log[b, :n].double().cpu().numpy()[None])
            qb, Kb, Vb = prepared[b]
            t0 = time.perf_counter()
            oracle.decode_attention(qb, Kb, Vb, np.array([n], np.int32), cfg.softmax_scale,
                                    nthreads=threads)
            t_spent += time.perf_counter() - t0
            done_bytes += n * cfg.kv_heads * cfg.head_dim * 2 * cfg.cache_elem_bytes
            seqs += 1
            if t_spent >= max_seconds:
                return done_bytes, t_spent, seqs, threads
        if not whole_passes:
            return done_bytes, t_spent, seqs, threads


def cpu_baseline(cfg, w, max_seconds=10.0, threads=0):
    b, t, seqs, threads = oracle_sample(cfg, w, max_seconds, threads=threads)
    return {"value": round(b / t / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{seqs} sequence passes over the {cfg.batch}-sequence batch (all "
                      f"{cfg.q_heads} query heads each), fp64 C oracle with OpenMP; "
                      f"{b / 1e6:.1f} MB of cache in {t:.2f} s"}


def run_reference(args, cfg):
    """The reference arm: the fp64 CPU oracle, as it stands, on the host cores.
    Each step is one pass over the workload's sequences (all query heads),
    cut short if it would exceed a per-step budget that keeps the whole run
    within a few minutes."""
    w = wl.generate(cfg, device="cpu")
    K, W = args.steps, args.warmup
    budget = max(0.5, 150.0 / max(1, K + W))
    for _ in range(W):
        oracle_sample(cfg, w, budget, whole_passes=False)
    total_b, total_t, seqs, threads = 0, 0.0, 0, 1
    for _ in range(K):
        b, t, seqs, threads = oracle_sample(cfg, w, budget, whole_passes=False)
        total_b += b
        total_t += t
    value = total_b / total_t / 1e9
    cb = {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
          "sample": f"per step {seqs} of the {cfg.batch} sequences of {cfg.name} (all query "
                    f"heads), fp64 C oracle with OpenMP; step budget {budget:.1f} s"}
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": 1, "steps": K, "warmup": W, "ms_per_step": round(1e3 * total_t / K, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, same generator as the native arm)",
            "config": {**workload_config(cfg, w.ctx),
                       "timing": "wall clock around each oracle pass on the host cores"},
            "cpu_baseline": cb,
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------- block copy
def run_copy_blocks(args, device):
    """pkv_copy_blocks alone: copy-on-write of whole blocks (8192 bf16 blocks of
    8 KV heads x 16 tokens x 128, K and V: 0.54 GB read + 0.54 GB written per
    step, far above L2), K steps in one CUDA graph, CUDA events around it."""
    NB, Hkv, d, n = 16384, 8, 128, 8192
    g = torch.Generator().manual_seed(7)
    perm = torch.randperm(NB, generator=g).to(torch.int32)
    src, dst = perm[:n].to(device), perm[n:2 * n].to(device)
    kc = torch.randn(NB, Hkv, wl.PAGE, d, device=device).to(torch.bfloat16)
    vc = torch.randn(NB, Hkv, wl.PAGE, d, device=device).to(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    desc = pkv.make_desc(NB, wl.PAGE, Hkv, Hkv, d, pkv.PKV_BF16, None, None, err)
    stream = torch.cuda.Stream(device)
    K, W = args.steps, args.warmup
    for _ in range(W):
        pkv.pkv_copy_blocks(desc, kc, vc, src, dst, stream=stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(K):
            pkv.pkv_copy_blocks(desc, kc, vc, src, dst, stream=stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    with torch.cuda.stream(stream):
        e0.record(stream)
        graph.replay()
        e1.record(stream)
    torch.cuda.synchronize(device)
    if int(err.item()) != 0:
        raise RuntimeError("device error word set")
    ms = e0.elapsed_time(e1) / K
    nbytes = 2 * 2 * n * Hkv * wl.PAGE * d * 2  # K and V, read and written
    value = nbytes / (ms * 1e-3) / 1e9
    peak, peak_kind = measured_peak()
    return {"metric": "block copy (copy-on-write) achieved HBM GB/s", "value": round(value, 1),
            "unit": "GB/s", "n_gpus": 1, "steps": K, "warmup": W,
            "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) blocks)",
            "config": {"workload": f"copy_blocks_{n}x_bf16_h{Hkv}_d{d}", "blocks": n,
                       "block_bytes_per_cache": Hkv * wl.PAGE * d * 2,
                       "l2": f"{2 * n * Hkv * wl.PAGE * d * 2 / 1e9:.2f} GB read and as much "
                             "written per call, far above L2",
                       "timing": "K copies in one CUDA graph, CUDA events on the stream"},
            "roofline": {"bound": "hbm", "achieved": round(value, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(value / peak, 4), "traffic": None,
                         "kernel": "copy_blocks_kernel", "peak_kind": peak_kind},
            "gpu_launches": K}


# ---------------------------------------------------------------- multi-query
def visible_tokens(ctx: torch.Tensor, qlen: int, window: int, sinks: int) -> int:
    """Cached positions at least one of a sequence's qlen new tokens sees
    under a sliding window with sinks (window 0: all of them)."""
    total = 0
    for n in ctx.tolist():
        if window <= 0:
            total += n
            continue
        lo = max(0, n - qlen - window + 1)  # first position token 0's window reaches
        total += (n - lo) + min(sinks, lo)
    return total


def run_multi_query(args, cfg, device, windowed: bool = False):
    """pkv_paged_decode_attention_multi (or, windowed, _window) alone on a
    workload's cache: q_len new tokens per sequence (already in the cache)
    attend at once, causal among themselves.  K calls in one CUDA graph over
    rotating pool copies (>= 4x L2), CUDA events around it; bytes as for one
    decode plus the extra q and output rows, counting under a window only the
    positions some token sees."""
    qlen = args.qlen
    if not 1 <= qlen <= 8:
        raise SystemExit(f"q_len {qlen}: 1 to 8 query tokens per sequence are built")
    hint = {"llama3_8b_b32_ctx1-4096_bf16": 4096}.get(cfg.name, 0)
    st = Step(cfg, device, 1, hint)
    pool_bytes = st.kc[0].numel() * st.kc[0].element_size() * 2
    R = max(1, min(8, -(-4 * L2_BYTES // pool_bytes)))
    st = Step(cfg, device, R, hint)
    # partials of group x q_len columns
    n = pkv.pkv_decode_workspace_bytes_multi(st.desc, cfg.batch, qlen, st.w.max_blocks_per_seq,
                                             hint)
    st.ws = torch.zeros(n, dtype=torch.uint8, device=device)
    g = torch.Generator().manual_seed(cfg.seed + 77)
    q = torch.randn(cfg.batch, qlen, cfg.q_heads, cfg.head_dim, generator=g).to(cfg.qdt).to(device)
    out = torch.empty(cfg.batch, qlen, cfg.q_heads, cfg.head_dim, dtype=st.out.dtype, device=device)
    stream = torch.cuda.Stream(device)

    def call(r):
        if windowed:
            pkv.pkv_paged_decode_attention_window(st.desc, q, st.kc[r], st.vc[r], st.tables,
                                                  st.ctx, args.window, args.sinks,
                                                  cfg.softmax_scale, out, st.ws, hint,
                                                  stream=stream)
        else:
            pkv.pkv_paged_decode_attention_multi(st.desc, q, st.kc[r], st.vc[r], st.tables,
                                                 st.ctx, cfg.softmax_scale, out, st.ws, hint,
                                                 stream=stream)
    K, W = args.steps, args.warmup
    for i in range(W):
        call(i % R)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(K):
            call(i % R)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    with torch.cuda.stream(stream):
        e0.record(stream)
        graph.replay()
        e1.record(stream)
    torch.cuda.synchronize(device)
    if int(st.err.item()) != 0:
        raise RuntimeError("device error word set")
    ms = e0.elapsed_time(e1) / K
    attn, _ = algorithmic_bytes(cfg, st.w.ctx)
    attn += (qlen - 1) * cfg.batch * cfg.q_heads * cfg.head_dim * 4  # more q and out rows
    extra = {"q_len": qlen}
    if windowed:
        kv_tok = cfg.kv_heads * cfg.head_dim * 2 * cfg.cache_elem_bytes
        seen = visible_tokens(st.w.ctx, qlen, args.window, args.sinks)
        attn -= (int(st.w.ctx.sum()) - seen) * kv_tok
        extra.update(window=args.window, sinks=args.sinks, visible_tokens=seen)
    value = attn / (ms * 1e-3) / 1e9
    peak, peak_kind = measured_peak()
    what = "windowed" if windowed else "multi-query"
    return {"metric": f"{what} decode-attention achieved HBM GB/s", "value": round(value, 1),
            "unit": "GB/s", "n_gpus": 1, "steps": K, "warmup": W, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": {"bf16": "bf16", "f16": "f16", "e4m3": "e4m3", "e4m3tok": "e4m3"}[cfg.cache],
            "data": "synthetic (seeded N(0,1) q/k/v, the workload's lengths and tables)",
            "config": {**workload_config(cfg, st.w.ctx), **extra,
                       "tokens_per_s_per_layer": round(cfg.batch * qlen / (ms * 1e-3), 1),
                       "l2": f"rotating {R} cache-pool copies ({R * pool_bytes / 1e6:.0f} MB, "
                             ">= 4x L2 where the pool allows); every call reads cold pages",
                       "timing": "K calls in one CUDA graph, CUDA events on the stream"},
            "roofline": {"bound": "hbm", "achieved": round(value, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(value / peak, 4), "traffic": None,
                         "kernel": (f"decode_kernel (q_len 1{', window' if windowed else ''})"
                                    if qlen == 1 else
                                    f"mq::decode_kernel (q_len {qlen}, {cfg.group * qlen} "
                                    f"(token, head) columns{', window' if windowed else ''})"),
                         "peak_kind": peak_kind},
            "gpu_launches": K}


def prefill_flops(ctx: torch.Tensor, chunk: int, q_heads: int, d: int) -> int:
    """Causal attention FLOPs of the prefill: the row at position p scores and
    weighs p + 1 positions, 4 d flops each (q.k and p.v), per query head."""
    total = 0
    for n in ctx.tolist():
        c = min(chunk, n)
        total += c * n - c * (c - 1) // 2  # sum of (p + 1) over the chunk's rows
    return 4 * d * q_heads * total


def run_prefill(args, cfg, device):
    """pkv_paged_prefill_attention alone: every sequence's last `chunk`
    positions (already in the cache) attend causally over its whole context.
    K calls in one CUDA graph, CUDA events around it; causal FLOPs (QK and PV)
    over the time, against the measured bf16 tensor peak."""
    st = Step(cfg, device, 1, 0)
    st.append(0, torch.cuda.current_stream(device))  # the newest position too
    torch.cuda.synchronize(device)
    chunks = [min(args.chunk, int(n)) for n in st.w.ctx.tolist()]
    starts = torch.tensor([0] + list(itertools.accumulate(chunks)), dtype=torch.int32,
                          device=device)
    total = int(starts[-1])
    g = torch.Generator().manual_seed(cfg.seed + 91)
    q = torch.randn(total, cfg.q_heads, cfg.head_dim, generator=g).to(cfg.qdt).to(device)
    out = torch.empty(total, cfg.q_heads, cfg.head_dim, dtype=st.out.dtype, device=device)
    stream = torch.cuda.Stream(device)

    def call():
        pkv.pkv_paged_prefill_attention(st.desc, q, st.kc[0], st.vc[0], st.tables, st.ctx,
                                        starts, max(chunks), cfg.softmax_scale, out,
                                        stream=stream)
    K, W = args.steps, args.warmup
    for _ in range(W):
        call()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(K):
            call()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    time.sleep(0.2)
    t0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        graph.replay()
        e1.record(stream)
    torch.cuda.synchronize(device)
    t1 = time.time()
    time.sleep(0.1)
    sampler.stop()
    if int(st.err.item()) != 0:
        raise RuntimeError("device error word set")
    ms = e0.elapsed_time(e1) / K
    pool_mb = st.kc[0].numel() * st.kc[0].element_size() * 2 / 1e6
    flops = prefill_flops(st.w.ctx, args.chunk, cfg.q_heads, cfg.head_dim)
    tflops = flops / (ms * 1e-3) / 1e12
    peak = measured_tensor_peak()
    return {"metric": "paged prefill attention TFLOP/s (causal QK and PV flops)",
            "value": round(tflops, 1), "unit": "TFLOP/s", "n_gpus": 1, "steps": K,
            "warmup": W, "ms_per_step": round(ms, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": {"bf16": "bf16", "f16": "f16"}[cfg.cache],
            "data": "synthetic (seeded N(0,1) q/k/v, the workload's lengths and tables)",
            "config": {**workload_config(cfg, st.w.ctx), "chunk": args.chunk,
                       "query_rows": total, "flops_per_call": flops,
                       "l2": f"one cache pool ({pool_mb:.0f} MB of K and V, above L2) read "
                             "by every call",
                       "timing": "K calls in one CUDA graph, CUDA events on the stream"},
            "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak[0],
                         "unit": "TFLOP/s", "frac": round(tflops / peak[0], 4),
                         "traffic": None, "kernel": "prefill_kernel (tcgen05)",
                         "peak_kind": peak[1]},
            "gpu_launches": K, "clocks": sampler.summary(t0, t1)}


# ---------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(wl.CONFIGS))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--op", default="decode_step",
                    choices=["decode_step", "copy_blocks", "multi_query", "window", "prefill"],
                    help="decode_step (the default line), copy_blocks, multi_query, window or "
                         "prefill alone")
    ap.add_argument("--chunk", type=int, default=2048,
                    help="prefill rows per sequence (its last positions)")
    ap.add_argument("--qlen", type=int, default=2,
                    help="query tokens per sequence (multi_query, window)")
    ap.add_argument("--window", type=int, default=4096, help="window length (window)")
    ap.add_argument("--sinks", type=int, default=4, help="sink positions (window)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    cfg = wl.CONFIGS[args.config]
    world, rank, local = dist_env()

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, cfg)), flush=True)
        return

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device for the native arm")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    pkv.load_library()
    if args.op == "copy_blocks":
        if rank == 0:
            print(json.dumps(run_copy_blocks(args, device)), flush=True)
        return
    if args.op == "prefill":
        if rank == 0:
            print(json.dumps(run_prefill(args, cfg, device)), flush=True)
        return
    if args.op in ("multi_query", "window"):
        if rank == 0:
            print(json.dumps(run_multi_query(args, cfg, device, args.op == "window")), flush=True)
        return
    res, st = run_native(args, cfg, rank, world, device)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            wcpu = wl.generate(cfg, device="cpu")
            res["cpu_baseline"] = cpu_baseline(cfg, wcpu)
            res["cpu_baseline_single_core"] = cpu_baseline(cfg, wcpu, 5.0, threads=1)
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
