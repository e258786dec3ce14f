"""Benchmark of the INT8-KV-cache attention hot path on GB300.

A step of the headline workload (decode_32k: one sequence, ctx 32768, 24 query / 4 KV heads,
head_dim 256, int8 K/V in 16-token pages behind a shuffled block table, K outliers) is one
pass of the decode path: kv_quant_write of the step's new token, then split-K decode over
the whole context (split-K with the library's split size for this GPU: stage 1, then the merge).
value = K/V bytes the step reads
(2080 B per token) / device time of the step, in GB/s, with the L2 flushed (256 MB write, then a
256 MB read of another buffer) before every timed step, outside its events.

Prints one JSON line.  --impl reference times the CPU oracle (the plain reference) on the
host cores on a bounded sample of the same workload.  Under torchrun (N > 1) every rank runs
an independent replica (the path has no cross-GPU exchange) and value sums the ranks' bytes
over the slowest rank's time.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode KV GB/s + µs/call at 32K ctx; prefill int8 TOPS; % of GB300 roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# DRAM bytes (read + written) of one decode_32k stage-1 launch, from an ncu capture of this
# kernel (dram__bytes_read.sum + dram__bytes_write.sum), and the SHA-256 prefix of the kernel's
# sources at that capture.  Once the sources differ, the figure no longer describes the kernel
# and the line reports null.
STAGE1_TRAFFIC_BYTES = 68232960 + 115712
STAGE1_TRAFFIC_SOURCES = ("int8_kv_cache_quant_gb300/csrc/decode.cu", "int8_kv_cache_quant_gb300/csrc/kvq_dev.cuh",
                          "int8_kv_cache_quant_gb300/csrc/quant_rule.cuh")
STAGE1_TRAFFIC_SHA = "9436c9bad45afc5c"


def stage1_traffic():
    import hashlib
    h = hashlib.sha256()
    for f in STAGE1_TRAFFIC_SOURCES:
        with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), f), "rb") as fh:
            h.update(fh.read())
    return STAGE1_TRAFFIC_BYTES if h.hexdigest()[:16] == STAGE1_TRAFFIC_SHA else None


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling (every 50 ms) in a background thread; summary()
    reports the samples taken between mark_begin() and mark_end() widened by `pad_s` on each
    side (a timed region of a few milliseconds is shorter than one sampling interval)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, pad_s=0.25):
        self.gpu, self.pad = gpu_index, pad_s
        self.proc, self.samples, self.t0, self.t1 = None, [], None, None

    def _reader(self):
        for line in self.proc.stdout:
            if line.strip():
                self.samples.append((time.perf_counter(), line))

    def __enter__(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._reader, daemon=True)
            self.thread.start()
            deadline = time.perf_counter() + 3.0
            while not self.samples and time.perf_counter() < deadline:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        return self

    def mark_begin(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        self.t1 = time.perf_counter()
        time.sleep(self.pad)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lo = (self.t0 or 0) - self.pad
        hi = (self.t1 or time.perf_counter()) + self.pad
        for t, l in self.samples:
            if not (lo <= t <= hi):
                continue
            parts = [p.strip() for p in l.split(",")]
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "window": "timed region +- %.2f s" % self.pad}


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """Largest x over all ranks (the slowest replica's time).  The reduction tensor lives where
    the process group's backend can reach it: device memory for NCCL, host memory for gloo."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(bytes_per_rank, ms_max, world):
    """Whole-job throughput of N independent replicas: every rank moves bytes_per_rank per step,
    and the job's step time is the slowest rank's."""
    return world * bytes_per_rank / (ms_max * 1e-3) / 1e9


# ----------------------------------------------------------------------------- kvq arm

def bench_decode_32k(args, world, rank, local, extra_out):
    import numpy as np
    import torch

    import int8_kv_cache_quant_gb300 as kvq
    import workloads as W
    from int8_kv_cache_quant_gb300 import build as kbuild

    kbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = W.make("decode_32k")
    D, Hq, Hkv = w["d"], w["hq"], w["hkv"]

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

    cache = kvq.KVCache(w["num_blocks"], Hkv, D, device=dev)
    bt = i32(w["block_table"])
    kvq.kvq_quant_write(cache, bf16(w["k_fill"]), bf16(w["v_fill"]), i32(w["fill_seq"]),
                        i32(w["fill_pos"]), bt)
    q = bf16(w["q"])
    k_new, v_new = bf16(w["k_new"]), bf16(w["v_new"])
    new_seq, new_pos = i32(w["new_seq"]), i32(w["new_pos"])
    ctx = i32(w["ctx_lens"])
    max_ctx = w["max_ctx"]
    # the library's default split (split_rows 0): sized so that stage 1 fills the GPU in one wave
    split = kvq.kvq_decode_auto_split_rows(1, Hkv, D, max_ctx, torch.cuda.get_device_properties(local).multi_processor_count)
    ws = torch.empty(kvq.kvq_decode_workspace_bytes(1, Hq, max_ctx, D),
                     dtype=torch.uint8, device=dev)
    out = torch.empty((1, Hq, D), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    sweep = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    s = torch.cuda.current_stream()

    def cold_l2(i):
        # write 256 MB (> the 129 MB L2), then read another 256 MB so that the L2 holds clean
        # lines of an unrelated buffer: the timed step then starts cold and pays no write-back.
        # A ~30 us device sleep follows, so that the host has queued the step's launches before
        # the GPU reaches the start event: the events then time device work, not the host's
        # argument marshalling (e2e below is the figure with the host in it).
        flush.fill_(i & 0xFF)
        sweep.sum()
        torch.cuda._sleep(60000)

    def step(ev=None):
        # the fused step: stage 1 writes the new token into its page, then attends
        kvq.kvq_decode_step_int8kv(cache, k_new, v_new, q, bt, ctx, max_ctx, w["softmax_scale"], out=out,
                                   workspace=ws, stage1_events=ev)

    def step_unfused():
        kvq.kvq_quant_write(cache, k_new, v_new, new_seq, new_pos, bt)
        kvq.kvq_attn_decode_int8kv(cache, q, bt, ctx, max_ctx, w["softmax_scale"], out=out, workspace=ws)

    for _ in range(args.warmup):
        cold_l2(1)
        step()
    torch.cuda.synchronize()
    assert kvq.kvq_device_status() == 0

    K = args.steps
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    k0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    k1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for e in k0 + k1:  # create the underlying CUDA events; the library re-records them
        e.record(s)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for _ in range(3):  # keep the GPU busy while the sampler starts (untimed)
            cold_l2(0)
            step()
        torch.cuda.synchronize()
        clk.mark_begin()
        t_wall = time.perf_counter()
        for i in range(K):
            cold_l2(i)
            ev0[i].record(s)
            step()
            ev1[i].record(s)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
        clk.mark_end()
    barrier(world)
    step_ms = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    # Stage-1 duration for the roofline: a second pass of K steps with events recorded on the
    # library's stream right around the stage-1 launch.  They are kept out of the headline
    # pass because an event between two launches ends the programmatic-dependent-launch
    # overlap of stage 1 -> merge.
    ev2 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev3 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        cold_l2(i)
        ev2[i].record(s)
        step((k0[i], k1[i]))
        ev3[i].record(s)
    torch.cuda.synchronize()
    kern_ms = [a.elapsed_time(b) for a, b in zip(k0, k1)]
    step_ms_events = statistics.mean(a.elapsed_time(b) for a, b in zip(ev2, ev3))
    # the same step as two calls (kvq_quant_write, then kvq_attn_decode_int8kv), for reference
    for i in range(K):
        cold_l2(i)
        ev2[i].record(s)
        step_unfused()
        ev3[i].record(s)
    torch.cuda.synchronize()
    step_ms_unfused = statistics.mean(a.elapsed_time(b) for a, b in zip(ev2, ev3))
    # kernels one step launches (stage 1 and the merge on the split route)
    import ctypes
    n_launch = ctypes.c_int32(0)
    kvq.kvq_decode_step_int8kv(cache, k_new, v_new, q, bt, ctx, max_ctx, w["softmax_scale"], out=out, workspace=ws,
                               launches=n_launch)
    torch.cuda.synchronize()
    launches_per_step = int(n_launch.value)

    def time_events(fn, with_stage1=False):
        t_all, t_s1 = [], []
        for i in range(K):
            cold_l2(i)
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            if with_stage1:
                e[2].record(s)
                e[3].record(s)
            e[0].record(s)
            fn((e[2], e[3]) if with_stage1 else None)
            e[1].record(s)
            torch.cuda.synchronize()
            t_all.append(e[0].elapsed_time(e[1]))
            if with_stage1:
                t_s1.append(e[2].elapsed_time(e[3]))
        return statistics.mean(t_all), (statistics.mean(t_s1) if with_stage1 else None)

    # The stream floor: decode stage 1's grid, rings and bulk copies of the same pages, with no
    # arithmetic (kvq_debug_stream_floor), timed like the step.
    floor_ms, _ = time_events(lambda ev: kvq.kvq_debug_stream_floor(cache, bt, ctx, max_ctx))
    # The stated configuration's 512-key splits (64 splits x 4 KV heads = 256 CTAs, two waves:
    # the split route then ends in the separate merge kernel), beside the automatic split above.
    ws512 = torch.empty(kvq.kvq_decode_workspace_bytes(1, Hq, max_ctx, D, split_rows=512), dtype=torch.uint8,
                        device=dev)

    def step512(ev):
        kvq.kvq_decode_step_int8kv(cache, k_new, v_new, q, bt, ctx, max_ctx, w["softmax_scale"], out=out,
                                   workspace=ws512, split_rows=512, stage1_events=ev)
    step512(None)
    torch.cuda.synchronize()
    ms512, _ = time_events(step512)
    _, s1_512 = time_events(step512, with_stage1=True)
    ms_step = statistics.mean(step_ms)
    ms_step_max = max_over_ranks(ms_step, world)
    kv_bytes = max_ctx * (2 * Hkv * D + 2 * Hkv * 4)  # 2080 B per token at 4 x 256

    # End to end through the public API with host buffers.  On GB300 the kernels read and write
    # page-locked host memory across the coherent host link, so the step takes its inputs (Q,
    # the new K and V rows) from pinned host buffers and writes its result into one (zero-copy):
    # the transfers run inside the call, overlapped with the K/V stream.  The timed steps cycle
    # through NSET buffer sets with different query rows, and afterwards every set's host result
    # is checked bit for bit against the same step with device buffers.  The same step with
    # explicit copies (one H2D of a staged input buffer, the call, one D2H of the result) is
    # timed as well.
    NSET = 4
    rng_e = np.random.default_rng(4242)
    sets = []
    for i in range(NSET):
        qi = w["q"] if i == 0 else W.normal_bf16(rng_e, w["q"].shape)
        parts = [np.ascontiguousarray(x).view(np.int16).ravel() for x in (qi, w["k_new"], w["v_new"])]
        buf = torch.from_numpy(np.concatenate(parts)).pin_memory()
        nq_el, nk_el = parts[0].size, parts[1].size
        views = (buf[:nq_el].view(torch.bfloat16).view(1, Hq, D),
                 buf[nq_el:nq_el + nk_el].view(torch.bfloat16).view(1, Hkv, D),
                 buf[nq_el + nk_el:].view(torch.bfloat16).view(1, Hkv, D))
        sets.append((buf, views, torch.empty((1, Hq, D), dtype=torch.float32).pin_memory()))
    h2d = sets[0][0].numel() * 2
    d2h = sets[0][2].numel() * 4

    def e2e_step(i):
        _, (qh, knh, vnh), oh = sets[i % NSET]
        kvq.kvq_decode_step_int8kv(cache, knh, vnh, qh, bt, ctx, max_ctx, w["softmax_scale"], out=oh, workspace=ws)

    in_d = torch.empty_like(sets[0][0], device=dev)
    q_d = in_d[:nq_el].view(torch.bfloat16).view(1, Hq, D)
    kn_d = in_d[nq_el:nq_el + nk_el].view(torch.bfloat16).view(1, Hkv, D)
    vn_d = in_d[nq_el + nk_el:].view(torch.bfloat16).view(1, Hkv, D)
    out_copy_h = torch.empty((1, Hq, D), dtype=torch.float32).pin_memory()

    def e2e_copy_step(i):
        in_d.copy_(sets[i % NSET][0], non_blocking=True)
        kvq.kvq_decode_step_int8kv(cache, kn_d, vn_d, q_d, bt, ctx, max_ctx, w["softmax_scale"], out=out,
                                   workspace=ws)
        out_copy_h.copy_(out, non_blocking=True)

    def time_e2e(fn):
        # no device sleep here: the host's work of each call (argument checks and marshalling)
        # stays inside the timed region
        for i in range(3):
            cold_l2(2)
            fn(i)
        torch.cuda.synchronize()
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        for i in range(K):
            flush.fill_(i & 0xFF)
            sweep.sum()
            e0[i].record(s)
            fn(i)
            e1[i].record(s)
        torch.cuda.synchronize()
        return max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in zip(e0, e1)), world)

    e2e_ms = time_e2e(e2e_step)
    e2e_copy_ms = time_e2e(e2e_copy_step)
    for i in range(NSET):  # each set's host result against the step with device buffers
        e2e_step(i)
        torch.cuda.synchronize()
        in_d.copy_(sets[i][0])
        kvq.kvq_decode_step_int8kv(cache, kn_d, vn_d, q_d, bt, ctx, max_ctx, w["softmax_scale"], out=out,
                                   workspace=ws)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy().view(np.uint32), sets[i][2].numpy().view(np.uint32)), i
    assert kvq.kvq_device_status() == 0

    hbm, _, peak_kind = load_peaks()
    kern_avg = statistics.mean(kern_ms)
    achieved = kv_bytes / (kern_avg * 1e-3) / 1e9
    res = {
        "metric": METRIC,
        "value": round(aggregate_gbs(kv_bytes, ms_step_max, world), 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step_max, 5),
        "ms_per_step_with_stage1_events": round(step_ms_events, 5),
        "ms_per_step_unfused": round(step_ms_unfused, 5),
        "us_per_call": round(ms_step_max * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int8",
        "data": "synthetic (seeded N(0,1) bf16 Q/K/V quantised to int8 codes + fp32 scales; K outliers x8 p=0.01)",
        "config": {"workload": "decode_32k", "batch": 1, "ctx": max_ctx, "q_heads": Hq, "kv_heads": Hkv,
                   "head_dim": D, "block_size": 16, "block_table": "random permutation",
                   "split_rows": split, "kv_bytes_per_step": kv_bytes,
                   "step": "kvq_decode_step_int8kv: the new token's quantise-and-write inside decode stage 1, then the merge",
                   "l2": "cold before every timed step: 256 MB write then 256 MB read of another buffer, outside the events",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": stage1_traffic(),
                     "kernel": "decode_stage1_kernel<256,warps=8,DEPTH=3,split,fused write>", "peak_kind": peak_kind,
                     "kernel_us": round(kern_avg * 1e3, 2)},
        "e2e": {"value": round(aggregate_gbs(kv_bytes, e2e_ms, world), 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "transfer": "zero-copy: the step's kernels read Q and the new K/V rows from, and write the "
                            "result into, page-locked host memory over the coherent host link; %d host "
                            "buffer sets with different queries, each result checked bit for bit" % NSET,
                "with_copies": {"value": round(aggregate_gbs(kv_bytes, e2e_copy_ms, world), 2),
                                "ms_per_step": round(e2e_copy_ms, 5),
                                "transfer": "one H2D copy of the staged inputs, the call, one D2H copy"}},
        "gpu_launches": launches_per_step * K,
        "launches_per_step": launches_per_step,
        "stream_floor": {"us": round(floor_ms * 1e3, 2), "GBps": round(kv_bytes / (floor_ms * 1e-3) / 1e9, 1),
                         "frac": round(kv_bytes / (floor_ms * 1e-3) / 1e9 / hbm, 4),
                         "what": "kvq_debug_stream_floor: stage 1's grid, rings and bulk copies of the same 68 MB "
                                 "of pages, no arithmetic, timed like the step (cold L2, CUDA events)",
                         "stage1_over_floor": round(kern_avg / floor_ms, 3)},
        "split_512": {"split_rows": 512, "us_per_step": round(ms512 * 1e3, 2),
                      "GBps": round(kv_bytes / (ms512 * 1e-3) / 1e9, 1),
                      "stage1_us": round(s1_512 * 1e3, 2),
                      "stage1_frac": round(kv_bytes / (s1_512 * 1e-3) / 1e9 / hbm, 4),
                      "what": "the stated 512-key splits: 256 stage-1 CTAs in two waves, then the merge kernel"},
        "clocks": clk.summary(),
        "wall_s_timed_region": round(t_wall, 4),
    }
    return res


def bench_extra(args, local, hbm, tflops, only=None):
    """Secondary figures on the other workloads (one JSON object, not the headline)."""
    import numpy as np
    import torch

    import int8_kv_cache_quant_gb300 as kvq
    import workloads as W
    dev = torch.device("cuda", local)

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    sweep = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    s = torch.cuda.current_stream()

    def cold_l2(i):
        flush.fill_(i & 0xFF)
        sweep.sum()
        torch.cuda._sleep(60000)  # the host's launches get ahead of the GPU (device-only timing)

    def timed(fn, reps, cold=True):
        """Median event time of one call; L2 flushed before each (cold) or still holding the
        previous call's inputs (warm: a ~50 us sleep kernel between that call and the timed
        one keeps the host's launches ahead of the GPU, so the events see device time only)."""
        for _ in range(3):
            cold_l2(1)
            fn()
        torch.cuda.synchronize()
        ms = []
        for i in range(reps):
            if cold:
                cold_l2(i)
            else:
                fn()
                torch.cuda._sleep(100000)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            fn()
            b.record(s)
            b.synchronize()
            ms.append(a.elapsed_time(b))
        return statistics.median(ms)

    res = {}
    reps = args.steps if only else None

    def want(name):
        return only is None or only == name

    # decode_1k: launch/latency bound
    if want("decode_1k"):
        res.update(_extra_decode_1k(kvq, W, bf16, i32, timed, dev, reps or 50))
    if want("decode_b64"):
        res.update(_extra_decode_b64(kvq, W, bf16, i32, timed, dev, reps or 20, hbm))
    if want("verify_32k"):
        res.update(_extra_verify_32k(kvq, W, bf16, i32, timed, dev, reps or 30, hbm))
    if want("rope_quant_write"):
        res.update(_extra_rope_quant_write(kvq, W, bf16, i32, timed, dev, reps or 20, hbm))
    if want("prefill_32k"):
        res.update(_extra_prefill_32k(kvq, W, bf16, i32, timed, dev, reps or 10, tflops))
    if want("prefill_first_4k"):
        res.update(_extra_prefill_first_4k(kvq, W, bf16, i32, timed, dev, reps or 10, tflops))
    if want("sparse_32k"):
        res.update(_extra_sparse_32k(kvq, W, bf16, i32, timed, dev, reps or 10))
    return res


def _extra_decode_1k(kvq, W, bf16, i32, timed, dev, reps):
    import torch
    res = {}
    w = W.make("decode_1k")
    cache = kvq.KVCache(w["num_blocks"], w["hkv"], w["d"], device=dev)
    bt = i32(w["block_table"])
    kvq.kvq_quant_write(cache, bf16(w["k_fill"]), bf16(w["v_fill"]), i32(w["fill_seq"]), i32(w["fill_pos"]), bt)
    q, ctx = bf16(w["q"]), i32(w["ctx_lens"])
    out = torch.empty((1, w["hq"], w["d"]), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, kvq.kvq_decode_workspace_bytes(1, w["hq"], w["max_ctx"], w["d"])), dtype=torch.uint8,
                     device=dev)

    def call():
        kvq.kvq_attn_decode_int8kv(cache, q, bt, ctx, w["max_ctx"], w["softmax_scale"], out=out, workspace=ws)
    split = kvq.kvq_decode_auto_split_rows(1, w["hkv"], w["d"], w["max_ctx"],
                                           torch.cuda.get_device_properties(dev).multi_processor_count)
    ms = timed(call, reps)
    ms_warm = timed(call, reps, cold=False)
    # the same call recorded once in a CUDA graph and replayed (no per-call host work)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    ms_graph = timed(g.replay, reps)
    ms_graph_warm = timed(g.replay, reps, cold=False)

    def back_to_back(fn, n=200):
        # n calls issued as fast as the host can: host-bound unless each call is cheap to launch
        fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(n):
            fn()
        b.record()
        b.synchronize()
        return a.elapsed_time(b) / n
    b2b, b2b_graph = back_to_back(call), back_to_back(g.replay)
    kvb = w["max_ctx"] * (2 * w["hkv"] * w["d"] + 8 * w["hkv"])
    res["decode_1k"] = {"us_per_call": round(ms * 1e3, 2), "kv_GBps": round(kvb / ms / 1e6, 1),
                        "us_per_call_warm_l2": round(ms_warm * 1e3, 2),
                        "us_per_call_graph": round(ms_graph * 1e3, 2),
                        "us_per_call_graph_warm_l2": round(ms_graph_warm * 1e3, 2),
                        "us_per_call_back_to_back": round(b2b * 1e3, 2),
                        "us_per_call_back_to_back_graph": round(b2b_graph * 1e3, 2),
                        "gpu_launches_per_call": 2 if split < w["max_ctx"] else 1}
    return res


def _extra_decode_b64(kvq, W, bf16, i32, timed, dev, reps, hbm):
    """decode_b64: one batched step (kv_quant_write of one new token per sequence, then decode)
    over 64 sequences of ctx 512..16384, 32 query / 8 KV heads, head_dim 128."""
    import numpy as np
    import torch
    res = {}
    w = W.make("decode_b64")
    cache = kvq.KVCache(w["num_blocks"], w["hkv"], w["d"], device=dev)
    bt = i32(w["block_table"])
    kvq.kvq_quant_write(cache, bf16(w["k_fill"]), bf16(w["v_fill"]), i32(w["fill_seq"]), i32(w["fill_pos"]), bt)
    q, ctx = bf16(w["q"]), i32(w["ctx_lens"])
    kn, vn, ns, npos = bf16(w["k_new"]), bf16(w["v_new"]), i32(w["new_seq"]), i32(w["new_pos"])
    B, Hq, D = w["batch"], w["hq"], w["d"]
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, kvq.kvq_decode_workspace_bytes(B, Hq, w["max_ctx"], D)), dtype=torch.uint8, device=dev)

    def step():
        kvq.kvq_decode_step_int8kv(cache, kn, vn, q, bt, ctx, w["max_ctx"], w["softmax_scale"], out=out,
                                   workspace=ws)

    def step_unfused():
        kvq.kvq_quant_write(cache, kn, vn, ns, npos, bt)
        kvq.kvq_attn_decode_int8kv(cache, q, bt, ctx, w["max_ctx"], w["softmax_scale"], out=out, workspace=ws)
    ms = timed(step, reps)
    ms_unfused = timed(step_unfused, reps)
    ms_write = timed(lambda: kvq.kvq_quant_write(cache, kn, vn, ns, npos, bt), reps)
    kvb = int(w["ctx_lens"].astype(np.int64).sum()) * w["hkv"] * (2 * D + 8)
    res["decode_b64"] = {"us_per_step": round(ms * 1e3, 2), "kv_bytes": kvb, "kv_GBps": round(kvb / ms / 1e6, 1),
                         "frac_of_hbm_peak": round(kvb / ms / 1e6 / hbm, 4),
                         "us_per_step_unfused": round(ms_unfused * 1e3, 2),
                         "us_quant_write": round(ms_write * 1e3, 2),
                         "step": "kvq_decode_step_int8kv: 64 new tokens written inside decode stage 1 (split route)"}
    return res


def _extra_verify_32k(kvq, W, bf16, i32, timed, dev, reps, hbm):
    """verify_32k: one speculative-verify step on decode_32k's cache shape (ctx 32768, 24/4,
    head_dim 256): the 4 drafted tokens written into the cache inside the 4-row verify decode
    (kvq_decode_step_int8kv, automatic split); the verify decode alone is timed too.  Bytes:
    the K/V codes and scales of all 32768 keys, read once for the 4 rows."""
    import torch
    w = W.make("verify_32k")
    cache = kvq.KVCache(w["num_blocks"], w["hkv"], w["d"], device=dev)
    bt = i32(w["block_table"])
    kvq.kvq_quant_write(cache, bf16(w["k_fill"]), bf16(w["v_fill"]), i32(w["fill_seq"]), i32(w["fill_pos"]), bt)
    q, ctx = bf16(w["q"]), i32(w["ctx_lens"])
    kn, vn = bf16(w["k_new"]), bf16(w["v_new"])
    B, nq, Hq, D = w["batch"], w["nq"], w["hq"], w["d"]
    out = torch.empty((B, nq, Hq, D), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, kvq.kvq_verify_workspace_bytes(B, nq, Hq, w["max_ctx"], D)), dtype=torch.uint8,
                     device=dev)

    def verify():
        kvq.kvq_attn_verify_int8kv(cache, q, bt, ctx, w["max_ctx"], w["softmax_scale"], out=out, workspace=ws)

    kn4 = kn.view(B, nq, w["hkv"], D)
    vn4 = vn.view(B, nq, w["hkv"], D)

    def step():
        kvq.kvq_decode_step_int8kv(cache, kn4, vn4, q, bt, ctx, w["max_ctx"], w["softmax_scale"], out=out,
                                   workspace=ws)
    ms = timed(step, reps)
    ms_verify = timed(verify, reps)
    kvb = w["max_ctx"] * (2 * w["hkv"] * D + 8 * w["hkv"])
    return {"verify_32k": {"us_per_step": round(ms * 1e3, 2), "us_verify": round(ms_verify * 1e3, 2),
                           "rows": nq, "kv_bytes": kvb, "kv_GBps": round(kvb / ms / 1e6, 1),
                           "verify_frac_of_hbm_peak": round(kvb / ms_verify / 1e6 / hbm, 4),
                           "step": "kvq_decode_step_int8kv: 4 drafted tokens written inside the 4-row verify decode"}}


def _extra_rope_quant_write(kvq, W, bf16, i32, timed, dev, reps, hbm):
    """The fused producer (RoPE on Q and K, quantisation of Q, K and V, paged K/V write) at two
    shapes: the prefill_32k chunk (2048 tokens at positions 30720..32767, 24/4 heads, head_dim
    256) and one decode_b64 step (64 tokens, 32/8 heads, head_dim 128).  Bytes: bf16 Q/K/V and
    the table rows read; K/V codes and scales, Q codes, Q scales and bf16 rotated Q written."""
    import numpy as np
    import torch
    res = {}
    rng = np.random.default_rng(77)
    for name, T, hq, hkv, d, max_pos, first in (("prefill_chunk", 2048, 24, 4, 256, 32768, 30720),
                                                ("decode_b64_step", 64, 32, 8, 128, 16384, None)):
        n_blocks = max_pos // 16
        cache = kvq.KVCache(n_blocks * (1 if first is not None else 1), hkv, d, device=dev)
        if first is not None:
            pos = np.arange(first, first + T, dtype=np.int32)
            seq = np.zeros(T, np.int32)
            table = rng.permutation(n_blocks).astype(np.int32)[None, :]
        else:  # one sequence per token, each with its own slice of pages
            per = n_blocks // T
            pos = rng.integers(0, per * 16, size=T).astype(np.int32)
            seq = np.arange(T, dtype=np.int32)
            table = rng.permutation(n_blocks)[: per * T].astype(np.int32).reshape(T, per)
        inv = 1.0e6 ** (-np.arange(0, d, 2, dtype=np.float64) / d)
        ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
        cs = torch.from_numpy(np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)).to(dev)
        q, k, v = (bf16(W.normal_bf16(rng, (T, h, d))) for h in (hq, hkv, hkv))
        qc = torch.empty((T, hq, d), dtype=torch.int8, device=dev)
        qs = torch.empty((T, hq), dtype=torch.float32, device=dev)
        qr = torch.empty((T, hq, d), dtype=torch.bfloat16, device=dev)
        pos_d, seq_d, tab_d = i32(pos), i32(seq), i32(table)
        ms = timed(lambda: kvq.kvq_rope_quant_write(cache, q, k, v, seq_d, pos_d, tab_d, cs, d, q_codes=qc,
                                                    q_scales=qs, q_rot=qr), reps)
        nbytes = T * ((hq + 2 * hkv) * d * 2 + d * 4 + 8 + 2 * hkv * (d + 4) + hq * (d + 4 + 2 * d))
        res[name] = {"us_per_call": round(ms * 1e3, 2), "bytes": nbytes, "GBps": round(nbytes / ms / 1e6, 1),
                     "frac_of_hbm_peak": round(nbytes / ms / 1e6 / hbm, 4)}
    return {"rope_quant_write": res}


def _extra_prefill_32k(kvq, W, bf16, i32, timed, dev, reps, tflops):
    """prefill_32k: the chunk's K/V written by kv_quant_write first (timed separately)."""
    import torch
    res = {}
    w = W.make("prefill_32k")
    cache = kvq.KVCache(w["num_blocks"], w["hkv"], w["d"], device=dev)
    bt = i32(w["block_table"])
    kvq.kvq_quant_write(cache, bf16(w["k_fill"]), bf16(w["v_fill"]), i32(w["fill_seq"]), i32(w["fill_pos"]), bt)
    q = bf16(w["q"])
    T, Hq, D = w["n_tokens"], w["hq"], w["d"]
    out = torch.empty((T, Hq, D), dtype=torch.float32, device=dev)
    ws = torch.empty(kvq.kvq_prefill_workspace_bytes(T, Hq, w["hkv"], w["history"], D), dtype=torch.uint8,
                     device=dev)
    row = bt[0]
    ms = timed(lambda: kvq.kvq_attn_prefill_int8(cache, q, w["history"], row, w["softmax_scale"], out=out,
                                                  workspace=ws), reps)
    hist = w["history"]
    triples = Hq * sum(hist + i + 1 for i in range(T))
    ops = 2.0 * 2 * D * triples
    chunk_seq = torch.zeros(T, dtype=torch.int32, device=dev)
    chunk_pos = torch.arange(hist, hist + T, dtype=torch.int32, device=dev)
    kc, vc = bf16(w["k_fill"][hist:]), bf16(w["v_fill"][hist:])
    ms_qw = timed(lambda: kvq.kvq_quant_write(cache, kc, vc, chunk_seq, chunk_pos, bt), reps)
    res["prefill_32k"] = {"ms_per_call": round(ms, 4), "int8_equiv_TOPS": round(ops / ms / 1e9, 1),
                          "frac_of_bf16_peak": round(ops / ms / 1e9 / tflops, 4), "peak_TFLOPS": tflops,
                          "chunk_kv_quant_write_ms": round(ms_qw, 4), "ops": ops}
    return res


def _extra_prefill_first_4k(kvq, W, bf16, i32, timed, dev, reps, tflops):
    """The first prefill chunk of a sequence, 4096 tokens at 24 query / 4 KV heads, head_dim 256
    (the page's 0 + 4K chunk): the chunk's K/V written into the int8 cache and the high-precision
    causal attention over its bf16 Q/K/V, one call.  Ops: 2 (QK, PV) x 2 x head_dim per visible
    (query head, query, key) triple."""
    import numpy as np
    import torch
    rng = np.random.default_rng(99)
    T, hq, hkv, d = 4096, 24, 4, 256
    nb = T // 16
    table = i32(rng.permutation(nb).astype(np.int32))
    q, k, v = (bf16(W.normal_bf16(rng, (T, h, d))) for h in (hq, hkv, hkv))
    cache = kvq.KVCache(nb, hkv, d, device=dev)
    out = torch.empty((T, hq, d), dtype=torch.float32, device=dev)
    ws = torch.empty(kvq.kvq_prefill_first_workspace_bytes(T, hq, hkv, d), dtype=torch.uint8, device=dev)
    ms = timed(lambda: kvq.kvq_attn_prefill_first_bf16(cache, q, k, v, table, 1.0 / 16, out=out, workspace=ws), reps)
    ops = 2.0 * 2 * d * hq * (T * (T + 1) / 2)
    return {"prefill_first_4k": {"ms_per_call": round(ms, 4), "TFLOPS": round(ops / ms / 1e9, 1),
                                 "frac_of_bf16_peak": round(ops / ms / 1e9 / tflops, 4), "ops": ops,
                                 "step": "kvq_attn_prefill_first_bf16: int8 K/V write + fp16-operand attention"}}


def _extra_sparse_32k(kvq, W, bf16, i32, timed, dev, reps):
    import torch
    res = {}
    w = W.make("sparse_32k")
    cache = kvq.KVCache(w["num_blocks"], w["hkv"], w["d"], device=dev)
    bt = i32(w["block_table"])
    kvq.kvq_quant_write(cache, bf16(w["k_fill"]), bf16(w["v_fill"]), i32(w["fill_seq"]), i32(w["fill_pos"]), bt)
    q, off, cells, row = bf16(w["q"]), i32(w["cell_offsets"]), i32(w["cells"]), i32(w["block_table"][0])
    out = torch.empty((w["n_queries"], w["hq"], w["d"]), dtype=torch.float32, device=dev)
    ws = torch.empty(kvq.kvq_sparse_workspace_bytes(int(row.numel()), w["hkv"], w["d"]), dtype=torch.uint8,
                     device=dev)
    ms = timed(lambda: kvq.kvq_attn_sparse_int8kv(cache, q, off, cells, row, w["softmax_scale"], out=out,
                                                  workspace=ws), reps)
    pairs = int(len(w["cells"]))
    fma = pairs * w["hq"] * w["d"] * 2
    res["sparse_32k"] = {"ms_per_call": round(ms, 4), "GFMA_per_s": round(fma / ms / 1e6, 1),
                         "pairs": pairs, "workspace_bytes": int(ws.numel())}
    return res


# ----------------------------------------------------------------------------- reference arm

def bench_reference(args, world, rank):
    """The CPU oracle (test infrastructure, the plain reference) on the host cores: each step is
    a bounded sample of decode_32k (the new token's quantise-and-write, then FP64 decode of a
    subset of the query heads over all 32768 keys)."""
    import numpy as np

    import oracle
    import workloads as W
    w = W.make("decode_32k")
    hc = oracle.HostCache(w["num_blocks"], w["hkv"], w["d"])
    oracle.kv_quant_write(hc, w["k_fill"], w["v_fill"], w["fill_seq"], w["fill_pos"], w["block_table"])
    cores = os.cpu_count() or 1
    heads = int(os.environ.get("KVQ_REF_HEADS", "24"))
    units = np.arange(heads, dtype=np.int64)
    kv_bytes = w["max_ctx"] * (2 * w["hkv"] * w["d"] + 8 * w["hkv"])
    frac = heads / w["hq"]

    def step():
        oracle.kv_quant_write(hc, w["k_new"], w["v_new"], w["new_seq"], w["new_pos"], w["block_table"])
        oracle.decode_f64(hc, w["q"], w["block_table"], w["ctx_lens"], w["softmax_scale"],
                          units=units, n_threads=cores)

    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t) / args.steps
    value = kv_bytes * frac / dt / 1e9
    sample = "%d of %d query heads (units 0..%d) of decode_32k per step, all 32768 keys" % (
        heads, w["hq"], heads - 1)
    return {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "impl": "reference",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "decode_32k", "ctx": w["max_ctx"], "q_heads": w["hq"],
                   "kv_heads": w["hkv"], "head_dim": w["d"], "sample_heads": heads},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def cpu_baseline_for_line(budget_s=12.0):
    """The oracle timed on the host cores on a bounded sample of decode_32k (reported beside
    the GPU number; not the target)."""
    import numpy as np

    import oracle
    import workloads as W
    w = W.make("decode_32k")
    hc = oracle.HostCache(w["num_blocks"], w["hkv"], w["d"])
    oracle.kv_quant_write(hc, w["k_fill"], w["v_fill"], w["fill_seq"], w["fill_pos"], w["block_table"])
    cores = os.cpu_count() or 1
    kv_bytes = w["max_ctx"] * (2 * w["hkv"] * w["d"] + 8 * w["hkv"])
    units = np.arange(w["hq"], dtype=np.int64)
    t = time.perf_counter()
    n = 0
    while True:
        oracle.decode_f64(hc, w["q"], w["block_table"], w["ctx_lens"], w["softmax_scale"], units=units,
                          n_threads=cores)
        n += 1
        if time.perf_counter() - t > budget_s or n >= 64:
            break
    dt = (time.perf_counter() - t) / n
    # one core: a few query heads single-threaded, scaled to a full call (every head costs the same)
    k1 = 4
    t1 = time.perf_counter()
    oracle.decode_f64(hc, w["q"], w["block_table"], w["ctx_lens"], w["softmax_scale"], units=units[:k1],
                      n_threads=1)
    dt1 = (time.perf_counter() - t1) * w["hq"] / k1
    return {"value": round(kv_bytes / dt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "%d full decode_32k calls (all 24 query heads, FP64 Part A), %.1f s" % (n, dt * n),
            "one_core": {"value": round(kv_bytes / dt1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                         "sample": "%d of %d query heads of one decode_32k call, single-threaded, scaled to the "
                                   "full call" % (k1, w["hq"])}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--no-extra", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default=None, choices=["prefill_32k", "sparse_32k", "decode_1k", "decode_b64", "verify_32k",
                             "rope_quant_write", "prefill_first_4k"],
                    help="time only this secondary workload (profiling runs); prints its figures")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world, rank, local = dist_setup()
    if args.only:
        import torch
        from int8_kv_cache_quant_gb300 import build as kbuild
        kbuild.build()
        torch.cuda.set_device(local)
        hbm, tflops, _ = load_peaks()
        print(json.dumps(bench_extra(args, local, hbm, tflops, only=args.only)))
        return
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(bench_reference(args, world, rank)))
        return
    res = bench_decode_32k(args, world, rank, local, None)
    if rank == 0:
        hbm, tflops, _ = load_peaks()
        if not args.no_extra:
            res["extra"] = bench_extra(args, local, hbm, tflops)
        if world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline_for_line()
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
