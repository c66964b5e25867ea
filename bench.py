#!/usr/bin/env python
"""Benchmark of the DSpark per-cycle draft step on GB300; prints one JSON line.

One step = one pass of the whole hot path over one batch of synthetic input:
  1. Markov block draft, full-vocab 27B-shaped lane (num_reqs x k=15 x vocab 248320,
     rank 256, bf16 markov weights, fp32 base logits, identity d2t) -- one graph launch
  2. 2048 confidence probes (2 per cycle x 1024 cycles), 7424-wide Q8_0, threshold 0.5
  3. the four M=7 fp16 weight-stationary projections of a Qwen3-8B-shaped draft
     (K,N) = (4096,4096), (4096,1024), (4096,12288), (12288,4096), as one grouped launch

value = microseconds per step (lower is better), device time from CUDA events around
each step's work; L2 is flushed before every step (256 MiB write, then a read of the
buffer so the write-back of dirty lines is not charged to the step), outside the events.
`e2e` times the same step through the C ABI's host-buffer forms: the step's inputs copied
from pinned host memory and its outputs copied back, inside the events.  `roofline` is for
the Markov kernel (the dominant one): algorithmic bytes per launch / mean launch time.

--impl reference times the CPU oracle on the host (the reference arm of this method).
With torchrun (--gpus N > 1) every rank runs an independent replica (the path has no
cross-GPU exchange); the timed region is bracketed by barriers and the max over ranks
is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

REPO = os.path.dirname(os.path.abspath(__file__))
if REPO not in sys.path:
    sys.path.insert(0, REPO)

from dspark_draft_sampling_gb300 import synth  # noqa: E402

METRIC = "Markov draft-step µs and achieved HBM GB/s vs GB300 peak (1 GPU)"
UNIT = "us"
N_PROBES = 2048
FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------- workload ---------------
_WORKLOADS = {}


def make_workload(num_reqs: int, seed: int = 0):
    """The step's synthetic inputs (cached: the 27B lane takes seconds to draw)."""
    if (num_reqs, seed) in _WORKLOADS:
        return _WORKLOADS[(num_reqs, seed)]
    mk = synth.markov_config("full_vocab_27b", num_reqs=num_reqs, seed=seed)
    pr = synth.probe_inputs(N_PROBES, synth.PROBE_K, seed=seed)
    ws = [synth.ws_inputs(7, N, K, seed=seed + K + N) for (K, N) in synth.WS_SHAPES]
    _WORKLOADS[(num_reqs, seed)] = (mk, pr, ws)
    return mk, pr, ws


def markov_bytes(B, k, V, R, d2t=False):
    """Algorithmic bytes of one draft: markov_w2 re-read at every position, the base rows,
    the gathered markov_w1 rows and the ids."""
    return k * (V * R * 2 + B * V * 4 + B * R * 2) + B * k * 8 + (V * 4 if d2t else 0)


def probe_bytes(n, K):
    return n * (K * 4 + 8) + (K // 32) * 34


def ws_bytes(M, N, K):
    return N * K * 2 + M * K * 2 + M * N * 2


def config_dict(B):
    k, V, R = 15, 248320, 256
    return {
        "workload": (f"dspark draft step: Markov draft full-vocab 27B lane (num_reqs={B}, k={k}, "
                     f"vocab={V}, rank={R}, bf16 markov_w1/w2, fp32 base, identity d2t) + "
                     f"{N_PROBES} Q8_0 confidence probes (K=7424, threshold 0.5) + 4 M=7 fp16 "
                     "weight-stationary matvecs (K,N)=(4096,4096),(4096,1024),(4096,12288),"
                     "(12288,4096) in one grouped launch"),
        "num_reqs": B, "k": k, "vocab": V, "rank": R, "probes": N_PROBES, "probe_K": 7424,
        "ws_M": 7, "ws_shapes_KN": [list(s) for s in synth.WS_SHAPES],
        "l2": ("flushed before every step: 256 MiB write then a read of the same buffer, "
               "so no dirty lines are left; outside the timed events"),
        "timing": ("CUDA events on the launch stream around each step's work only (one CUDA graph "
                   "of the step's three calls, captured once and replayed); mean over steps; the "
                   "per-part breakdown comes from a separate loop of direct calls with events "
                   "between the parts"),
        "parallelism": "replicas",
    }


# ---------------------------------------------------------------- helpers ----------------
def max_over_ranks(values, device):
    """Element-wise max of per-rank timings (the job is as slow as its slowest replica)."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_value_us(max_ms_per_step, world):
    """Whole-job microseconds per draft step: every rank completes one step per max time."""
    return max_ms_per_step * 1000.0 / world


def read_peak():
    p = os.path.join(REPO, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def markov_source_hash():
    h = hashlib.sha256()
    for f in ("markov_tc.cu", "markov.cu", "markov.cuh", "tc.cuh", "common.cuh"):
        with open(os.path.join(REPO, "dspark_draft_sampling_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


MARKOV_PROFILE = os.path.join("profiles", "markov_draft_full_vocab_27b.md")


def recorded_traffic(B, what="traffic_bytes_per_launch"):
    """Bytes per Markov launch from the committed ncu summary (DRAM read + write for
    `traffic_bytes_per_launch`, L2-to-SM reads for `l2_to_sm_bytes_per_launch`), if it was
    taken on the current kernel source and this num_reqs; else None."""
    p = os.path.join(REPO, MARKOV_PROFILE)
    if not os.path.exists(p):
        return None
    text = open(p).read()
    src = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    if not src or src.group(1) != markov_source_hash():
        return None
    m = re.search(rf"{what}\[num_reqs={B}\]:\s*([0-9.eE+]+)", text)
    return float(m.group(1)) if m else None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- ceilings ---------------
def load_bench_library():
    """libdspark_bench.so: the measurement kernels (read bandwidth, empty launch)."""
    import ctypes

    from dspark_draft_sampling_gb300 import build

    lib = ctypes.CDLL(build.bench_lib_file())
    lib.dspark_bench_read.restype = ctypes.c_int
    lib.dspark_bench_read.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    lib.dspark_bench_empty.restype = ctypes.c_int
    lib.dspark_bench_empty.argtypes = [ctypes.c_void_p]
    lib.dspark_bench_empty_smem.restype = ctypes.c_int
    lib.dspark_bench_empty_smem.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    return lib


def measure_ceilings(dev, reps: int = 10):
    """Ceilings measured on this GPU in this run, with the same CUDA-event method as the
    kernels: the L2-to-SM read bandwidth (a 64 MiB buffer, well inside L2, read 20 times in
    one launch after a warming pass; best of `reps`), the DRAM read bandwidth (a 2 GiB buffer
    read once; best of `reps`) and the event floor (two events around one empty launch after
    an L2 flush; median of 50)."""
    import ctypes

    import torch

    lib = load_bench_library()
    stream = torch.cuda.current_stream(dev)
    s = ctypes.c_void_p(stream.cuda_stream)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sink = torch.zeros(1, dtype=torch.int64, device=dev)
    out = {}

    def best_read(buf, passes, warm):
        nbytes = buf.numel()
        best = None
        for _ in range(reps):
            if warm:
                rc = lib.dspark_bench_read(ctypes.c_void_p(buf.data_ptr()), nbytes, 1,
                                           ctypes.c_void_p(sink.data_ptr()), sms * 4, 512, s)
                assert rc == 0, rc
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            rc = lib.dspark_bench_read(ctypes.c_void_p(buf.data_ptr()), nbytes, passes,
                                       ctypes.c_void_p(sink.data_ptr()), sms * 4, 512, s)
            b.record(stream)
            b.synchronize()
            assert rc == 0, rc
            gbs = nbytes * passes / (a.elapsed_time(b) * 1e-3) / 1e9
            best = gbs if best is None else max(best, gbs)
        return best

    l2buf = torch.ones(64 << 20, dtype=torch.uint8, device=dev)
    out["l2_read_gbs"] = best_read(l2buf, 20, True)
    del l2buf
    big = torch.ones(2 << 30, dtype=torch.uint8, device=dev)
    out["dram_read_gbs"] = best_read(big, 1, False)
    del big
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    sinkf = torch.empty((), dtype=torch.int32, device=dev)
    def floor(launch):
        ts = []
        for r in range(53):
            flush.fill_(r & 0xFF)
            torch.amax(flush.view(torch.int32), dim=0, out=sinkf)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            assert launch() == 0
            b.record(stream)
            b.synchronize()
            if r >= 3:
                ts.append(a.elapsed_time(b) * 1000.0)
        return {"median": statistics.median(ts), "mean": statistics.mean(ts), "min": min(ts), "max": max(ts)}

    out["event_floor_us"] = floor(lambda: lib.dspark_bench_empty(s))
    # the same with one CTA per SM holding 200 KB of shared memory, like the draft-step kernels
    out["event_floor_200KB_smem_us"] = floor(lambda: lib.dspark_bench_empty_smem(sms, 200 * 1024, s))
    out["method"] = ("libdspark_bench read kernel (16-byte ld.global.cg, grid = 4 x SMs x 512 "
                     "threads): 64 MiB read 20 times per launch after a warming pass (L2) and "
                     "2 GiB read once (DRAM), best of 10; empty launch between two events "
                     "after an L2 flush (1 CTA; and one CTA per SM with 200 KB of shared memory), "
                     "50 samples")
    return out


# ---------------------------------------------------------------- GPU arm ----------------
def run_gpu(args, rank, world):
    import torch

    from dspark_draft_sampling_gb300 import api

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    api.load_library()
    B = args.num_reqs
    mk, pr, ws = make_workload(B, seed=0)
    k, V, R = mk["k"], mk["vocab"], mk["rank"]

    # resident inputs
    base = torch.from_numpy(mk["base"]).to(dev)
    w1 = torch.from_numpy(mk["w1"].view(np.int16)).to(dev)
    w2 = torch.from_numpy(mk["w2"].view(np.int16)).to(dev)
    prev = torch.from_numpy(mk["prev0"].copy()).to(dev)
    out_ids = torch.empty((B, k), dtype=torch.int64, device=dev)
    wsp = api.new_markov_workspace(B, k, V, R, dev)
    plan = api.MarkovPlan(base, w1, w2, None, prev, out_ids, wsp)
    wq = torch.from_numpy(pr["wq"]).to(dev)
    hid = torch.from_numpy(pr["hidden"]).to(dev)
    z = torch.empty(N_PROBES, dtype=torch.float32, device=dev)
    gate = torch.empty(N_PROBES, dtype=torch.int32, device=dev)
    Ws = [torch.from_numpy(w["W"].view(np.int16)).to(dev).view(torch.float16) for w in ws]
    Xs = [torch.from_numpy(w["X"].view(np.int16)).to(dev).view(torch.float16) for w in ws]
    Ys = [torch.empty((7, w["N"]), dtype=torch.float16, device=dev) for w in ws]
    WSs = [api.new_ws_workspace(7, w["N"], w["K"], dev) for w in ws]
    ws_group = list(zip(Ws, Xs, Ys))  # the four projections as one grouped launch
    ws_group_ws = torch.zeros(api.ws_matvec_grouped_workspace_bytes(ws_group), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_sink = torch.empty((), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush_l2(s):
        """Evict L2 (write a buffer twice its size), then read it back so the lines left
        behind are clean: otherwise the write-back of ~126 MB of dirty lines would be
        charged to the first kernel of the timed step."""
        flush.fill_(s & 0xFF)
        torch.amax(flush.view(torch.int32), dim=0, out=flush_sink)

    def step_calls(s_):
        api.markov_draft(base, w1, w2, None, prev, out_ids=out_ids, workspace=wsp, stream=s_)
        api.conf_probe(wq, hid, pr["bias"], pr["threshold"], logit_out=z, gate_out=gate, stream=s_)
        api.ws_matvec_grouped(ws_group, workspace=ws_group_ws, stream=s_)

    # The timed step is one CUDA graph of the three calls, captured once and replayed every
    # step, as a decoder replays its draft step each cycle (one graph launch instead of three;
    # the memset node and the programmatic-dependent-launch edges are kept in the graph).
    step_calls(stream)
    torch.cuda.synchronize()
    step_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(step_graph):
        step_calls(torch.cuda.current_stream())

    def step_work():
        step_graph.replay()

    kernels_per_step = 3  # Markov draft, probe batch, grouped WS matvec
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]

    for _ in range(args.warmup):
        flush_l2(1)
        step_work()
    torch.cuda.synchronize()
    if api.markov_status(wsp) != 0:
        raise RuntimeError("markov draft reported a device-side error during warm-up")

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    clocks = ClockSampler(dev.index)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    t0 = time.perf_counter()
    for s in range(args.steps):
        flush_l2(s)
        e = ev[s]
        e[0].record(stream)
        step_work()
        e[3].record(stream)
    torch.cuda.synchronize()
    barrier()
    wall = time.perf_counter() - t0
    clk = clocks.stop()
    step_ms = [ev[s][0].elapsed_time(ev[s][3]) for s in range(args.steps)]
    if api.markov_status(wsp) != 0:
        raise RuntimeError("markov draft reported a device-side error")

    # Breakdown by part, in a separate loop: events between the kernels would cut the
    # programmatic-dependent-launch overlap the timed steps above keep.
    n_parts = min(args.steps, 100)
    for s in range(n_parts):
        flush_l2(s)
        e = ev[s]
        e[0].record(stream)
        plan.launch(stream)
        e[1].record(stream)
        api.conf_probe(wq, hid, pr["bias"], pr["threshold"], logit_out=z, gate_out=gate,
                       stream=stream)
        e[2].record(stream)
        api.ws_matvec_grouped(ws_group, workspace=ws_group_ws, stream=stream)
        e[3].record(stream)
    torch.cuda.synchronize()
    markov_ms = [ev[s][0].elapsed_time(ev[s][1]) for s in range(n_parts)]
    probe_ms = [ev[s][1].elapsed_time(ev[s][2]) for s in range(n_parts)]
    ws_ms = [ev[s][2].elapsed_time(ev[s][3]) for s in range(n_parts)]
    ms_step = statistics.mean(step_ms)

    # ---- end to end through the C ABI's host-buffer forms ----
    # Every step copies its per-call inputs from pinned host memory and its results back,
    # inside the timed events.  Three lanes: the Markov draft on the launch stream, the
    # grouped WS matvec and the probe batch on two more streams.  Pinned copies are served in
    # the order they become ready, so the inputs are ordered small and urgent first: the
    # draft's 15 MB, then the projections' 0.2 MB, then the probes' 61 MB, each lane's
    # kernels overlapping the later copies.  Every lane starts after the step's start event.
    # (Splitting the probe batch into pieces on two alternating streams, so that each piece's
    # probes overlap the next piece's copy, was measured slower: 424 / 535 / 625 us for 1 / 4 /
    # 8 pieces.)
    e2e = None
    if not args.no_e2e:
        base_h = torch.from_numpy(mk["base"]).pin_memory()
        prev_h = torch.from_numpy(mk["prev0"].copy()).pin_memory()
        hid_h = torch.from_numpy(pr["hidden"]).pin_memory()
        X_h = [torch.from_numpy(w["X"].view(np.int16)).view(torch.float16).pin_memory() for w in ws]
        ids_h = torch.empty((B, k), dtype=torch.int64).pin_memory()
        gate_h = torch.empty(N_PROBES, dtype=torch.int32).pin_memory()
        Y_h = [torch.empty((7, w["N"]), dtype=torch.float16).pin_memory() for w in ws]
        ws_host = list(zip(Ws, X_h, Y_h))
        scr_m = torch.empty(api.markov_draft_host_scratch_bytes(B, k, V, R), dtype=torch.uint8, device=dev)
        scr_p = torch.empty(api.conf_probe_host_scratch_bytes(synth.PROBE_K, N_PROBES), dtype=torch.uint8,
                            device=dev)
        scr_w = torch.zeros(api.ws_matvec_grouped_host_scratch_bytes(ws_host), dtype=torch.uint8, device=dev)
        lane_w = torch.cuda.Stream(dev)
        lane_p = torch.cuda.Stream(dev)
        base_in = torch.cuda.Event()
        x_in = torch.cuda.Event()
        base_in.record(stream)  # create both events; the library records them inside each step
        x_in.record(stream)
        h2d = (base_h.numel() * 4 + prev_h.numel() * 8 + hid_h.numel() * 4
               + sum(x.numel() * 2 for x in X_h))
        d2h = ids_h.numel() * 8 + prev_h.numel() * 8 + gate_h.numel() * 4 + sum(y.numel() * 2 for y in Y_h)

        def e2e_step():
            api.markov_draft_host(base_h, w1, w2, None, prev_h, ids_h, scr_m, inputs_copied=base_in,
                                  stream=stream)
            lane_w.wait_event(base_in)
            api.ws_matvec_grouped_host(ws_host, scr_w, inputs_copied=x_in, stream=lane_w)
            lane_p.wait_event(x_in)
            api.conf_probe_host(wq, hid_h, pr["bias"], pr["threshold"], gate_h, scr_p, stream=lane_p)
            for lane in (lane_w, lane_p):
                join = torch.cuda.Event()
                join.record(lane)
                stream.wait_event(join)

        for _ in range(max(1, args.warmup)):
            flush_l2(2)
            e2e_step()
        torch.cuda.synchronize()
        e2e_ms, enqueue_s = [], []
        for s in range(args.steps):
            flush_l2(s)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            h0 = time.perf_counter()
            e2e_step()
            enqueue_s.append(time.perf_counter() - h0)
            b.record(stream)
            b.synchronize()
            e2e_ms.append(a.elapsed_time(b))
        e2e = {"value": statistics.mean(e2e_ms) * 1000.0, "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "host_enqueue_us": statistics.median(enqueue_s) * 1e6,
               "api": "dspark_markov_draft_host, dspark_ws_matvec_grouped_host and "
                      "dspark_conf_probe_host on three streams, pinned host buffers, input copies "
                      "ordered by the calls' inputs_copied events"}
    plan.close()

    ceilings = None if args.no_ceilings else measure_ceilings(dev)
    res = dict(ms_step=ms_step, wall=wall, markov_ms=statistics.mean(markov_ms), ceilings=ceilings,
               probe_ms=statistics.mean(probe_ms), ws_ms=statistics.mean(ws_ms),
               clocks=clk, e2e=e2e, kernels=kernels_per_step * args.steps,
               markov_ms_min=min(markov_ms))
    return res


def run_next_rows(dev, reps: int = 20):
    """Device times of the rows built beyond the headline step, each timed alone after an L2
    flush (median of `reps`): the Q8_0 weight-stationary matvec on the Qwen3-8B projection
    shapes and on a 4096 -> 151936 lm_head, the lm_head -> Markov draft graph (Qwen3-8B lane),
    and the probe-gated Markov draft (27B lane) with the gate open and closed.  Weights are
    drawn on the device from a seeded generator: only timing is reported here, parity is
    covered by the tests."""
    import torch

    from dspark_draft_sampling_gb300 import api

    gen = torch.Generator(device=dev)
    gen.manual_seed(1234)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    sink = torch.empty((), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    peak, _ = read_peak()

    def timed(fn):
        for _ in range(3):
            fn()
        ts = []
        for r in range(reps):
            flush.fill_(r & 0xFF)
            torch.amax(flush.view(torch.int32), dim=0, out=sink)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b) * 1000.0)
        return statistics.median(ts)

    def q8_weights(N, K):
        q = torch.randint(-127, 128, (N, K), generator=gen, device=dev, dtype=torch.int8)
        d = (torch.rand((N, K // 32), generator=gen, device=dev) * 4e-4).half().view(torch.int16)
        return q, d

    def f16(shape, sd):
        return (torch.randn(shape, generator=gen, device=dev) * sd).half()

    out = {}
    # Q8_0 projections, M = 7: each shape alone, and the four back to back in one timed region
    # (a layer's projections: programmatic dependent launch overlaps each launch's prologue
    # with the previous one's tail)
    q8_us, q8_bytes, q8_calls, q8_probs = 0.0, 0, [], []
    for (K, N) in synth.WS_SHAPES:
        q, d = q8_weights(N, K)
        X = f16((7, K), 1.0)
        Y = torch.empty((7, N), dtype=torch.float16, device=dev)
        wsq = api.new_ws_q8_workspace(7, N, K, dev)
        call = (lambda q=q, d=d, X=X, Y=Y, wsq=wsq: api.ws_matvec_q8(q, d, X, out=Y, workspace=wsq, stream=stream))
        us = timed(call)
        nb = N * K + N * (K // 32) * 2 + 7 * K * 2 + 7 * N * 2
        out[f"ws_q8_m7_{K}x{N}_us"] = us
        out[f"ws_q8_m7_{K}x{N}_frac_of_hbm"] = nb / (us * 1e-6) / 1e9 / peak
        q8_us += us
        q8_bytes += nb
        q8_calls.append(call)
        q8_probs.append((q, d, X, Y))
    out["ws_q8_qwen3_8b_4_shapes_us"] = q8_us
    out["ws_q8_qwen3_8b_GBps"] = q8_bytes / (q8_us * 1e-6) / 1e9
    seq = timed(lambda: [c() for c in q8_calls])
    out["ws_q8_qwen3_8b_4_shapes_back_to_back_us"] = seq
    out["ws_q8_qwen3_8b_back_to_back_frac_of_hbm"] = q8_bytes / (seq * 1e-6) / 1e9 / peak
    # the four as one grouped launch (dspark_ws_matvec_q8_grouped)
    wsg = api.new_ws_q8_grouped_workspace(dev)
    grp = timed(lambda: api.ws_matvec_q8_grouped(q8_probs, workspace=wsg, stream=stream))
    out["ws_q8_qwen3_8b_4_shapes_grouped_us"] = grp
    out["ws_q8_qwen3_8b_grouped_frac_of_hbm"] = q8_bytes / (grp * 1e-6) / 1e9 / peak
    del q8_calls, q8_probs
    K, N = 4096, 151936
    q, d = q8_weights(N, K)
    X = f16((7, K), 1.0)
    Y = torch.empty((7, N), dtype=torch.float16, device=dev)
    wsq = api.new_ws_q8_workspace(7, N, K, dev)
    us = timed(lambda: api.ws_matvec_q8(q, d, X, out=Y, workspace=wsq, stream=stream))
    byts = N * K + N * (K // 32) * 2 + 7 * K * 2 + 7 * N * 2
    out["ws_q8_lm_head_4096x151936_us"] = us
    out["ws_q8_lm_head_frac_of_hbm"] = byts / (us * 1e-6) / 1e9 / peak
    del q, d, wsq
    # lm_head (fp16) -> Markov draft, Qwen3-8B lane (num_reqs 1, k 7, vocab 151936, rank 256)
    k, V, R, H = 7, 151936, 256, 4096
    lm_head = f16((V, H), 0.02)
    hidden = f16((k, H), 1.0)
    w1 = f16((V, R), 0.02).view(torch.int16)
    w2 = f16((V, R), 0.02).view(torch.int16)
    prev = torch.zeros(1, dtype=torch.int64, device=dev)
    dp = api.DraftPlan(lm_head, hidden, w1, w2, None, prev, k)
    out["draft_plan_qwen3_8b_us"] = timed(lambda: dp.launch(stream))
    dp.close()
    del lm_head, dp
    # probe-gated Markov draft, 27B lane
    k, V = 15, 248320
    base = torch.randn((1, k, V), generator=gen, device=dev) * 2.0
    w1 = f16((V, R), 0.02).view(torch.int16)
    w2 = f16((V, R), 0.02).view(torch.int16)
    wq = torch.randint(0, 256, ((synth.PROBE_K // 32) * 34,), generator=gen, device=dev,
                       dtype=torch.uint8)
    wq.view(-1, 34)[:, 0] = 0x00
    wq.view(-1, 34)[:, 1] = 0x14  # every block scale = fp16 0x1400 (2^-10)
    pin = torch.randn(synth.PROBE_K, generator=gen, device=dev)
    for name, bias in (("open", 100.0), ("closed", -100.0)):  # z = bias + w.x, |w.x| << 100
        gp = api.GatedDraftPlan(wq, pin, bias, 0.5, base, w1, w2, None, prev)
        out[f"gated_plan_gate_{name}_us"] = timed(lambda: gp.launch(stream))
        gp.close()
    return out


def run_configs(dev, mk27, reps: int = 30):
    """Every configuration of the workload table timed on its own: median / p10 / p90 of
    `reps` single calls with the L2 flushed before each (cold) and without (warm, back to
    back), plus the algorithmic GB/s and the fraction of the measured HBM bandwidth (cold
    median).  Markov lanes tiny / reduced_vocab / qwen3_8b / full_vocab_27b (num_reqs 1, 4,
    8), the probe in latency mode (one probe, 4-byte readback, stream synchronization; host
    clock) and batched (2048), and the four M = 7 WS matvecs."""
    import torch

    from dspark_draft_sampling_gb300 import api

    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    sink = torch.empty((), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    peak, _ = read_peak()

    def stats(ts):
        # CUDA event timestamps on this GPU step in about 2 us, so a median of short launches
        # sits on that grid; the mean of many samples averages the step out
        ts = sorted(ts)
        q = lambda f: ts[min(len(ts) - 1, int(round(f * (len(ts) - 1))))]
        return {"median": q(0.5), "p10": q(0.1), "p90": q(0.9), "mean": statistics.mean(ts)}

    def timed(fn, cold):
        for _ in range(3):
            fn()
        ts = []
        for r in range(reps):
            if cold:
                flush.fill_(r & 0xFF)
                torch.amax(flush.view(torch.int32), dim=0, out=sink)
            else:
                # keep the GPU busy while the host enqueues the call, so the events time the
                # kernel and not the host's enqueue latency (the flush does this when cold)
                torch.cuda._sleep(100000)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b) * 1000.0)
        return stats(ts)

    def entry(fn, nbytes):
        cold, warm = timed(fn, True), timed(fn, False)
        return {"us_cold": cold, "us_warm": warm, "algorithmic_bytes": nbytes,
                "GBps_cold": nbytes / (cold["median"] * 1e-6) / 1e9,
                "frac_of_hbm_cold": nbytes / (cold["median"] * 1e-6) / 1e9 / peak,
                "frac_of_hbm_cold_mean": nbytes / (cold["mean"] * 1e-6) / 1e9 / peak}

    out = {}
    w1_27 = torch.from_numpy(mk27["w1"].view(np.int16)).to(dev)
    w2_27 = torch.from_numpy(mk27["w2"].view(np.int16)).to(dev)
    lanes = [(name, None) for name in ("tiny", "reduced_vocab", "qwen3_8b")] + [("full_vocab_27b", b) for b in (1, 4, 8)]
    for name, nreq in lanes:
        if name == "full_vocab_27b":
            c = synth.MARKOV_CONFIGS[name]
            base = torch.from_numpy(synth.markov_base(nreq, c["k"], c["vocab"], base_sd=c["base_sd"])).to(dev)
            w1, w2, d2t = w1_27, w2_27, None
            prev = torch.from_numpy(np.random.default_rng(nreq).integers(0, c["vocab"], nreq)).to(dev)
            B, k, V, R = nreq, c["k"], c["vocab"], c["rank"]
            key = f"markov_{name}_num_reqs_{nreq}"
        else:
            mk = synth.markov_config(name)
            base = torch.from_numpy(mk["base"]).to(dev)
            w1 = torch.from_numpy(mk["w1"].view(np.int16)).to(dev)
            w2 = torch.from_numpy(mk["w2"].view(np.int16)).to(dev)
            d2t = None if mk["d2t"] is None else torch.from_numpy(mk["d2t"]).to(dev)
            prev = torch.from_numpy(mk["prev0"].copy()).to(dev)
            B, k, V, R = mk["num_reqs"], mk["k"], mk["vocab"], mk["rank"]
            key = f"markov_{name}"
        # one dspark_markov_draft call (what a caller of the C ABI pays on the device); the
        # same call recorded in a CUDA graph (MarkovPlan) is reported beside it
        nbytes = markov_bytes(B, k, V, R, d2t is not None)
        wsd = api.new_markov_workspace(B, k, V, R, dev)
        ids = torch.empty((B, k), dtype=torch.int64, device=dev)
        out[key] = entry(lambda: api.markov_draft(base, w1, w2, d2t, prev, out_ids=ids, workspace=wsd,
                                                  stream=stream), nbytes)
        out[key]["us_per_position_cold"] = out[key]["us_cold"]["median"] / k
        out[key]["kernel"] = api.markov_kernel_for(B, k, V, R)
        plan = api.MarkovPlan(base, w1, w2, d2t, prev)
        pl = entry(lambda: plan.launch(stream), nbytes)
        out[key]["graph_plan"] = {"us_cold": pl["us_cold"], "us_warm": pl["us_warm"]}
        plan.close()
        if out[key]["kernel"] == "cluster":
            # the same lane on the grid kernel, for comparison (direct calls)
            out[key]["grid_kernel"] = entry(
                lambda: api.markov_draft(base, w1, w2, d2t, prev, out_ids=ids, workspace=wsd, stream=stream,
                                         kernel="grid"), nbytes)
        del plan, base
    pr = synth.probe_inputs(N_PROBES, synth.PROBE_K, seed=0)
    wq = torch.from_numpy(pr["wq"]).to(dev)
    hid = torch.from_numpy(pr["hidden"]).to(dev)
    z = torch.empty(N_PROBES, dtype=torch.float32, device=dev)
    g = torch.empty(N_PROBES, dtype=torch.int32, device=dev)
    out["probe_batched_2048"] = entry(
        lambda: api.conf_probe(wq, hid, pr["bias"], pr["threshold"], logit_out=z, gate_out=g, stream=stream),
        probe_bytes(N_PROBES, synth.PROBE_K))
    g_h = torch.empty(1, dtype=torch.int32).pin_memory()
    h1 = hid[:1].contiguous()
    lat = []
    for r in range(reps + 3):
        t0 = time.perf_counter()
        api.conf_probe(wq, h1, pr["bias"], pr["threshold"], gate_out=g[:1], stream=stream)
        g_h.copy_(g[:1], non_blocking=True)
        stream.synchronize()
        if r >= 3:
            lat.append((time.perf_counter() - t0) * 1e6)
    out["probe_latency_1_with_4B_readback"] = {"us_host_clock": stats(lat),
                                                "how": "launch, 4-byte cudaMemcpyAsync to pinned memory, stream sync"}
    # the same probe with the gate stored by the kernel straight into pinned host memory and
    # the host polling that word: no copy and no stream synchronization on the host path
    g_map = torch.empty(1, dtype=torch.int32).pin_memory()
    g_np = g_map.numpy()
    lat = []
    for r in range(reps + 3):
        g_np[0] = -1
        t0 = time.perf_counter()
        api.conf_probe(wq, h1, pr["bias"], pr["threshold"], gate_out=g_map, stream=stream)
        while g_np[0] == -1:
            pass
        if r >= 3:
            lat.append((time.perf_counter() - t0) * 1e6)
    stream.synchronize()
    out["probe_latency_1_mapped_gate"] = {"us_host_clock": stats(lat),
                                          "how": "api.conf_probe (Python wrapper), the kernel stores the gate "
                                                 "into pinned host memory, the host polls the 4-byte word"}
    # the same through the C ABI with the arguments marshalled once (what a C caller pays)
    import ctypes

    lib = api.load_library()
    cargs = (ctypes.c_void_p(wq.data_ptr()), ctypes.c_void_p(h1.data_ptr()), ctypes.c_float(pr["bias"]),
             ctypes.c_float(pr["threshold"]), synth.PROBE_K, 1, None, ctypes.c_void_p(g_map.data_ptr()),
             ctypes.c_void_p(stream.cuda_stream))
    fn = lib.dspark_conf_probe
    lat = []
    for r in range(reps + 3):
        g_np[0] = -1
        t0 = time.perf_counter()
        rc = fn(*cargs)
        while g_np[0] == -1:
            pass
        if r >= 3:
            lat.append((time.perf_counter() - t0) * 1e6)
        assert rc == 0
    stream.synchronize()
    out["probe_latency_1_mapped_gate_c_abi"] = {"us_host_clock": stats(lat),
                                                "how": "dspark_conf_probe through ctypes with prepared arguments, "
                                                       "gate stored into pinned host memory, host polls"}
    # the same through the Python API's prepared call (api.ProbeCall.decide)
    call = api.ProbeCall(wq, h1, pr["bias"], pr["threshold"], gate_out=g_map, stream=stream)
    lat = []
    for r in range(reps + 3):
        t0 = time.perf_counter()
        call.decide()
        if r >= 3:
            lat.append((time.perf_counter() - t0) * 1e6)
    stream.synchronize()
    out["probe_latency_1_probecall"] = {"us_host_clock": stats(lat),
                                        "how": "api.ProbeCall.decide(): arguments marshalled once, gate stored "
                                               "into pinned host memory, host polls"}
    for (K, N) in synth.WS_SHAPES:
        w = synth.ws_inputs(7, N, K)
        W = torch.from_numpy(w["W"].view(np.int16)).to(dev).view(torch.float16)
        X = torch.from_numpy(w["X"].view(np.int16)).to(dev).view(torch.float16)
        Y = torch.empty((7, N), dtype=torch.float16, device=dev)
        wsp = api.new_ws_workspace(7, N, K, dev)
        out[f"ws_matvec_m7_{K}x{N}"] = entry(lambda: api.ws_matvec(W, X, out=Y, workspace=wsp, stream=stream),
                                             ws_bytes(7, N, K))
        # the prior-art library path beside it (cuBLAS through torch.matmul, fp16, M = 7):
        # context only, not part of the draft step
        Wt = W.t()
        out[f"cublas_matmul_m7_{K}x{N}"] = entry(lambda: torch.matmul(X, Wt, out=Y), ws_bytes(7, N, K))
    return out


def cpu_oracle_step(mk, pr, ws):
    """One step of the oracle on the host: the same three parts, single-threaded fp64."""
    import oracle

    t0 = time.perf_counter()
    oracle.markov_draft(mk["base"], mk["w1"], mk["w2"], mk["d2t"], mk["prev0"])
    t1 = time.perf_counter()
    oracle.conf_probe(pr["wq"], pr["hidden"], pr["bias"], pr["threshold"])
    t2 = time.perf_counter()
    for w in ws:
        oracle.ws_matvec(w["W"], w["X"])
    t3 = time.perf_counter()
    return t3 - t0, (t1 - t0, t2 - t1, t3 - t2)


def oracle_sample(mk, pr, ws, f):
    """The workload cut to about a fraction f of a step, for timing the oracle within a
    budget: the first k' of the k draft positions, the first n' probes and the first N' rows
    of each projection (contiguous copies, made outside any timing).  Returns the sample and
    the factor that scales each part's time back to the full step."""
    k = mk["base"].shape[1]
    kk = max(1, min(k, round(k * f)))
    n = pr["hidden"].shape[0]
    nn = max(1, min(n, round(n * f)))
    mk_s = dict(mk, base=np.ascontiguousarray(mk["base"][:, :kk]))
    pr_s = dict(pr, hidden=np.ascontiguousarray(pr["hidden"][:nn]))
    ws_s = []
    for w in ws:
        nr = max(1, min(w["N"], round(w["N"] * f)))
        ws_s.append(dict(w, W=np.ascontiguousarray(w["W"][:nr]), N=nr))
    full_ws = sum(w["N"] * w["K"] for w in ws)
    part_ws = sum(w["N"] * w["K"] for w in ws_s)
    desc = (f"{kk}/{k} draft positions, {nn}/{n} probes and {ws_s[0]['N']}/{ws[0]['N']} .. "
            f"{ws_s[-1]['N']}/{ws[-1]['N']} rows of the projections")
    return mk_s, pr_s, ws_s, (k / kk, n / nn, full_ws / part_ws), desc


def cpu_baseline(B):
    import oracle

    oracle.build()
    mk, pr, ws = make_workload(B, seed=0)
    total, parts = cpu_oracle_step(mk, pr, ws)
    return {"value": total * 1e6, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": ("one full step of the same workload (Markov draft + 2048 probes + 4 WS "
                       "matvecs), single-threaded fp64 C oracle"),
            "parts_s": {"markov": parts[0], "probe": parts[1], "ws": parts[2]},
            "host_cpus": os.cpu_count()}


def markov_roofline(B, mb, t_s, peak, peak_kind, ceil):
    """Roofline of the Markov kernel.  `achieved` / `frac` follow the pages' accounting
    (markov_w2 re-read whole at every position) against the measured HBM copy bandwidth;
    because each position starts on rows the previous one left in L2, that accounting can
    exceed 1.  So the line also states the two ceilings the kernel actually streams against:
    its DRAM bytes (ncu, committed summary) over the HBM peak, and its L2-to-SM bytes over
    the L2 read bandwidth measured in this run, and names the one that binds (or neither)."""
    traffic = recorded_traffic(B)
    l2b = recorded_traffic(B, "l2_to_sm_bytes_per_launch")
    l2_src = "ncu l1tex__m_xbar2l1tex_read_bytes (committed summary)"
    if l2b is None:
        l2b, l2_src = float(mb), "algorithmic bytes (every byte reaches the SMs from L2 once)"
    achieved = mb / t_s / 1e9
    r = {"kernel": "markov_tc_kernel (k=15 positions, one launch)",
         "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
         "frac": achieved / peak, "peak_source": peak_kind,
         "algorithmic_bytes_per_launch": mb, "traffic": traffic,
         "traffic_source": (f"dram__bytes_read.sum + dram__bytes_write.sum from {MARKOV_PROFILE}, "
                            "used only while the kernel sources hash to the value recorded there"),
         "l2_to_sm_bytes_per_launch": l2b, "l2_to_sm_source": l2_src}
    l2_peak = ceil.get("l2_read_gbs") if ceil else None
    if r["frac"] > 1.0:
        r["frac_note"] = ("frac counts markov_w2 once per position (the pages' accounting); after the "
                          "first position about half of it is served from L2, so frac exceeds 1. "
                          "frac_dram and frac_l2 divide the kernel's measured DRAM and L2-to-SM bytes by "
                          "the HBM copy peak and the L2 read bandwidth measured in this run")
    fr = {}
    if traffic:
        fr["dram"] = traffic / t_s / 1e9 / peak
        r["frac_dram"] = fr["dram"]
    if l2_peak:
        fr["l2"] = l2b / t_s / 1e9 / l2_peak
        r["frac_l2"] = fr["l2"]
        r["l2_peak"] = l2_peak
    if fr:
        name = max(fr, key=fr.get)
        t_min = max((traffic / (peak * 1e9)) if traffic else 0.0,
                    (l2b / (l2_peak * 1e9)) if l2_peak else 0.0)
        r["frac_ceiling"] = t_min / t_s
        if fr[name] >= 0.75:
            r["binding"] = name
        else:
            r["binding"] = ("neither DRAM nor L2 bandwidth: the chain of k grid-wide argmax "
                            "barriers and the bytes each SM keeps in flight bound the kernel")
    return r


def run_one_kernel(name: str) -> int:
    """Runs one kernel of the workload twice on cuda:0 and exits, for a profiler capture of a
    single launch (`ncu -k ... -s 1 -c 1`): `ws_4096x4096` (the fp16 weight-stationary matvec,
    M = 7), `ws_grouped_qwen3_8b` (the four fp16 projections in one launch), `probe_2048` (the
    batched confidence probe), `q8_lm_head` (the Q8_0 matvec,
    4096 -> 151936, M = 7), `q8_grouped_qwen3_8b` (the four Q8_0 projections in one launch),
    `markov_tiny` (the tiny Markov lane on the single-cluster kernel).  No timing is taken."""
    import torch

    from dspark_draft_sampling_gb300 import api

    api.load_library()
    dev = torch.device("cuda", 0)
    if name == "ws_4096x4096":
        w = synth.ws_inputs(7, 4096, 4096, seed=4096 + 4096)
        W = torch.from_numpy(w["W"].view(np.int16)).to(dev).view(torch.float16)
        X = torch.from_numpy(w["X"].view(np.int16)).to(dev).view(torch.float16)
        Y = torch.empty((7, 4096), dtype=torch.float16, device=dev)
        wsp = api.new_ws_workspace(7, 4096, 4096, dev)
        call = lambda: api.ws_matvec(W, X, out=Y, workspace=wsp)
    elif name == "probe_2048":
        pr = synth.probe_inputs(N_PROBES, synth.PROBE_K, seed=0)
        wq = torch.from_numpy(pr["wq"]).to(dev)
        hid = torch.from_numpy(pr["hidden"]).to(dev)
        call = lambda: api.conf_probe(wq, hid, pr["bias"], pr["threshold"])
    elif name == "q8_grouped_qwen3_8b":
        gen = torch.Generator(device=dev)
        gen.manual_seed(1)
        probs = []
        for (K, N) in synth.WS_SHAPES:
            q = torch.randint(-127, 128, (N, K), generator=gen, device=dev, dtype=torch.int8)
            d = (torch.rand((N, K // 32), generator=gen, device=dev) * 4e-4).half().view(torch.int16)
            X = torch.randn((7, K), generator=gen, device=dev).half()
            probs.append((q, d, X, torch.empty((7, N), dtype=torch.float16, device=dev)))
        wsg = api.new_ws_q8_grouped_workspace(dev)
        call = lambda: api.ws_matvec_q8_grouped(probs, workspace=wsg)
    elif name == "ws_grouped_qwen3_8b":
        gen = torch.Generator(device=dev)
        gen.manual_seed(1)
        probs = []
        for (K, N) in synth.WS_SHAPES:
            W = (torch.randn((N, K), generator=gen, device=dev) * 0.02).half()
            X = torch.randn((7, K), generator=gen, device=dev).half()
            probs.append((W, X, torch.empty((7, N), dtype=torch.float16, device=dev)))
        wsg = torch.zeros(api.ws_matvec_grouped_workspace_bytes(probs), dtype=torch.uint8, device=dev)
        call = lambda: api.ws_matvec_grouped(probs, workspace=wsg)
    elif name == "markov_tiny":
        mk = synth.markov_config("tiny")
        base = torch.from_numpy(mk["base"]).to(dev)
        w1 = torch.from_numpy(mk["w1"].view(np.int16)).to(dev)
        w2 = torch.from_numpy(mk["w2"].view(np.int16)).to(dev)
        prev = torch.from_numpy(mk["prev0"].copy()).to(dev)
        wsm = api.new_markov_workspace(1, 4, 4096, 64, dev)
        call = lambda: api.markov_draft(base, w1, w2, None, prev, workspace=wsm)
    elif name == "q8_lm_head":
        gen = torch.Generator(device=dev)
        gen.manual_seed(1)
        N, K = 151936, 4096
        q = torch.randint(-127, 128, (N, K), generator=gen, device=dev, dtype=torch.int8)
        d = (torch.rand((N, K // 32), generator=gen, device=dev) * 4e-4).half().view(torch.int16)
        X = torch.randn((7, K), generator=gen, device=dev).half()
        Y = torch.empty((7, N), dtype=torch.float16, device=dev)
        wsq = api.new_ws_q8_workspace(7, N, K, dev)
        call = lambda: api.ws_matvec_q8(q, d, X, out=Y, workspace=wsq)
    else:
        raise SystemExit(f"unknown --kernel {name}")
    for _ in range(2):
        call()
    torch.cuda.synchronize()
    print(f"{name}: ok")
    return 0


# ---------------------------------------------------------------- main -------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--reference-budget-s", type=float, default=90.0,
                    help="--impl reference: seconds of oracle time the timed steps may take")
    ap.add_argument("--num-reqs", type=int, default=8,
                    help="requests of the Markov draft (the 27B lane's largest configuration is 8)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-ceilings", action="store_true",
                    help="skip the in-run L2 / DRAM read bandwidth and event-floor measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-next-rows", action="store_true",
                    help="skip the separately timed rows beyond the headline step")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration sweep (median/p10/p90, cold and warm L2)")
    ap.add_argument("--kernel", choices=["ws_4096x4096", "ws_grouped_qwen3_8b", "probe_2048", "q8_lm_head",
                                         "q8_grouped_qwen3_8b", "markov_tiny"],
                    help="run only this kernel of the workload twice, untimed (for a profiler)")
    args = ap.parse_args()
    if args.kernel:
        return run_one_kernel(args.kernel)
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)

    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", args.gpus))
    B = args.num_reqs

    if args.impl == "reference":
        if rank != 0:
            return 0
        import oracle

        oracle.build()
        mk, pr, ws = make_workload(B, seed=0)
        # One full step first (also a warm-up).  If the requested steps would take longer
        # than the budget, every step then times a proportional sample of the workload and
        # scales each part's time back to a full step (the oracle's cost is linear in the
        # positions, the probes and the projection rows).
        full_s, _ = cpu_oracle_step(mk, pr, ws)
        f = min(1.0, args.reference_budget_s / (max(1, args.steps + args.warmup) * full_s))
        if f < 1.0:
            mk_s, pr_s, ws_s, scale, desc = oracle_sample(mk, pr, ws, f)
            sample = (f"each step times {desc} of the workload (about {f:.3f} of it, so that the "
                      f"run fits a {args.reference_budget_s:.0f} s budget) and scales each part to "
                      "the full step; single-threaded fp64 C oracle")
        else:
            mk_s, pr_s, ws_s, scale = mk, pr, ws, (1.0, 1.0, 1.0)
            sample = "each step is one full step of the workload, single-threaded fp64 C oracle"
        for _ in range(args.warmup):
            cpu_oracle_step(mk_s, pr_s, ws_s)
        times = []
        for _ in range(args.steps):
            _, parts = cpu_oracle_step(mk_s, pr_s, ws_s)
            times.append(sum(p * c for p, c in zip(parts, scale)))
        us = statistics.mean(times) * 1e6
        line = {
            "impl": "reference", "metric": METRIC, "value": us, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": us / 1000.0, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(B),
            "cpu_baseline": {"value": us, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample, "full_step_us": full_s * 1e6},
            "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line))
        return 0

    import torch

    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    res = run_gpu(args, rank, world)

    ms_step = res["ms_step"]
    markov_ms = res["markov_ms"]
    if world > 1:
        ms_step, markov_ms, _ = max_over_ranks([ms_step, markov_ms, res["wall"]], "cuda")
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    k, V, R = 15, 248320, 256
    mb = markov_bytes(B, k, V, R)
    pb = probe_bytes(N_PROBES, synth.PROBE_K)
    wb = sum(ws_bytes(7, N, K) for (K, N) in synth.WS_SHAPES)
    peak, peak_kind = read_peak()
    achieved = mb / (markov_ms * 1e-3) / 1e9
    roof = markov_roofline(B, mb, markov_ms * 1e-3, peak, peak_kind, res["ceilings"])
    line = {
        "metric": METRIC,
        "value": job_value_us(ms_step, world),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded numpy PCG64; shapes and distributions of the pages' lanes)",
        "config": config_dict(B),
        "roofline": roof,
        "ceilings": res["ceilings"],
        "parts": {
            "markov_draft_us": markov_ms * 1000.0,
            "markov_us_per_position": markov_ms * 1000.0 / k,
            "markov_GBps": achieved,
            "conf_probe_batch_us": res["probe_ms"] * 1000.0,
            "conf_probe_us_per_probe": res["probe_ms"] * 1000.0 / N_PROBES,
            "conf_probe_GBps": pb / (res["probe_ms"] * 1e-3) / 1e9,
            "ws_matvec_4_shapes_grouped_us": res["ws_ms"] * 1000.0,
            "ws_matvec_GBps": wb / (res["ws_ms"] * 1e-3) / 1e9,
        },
        "gpu_launches": res["kernels"],
        "clocks": res["clocks"],
        "e2e": res["e2e"],
        "wall_s_timed_region": res["wall"],
    }
    if not args.no_next_rows:
        line["next_rows"] = run_next_rows(torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0))))
    if not args.no_configs:
        line["configs"] = run_configs(torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0))),
                                      make_workload(B, seed=0)[0])
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(B)
    print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
