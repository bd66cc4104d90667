"""Benchmark of one decode step of paged GQA attention: RoPE + KV store of the new token, then
decode over the paged cache.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload mix64] [--impl reference]
                    [--split-step]

A step is one pass of the whole hot path over one batch, for each layer of the workload:
pa_decode_step, which rotates and stores every sequence's new token and attends over every
cached context in one launch (plus the merge of split contexts); or, with --split-step,
pa_rope_kv_store followed by pa_decode.  The fused step sets PA_STEP_EARLY_METADATA on every
layer after the first (lengths and block tables are written before the timed steps, never by
a kernel), so each such layer's kernel resolves its work while the previous one finishes.  The metric is KV-cache bytes read
per second: sum(context_lens) * Hkv * D * 2 B (K and V) per layer per step, over the step's
device time.  L2 is flushed between timed steps,
outside the timed events, because the workloads' caches fit in L2: a 512 MiB write, then a
read of the same buffer so that no dirty flush lines are written back inside the timed step.

The printed JSON line carries:
  value / ms_per_step  from CUDA events around each step, inputs resident in HBM;
  e2e                  the same metric when every step also copies its inputs (new-token
                       q/k/v, positions, slots, block tables, lengths) from pinned host
                       memory and reads the output back, all inside the timed region (the
                       copies and calls replayed as one CUDA graph, like the device step); the
                       two copies are pa_stage_copy kernels, and e2e.copy_engine repeats the
                       step with cudaMemcpyAsync transfers instead;
  roofline             the step's decode call (its partition kernel plus the merge kernel)
                       on one layer, timed alone with CUDA events, against the measured HBM
                       copy bandwidth; beside it gather_floor_*: pa_gather_checksum on the same
                       layer, the same tile gather with no attention and no merge;
  configs              every named workload's step (tiny, qwen_b1 with its 28 layers, mix64,
                       prefix32, long4 with 512-token partitions): time, GB/s, fraction of the
                       HBM peak, decode tokens/s; and mix64_x28, the mix64 layer as the attention
                       of a 28-layer model step, 28 device copies of its caches (--no-configs
                       skips it);
  cpu_baseline         the fp64 oracle on the host cores over a bounded sample;
  fp8_kv               the step's decode on E4M3 caches (pa_decode_fp8, pa_decode_step_fp8),
                       bandwidth counted on the E4M3 bytes, and beside it gather_floor_*:
                       pa_gather_checksum_fp8, the same tile gather alone; fp8_kv.x28: the
                       layer as the attention of a 28-layer step (--no-fp8 skips it);
  prefill              pa_prefill on two prefill workloads, TFLOP/s against the measured bf16
                       dense peak, and pa_rope_kv_store of their new tokens against the HBM
                       copy bandwidth (--no-prefill skips it);
  block_ops            pa_copy_blocks over K and V of 28 layers: copy-on-write inside the
                       device pools, swap out / in of a 2048-token sequence to page-locked
                       host pools, beside a plain memcpy of the same bytes (--no-block-ops
                       skips it).
With --gpus N under torchrun each rank runs its own batch (weak scaling, no collective on
the data path); value is all ranks' bytes over the slowest rank's time.
`--impl reference` times the oracle instead, on the host cores (rank 0 only).
"""

from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

from paged_kv_cache_244_gb300 import workloads as W  # noqa: E402

METRIC = "paged GQA decode: KV-cache HBM GB/s (% of GB300 peak) and attention tokens/s"

# DRAM bytes (read + write) of one call of the step's decode (partition + merge kernels), from
# an ncu capture of `bench.py --steps 5 --warmup 3 --no-cpu-baseline`, keyed by the workload,
# the step form and a hash of the CUDA sources it was taken on: once a kernel changes, the
# hash no longer matches and roofline.traffic is reported as null until it is captured again.
MEASURED_TRAFFIC = {
    ("mix64", "fused", "66bc39d37e6f7fac"): 122108928 + 3006464 + 4185600,
    ("prefix32", "fused", "66bc39d37e6f7fac"): 4348672 + 0 + 3823360,
    ("long4", "fused", "66bc39d37e6f7fac"): 83981056 + 2105088 + 4823040,
}
FLUSH_BYTES = 512 << 20
FALLBACK_HBM_GBS = 6800.0


def kernel_source_hash() -> str:
    """Hash of the code the decode kernels compile from (their file, the device helpers, the
    launch header), with comments and whitespace removed: editing a comment keeps the hash."""
    import hashlib
    import re
    csrc = ROOT / "paged_kv_cache_244_gb300" / "csrc"
    h = hashlib.sha256()
    for name in ("paged_decode.cu", "pa_device.cuh", "pa_launch.h"):
        text = (csrc / name).read_text()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(name.encode())
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def bf16_peak():
    try:
        d = json.loads((ROOT / "MEASURED_PEAKS.json").read_text())
        return float(d["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def hbm_peak():
    p = ROOT / "MEASURED_PEAKS.json"
    try:
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------------ clocks ----

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the benchmark runs."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        inside = [r for t, r in self.rows if t0 <= t <= t1]
        note = "samples inside the timed region"
        if not inside:  # timed region shorter than the sampling period: nearest samples
            inside = [r for t, r in self.rows if t0 - 0.5 <= t <= t1 + 0.5]
            note = "timed region shorter than the 100 ms sampling period; nearest samples"
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            try:
                sm.append(float(r[2]))
                smax.append(float(r[3]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, r[6:10]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "note": note}


# --------------------------------------------------------------------- GPU path ----

class DeviceStep:
    """A workload resident on the GPU and one step of the hot path over it."""

    def __init__(self, w: W.Workload, torch, binding, fused: bool = True, early: bool = True,
                 replicate_layers: int = 0):
        """replicate_layers > 0: run that many layers, each with its own device copy of the
        workload's first layer (inputs and caches), instead of the workload's own layers."""
        self.w, self.torch, self.pa, self.fused, self.early = w, torch, binding, fused, early
        dev = torch.device("cuda")

        def bf(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

        L = w.num_layers
        src = [0] * replicate_layers if replicate_layers else list(range(L))
        self.num_layers = len(src)
        first = {}

        def layer(arr, i):
            if i not in first.setdefault(id(arr), {}):
                first[id(arr)][i] = bf(arr[i])
                return first[id(arr)][i]
            return first[id(arr)][i].clone()

        self.q = [layer(w.q, i) for i in src]
        self.q_src = [bf(w.q[i]) for i in src]
        self.k = [layer(w.k, i) for i in src]
        self.v = [layer(w.v, i) for i in src]
        self.k_cache = [layer(w.k_cache, i) for i in src]
        self.v_cache = [layer(w.v_cache, i) for i in src]
        self.positions = torch.from_numpy(w.positions).to(dev)
        self.slots = torch.from_numpy(w.slot_mapping).to(dev)
        self.cos_sin = torch.from_numpy(w.cos_sin).to(dev)
        self.block_tables = torch.from_numpy(w.block_tables).to(dev)
        self.context_lens = torch.from_numpy(w.context_lens).to(dev)
        self.out = [torch.empty_like(q) for q in self.q]
        self.P = binding.decode_partition_tokens(w.num_q_heads, w.num_kv_heads, w.num_seqs,
                                                 w.max_context_len, w.partition_tokens)
        self.workspace = binding.decode_workspace(self.q[0], self.k_cache[0], w.max_context_len, self.P)
        # per layer: the (fused) decode kernel and the merge kernel, plus the RoPE + store
        # kernel when it runs apart
        self.launches_per_step = self.num_layers * (2 if fused else 3)

    def rope_store(self, i):
        self.pa.rope_kv_store(self.q[i], self.k[i], self.v[i], self.positions, self.cos_sin,
                              self.slots, self.k_cache[i], self.v_cache[i])

    def decode(self, i):
        w = self.w
        self.pa.decode(self.q[i], self.k_cache[i], self.v_cache[i], self.block_tables,
                       self.context_lens, w.max_context_len, w.scale, partition_tokens=self.P,
                       workspace=self.workspace, out=self.out[i])

    def decode_step(self, i):
        # Early metadata on every layer after the first: the lengths and block table are written
        # before the timed steps and never by a kernel, so such a layer's kernel may resolve its
        # work while the previous layer's kernels finish.  The first layer follows whatever ran
        # before the step (here the L2 flush), with nothing of ours to overlap.
        w = self.w
        self.pa.decode_step(self.q[i], self.k[i], self.v[i], self.cos_sin, self.k_cache[i],
                            self.v_cache[i], self.block_tables, self.context_lens,
                            w.max_context_len, w.scale, partition_tokens=self.P,
                            workspace=self.workspace, out=self.out[i],
                            early_metadata=self.early and i > 0)

    def step(self):
        for i in range(self.num_layers):
            if self.fused:
                self.decode_step(i)
            else:
                self.rope_store(i)
                self.decode(i)


def run_gpu(args, rank, world, dist):
    import torch

    from paged_kv_cache_244_gb300 import _build, binding

    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local_rank)
    if rank == 0:
        _build.build()
    if dist is not None:
        dist.barrier()
    base = W.make(args.workload)
    w = base if rank == 0 else W.make(args.workload, seed=base.seed + 1000 * rank)
    if args.partition_tokens is not None:
        w.partition_tokens = args.partition_tokens
    st = DeviceStep(w, torch, binding, fused=not args.split_step, early=not args.no_early_metadata)
    stream = torch.cuda.current_stream()
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    sink = torch.empty(1, dtype=torch.float32, device="cuda")

    def flush_l2():
        # Write a buffer larger than L2, then read it back: the write evicts the inputs, the
        # read evicts the written (dirty) lines so that their write-back is not billed to
        # the timed step.
        flush.fill_(1.0)
        torch.sum(flush.view(1, -1), dim=1, out=sink)
    bytes_step = w.kv_bytes_per_layer() * w.num_layers

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    def timed_loop(fn, steps):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for a, b in evs:
            flush_l2()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    # warm-up (also builds the library state and the kernels' shared-memory attributes)
    for _ in range(args.warmup):
        st.step()
    rc, flags = binding.get_device_status()
    if rc != 0:
        raise RuntimeError(f"device status after warm-up: {rc} flags {flags:#x}")

    # The step as a CUDA graph (all its launches recorded once, replayed per step), as a serving
    # engine runs a decode step; --no-graph launches every call from Python instead.
    step_fn, graph_note = st.step, "eager launches"
    if not args.no_graph:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                st.step()
            graph.replay()
            torch.cuda.synchronize()
            step_fn, graph_note = graph.replay, "CUDA graph of the step's launches"
        except Exception as e:  # capture unsupported here: keep eager launches
            graph_note = f"eager launches (graph capture failed: {type(e).__name__})"
    rc, flags = binding.get_device_status()
    if rc != 0:
        raise RuntimeError(f"device status after capture: {rc} flags {flags:#x}")

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    barrier()
    t_wall0 = time.time()
    step_ms = timed_loop(step_fn, args.steps)
    barrier()
    t_wall1 = time.time()
    time.sleep(0.25)
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)
    total_ms = float(np.sum(step_ms))

    # the step's decode call on one layer alone (roofline of the dominant kernel), same flush
    # discipline; then the unfused calls for comparison
    dec_ms = timed_loop(lambda: (st.decode_step(0) if st.fused else st.decode(0)), args.steps)
    dec_avg = float(np.mean(dec_ms))
    rope_ms = timed_loop(lambda: st.rope_store(0), max(3, args.steps // 4))
    plain_ms = timed_loop(lambda: st.decode(0), max(3, args.steps // 4))
    # the floor of the decode's access pattern: the same gather of K/V tiles (same kernel shape,
    # block tables, TMA boxes, stage ring, persistent grid) with no attention and no merge
    xor_buf = torch.zeros((w.num_seqs, w.num_kv_heads), dtype=torch.int32, device="cuda")
    floor_ms = timed_loop(lambda: binding.gather_checksum(st.k_cache[0], st.v_cache[0], st.block_tables,
                                                          st.context_lens, w.max_context_len,
                                                          w.num_q_heads, out_xor=xor_buf), args.steps)
    floor_avg = float(np.mean(floor_ms))

    # end to end through the public API with host buffers
    e2e = run_e2e(args, st, torch, binding, flush_l2)
    e2e_ce = run_e2e(args, st, torch, binding, flush_l2, copy_engine=True)
    configs = None if args.no_configs else all_configs(args, torch, binding, flush_l2, timed_loop, world)
    blocks = None if args.no_block_ops else block_ops(torch, binding, flush_l2, timed_loop, w)
    fp8 = None if args.no_fp8 else fp8_kv(torch, binding, timed_loop, st, args.steps)
    pre = None if args.no_prefill else prefill_runs(torch, binding, timed_loop, max(5, args.steps // 4))

    rc, flags = binding.get_device_status()
    if rc != 0:
        raise RuntimeError(f"device status after timing: {rc} flags {flags:#x}")

    # max over ranks of the timed device time; sum of bytes
    (total_ms_max, e2e_ms_max, e2e_ce_ms_max), (all_bytes,) = reduce_over_ranks(
        [total_ms, e2e["ms"], e2e_ce["ms"]], [float(bytes_step)], dist, torch.device("cuda"))
    if rank != 0:
        return None

    peak, peak_kind = hbm_peak()
    if args.traffic is not None:
        traffic, traffic_note = args.traffic, "--traffic"
    else:
        traffic = MEASURED_TRAFFIC.get((w.name, "fused" if st.fused else "split", kernel_source_hash()))
        traffic_note = ("ncu dram__bytes_read.sum + dram__bytes_write.sum of the decode kernels, "
                        "same sources" if traffic is not None else "no ncu capture of these sources")
    gbs = all_bytes * args.steps / (total_ms_max * 1e-3) / 1e9
    dec_bytes = w.kv_bytes_per_layer()
    achieved = dec_bytes / (dec_avg * 1e-3) / 1e9
    tokens_per_s = world * w.num_seqs * args.steps / (total_ms_max * 1e-3)
    cfg = config_of(w, st, world)
    cfg["launch"] = graph_note
    line = {
        "metric": METRIC,
        "value": round(gbs, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms_max / args.steps, 6),
        # spread of this rank's per-step event times (each step timed alone after the flush)
        "step_us_percentiles": {k: round(1e3 * float(v), 3) for k, v in
                                zip(("p10", "p50", "p90"), np.percentile(step_ms, [10, 50, 90]))},
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded splitmix64 -> Box-Muller -> bf16)",
        "pct_of_peak": round(100.0 * gbs / peak, 2),
        "tokens_per_s": round(tokens_per_s, 1),
        "config": cfg,
        "roofline": {
            "kernel": ("pa_decode_step (decode_partition_kernel<fused> + decode_merge_kernel)"
                       if st.fused else "pa_decode (decode_partition_kernel + decode_merge_kernel)"),
            "bound": "hbm",
            "achieved": round(achieved, 2),
            "peak": peak,
            "peak_kind": f"{peak_kind} hbm_gbs (copy, burst)",
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "traffic_source": traffic_note,
            "algorithmic_bytes_per_launch": dec_bytes,
            "avg_launch_ms": round(dec_avg, 6),
            # pa_gather_checksum on the same layer: the decode's tile gather alone
            "gather_floor_us": round(floor_avg * 1e3, 3),
            "gather_floor_GBps": round(dec_bytes / (floor_avg * 1e-3) / 1e9, 2),
            "gather_floor_frac": round(dec_bytes / (floor_avg * 1e-3) / 1e9 / peak, 4),
            "decode_over_floor": round(dec_avg / floor_avg, 4),
        },
        "rope_kv_store_us": round(1e3 * float(np.median(rope_ms)), 3),
        "pa_decode_us": round(1e3 * float(np.mean(plain_ms)), 3),
        "e2e": {"value": round(all_bytes * args.steps / (e2e_ms_max * 1e-3) / 1e9, 2),
                "unit": "GB/s", "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": round(e2e_ms_max / args.steps, 6), "launch": e2e["launch"],
                "copy_engine": {"value": round(all_bytes * args.steps / (e2e_ce_ms_max * 1e-3) / 1e9, 2),
                                "ms_per_step": round(e2e_ce_ms_max / args.steps, 6),
                                "launch": e2e_ce["launch"]}},
        "gpu_launches": st.launches_per_step * args.steps,
        "configs": configs,
        "block_ops": blocks,
        "fp8_kv": fp8,
        "prefill": pre,
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_seconds)
    return line


def all_configs(args, torch, binding, flush_l2, timed_loop, world):
    """Every named workload's step (fused RoPE + store + decode for each of its layers, early
    metadata on layers after the first, replayed as a CUDA graph), L2 flushed before each
    step: step time, KV bytes per second against the measured HBM copy peak, and decode
    tokens per second (sequences per step over the step time).  prefix32 also reports the
    bandwidth over its unique KV bytes (the shared prefix is read once from HBM, then from L2).

    mix64_x28 is the batch-64 mixed-length layer run as the attention of a 28-layer model step
    (Qwen2.5-1.5B's depth): 28 layers, each with its own copy of the layer's caches in HBM
    (3.4 GB of KV read per step, far past L2), so that layers 2-28 resolve their work beside
    the layer before, as in a real decode step."""
    peak, kind = hbm_peak()
    res = {}
    runs = [(name, W.make(name), 0) for name in W.WORKLOADS]
    runs.append(("mix64_x28", None, 28))
    for name, w, rep in runs:
        if w is None:
            w = W.make("mix64")
        st = DeviceStep(w, torch, binding, fused=True, early=True, replicate_layers=rep)
        for _ in range(3):
            st.step()
        fn = st.step
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                st.step()
            for _ in range(max(3, args.warmup)):   # untimed replays, as the main step's warm-up
                graph.replay()
            torch.cuda.synchronize()
            fn = graph.replay
        except Exception:
            pass
        ms = float(np.mean(timed_loop(fn, max(10, args.steps // 4))))
        rc, flags = binding.get_device_status()
        if rc != 0:
            raise RuntimeError(f"device status after the {name} step: {rc} flags {flags:#x}")
        layers = st.num_layers
        nbytes = w.kv_bytes_per_layer() * layers
        gbs = nbytes / (ms * 1e-3) / 1e9
        entry = {"layers": layers, "num_seqs": w.num_seqs,
                 "partition_tokens": st.P or "0 (even split)",
                 "step_us": round(ms * 1e3, 3), "kv_bytes_per_step": nbytes,
                 "GB/s": round(gbs, 1), "frac_of_hbm_peak": round(gbs / peak, 4),
                 "decode_tokens_per_s": round(world * w.num_seqs / (ms * 1e-3), 1)}
        if layers > 1:
            entry["per_layer_us"] = round(ms * 1e3 / layers, 3)
        if rep:
            entry["layer_caches"] = f"{rep} device copies of one layer's inputs and caches"
        if w.meta.get("shared_prefix_blocks"):
            ub = w.unique_kv_bytes_per_layer() * layers
            entry["unique_kv_bytes_per_step"] = ub
            entry["unique_GB/s"] = round(ub / (ms * 1e-3) / 1e9, 1)
        res[name] = entry
        del st, fn
        torch.cuda.empty_cache()
    res["peak"] = {"hbm_GB/s": peak, "kind": f"{kind} hbm_gbs"}
    return res


def block_ops(torch, binding, flush_l2, timed_loop, w, layers=28, pool_blocks=1024, reps=20):
    """pa_copy_blocks on the model's whole cache: K and V of `layers` layers, pools of
    `pool_blocks` blocks each.  copy_on_write: pool_blocks / 2 pairs inside each device pool;
    swap_out / swap_in: one 2048-token sequence (128 blocks) to page-locked host pools and
    back, against a plain device<->host memcpy of the same bytes.  L2 flushed before each."""
    dev = torch.device("cuda")
    shape = (pool_blocks, w.num_kv_heads, W.BLOCK_SIZE, W.HEAD_DIM)
    pools = [torch.randn(shape, device=dev).to(torch.bfloat16) for _ in range(2 * layers)]
    block_bytes = w.num_kv_heads * W.BLOCK_SIZE * W.HEAD_DIM * 2
    rng = np.random.default_rng(0x244)
    half = pool_blocks // 2
    cow = np.stack([rng.permutation(half), half + rng.permutation(half)], 1).astype(np.int64)
    cow_pairs = torch.from_numpy(cow).to(dev)
    nseq = 128
    host = [torch.empty((nseq,) + shape[1:], dtype=torch.bfloat16).pin_memory() for _ in pools]
    out_pairs = torch.from_numpy(np.stack([rng.permutation(pool_blocks)[:nseq], np.arange(nseq)],
                                          1).astype(np.int64)).to(dev)
    in_pairs = torch.from_numpy(np.stack([np.arange(nseq), rng.permutation(pool_blocks)[:nseq]],
                                         1).astype(np.int64)).to(dev)
    flat_dev = torch.empty(nseq * block_bytes * len(pools), dtype=torch.uint8, device=dev)
    flat_host = torch.empty(flat_dev.numel(), dtype=torch.uint8).pin_memory()

    def rate(fn, nbytes):
        ms = float(np.median(timed_loop(fn, reps)))
        return round(nbytes / (ms * 1e-3) / 1e9, 1), round(ms * 1e3, 2)

    cow_bytes = 2 * cow.shape[0] * len(pools) * block_bytes          # read + write
    swap_bytes = nseq * len(pools) * block_bytes                      # each way
    cow_gbs, cow_us = rate(lambda: binding.copy_blocks(pools, pools, cow_pairs), cow_bytes)
    out_gbs, out_us = rate(lambda: binding.copy_blocks(pools, host, out_pairs), swap_bytes)
    in_gbs, in_us = rate(lambda: binding.copy_blocks(host, pools, in_pairs), swap_bytes)
    d2h, _ = rate(lambda: flat_host.copy_(flat_dev, non_blocking=True), swap_bytes)
    h2d, _ = rate(lambda: flat_dev.copy_(flat_host, non_blocking=True), swap_bytes)
    rc, flags = binding.get_device_status()
    if rc != 0:
        raise RuntimeError(f"device status after block copies: {rc} flags {flags:#x}")
    peak, kind = hbm_peak()
    return {
        "caches": len(pools), "pool_blocks": pool_blocks, "block_bytes_per_cache": block_bytes,
        "copy_on_write": {"pairs": int(cow.shape[0]), "GB/s": cow_gbs, "us": cow_us,
                          "bytes": cow_bytes, "frac_of_hbm_copy_peak": round(cow_gbs / peak, 4)},
        "swap_out": {"blocks": nseq, "GB/s": out_gbs, "us": out_us, "bytes": swap_bytes,
                     "memcpy_d2h_GB/s": d2h},
        "swap_in": {"blocks": nseq, "GB/s": in_gbs, "us": in_us, "bytes": swap_bytes,
                    "memcpy_h2d_GB/s": h2d},
    }


def fp8_kv(torch, binding, timed_loop, st, steps):
    """The step's decode on E4M3 caches (one byte per element, one scale per KV head), layer 0
    of the workload: pa_decode_fp8 and pa_decode_step_fp8, L2 flushed before each call, and
    pa_gather_checksum_fp8 (the same tile gather without attention or merge) as their floor.
    The codes are made once on the GPU with torch's float8 cast from the bf16 caches (set-up,
    not timed); achieved bandwidth counts the E4M3 bytes, half the bf16 bytes."""
    w = st.w

    def codes(cache):
        amax = cache.float().abs().nan_to_num(0.0).amax(dim=(0, 2, 3)).clamp_min(1e-3)
        scale = (amax / 448.0).float().contiguous()
        c = (cache.float() / scale[None, :, None, None]).clamp(-448, 448).to(torch.float8_e4m3fn)
        return c.view(torch.uint8).contiguous(), scale

    k8, ks = codes(st.k_cache[0])
    v8, vs = codes(st.v_cache[0])
    out = torch.empty_like(st.q[0])
    dec = lambda: binding.decode_fp8(st.q[0], k8, v8, ks, vs, st.block_tables, st.context_lens,
                                     w.max_context_len, w.scale, partition_tokens=st.P,
                                     workspace=st.workspace, out=out)
    stp = lambda: binding.decode_step_fp8(st.q[0], st.k[0], st.v[0], st.cos_sin, k8, v8, ks, vs,
                                          st.block_tables, st.context_lens, w.max_context_len,
                                          w.scale, partition_tokens=st.P, workspace=st.workspace,
                                          out=out)
    # the floor of the E4M3 decode's access pattern: its tile gather alone, same kernel shape
    gx = torch.zeros((w.num_seqs, w.num_kv_heads), dtype=torch.int32, device=k8.device)
    gat = lambda: binding.gather_checksum(k8, v8, st.block_tables, st.context_lens, w.max_context_len,
                                          w.num_q_heads, out_xor=gx)
    dec()
    stp()
    gat()
    dec_ms = float(np.mean(timed_loop(dec, steps)))
    stp_ms = float(np.mean(timed_loop(stp, steps)))
    gat_ms = float(np.mean(timed_loop(gat, steps)))
    rc, flags = binding.get_device_status()
    if rc != 0:
        raise RuntimeError(f"device status after the E4M3 decode: {rc} flags {flags:#x}")
    nbytes = w.kv_bytes_per_layer() // 2
    peak, _ = hbm_peak()
    gbs = nbytes / (dec_ms * 1e-3) / 1e9

    # The same layer as the attention of a 28-layer step: 28 device copies of its E4M3 caches
    # (each layer's kernel resolves its work beside the layer before), one CUDA graph per step.
    L28 = 28
    k8s = [k8] + [k8.clone() for _ in range(L28 - 1)]
    v8s = [v8] + [v8.clone() for _ in range(L28 - 1)]
    outs = [torch.empty_like(st.q[0]) for _ in range(L28)]

    def chain():
        for i in range(L28):
            binding.decode_step_fp8(st.q[0], st.k[0], st.v[0], st.cos_sin, k8s[i], v8s[i], ks, vs,
                                    st.block_tables, st.context_lens, w.max_context_len, w.scale,
                                    partition_tokens=st.P, workspace=st.workspace, out=outs[i],
                                    early_metadata=i > 0)

    chain()
    x28_fn = chain
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            chain()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        x28_fn = graph.replay
    except Exception:
        pass
    x28_ms = float(np.mean(timed_loop(x28_fn, max(10, steps // 4))))
    rc, flags = binding.get_device_status()
    if rc != 0:
        raise RuntimeError(f"device status after the 28-layer E4M3 step: {rc} flags {flags:#x}")
    x28_gbs = L28 * nbytes / (x28_ms * 1e-3) / 1e9
    del k8s, v8s, outs
    return {"algorithmic_bytes_per_launch": nbytes,
            "pa_decode_fp8_us": round(dec_ms * 1e3, 3), "GB/s": round(gbs, 1),
            "frac_of_hbm_copy_peak": round(gbs / peak, 4),
            "pa_decode_step_fp8_us": round(stp_ms * 1e3, 3),
            "gather_floor_us": round(gat_ms * 1e3, 3),
            "gather_floor_frac": round(nbytes / (gat_ms * 1e-3) / 1e9 / peak, 4),
            "decode_over_floor": round(dec_ms / gat_ms, 4),
            "context_tokens_per_s": round(int(w.context_lens.astype(np.int64).sum()) / (dec_ms * 1e-3), 1),
            "x28": {"layers": L28, "step_us": round(x28_ms * 1e3, 3),
                    "per_layer_us": round(x28_ms * 1e3 / L28, 3), "GB/s": round(x28_gbs, 1),
                    "frac_of_hbm_copy_peak": round(x28_gbs / peak, 4),
                    "layer_caches": f"{L28} device copies of the layer's E4M3 caches, pa_decode_step_fp8 "
                                    "with early metadata on layers after the first, one CUDA graph"}}


def prefill_runs(torch, binding, timed_loop, steps):
    """pa_prefill on the named prefill workloads (4 whole 2048-token prompts; 16 chunks of 256
    tokens continuing 1792 cached ones), Qwen2.5-1.5B attention shape, one layer, L2 flushed
    before each call.  Tensor roofline: attention flops (4 Hq D per causal (query, key) pair)
    over the measured bf16 dense peak."""
    dev = torch.device("cuda")
    peak, kind = bf16_peak()

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    res = {}
    for name in W.PREFILL_WORKLOADS:
        w = W.make_prefill(name)
        q, kc, vc = bf(w.q), bf(w.k_cache), bf(w.v_cache)
        qs = torch.from_numpy(w.q_start).to(dev)
        bt = torch.from_numpy(w.block_tables).to(dev)
        ctx = torch.from_numpy(w.context_lens).to(dev)
        out = torch.empty_like(q)
        call = lambda: binding.prefill(q, qs, kc, vc, bt, ctx, w.max_query_len, w.max_context_len,
                                       w.scale, out=out)
        call()
        ms = float(np.mean(timed_loop(call, steps)))
        rc, flags = binding.get_device_status()
        if rc != 0:
            raise RuntimeError(f"device status after pa_prefill: {rc} flags {flags:#x}")
        tf = w.attention_flops() / (ms * 1e-3) / 1e12
        res[name] = {"num_seqs": w.num_seqs, "new_tokens": w.num_tokens,
                     "max_context_len": w.max_context_len, "us": round(ms * 1e3, 2),
                     "attention_flops": w.attention_flops(), "TFLOP/s": round(tf, 1),
                     "roofline": {"bound": "tensor", "peak": peak, "peak_kind": f"{kind} bf16_tflops",
                                  "unit": "TFLOP/s", "frac": round(tf / peak, 4)},
                     "new_tokens_per_s": round(w.num_tokens / (ms * 1e-3), 1)}
        res[name]["rope_kv_store"] = prefill_store(torch, binding, timed_loop, steps, w, kc, vc, bt)
    return res


def prefill_store(torch, binding, timed_loop, steps, w, kc, vc, bt):
    """pa_rope_kv_store of a prefill workload's new tokens (their k and v drawn from a seeded
    generator, each at its position ctx - n + i and that position's slot), timed after the
    prefill runs: bytes = q read and written, k and v read and written to the caches, one
    cos/sin row read, per token, over the measured HBM copy bandwidth."""
    dev = torch.device("cuda")
    T, Hq, D = w.q.shape
    Hkv = kc.shape[1]
    pos = np.concatenate([np.arange(w.context_lens[s] - (w.q_start[s + 1] - w.q_start[s]),
                                    w.context_lens[s]) for s in range(w.num_seqs)]).astype(np.int32)
    seq = np.repeat(np.arange(w.num_seqs), np.diff(w.q_start))
    slots = w.block_tables[seq, pos // W.BLOCK_SIZE].astype(np.int64) * W.BLOCK_SIZE + pos % W.BLOCK_SIZE
    gen = torch.Generator(device="cpu").manual_seed(0x244)
    q = torch.from_numpy(np.ascontiguousarray(w.q).view(np.int16)).view(torch.bfloat16).to(dev)
    k = torch.randn(T, Hkv, D, generator=gen).to(torch.bfloat16).to(dev)
    v = torch.randn(T, Hkv, D, generator=gen).to(torch.bfloat16).to(dev)
    cs = torch.from_numpy(W.rope_cos_sin_table(int(w.max_context_len))).to(dev)
    pos_d, slots_d = torch.from_numpy(pos).to(dev), torch.from_numpy(slots).to(dev)
    call = lambda: binding.rope_kv_store(q, k, v, pos_d, cs, slots_d, kc, vc)
    call()
    ms = float(np.mean(timed_loop(call, steps)))
    rc, flags = binding.get_device_status()
    if rc != 0:
        raise RuntimeError(f"device status after pa_rope_kv_store: {rc} flags {flags:#x}")
    nbytes = T * ((2 * Hq + 4 * Hkv) * D * 2 + D * 4)
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak, _ = hbm_peak()
    return {"tokens": int(T), "us": round(ms * 1e3, 2), "bytes": int(nbytes), "GB/s": round(gbs, 1),
            "frac_of_hbm_copy_peak": round(gbs / peak, 4)}


def reduce_over_ranks(maxes, sums, dist, device):
    """Max of `maxes` and sum of `sums` over all ranks (no-op on one rank).  Only timings and
    byte counts cross ranks: the decode itself has no collective."""
    import torch
    t = torch.tensor(maxes, dtype=torch.float64, device=device)
    b = torch.tensor(sums, dtype=torch.float64, device=device)
    if dist is not None and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return [float(x) for x in t.cpu()], [float(x) for x in b.cpu()]


def run_e2e(args, st, torch, binding, flush_l2, copy_engine=False):
    """Every step: one host -> device copy of all the step's inputs (new-token q/k/v of every
    layer, block tables, lengths, and for the split step positions and slots), packed in one
    pinned buffer, then the C-ABI calls on views of the device copy, then one device -> host
    copy of every layer's output, all between the CUDA events.  The KV caches stay resident,
    as in a serving engine.  The two copies are pa_stage_copy kernels (the library's loads and
    stores over the CPU-GPU link), or with copy_engine cudaMemcpyAsync transfers."""
    w = st.w
    stream = torch.cuda.current_stream()
    L = w.num_layers
    items = [st.positions, st.slots, st.block_tables, st.context_lens]
    for i in range(L):
        items += [st.q_src[i], st.k[i], st.v[i]]
    if st.fused:  # the fused step derives positions and slots from the lengths and tables
        items[0] = items[1] = None
    offs, total = [], 0
    for t in items:
        offs.append(total)
        if t is not None:
            total += (t.numel() * t.element_size() + 255) // 256 * 256
    h_in = torch.empty(total, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(total, dtype=torch.uint8, device="cuda")
    views = []
    for t, o in zip(items, offs):
        if t is None:
            views.append(None)
            continue
        n = t.numel() * t.element_size()
        h_in[o:o + n].copy_(t.detach().reshape(-1).view(torch.uint8).cpu())
        views.append(d_in[o:o + n].view(t.dtype).view(t.shape))
    pos, slots, bt, ctx = views[:4]
    q = [views[4 + 3 * i] for i in range(L)]
    k = [views[5 + 3 * i] for i in range(L)]
    v = [views[6 + 3 * i] for i in range(L)]
    d_out = torch.empty((L,) + tuple(st.out[0].shape), dtype=torch.bfloat16, device="cuda")
    h_out = torch.empty(d_out.shape, dtype=torch.bfloat16).pin_memory()

    def h2d():
        if copy_engine:
            d_in.copy_(h_in, non_blocking=True)
        else:
            binding.stage_copy(d_in, h_in)

    def d2h():
        if copy_engine:
            h_out.copy_(d_out, non_blocking=True)
        else:
            binding.stage_copy(h_out, d_out)

    def one():
        h2d()
        for i in range(L):
            if st.fused:
                # layers after the first follow a decode kernel, and the copy that wrote the
                # tables precedes them all: they may start early
                binding.decode_step(q[i], k[i], v[i], st.cos_sin, st.k_cache[i], st.v_cache[i], bt,
                                    ctx, w.max_context_len, w.scale, partition_tokens=st.P,
                                    workspace=st.workspace, out=d_out[i],
                                    early_metadata=st.early and i > 0)
                continue
            binding.rope_kv_store(q[i], k[i], v[i], pos, st.cos_sin, slots, st.k_cache[i],
                                  st.v_cache[i])
            binding.decode(q[i], st.k_cache[i], st.v_cache[i], bt, ctx, w.max_context_len, w.scale,
                           partition_tokens=st.P, workspace=st.workspace, out=d_out[i])
        d2h()

    for _ in range(2):
        one()
    torch.cuda.synchronize()
    # As for the device-only step: the whole step -- the H2D copy, every layer's call, the D2H
    # copy -- recorded once as a CUDA graph and replayed, unless --no-graph.
    step_fn, how = one, "eager calls"
    if not args.no_graph:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                one()
            graph.replay()
            torch.cuda.synchronize()
            step_fn, how = graph.replay, "CUDA graph of the H2D copy, the calls and the D2H copy"
            how += " (cudaMemcpyAsync)" if copy_engine else " (pa_stage_copy kernels)"
        except Exception as e:  # capture unsupported here: keep eager calls
            how = f"eager calls (graph capture failed: {type(e).__name__})"
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, b in evs:
        flush_l2()
        a.record(stream)
        step_fn()
        b.record(stream)
    torch.cuda.synchronize()
    ms = float(np.sum([a.elapsed_time(b) for a, b in evs]))
    return {"ms": ms, "h2d": int(total), "d2h": int(h_out.numel() * h_out.element_size()),
            "launch": how}


def config_of(w, st, world):
    c = {
        "workload": w.name,
        "num_seqs_per_gpu": w.num_seqs,
        "num_layers": w.num_layers,
        "context_lens": describe_ctx(w),
        "num_q_heads": w.num_q_heads,
        "num_kv_heads": w.num_kv_heads,
        "head_dim": W.HEAD_DIM,
        "block_size": W.BLOCK_SIZE,
        "pool_blocks": w.num_blocks,
        "partition_tokens": (st.P if st is not None else w.partition_tokens) or "0 (even split)",
        "kv_bytes_per_step_per_gpu": w.kv_bytes_per_layer() * w.num_layers,
        "l2": "flushed between timed steps (512 MiB write then read back, outside the events)",
        "parallelism": f"replicas x{world} (independent batches)",
    }
    if st is not None:
        c["step"] = ("pa_decode_step (RoPE + KV store fused into the decode launch)" if st.fused
                     else "pa_rope_kv_store then pa_decode")
        if st.fused:
            c["early_metadata"] = "layers after the first" if st.early else "off"
    if w.meta.get("shared_prefix_blocks"):
        c["unique_kv_bytes_per_step_per_gpu"] = w.unique_kv_bytes_per_layer() * w.num_layers
    return c


def describe_ctx(w):
    c = w.context_lens
    if w.name == "mix64":
        return f"uniform[64,4096] seeded: sum {int(c.sum())}, min {int(c.min())}, max {int(c.max())}"
    return [int(x) for x in c[:8]] + (["..."] if len(c) > 8 else [])


# ------------------------------------------------------------------ CPU oracle ----

def oracle_step(orc, w, sample_seqs, nthreads):
    """The oracle's RoPE + store and decode over the first `sample_seqs` sequences of every
    layer.  Returns the KV bytes the decode read."""
    n = min(sample_seqs, w.num_seqs)
    total = 0
    for layer in range(w.num_layers):
        kc, vc = w.k_cache[layer].copy(), w.v_cache[layer].copy()
        q = orc.rope_kv_store(w.q[layer, :n], w.k[layer, :n], w.v[layer, :n], w.positions[:n],
                              w.cos_sin, w.slot_mapping[:n], kc, vc)
        orc.decode(q, kc, vc, w.block_tables[:n], w.context_lens[:n], w.scale, nthreads=nthreads)
        total += int(w.context_lens[:n].astype(np.int64).sum()) * w.num_kv_heads * W.HEAD_DIM * 4
    return total


def choose_sample(orc, w, budget_s, nthreads):
    """Number of sequences whose oracle step takes about budget_s (at least 1)."""
    n = max(1, min(w.num_seqs, 4))
    t0 = time.perf_counter()
    oracle_step(orc, w, n, nthreads)
    dt = max(time.perf_counter() - t0, 1e-3)
    return max(1, min(w.num_seqs, int(n * budget_s / dt)))


def cpu_baseline(w, budget_s=10.0):
    import oracle
    orc = oracle.default()
    cores = orc.hardware_threads()
    n = choose_sample(orc, w, budget_s, 0)
    # the sample, repeated until about budget_s of CPU time has run (at least once)
    t0 = time.perf_counter()
    nbytes, reps = 0, 0
    while reps == 0 or time.perf_counter() - t0 < budget_s:
        nbytes += oracle_step(orc, w, n, 0)
        reps += 1
    dt = time.perf_counter() - t0
    # the same oracle on one thread, for about a quarter of the budget
    n1 = choose_sample(orc, w, budget_s / 4, 1)
    t1 = time.perf_counter()
    b1, reps1 = 0, 0
    while reps1 == 0 or time.perf_counter() - t1 < budget_s / 4:
        b1 += oracle_step(orc, w, n1, 1)
        reps1 += 1
    dt1 = time.perf_counter() - t1
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"fp64 oracle RoPE+store and decode of the first {n} of {w.num_seqs} "
                      f"sequences x {w.num_layers} layer(s), {reps} time(s), {dt:.1f} s on "
                      f"{cores} threads",
            "single_thread": {"value": round(b1 / dt1 / 1e9, 4), "unit": "GB/s",
                              "sample": f"the first {n1} sequences, {reps1} time(s), {dt1:.1f} s "
                                        f"on 1 thread"}}


def run_reference(args, world):
    import oracle
    orc = oracle.default()
    cores = orc.hardware_threads()
    w = W.make(args.workload)
    per_step = max(0.2, min(5.0, 120.0 / max(1, args.steps + args.warmup)))
    n = choose_sample(orc, w, per_step, 0)
    for _ in range(args.warmup):
        oracle_step(orc, w, n, 0)
    t0 = time.perf_counter()
    nbytes = 0
    for _ in range(args.steps):
        nbytes += oracle_step(orc, w, n, 0)
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    sample = (f"fp64 oracle RoPE+store and decode of the first {n} of {w.num_seqs} sequences x "
              f"{w.num_layers} layer(s) per step, on {cores} host threads")
    cfg = config_of(w, None, world)
    cfg["l2"] = "not flushed (host cores)"
    return {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * dt / max(1, args.steps), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference", "config": cfg,
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="mix64", choices=W.WORKLOADS)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch each call instead of a CUDA graph")
    ap.add_argument("--no-early-metadata", action="store_true",
                    help="run the step without PA_STEP_EARLY_METADATA")
    ap.add_argument("--no-fp8", action="store_true", help="skip the E4M3-cache decode measurement")
    ap.add_argument("--no-prefill", action="store_true", help="skip the pa_prefill measurement")
    ap.add_argument("--no-block-ops", action="store_true",
                    help="skip the pa_copy_blocks measurements (copy-on-write, swap out / in)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the step measurement of every named workload")
    ap.add_argument("--split-step", action="store_true",
                    help="pa_rope_kv_store then pa_decode instead of the fused pa_decode_step")
    ap.add_argument("--partition-tokens", type=int, default=None,
                    help="Flash-Decode partition size (default: the workload's, 0 = library choice)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes read+written per pa_decode call from an ncu capture")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, world)), flush=True)
        return
    dist = None
    if world > 1:
        import torch
        import torch.distributed as td
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        td.init_process_group("nccl")
        dist = td
    line = run_gpu(args, rank, world, dist)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
