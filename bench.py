"""Benchmark: paged decode attention on one GB300 (replicas on N GPUs).

A step is one decode step of the whole hot path over one batch: for each of
the 16 layers, the fused append-then-attend launch (append the new token's
K/V into its block-table slot, then paged GQA decode attention with split-KV
and the in-launch merge). The headline workload is the largest
configuration that fits one GPU, the large ragged batch: 256 sequences with
lengths uniform in [1, 2048] (1, 16, 32, 2048, 17 and 1024 among them), a
pool sized to fit them, BF16 N(0,1) inputs with K scaled by 4, 32q/8kv heads,
head_dim 64, 16-token pages. Beside it ("per_config") every other
configuration is timed the same way for at least a second each: the
Llama-3.2-1B default step (batch 2 at 2,048 tokens, 128 MiB pool), the
batch-64 continuous-batching mix, and the long-context batches 1 and 4.

Timing: the 16 launches of a step are captured in a CUDA graph with
GPU-timestamped events before and after them; before every step an untimed
read of a buffer twice the L2 size evicts the cache. A second graph of the
same step with events between the launches gives the per-launch durations of
the kernel for the roofline. value = KV GB/s
= algorithmic bytes per step / step time, with algorithmic bytes per
(sequence, layer) = seq_len x 2048 (every cached K/V row read once) + 2048
(the new row written) + 4096 (q) + 8192 (FP32 out). With --rope the
launches also rotate the appended key and the queries to their position
(pkv_append_attend_rope; angle tables for base 500000), adding 256 bytes (the
position's cos and sin rows) per (sequence, layer).

e2e: the same step with its inputs copied from pinned host memory and its
output copied back inside the timed region, (a) replaying a CUDA graph that
holds the copies and the launches, (b) issuing the C-ABI calls from the host
every step (what a decode loop without graphs pays).

--impl reference times the CPU oracle (FP64 C++) on the host cores on a
bounded sample of the same workload and prints the same line with
"impl": "reference". cpu_baseline reports the oracle single-threaded and on
every host core, with the core count and CPU model.
"""

import argparse
import concurrent.futures
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged decode attention KV GB/s and seq-layer steps/s; % of GB300 HBM peak"
NOMINAL_HBM_GBS = 8000.0
# each takes the number of layers (16: the model's; fewer only for profiling
# captures, which launch the same per-layer kernels on a smaller pool)
WORKLOADS = {
    "llama-b2-2048": lambda n=16: W.llama_default(num_layers=n),
    "mix-b64": lambda n=16: W.continuous_mix(num_layers=n),
    "ragged-b256": lambda n=16: W.large_ragged(num_layers=n),
    "long-b1": lambda n=16: W.long_context(1, num_layers=n),
    "long-b4": lambda n=16: W.long_context(4, num_layers=n),
    "long-b8": lambda n=16: W.long_context(8, num_layers=n),
    "long-b16": lambda n=16: W.long_context(16, num_layers=n),
}
# the workloads timed beside the headline (every configuration of the task
# that fits one GPU: the default decode step, the continuous-batching mix, the
# large ragged batch, and the long-context batches 1 and 4)
PER_CONFIG = ["llama-b2-2048", "mix-b64", "ragged-b256", "long-b1", "long-b4"]
DESCRIPTIONS = {
    "llama-b2-2048": "Llama-3.2-1B decode step at the default 128 MiB pool: 16 layers, batch 2 at "
                     "seq_len 2048, 32q/8kv heads, head_dim 64, 4096 shuffled 16-token pages",
    "mix-b64": "continuous-batching mix: 16 layers, batch 64, seq_lens log-uniform in "
               "[16, 2048], 4 GiB pool, fragmented free list",
    "ragged-b256": "large ragged batch: 16 layers, batch 256, seq_lens uniform in [1, 2048], "
                   "K x 4",
    "long-b1": "long context: 16 layers, batch 1 at 2048, 1 GiB pool",
    "long-b4": "long context: 16 layers, batch 4 at 2048, 1 GiB pool",
    "long-b8": "long context: 16 layers, batch 8 at 2048, 1 GiB pool",
    "long-b16": "long context: 16 layers, batch 16 at 2048, 1 GiB pool (every page used)",
}


ROPE_BASE = 500000.0


def step_bytes(wl, rope=False):
    """Algorithmic bytes of one fused step over all layers."""
    per_seq = wl.seq_lens.astype(np.int64) * 2048 + 2048 + 4096 + 8192 + (256 if rope else 0)
    return int(per_seq.sum()) * wl.num_layers


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0}, "fallback"


KERNEL_SOURCES = {
    "decode": ("paged_kv_cache_210_gb300/csrc/pkv.cu",
               "paged_kv_cache_210_gb300/csrc/decode_device.cuh"),
    "layers": ("paged_kv_cache_210_gb300/csrc/layers.cu",
               "paged_kv_cache_210_gb300/csrc/decode_device.cuh"),
    "prefill": ("paged_kv_cache_210_gb300/csrc/prefill.cu", "include/pkv_prefill.h"),
}


def kernel_source_hash(component="decode"):
    """First 16 hex digits of the SHA-256 over the sources one kernel family is
    compiled from (its .cu file, the shared device and pool headers, pkv.h)."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[component] + ("paged_kv_cache_210_gb300/csrc/device_common.cuh",
                                            "paged_kv_cache_210_gb300/csrc/pool_internal.h",
                                            "include/pkv.h"):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(profile, component="decode"):
    """DRAM bytes per launch of a kernel from its committed ncu summary
    (profiles/<profile>.md), or None when there is none for the current
    kernel source."""
    path = os.path.join(ROOT, "profiles", f"{profile}.md")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if line.startswith("- ") and ": " in line:
                k, v = line[2:].split(": ", 1)
                fields[k.strip()] = v.strip().strip("`")
    if fields.get("kernel_source_sha256_16") != kernel_source_hash(component):
        return None
    try:
        return int(float(fields["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        self.lines = []
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            target = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            target = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"] + target, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
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
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(n_gpus, backend=None):
    """One process per GPU (torchrun sets RANK/LOCAL_RANK/WORLD_SIZE/MASTER_*);
    NCCL on GPUs, gloo where there is none (the CPU tests of this path)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = backend or ("nccl" if torch.cuda.is_available() else "gloo")
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """The slowest rank's figure (the whole job ends with it)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world, bytes_per_step, steps, total_ms_max):
    """Replicas: every rank moves bytes_per_step per step; the job takes as
    long as its slowest rank. GB/s over all ranks."""
    return world * bytes_per_step * steps / (total_ms_max * 1e-3) / 1e9


# ---------------------------------------------------------------- CPU oracle
def oracle_inputs(wl):
    kp, vp = wl.pools("cpu", "zero")

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()

    return bits(kp), bits(vp), bits(wl.q()), bits(wl.k_new()), bits(wl.v_new())


def oracle_sample(wl, max_seqs=64, max_layers=4):
    """A bounded sample of a workload for timing the CPU oracle: its first
    `max_seqs` sequences (the same lengths, so the same length mix for the
    ragged and log-uniform workloads) over `max_layers` layers, with a pool
    of just their pages. Bytes per (sequence, layer) are those of the
    workload, so GB/s compares directly."""
    if wl.batch <= max_seqs and wl.num_layers <= max_layers:
        return wl
    return W.custom(wl.seq_lens[:max_seqs], num_layers=min(wl.num_layers, max_layers),
                    seed=wl.seed, k_scale=wl.k_scale, name=wl.name + "-sample")


def time_oracle(wl, layers_per_step, n_steps, threads, rope=False, inputs=None):
    """Runs the oracle (append + attention, rotated when `rope`) on
    `layers_per_step` layers per step over `threads` host threads: layers in
    parallel, and within a layer sequences spread over the layer's share of
    the threads. Returns (seconds, bytes, layer-steps, threads used)."""
    import oracle
    orc = oracle.load()
    kp, vp, q, kn, vn = inputs if inputs is not None else oracle_inputs(wl)
    g = oracle.geometry(wl.num_layers, wl.num_pages, wl.batch)
    pos = wl.positions
    bytes_per_layer = step_bytes(wl, rope) // wl.num_layers
    cos_t, sin_t = W.rope_tables(base=ROPE_BASE)
    workers = max(1, min(threads, layers_per_step))
    per_layer = max(1, threads // workers)
    used = workers * (1 if rope else min(per_layer, wl.batch))

    def one_layer(layer):
        if rope:
            st = orc.append_rope(g, layer, kn[layer].copy(), vn[layer].copy(), kp, vp,
                                 wl.block_tables, pos, cos_t, sin_t)
            st1, q64 = orc.rope_queries(q[layer].copy(), pos, cos_t, sin_t)
            st2, _ = orc.decode_attention_q64(g, layer, q64, kp, vp, wl.block_tables,
                                              wl.seq_lens)
            assert st == st1 == st2 == oracle.OK
            return layer
        st = orc.append(g, layer, kn[layer].copy(), vn[layer].copy(), kp, vp, wl.block_tables,
                        pos)
        st2, _ = orc.decode_attention_mt(g, layer, q[layer].copy(), kp, vp, wl.block_tables,
                                         wl.seq_lens, per_layer)
        assert st == st2 == oracle.OK
        return layer

    total_layers = 0
    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        for s in range(n_steps):
            layers = [(s * layers_per_step + i) % wl.num_layers for i in range(layers_per_step)]
            list(ex.map(one_layer, layers))
            total_layers += len(layers)
    dt = time.perf_counter() - t0
    return dt, total_layers * bytes_per_layer, total_layers, used


def cpu_threads():
    return max(1, os.cpu_count() or 1)


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(wl, rope=False, seconds=8.0):
    """The oracle as it stands, timed on this host's cores on a bounded
    sample of the workload: single-threaded, and on all cores (about
    `seconds` of wall time each). Returns the cpu_baseline object."""
    sw = oracle_sample(wl)
    inputs = oracle_inputs(sw)
    nproc = cpu_threads()
    result = {"unit": "GB/s", "kind": "oracle", "nproc": nproc, "cpu_model": cpu_model()}
    for key, threads in (("single_thread", 1), ("all_cores", nproc)):
        per_step = min(sw.num_layers, threads) if threads > 1 else 1
        probe, _, _, _ = time_oracle(sw, per_step, 1, threads, rope, inputs)
        n_steps = max(1, int(seconds / max(probe, 1e-6)))
        dt, nbytes, n_layers, used = time_oracle(sw, per_step, n_steps, threads, rope, inputs)
        result[key] = {"value": round(nbytes / dt / 1e9, 4), "cores": used,
                       "sample": f"{n_layers} layer-steps of {sw.batch} sequences "
                                 f"(lengths as the workload's first {sw.batch}), "
                                 f"{per_step} layer(s) at a time, {dt:.1f} s wall"}
    result["value"] = result["all_cores"]["value"]
    result["cores"] = result["all_cores"]["cores"]
    result["sample"] = result["all_cores"]["sample"]
    return result


def decode_config(wl, args, world=1):
    return {"workload": f"{wl.name}: {DESCRIPTIONS[wl.name]}",
            "batch": wl.batch, "layers": wl.num_layers,
            "seq_lens": "all 2048" if np.all(wl.seq_lens == 2048)
            else f"mean {float(wl.seq_lens.mean()):.1f}",
            "rope": f"key and queries rotated in the launch, base {ROPE_BASE:g}" if args.rope
            else "none (keys arrive rotated)",
            "l2": "flushed before every step (read of a buffer twice the L2 size, outside the "
                  "timed events)",
            "bytes_per_step": step_bytes(wl, args.rope),
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    wl = WORKLOADS[args.workload]()
    sw = oracle_sample(wl)
    inputs = oracle_inputs(sw)
    threads = cpu_threads()
    per_step = min(sw.num_layers, threads)
    # size a step so the whole run stays within about a minute and a half
    probe_dt, _, probe_layers, _ = time_oracle(sw, per_step, 1, threads, args.rope, inputs)
    per_layer = probe_dt / probe_layers
    budget = 90.0 / max(1, args.steps + args.warmup)
    layers = max(1, min(4 * per_step, int(budget / max(per_layer, 1e-9))))
    time_oracle(sw, layers, args.warmup, threads, args.rope, inputs)
    dt, nbytes, n_layers, used = time_oracle(sw, layers, args.steps, threads, args.rope, inputs)
    value = nbytes / dt / 1e9
    sample = (f"{layers} layer-steps per step, each over {sw.batch} sequences (the workload's "
              f"first {sw.batch} lengths), on {used} of {threads} host threads, "
              f"{args.steps} steps")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": decode_config(wl, args, world),
        "seq_layer_steps_per_s": round(n_layers * sw.batch / dt, 2),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": used,
                         "kind": "oracle", "sample": sample, "nproc": threads,
                         "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU path
def make_event():
    try:
        return torch.cuda.Event(enable_timing=True, external=True), True
    except TypeError:
        return torch.cuda.Event(enable_timing=True), False


def nvtx_push(name):
    try:
        torch.cuda.nvtx.range_push(name)
    except Exception:
        pass


def nvtx_pop():
    try:
        torch.cuda.nvtx.range_pop()
    except Exception:
        pass


class DecodeRun:
    """One workload's decode step on the device: inputs resident in HBM, the
    pool handle, and CUDA graphs of the step (events around it, and events
    between its launches)."""

    def __init__(self, pkv, wl, dev, args, stream, flush):
        self.pkv, self.wl, self.dev, self.args = pkv, wl, dev, args
        self.stream, self.flush = stream, flush
        L, B = wl.num_layers, wl.batch
        self.k_pool, self.v_pool = wl.pools(dev, "zero")
        self.q = wl.q(dev)
        self.k_new, self.v_new = wl.k_new(dev), wl.v_new(dev)
        self.table = torch.from_numpy(wl.block_tables).to(dev)
        self.lens = torch.from_numpy(wl.seq_lens).to(dev)
        self.out = torch.zeros((L, B, W.NUM_Q_HEADS, W.HEAD_DIM), device=dev)
        self.pool = pkv.pkv_pool_create(L, wl.num_pages, B,
                                        flags=0 if args.no_pdl else pkv.PKV_FLAG_PDL)
        self.rope_cos, self.rope_sin = (torch.from_numpy(t).to(dev)
                                        for t in W.rope_tables(base=ROPE_BASE))
        self.launches = 1 if args.persistent else L
        made = [make_event() for _ in range(self.launches + 3)]
        self.external = all(e[1] for e in made)
        self.events = [e[0] for e in made[:self.launches + 1]]
        self.t_start, self.t_end = made[self.launches + 1][0], made[self.launches + 2][0]
        with torch.cuda.stream(stream):
            self.step()
        torch.cuda.synchronize()
        assert pkv.pkv_get_error(self.pool) == pkv.PKV_OK
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=stream):
            self.step([self.t_start, self.t_end] if self.external else None)
        self.launch_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.launch_graph, stream=stream):
            self.step(self.events if self.external else None)

    def plan(self):
        p = self.pkv.pkv_plan_decode(self.pkv.pkv_pool_device_figures(self.pool), self.wl.batch,
                                     self.args.splits)
        shape = {0: "ticket merge", 1: "narrow cluster", 2: "wide cluster"}[p.shape]
        if self.args.persistent:
            return "one persistent launch for all layers (cluster per (sequence, kv head))"
        if p.cluster:
            return f"{shape}, S = {p.num_splits} ({p.grid_splits * 8 * self.wl.batch} blocks)"
        if p.longest_first and p.range_div == 0:
            return (f"{shape}, whole sequences longest first, {p.grid_units * 8} blocks")
        if p.longest_first:
            return (f"{shape}, (sequence, range) units longest first, ranges of at least "
                    f"{p.chunk_pages} pages sized to the batch (pages / {p.range_div}), "
                    f"{p.grid_units * 8} blocks")
        ranges = (f"{p.num_splits} ranges" if p.num_splits else
                  f"ranges of {p.chunk_pages} pages")
        return f"{shape}, {ranges}, {p.grid_splits * 8 * self.wl.batch} blocks"

    def step(self, marks=None, stream=None, before=None, after=None):
        """The 16 launches (or the one multi-layer launch); `marks` = events
        recorded before, between and after; `before(layer)` / `after(layer)`
        run around each per-layer launch (stream work such as event waits)."""
        pkv, a = self.pkv, self.args
        s = stream if stream is not None else torch.cuda.current_stream()
        if marks:
            marks[0].record(s)
        if a.persistent:
            pkv.pkv_append_attend_layers(self.pool, 0, self.q, self.k_new, self.v_new,
                                         self.k_pool, self.v_pool, self.table, self.lens,
                                         self.out, stream=s)
            if marks:
                marks[-1].record(s)
            return
        for layer in range(self.wl.num_layers):
            if before:
                before(layer)
            if a.rope:
                pkv.pkv_append_attend_rope(self.pool, layer, self.q[layer], self.k_new[layer],
                                           self.v_new[layer], self.k_pool, self.v_pool,
                                           self.table, self.lens, self.rope_cos, self.rope_sin,
                                           self.out[layer], num_splits=a.splits, stream=s)
            else:
                pkv.pkv_append_attend(self.pool, layer, self.q[layer], self.k_new[layer],
                                      self.v_new[layer], self.k_pool, self.v_pool, self.table,
                                      self.lens, self.out[layer], num_splits=a.splits, stream=s)
            if after:
                after(layer)
            if marks and len(marks) > 2:
                marks[layer + 1].record(s)
        if marks and len(marks) == 2:
            marks[1].record(s)

    def replay(self, g, ev0, ev1):
        with torch.cuda.stream(self.stream):
            self.flush()
            if self.external:
                g.replay()
            else:
                ev0.record(self.stream)
                g.replay()
                ev1.record(self.stream)

    def time_steps(self, n):
        """n timed steps (L2 flushed before each), device ms per step."""
        ms = []
        for _ in range(n):
            self.replay(self.graph, self.t_start, self.t_end)
            self.stream.synchronize()
            ms.append(self.t_start.elapsed_time(self.t_end))
        return ms

    def time_launches(self, n):
        """Per-launch device ms from the graph with events between launches."""
        out = []
        if not self.external:
            return out
        for _ in range(n):
            self.replay(self.launch_graph, self.events[0], self.events[self.launches])
            self.stream.synchronize()
            out.extend(self.events[i].elapsed_time(self.events[i + 1])
                       for i in range(self.launches))
        return out

    def check(self):
        assert self.pkv.pkv_get_error(self.pool) == self.pkv.PKV_OK

    def close(self):
        self.pool.close()
        for name in ("graph", "launch_graph", "k_pool", "v_pool", "q", "k_new", "v_new",
                     "table", "lens", "out"):
            setattr(self, name, None)


def gbs(nbytes, ms):
    return nbytes / (ms * 1e-3) / 1e9


def per_config_entry(run, hbm_peak, min_seconds, min_steps):
    """One workload timed over at least `min_seconds` of replays (and at least
    `min_steps` steps) with its own clock samples."""
    nbytes = step_bytes(run.wl, run.args.rope)
    for _ in range(3):
        run.replay(run.graph, run.t_start, run.t_end)
    torch.cuda.synchronize()
    probe = statistics.median(run.time_steps(5))
    n = max(min_steps, int(min_seconds * 1e3 / max(probe, 1e-3)))
    sampler = ClockSampler(run.dev)
    time.sleep(0.2)
    nvtx_push(f"per-config {run.wl.name}")
    ms = run.time_steps(n)
    nvtx_pop()
    clocks = sampler.stop()
    launch_ms = run.time_launches(max(3, min(200, n // 4)))
    run.check()
    mean = float(np.mean(ms))
    value = gbs(nbytes, mean)
    return {"gbs": round(value, 2), "pct_of_measured_hbm": round(100 * value / hbm_peak, 2),
            "pct_of_nominal_hbm": round(100 * value / NOMINAL_HBM_GBS, 2),
            "ms_per_step": round(mean, 5),
            "step_ms_p10_p50_p90": [round(float(np.percentile(ms, p)), 5) for p in (10, 50, 90)],
            "per_launch_us": round(1e3 * mean / run.launches, 3),
            "per_launch_us_events_between_launches":
                round(1e3 * float(np.mean(launch_ms)), 3) if launch_ms else None,
            "seq_layer_steps_per_s": round(run.wl.batch * run.wl.num_layers / (mean * 1e-3), 1),
            "steps": n, "timed_s": round(sum(ms) * 1e-3, 3), "plan": run.plan(),
            "bytes_per_step": nbytes, "clocks": clocks}


def run_ours(args, world, rank, local):
    import paged_kv_cache_210_gb300 as pkv
    from paged_kv_cache_210_gb300 import build as lib_build

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib_build.build()
    pkv.load()
    wl = WORKLOADS[args.workload](args.layers)
    L, B = wl.num_layers, wl.batch
    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.ones(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)

    def flush():
        return flush_buf.sum()

    stream = torch.cuda.Stream(device=dev)
    run = DecodeRun(pkv, wl, dev, args, stream, flush)
    launches = run.launches

    # e2e: the same step through the public API with host buffers (pinned),
    # copies inside the timed region; (a) the step's CUDA graph with the
    # copies captured in it, (b) direct calls from the host every step
    q_h = run.q.cpu().pin_memory()
    kn_h, vn_h = run.k_new.cpu().pin_memory(), run.v_new.cpu().pin_memory()
    lens_h = run.lens.cpu().pin_memory()
    out_h = torch.empty(run.out.shape, dtype=run.out.dtype).pin_memory()
    e2e_start, _ = make_event()
    e2e_end, _ = make_event()

    # With large layers the copies overlap the layers: the inputs go over on
    # a copy stream in three parts (layer 0's, which the first launch waits
    # for; layers 1-3, copied while layer 0 runs; the rest, copied while
    # layers 1-3 run), each launch waiting for the part holding its layer;
    # layer l's output comes back on a second copy stream once layer l is
    # done, while the later layers run (measured at batch 256: one copy per
    # layer cost more per copy than it hid). With
    # small layers (under 1 MiB of output each) the fixed cost of the extra
    # copies and, in the direct calls, of issuing them exceeds what they
    # hide, so all inputs go first and all outputs come back at the end, as
    # with the one multi-layer launch.
    h2d_stream = torch.cuda.Stream(device=dev)
    d2h_stream = torch.cuda.Stream(device=dev)
    n_layers = wl.num_layers
    # input parts: layer 0, then layers 1-3 (copied while layer 0 runs), then
    # the rest (copied while layers 1-3 run)
    in_parts = [slice(0, 1), slice(1, min(4, n_layers)), slice(min(4, n_layers), n_layers)]
    in_parts = [p for p in in_parts if p.start < p.stop]
    in_ev = [torch.cuda.Event() for _ in in_parts]
    out_ev = [torch.cuda.Event() for _ in range(n_layers)]

    pipelined = (not args.persistent and
                 run.out[0].numel() * run.out.element_size() >= (1 << 20))

    def e2e_body(s):
        if not pipelined:
            run.q.copy_(q_h, non_blocking=True)
            run.k_new.copy_(kn_h, non_blocking=True)
            run.v_new.copy_(vn_h, non_blocking=True)
            run.lens.copy_(lens_h, non_blocking=True)
            run.step(stream=s)
            out_h.copy_(run.out, non_blocking=True)
            return
        h2d_stream.wait_stream(s)
        d2h_stream.wait_stream(s)
        with torch.cuda.stream(h2d_stream):
            run.lens.copy_(lens_h, non_blocking=True)
            for part, rows in enumerate(in_parts):
                run.q[rows].copy_(q_h[rows], non_blocking=True)
                run.k_new[rows].copy_(kn_h[rows], non_blocking=True)
                run.v_new[rows].copy_(vn_h[rows], non_blocking=True)
                in_ev[part].record(h2d_stream)

        def before(layer):
            for part, rows in enumerate(in_parts):
                if layer == rows.start:
                    s.wait_event(in_ev[part])

        def after(layer):
            out_ev[layer].record(s)
            d2h_stream.wait_event(out_ev[layer])
            with torch.cuda.stream(d2h_stream):
                out_h[layer].copy_(run.out[layer], non_blocking=True)

        run.step(stream=s, before=before, after=after)
        s.wait_stream(d2h_stream)

    e2e_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(e2e_graph, stream=stream):
        s = torch.cuda.current_stream()
        if run.external:
            e2e_start.record(s)
        e2e_body(s)
        if run.external:
            e2e_end.record(s)
    h2d = sum(t.numel() * t.element_size() for t in (q_h, kn_h, vn_h, lens_h))
    d2h = out_h.numel() * out_h.element_size()

    # warm-up
    for _ in range(args.warmup):
        run.replay(run.graph, run.t_start, run.t_end)
    torch.cuda.synchronize()

    # timed region: exactly args.steps steps
    barrier(world)
    torch.cuda.synchronize()
    sampler = ClockSampler(dev)
    time.sleep(0.3)
    wall0 = time.perf_counter()
    nvtx_push(f"timed steps {wl.name}")
    step_ms = run.time_steps(args.steps)
    nvtx_pop()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(world)
    clocks = sampler.stop()
    total_ms = max_over_ranks(sum(step_ms), world)
    run.check()

    # per-launch durations of the dominant kernel (same launches, same flush)
    launch_ms = run.time_launches(max(3, min(args.steps, 400)))

    # e2e (a): graph with the copies
    e2e_ms = []
    for _ in range(max(3, args.steps // 4)):
        run.replay(e2e_graph, e2e_start, e2e_end)
        stream.synchronize()
        e2e_ms.append(e2e_start.elapsed_time(e2e_end))
    run.check()
    e2e_total = max_over_ranks(sum(e2e_ms), world)
    # e2e (b): direct C-ABI calls from the host each step, host wall clock
    direct_s = []
    for i in range(3 + max(3, args.steps // 4)):
        with torch.cuda.stream(stream):
            flush()
        stream.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            e2e_body(stream)
        stream.synchronize()
        if i >= 3:
            direct_s.append(time.perf_counter() - t0)
    run.check()
    direct_ms = max_over_ranks(1e3 * statistics.median(direct_s), world)

    nbytes = step_bytes(wl, args.rope)
    ms_per_step = total_ms / args.steps
    value = whole_job_gbs(world, nbytes, args.steps, total_ms)
    e2e_value = whole_job_gbs(world, nbytes, len(e2e_ms), e2e_total)

    # average launch duration: the timed region's events / launches (includes
    # the graph's gaps between launches, so an upper bound on kernel time)
    per_launch_ms = ms_per_step / launches
    launch_source = (f"timed-region CUDA events (start/end of each step) / {launches} launch"
                     + ("es" if launches > 1 else ""))
    events_between = (round(statistics.mean(launch_ms), 6) if launch_ms else None)
    achieved = (nbytes / launches) / (per_launch_ms * 1e-3) / 1e9
    if args.persistent:
        kernel_name = "decode_layers_kernel"
        traffic = recorded_traffic("decode_layers_" + args.workload, "layers")
        step_note = ("16 layers of fused append+attend in one persistent launch (per-sequence "
                     "layer order kept by device-side waits), CUDA graph")
    else:
        kernel_name = "decode_kernel<fused>"
        traffic = recorded_traffic("decode_fused_" + args.workload +
                                   ("-rope" if args.rope else ""))
        step_note = ("16 x fused append+attend (one launch per layer), CUDA graph" +
                     ("" if args.no_pdl else ", programmatic dependent launch between layers"))
    plan = run.plan()
    run.close()
    del run

    # every other workload of the set, each timed over at least a second
    per_config = {}
    if not args.no_per_config:
        for name in PER_CONFIG:
            torch.cuda.empty_cache()
            other = DecodeRun(pkv, WORKLOADS[name](args.layers), dev, args, stream, flush)
            per_config[name] = per_config_entry(other, hbm_peak, args.per_config_seconds,
                                                args.steps)
            other.close()
            del other

    if rank != 0:
        return
    chunk_note = "library's choice" if args.splits == 0 else f"{args.splits} splits per sequence"
    config = decode_config(wl, args, world)
    config.update({"step": step_note, "splits": chunk_note, "plan": plan})
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "storage_dtype": "bf16", "data": "synthetic", "config": config,
        "seq_layer_steps_per_s": round(world * B * L * args.steps / (total_ms * 1e-3), 1),
        "pct_of_measured_hbm": round(100 * value / world / hbm_peak, 2),
        "pct_of_nominal_hbm": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "step_ms_p10_p50_p90": [round(float(np.percentile(step_ms, p)), 5) for p in (10, 50, 90)],
        "clocks": clocks,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_total / len(e2e_ms), 5),
                "how": ("step's CUDA graph replayed with the pinned host->device input copies "
                        "and the device->host output copies captured in it (device events)"
                        + ("" if not pipelined else
                           "; inputs on a copy stream in three parts (layer 0, layers "
                           "1-3 while layer 0 runs, the rest while layers 1-3 run), each "
                           "layer's output back on a second copy stream while the later "
                           "layers run")),
                "ms_per_step_direct_calls": round(direct_ms, 5),
                "gbs_direct_calls": round(world * gbs(nbytes, direct_ms), 2),
                "direct_calls_how": f"{launches} C-ABI calls issued from Python each step "
                                    "(ctypes binding, argument checks, launch) plus the same "
                                    "copies, host wall clock around the step, median"},
        "gpu_launches": launches * args.steps,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                     "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "traffic": traffic, "kernel": kernel_name,
                     "per_launch_ms": round(per_launch_ms, 6), "per_launch_source": launch_source,
                     "per_launch_ms_with_events_between_launches": events_between,
                     "bytes_per_launch": nbytes // launches},
        "wall_s_timed_loop": round(wall, 3),
    }
    if per_config:
        line["per_config"] = per_config
    if not args.no_cpu_baseline and rank == 0:
        line["cpu_baseline"] = cpu_baseline(wl, args.rope)
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- admission scheduler (host)
def scheduler_trace(n_steps, seed=W.BASE_SEED + 20):
    """A continuous-batching trace at the 4 GiB pool: requests with prompts
    log-uniform in [16, 1024] and allowances log-uniform in [16, 1024],
    submitted two per step, some ending early; returns per-step actions."""
    rng = np.random.default_rng(seed)
    lo, hi = np.log(16), np.log(1024)
    steps = []
    for _ in range(n_steps):
        subs = [(int(np.exp(rng.uniform(lo, hi))), int(np.exp(rng.uniform(lo, hi))))
                for _ in range(2)]
        steps.append((subs, float(rng.random())))
    return steps


def drive_scheduler(api, pool_pages, trace, max_batch=256):
    """Runs the trace through a scheduler API (native or oracle); returns
    (seconds of scheduler calls on the decode path, steps, batch sizes)."""
    s = api["create"](pool_pages)
    length, prefix = {}, {}
    t_decode = 0.0
    batches = []
    for subs, early in trace:
        for p, n in subs:
            rid = api["submit"](s, p, n)
            if rid is not None:
                prefix[rid] = p + min(n, 2048 - p) - 1
                length[rid] = p
        admitted = api["admit"](s)
        t0 = time.perf_counter()
        batch = api["batch"](s)[:max_batch]
        api["extend"](s, batch, [length[r] for r in batch])
        api["tables"](s, batch, max_batch)
        t_decode += time.perf_counter() - t0
        batches.append(len(batch))
        for i, rid in enumerate(batch):
            if length[rid] >= prefix[rid] or (i == 0 and early < 0.05):
                api["finish"](s, rid)
                del length[rid]
            else:
                length[rid] += 1
        del admitted
    return t_decode, len(trace), batches


def run_scheduler_bench(args):
    import paged_kv_cache_210_gb300 as pkv
    from paged_kv_cache_210_gb300 import build as lib_build
    lib_build.build()
    pkv.load()
    pool_pages = W.pages_for_pool_mib(4096)

    def native_submit(s, p, n):
        try:
            return pkv.pkv_sched_submit(s, p, n)
        except pkv.PkvError:
            return None
    tables = {}

    def native_tables(s, batch, max_batch):
        out = tables.get(max_batch)
        if out is None:
            out = tables[max_batch] = np.empty((16, max_batch, 128), np.int32)
        return pkv.pkv_sched_block_tables(s, batch, max_batch, 128, out, clear_tail=False)
    native = {"create": lambda n: pkv.pkv_sched_create(n), "submit": native_submit,
              "admit": pkv.pkv_sched_admit, "batch": pkv.pkv_sched_decode_batch,
              "extend": pkv.pkv_sched_extend_batch, "finish": pkv.pkv_sched_finish,
              "tables": native_tables}
    trace = scheduler_trace(args.warmup + args.steps)
    drive_scheduler(native, pool_pages, trace[:args.warmup])
    t, n, batches = drive_scheduler(native, pool_pages, trace)
    us = t / n * 1e6
    line = {
        "metric": "admission scheduler host time per decode step (batch, page growth, block "
                  "tables)", "value": round(us, 3), "unit": "us/step", "n_gpus": 0,
        "steps": n, "warmup": args.warmup, "higher_is_better": False, "dtype": "int32",
        "data": "synthetic",
        "config": {"workload": "continuous batching at the 4 GiB pool (131072 pages), 16 layers, "
                               "prompts and allowances log-uniform in [16, 1024], 2 submissions "
                               "per step, decode batch capped at 256",
                   "mean_batch": round(float(np.mean(batches)), 1),
                   "max_batch": int(np.max(batches)),
                   "tables_bytes_per_step": 16 * 256 * 128 * 4},
    }
    if not args.no_cpu_baseline:
        from oracle import admission as A

        def o_submit(s, p, n):
            st, rid = s.submit(p, n)
            return rid
        orc = {"create": lambda n: A.AdmissionScheduler(n), "submit": o_submit,
               "admit": lambda s: s.admit(), "batch": lambda s: s.decode_batch(),
               "extend": lambda s, rs, ls: [s.extend(r, l) for r, l in zip(rs, ls)],
               "finish": lambda s, r: s.finish(r),
               "tables": lambda s, b, mb: s.block_tables(b, 128)}
        sample = min(len(trace), 400)
        to, no, _ = drive_scheduler(orc, pool_pages, trace[:sample])
        line["cpu_baseline"] = {"value": round(to / no * 1e6, 3), "unit": "us/step", "cores": 1,
                                "kind": "oracle", "sample": f"first {sample} steps of the trace"}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- prefill over pages
def prefill_flops(wl):
    """Algorithmic FLOPs of one prefill attention launch: for every chunk
    token at position p and each of the 32 query heads, (p + 1) keys of
    64-dim dot products and (p + 1) value rows of 64: 4 * 64 * (p + 1)."""
    total = 0
    for s0, n in zip(wl.start_pos.tolist(), wl.chunk_lens.tolist()):
        keys = n * s0 + n * (n + 1) // 2
        total += keys
    return total * W.NUM_Q_HEADS * W.HEAD_DIM * 4


def run_prefill_bench(args):
    import paged_kv_cache_210_gb300 as pkv
    from paged_kv_cache_210_gb300 import build as lib_build
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    lib_build.build()
    pkv.load()
    wl = W.prefill_prompt(args.prompt_len)
    L, T = wl.num_layers, wl.total_tokens
    k_pool, v_pool = wl.pools(dev, "zero")
    q, k, v = wl.q(dev), wl.k(dev), wl.v(dev)
    table = torch.from_numpy(wl.block_tables).to(dev)
    cu = torch.from_numpy(wl.cu_tokens).to(dev)
    start = torch.from_numpy(wl.start_pos).to(dev)
    out = torch.zeros((L, T, W.NUM_Q_HEADS, W.HEAD_DIM), device=dev)
    pool = pkv.pkv_pool_create(L, wl.num_pages, wl.batch)
    max_chunk = int(wl.chunk_lens.max())
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.ones(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    made = [make_event() for _ in range(2 * L + 3)]
    external = all(e[1] for e in made)
    marks = [e[0] for e in made[:2 * L + 1]]
    t0, t1 = made[2 * L + 1][0], made[2 * L + 2][0]

    def step(events=None):
        s = torch.cuda.current_stream()
        if events:
            events[0].record(s)
        for layer in range(L):
            pkv.pkv_prefill_fill(pool, layer, k[layer], v[layer], k_pool, v_pool, table, cu, start,
                                 max_chunk, stream=s)
            if events and len(events) > 2:
                events[2 * layer + 1].record(s)
            pkv.pkv_prefill_attention(pool, layer, q[layer], k_pool, v_pool, table, cu, start,
                                      out[layer], max_chunk, stream=s)
            if events and len(events) > 2:
                events[2 * layer + 2].record(s)
        if events and len(events) == 2:
            events[1].record(s)

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    graph, per_launch = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step([t0, t1] if external else None)
    with torch.cuda.graph(per_launch, stream=stream):
        step(marks if external else None)

    def replay(g, a, b):
        with torch.cuda.stream(stream):
            flush_buf.sum()
            if external:
                g.replay()
            else:
                a.record(stream)
                g.replay()
                b.record(stream)

    for _ in range(args.warmup):
        replay(graph, t0, t1)
    torch.cuda.synchronize()
    sampler = ClockSampler(dev)
    time.sleep(0.3)
    step_ms = []
    for _ in range(args.steps):
        replay(graph, t0, t1)
        stream.synchronize()
        step_ms.append(t0.elapsed_time(t1))
    clocks = sampler.stop()
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    fill_ms, attn_ms = [], []
    if external:
        for _ in range(max(3, min(args.steps, 100))):
            replay(per_launch, marks[0], marks[-1])
            stream.synchronize()
            for layer in range(L):
                fill_ms.append(marks[2 * layer].elapsed_time(marks[2 * layer + 1]))
                attn_ms.append(marks[2 * layer + 1].elapsed_time(marks[2 * layer + 2]))
    ms = float(np.mean(step_ms))
    flops = prefill_flops(wl)
    peaks, kind = measured_peaks()
    peak = float(peaks.get("bf16_tflops", 1900.0))
    attn_launch_ms = float(np.mean(attn_ms)) if attn_ms else ms / L
    achieved = flops / (attn_launch_ms * 1e-3) / 1e12
    line = {
        "metric": "prefill over pages: causal attention TFLOP/s (algorithmic) and prompt "
                  "tokens/s", "value": round(flops * L / (ms * 1e-3) / 1e12, 2),
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 operands, f32 accumulate", "data": "synthetic",
        "config": {"workload": f"prefill-{args.prompt_len}: one {args.prompt_len}-token prompt, "
                               "16 layers, 32q/8kv heads, head_dim 64, 128 MiB pool, shuffled "
                               "pages; per layer the page fill then causal attention over the "
                               "pages",
                   "l2": "flushed before every step (read of a buffer twice the L2 size)",
                   "flops_per_layer": flops},
        "prompt_tokens_per_s": round(T / (ms * 1e-3), 1),
        "step_ms_p10_p50_p90": [round(float(np.percentile(step_ms, p)), 4) for p in (10, 50, 90)],
        "clocks": clocks,
        "gpu_launches": 2 * L * args.steps,
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "peak_kind": f"{kind} cuBLAS bf16 burst (MEASURED_PEAKS bf16_tflops)",
                     "traffic": recorded_traffic(f"prefill_attention_{wl.name}", "prefill"),
                     "kernel": "prefill_attention_kernel",
                     "per_launch_ms": round(attn_launch_ms, 5),
                     "fill_per_launch_ms": round(float(np.mean(fill_ms)), 5) if fill_ms else None},
    }
    if not args.no_cpu_baseline:
        import oracle
        orc = oracle.load()
        g = oracle.geometry(L, wl.num_pages, wl.batch)
        kp, vp = (t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()
                  for t in wl.pools("cpu", "zero"))

        def b16(t):
            return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()
        qc, kc, vc = b16(wl.q()[0]), b16(wl.k()[0]), b16(wl.v()[0])
        threads = cpu_threads()
        tt = time.perf_counter()
        assert orc.prefill_fill(g, 0, kc, vc, kp, vp, wl.block_tables, wl.cu_tokens,
                                wl.start_pos) == oracle.OK
        st, _ = orc.prefill_attention(g, 0, qc, kp, vp, wl.block_tables, wl.cu_tokens,
                                      wl.start_pos, threads=threads)
        dt = time.perf_counter() - tt
        assert st == oracle.OK
        line["cpu_baseline"] = {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s",
                                "cores": min(threads, wl.batch * W.NUM_KV_HEADS),
                                "kind": "oracle",
                                "sample": f"1 of {L} layers (fill + attention), {dt:.1f} s"}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(WORKLOADS), default="ragged-b256",
                    help="the headline workload (default: the largest configuration)")
    ap.add_argument("--layers", type=int, default=16,
                    help="layers per step (16, the model's; fewer only for profiling captures "
                         "on a smaller pool: the per-layer launches are the same)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip timing the other workloads beside the headline")
    ap.add_argument("--per-config-seconds", type=float, default=1.0,
                    help="minimum timed seconds per workload in per_config")
    ap.add_argument("--splits", type=int, default=0, help="0: the library chooses")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--rope", action="store_true",
                    help="rotate the appended key and the queries inside the launches")
    ap.add_argument("--persistent", action="store_true",
                    help="decode: all 16 layers in one persistent launch "
                         "(pkv_append_attend_layers)")
    ap.add_argument("--no-pdl", action="store_true",
                    help="launch without programmatic dependent launch")
    ap.add_argument("--component", choices=["decode", "scheduler", "prefill"], default="decode",
                    help="scheduler: the host admission scheduler; prefill: prefill over pages")
    ap.add_argument("--prompt-len", type=int, default=2048, help="prefill prompt length")
    args = ap.parse_args()
    if args.persistent and args.rope:
        ap.error("--persistent runs the unrotated fused step; drop --rope")
    if args.persistent and args.splits:
        ap.error("--persistent plans its own clusters; drop --splits")
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if not 1 <= args.layers <= 16:
        ap.error("--layers must be in 1..16")
    if args.component == "scheduler":
        run_scheduler_bench(args)
        return
    if args.component == "prefill":
        run_prefill_bench(args)
        return
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
