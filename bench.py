"""Benchmark: materialized GB/s (destination bytes) and fraction of the HBM
roofline for st_materialize on one GB300, next to the CPU oracle.

One step = one pass of the whole path over one checkpoint: every selected
tensor gathered from the device-resident data section and cast into its
destination (one kernel launch for the default single-chunk plan).  The
headline workload is the largest single-GPU configuration, the scaled-FP8
checkpoint: 57 blocks of E4M3 linears (570 weights of [3072,3072] and
[12288,3072], 11.83 GB) with one F32 scale each, dequantized to BF16
(23.67 GB out, 35.50 GB moved per launch).  The line also carries, under
"configs", the same kernel measurement for the other checkpoints (16 tiny
mixed tensors, the UNet-shaped F16 checkpoint, the 8B LLM's 4 joined shards to
BF16 and to F16, 100k misaligned tiny tensors) and for the sliced and
block-scaled loads, each timed in this process.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload scaled_fp8|unet|tiny|llm8b|llm8b_f16|stress|...]
                  [--configs auto|all|none] [--split replica|partition]

Prints one JSON line (rank 0).  Under torchrun each rank materializes its own
replica (--split replica, weak scaling) or its byte-balanced part of the
outputs (--split partition); no data-path collective; timings are
max-reduced.  --gpus N > 1 without torchrun re-launches this script under
torchrun with N processes.
"""
import argparse
import concurrent.futures as cf
import json
import os
import socket
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PROFILES = os.path.join(ROOT, "profiles")
TRAFFIC = os.path.join(PROFILES, "traffic.json")
KERNEL_SRC = os.path.join(ROOT, "safetensors_materialization_gb300", "csrc", "st_kernels.cu")

HEADLINE = "scaled_fp8"
# the other configurations of the metric, then the sliced and block-scaled loads
CONFIG_ROWS = ["tiny", "unet", "llm8b", "llm8b_f16", "stress", "llm8b_tp4", "block_fp8", "nvfp4"]


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--dst", default=None, help="output dtype (default: the workload's)")
    ap.add_argument("--configs", choices=["auto", "all", "none"], default="auto",
                    help="also time the other configurations (auto: with the default headline on one GPU)")
    ap.add_argument("--split", choices=["replica", "partition"], default="replica",
                    help="multi-GPU: every rank loads everything, or its byte-balanced part")
    ap.add_argument("--e2e-chunk-mb", type=int, default=128)
    ap.add_argument("--workers", type=int, default=0, help="warps to balance over (0: from --blocks-per-sm)")
    ap.add_argument("--blocks-per-sm", type=int, default=0, help="resident 8-warp blocks per SM (0: library default)")
    ap.add_argument("--unit-bytes", type=int, default=0, help="traffic per interleaved unit (0: library default)")
    ap.add_argument("--kernel", type=int, default=0, help="kernel build: 0 auto, 1 streaming, 2 latency, 3 tma, 4 wide tma")
    ap.add_argument("--order", type=int, default=0, help="unit order: 0 the build's default, 1 source, 2 class-major")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-files", choices=["auto", "on", "off"], default="auto",
                    help="also time st_load_files from shard files written to a temp dir (auto: below 8 GB)")
    ap.add_argument("--io-threads", type=int, default=16)
    ap.add_argument("--lazy", choices=["auto", "on", "off"], default="auto",
                    help="also time the lazy one-tensor-at-a-time path (auto: up to 2000 tensors, below 8 GB)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launch_command(args, world, argv):
    """None when this process runs as it is; else the torchrun command that
    runs --gpus ranks (one process per GPU).  Raises SystemExit when --gpus
    contradicts an existing WORLD_SIZE or the GPUs are not there."""
    if args.gpus < 1:
        raise SystemExit("bench.py: --gpus must be at least 1")
    if "WORLD_SIZE" in os.environ:
        if world != args.gpus:
            raise SystemExit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}: launch with --nproc-per-node "
                             f"{args.gpus} or pass --gpus {world}")
        return None
    if args.gpus == 1:
        return None
    if args.impl == "ours":
        import torch
        have = torch.cuda.device_count() if torch.cuda.is_available() else 0
        if have < args.gpus:
            raise SystemExit(f"bench.py: --gpus {args.gpus} needs {args.gpus} GPUs, this node has {have}")
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
            "--master-addr", "127.0.0.1", "--master-port", str(free_port()), os.path.abspath(__file__), *argv]


def host_cpu_model():
    """The host CPU's model name (lscpu's, from /proc/cpuinfo or the platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, burst copy)"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback 6.8 TB/s"


def kernel_code(text):
    """The kernel source without its comments and blank space: what a DRAM
    traffic record depends on (a comment edit leaves the kernel unchanged)."""
    import re
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"' or c == "'":                      # a literal, kept whole
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
        else:
            out.append(c)
            i += 1
    return re.sub(r"\s+", " ", "".join(out)).strip()


def kernel_sha():
    """sha256 prefix of the kernel code (st_kernels.cu, comments and blank
    space removed) that profiles/traffic.json records are keyed to."""
    import hashlib
    with open(KERNEL_SRC, encoding="utf-8") as f:
        return hashlib.sha256(kernel_code(f.read()).encode()).hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM read + write bytes per launch of `workload` from the committed
    1-pass ncu record (profiles/traffic.json), if it was taken on the current
    kernel source; else None."""
    try:
        with open(TRAFFIC) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    r = rec.get("workloads", {}).get(workload)
    if not r or r.get("kernel_sha256") != kernel_sha():
        return None
    return int(r["traffic_per_launch"])


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self, lead=1.5):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(lead)  # let nvidia-smi start sampling before the timed region
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def build_workload(name, dst=None):
    from safetensors_materialization_gb300 import synth
    w = synth.WORKLOADS[name]()
    if dst and dst != w.dst[0]:
        w.dst = [dst]
        w.name += "_to_" + dst.lower()
        if dst == "KEEP":
            w.scale_suffix = None
    return w


def source_bytes(ix, infos):
    """Algorithmic source bytes of a plan's outputs: each output's source
    elements once (a slice reads only its elements), plus the block scales of
    block-scaled outputs."""
    size = {"F16": 2, "BF16": 2, "F32": 4, "F8_E4M3": 1, "F8_E5M2": 1, "I64": 8, "BOOL": 1, "U8": 1}
    total = 0
    for o in infos:
        if o.get("quant") == "nvfp4":
            total += o["numel"] // 2
        else:
            total += o["numel"] * size.get(o["src_dtype"], 1)
        if o.get("quant"):
            e = ix.entry(ix.find(o["scale"]))
            total += e["end"] - e["begin"]
    return total


def host_image(w, stmat, torch):
    """(root index, pinned host tensor, offset of the data section in it).
    One shard: the whole file image.  Several: one arena holding every shard's
    data section at the bases st_index_concat gives, under one joined index,
    so that one plan and one launch cover all shards."""
    from safetensors_materialization_gb300 import synth
    if len(w.files) == 1:
        lay = w.files[0]
        host = torch.empty(lay.file_bytes, dtype=torch.uint8, pin_memory=True)
        synth.build_workload_file(w, 0, out=host.numpy())
        return stmat.Index.from_file(host.numpy()), host, lay.data_start
    parts = [stmat.Index.from_header(lay.header, lay.data_bytes) for lay in w.files]
    ix, bases = stmat.Index.concat(parts)
    host = torch.empty(ix.sizes()[1], dtype=torch.uint8, pin_memory=True)
    arena = host.numpy()
    for k, lay in enumerate(w.files):
        synth.build_workload_data(w, k, arena[bases[k]:bases[k] + lay.data_bytes])
    return ix, host, 0


# ------------------------------------------------------------------ oracle

def oracle_selection(w):
    """The oracle's selection of the workload (first shard for a sharded
    checkpoint) and that shard's layout."""
    from oracle import oracle as O
    lay = w.files[0]
    ix = w.view(O.parse_header(lay.header, lay.data_bytes))
    return ix.select(dst=w.dst[0], scale_suffix=w.scale_suffix, **w.selection(ix)), lay


def oracle_sample(w, seconds, data):
    """Times the oracle, single thread, on a bounded sample of the workload:
    whole outputs in plan order until about `seconds` of work.  `data`: the
    (first shard's) data section in host memory.  Returns (dst GB/s,
    description, bytes, seconds, outputs timed, every output's bytes)."""
    sel, lay = oracle_selection(w)
    outs = sel.outputs()
    # calibrate on the first output, then pick a prefix of outputs
    t0 = time.perf_counter()
    sel.materialize(0, data)
    rate = outs[0]["bytes"] / max(1e-9, time.perf_counter() - t0)
    budget = rate * seconds
    k, acc = 0, 0
    while k < len(outs) and acc < budget:
        acc += outs[k]["bytes"]
        k += 1
    t0 = time.perf_counter()
    for i in range(k):
        sel.materialize(i, data)
    dt = time.perf_counter() - t0
    where = w.name if len(w.files) == 1 else f"shard 0 of {w.name}"
    desc = f"first {k} of {len(outs)} outputs ({acc / 1e6:.1f} MB dst) of {where}, single thread"
    return acc / dt / 1e9, desc, acc, dt, k, [o["bytes"] for o in outs]


class OracleThreads:
    """The oracle (unchanged) on every host core: its C calls release the
    GIL, so a pool of threads, one per core, materializes outputs side by
    side from one shared copy of the data section.  run(k) materializes the
    first k outputs, dealt largest first to the least-loaded thread."""

    def __init__(self, sel, data, cores):
        self.sel, self.data, self.cores = sel, data, cores
        self.sizes = [o["bytes"] for o in sel.outputs()]
        self.pool = cf.ThreadPoolExecutor(cores)

    def _share(self, indices):
        n = 0
        for i in indices:
            self.sel.materialize(i, self.data)
            n += self.sizes[i]
        return n

    def run(self, k):
        shares = [[] for _ in range(self.cores)]
        load = [0] * self.cores
        for i in sorted(range(k), key=lambda i: -self.sizes[i]):
            j = load.index(min(load))
            shares[j].append(i)
            load[j] += self.sizes[i]
        t0 = time.perf_counter()
        n = sum(self.pool.map(self._share, shares))
        return n, time.perf_counter() - t0

    def close(self):
        self.pool.shutdown()


def run_reference(args, rank, world):
    """The reference arm is the oracle (no reference implementation exists):
    each step materializes a bounded sample of the workload with the oracle
    on every host core (OracleThreads)."""
    if rank != 0:
        return
    from safetensors_materialization_gb300 import synth
    w = build_workload(args.workload, args.dst)
    per_step = max(0.5, min(8.0, 30.0 / max(1, args.steps + args.warmup)))
    cores = max(1, len(os.sched_getaffinity(0)))
    sel, lay = oracle_selection(w)
    data = np.empty(lay.data_bytes, np.uint8)
    synth.build_workload_data(w, 0, data)
    outs = sel.outputs()
    op = OracleThreads(sel, data, cores)
    try:
        # calibrate: double a prefix of outputs until one run takes a quarter second, then take the
        # prefix that fills the step budget at that rate
        k = min(len(outs), cores)
        while True:
            nb, dt0 = op.run(k)
            if dt0 >= 0.25 or k >= len(outs):
                break
            k = min(len(outs), 2 * k)
        rate = max(1, nb) / max(1e-9, dt0)
        k, acc = 0, 0
        while k < len(outs) and acc < rate * per_step:
            acc += outs[k]["bytes"]
            k += 1
        for _ in range(args.warmup):
            op.run(k)
        total = 0.0
        for _ in range(args.steps):
            nbytes, dt = op.run(k)
            total += dt
    finally:
        op.close()
    dt = total / max(1, args.steps)
    value = nbytes / dt / 1e9
    where = w.name if len(w.files) == 1 else f"shard 0 of {w.name}"
    sample = f"first {k} of {len(outs)} outputs ({nbytes / 1e6:.1f} MB dst) of {where} per step, {cores} threads"
    line = {
        "impl": "reference", "metric": "materialized GB/s (dst bytes)", "value": round(value, 4),
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "sample": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------------- ours

def write_shards(w, host, data_start, stmat, tmp):
    """The workload's shard files (header + data section) under `tmp`."""
    paths = []
    hb = host.numpy()
    bases = None
    if len(w.files) > 1:
        _, bases = stmat.Index.concat([stmat.Index.from_header(x.header, x.data_bytes) for x in w.files])
    for k, lay in enumerate(w.files):
        path = os.path.join(tmp, f"shard{k}.safetensors")
        lo = data_start if bases is None else bases[k]
        with open(path, "wb") as f:
            f.write(lay.header)
            f.write(memoryview(hb[lo:lo + lay.data_bytes]))
        paths.append(path)
    return paths


def time_lazy(args, w, host, data_start, stmat, torch):
    """The lazy path: every output loaded alone through StreamStateDict
    (st_load_tensors) from the workload's files in the page cache; a cold
    pass (every tensor read into the RAM tier), a warm pass (every tensor a
    RAM-tier hit), a pass without a RAM tier (each tensor copied straight
    from the files' mappings) and a warm pass in batches (StreamStateDict.
    load_many).  Reports tensors/s and dst GB/s per pass."""
    import shutil
    import tempfile
    tmp = tempfile.mkdtemp(prefix="stmat_lazy_")
    try:
        paths = write_shards(w, host, data_start, stmat, tmp)
        sd = stmat.StreamStateDict(paths, dst=w.dst[0], ram_cache_bytes=1 << 34, threads=args.io_threads,
                                   rename=w.rename or None, prefix=w.prefix, scale_suffix=w.scale_suffix,
                                   quant=w.quant)
        names = [o for o in sd.keys()]
        if w.scale_suffix:   # scales are consumed by their weights
            names = [n for n in names if not n.endswith(w.scale_suffix[1])]
        if w.quant:
            names = [n for n in names if n in w.quant]
        sd0 = stmat.StreamStateDict(paths, dst=w.dst[0], ram_cache_bytes=0, threads=args.io_threads,
                                    rename=w.rename or None, prefix=w.prefix, scale_suffix=w.scale_suffix,
                                    quant=w.quant)
        res = {}
        for label, d in (("cold", sd), ("warm", sd), ("no_ram_tier", sd0)):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            nbytes = 0
            for n in names:
                t = d[n]
                nbytes += t.numel() * t.element_size()
                del t
            torch.cuda.synchronize()
            dt = time.perf_counter() - t0
            res[label] = {"tensors_per_s": round(len(names) / dt, 1), "gbs_dst": round(nbytes / dt / 1e9, 3),
                          "ms": round(dt * 1e3, 1)}
        if sd.check() != 0:
            raise RuntimeError("a lazy load left a device flag")
        # the same tensors in batches (one copy and one launch per batch), RAM tier warm; one
        # untimed pass first, so that the device allocator already holds the outputs' memory
        # (the one-at-a-time passes free each output at once and reuse one block)
        del sd0
        sd.load_many(names)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        got = sd.load_many(names)
        nbytes = sum(t.numel() * t.element_size() for t in got.values())
        del got
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        res["warm_batched"] = {"tensors_per_s": round(len(names) / dt, 1), "gbs_dst": round(nbytes / dt / 1e9, 3),
                               "ms": round(dt * 1e3, 1)}
        st = sd.cache.stats()
        res.update({"tensors": len(names), "ram_tier": {"hits": st["hits"], "misses": st["misses"],
                                                         "bytes": st["bytes"]},
                    "source": "one st_load_tensors per tensor (header-only index, pread into the pinned RAM "
                              "tier or, without it, a copy from the files' mappings; staged copy, one launch); "
                              "files in the page cache"})
        return res
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


def time_load_files(args, c, dist, world):
    """st_load_files from the workload's shard files, written to a temp dir
    just before (so they are read from the page cache): dst GB/s per step.
    Ring-less (copies straight from the files' mappings) where the GPU reads
    pageable memory through the host's page tables, else through a pinned
    ring filled by pread threads; the other mode and a first load (files
    opened, loaded once and closed inside each step: fresh mappings) are
    listed beside it."""
    import shutil
    import tempfile
    torch, stmat, w = c.torch, c.stmat, c.w
    tmp = tempfile.mkdtemp(prefix="stmat_bench_")
    try:
        paths = write_shards(w, c.host, c.data_start, stmat, tmp)
        files, fix = stmat.Files.of_checkpoint(paths)
        opened = [stmat.Index.open(p) for p in paths]
        _, bases = stmat.Index.concat([o[0] for o in opened])
        parts = [(p, off, o.sizes()[1], b) for p, (o, off), b in zip(paths, opened, bases)]
        chunk = args.e2e_chunk_mb << 20
        fplan = w.view(fix).plan(dst=w.dst[0], scale_suffix=w.scale_suffix, chunk_bytes=chunk, **c.plan_kw)
        ring = torch.empty(3 * chunk, dtype=torch.uint8).pin_memory()
        copy = torch.cuda.Stream()
        ddata = c.dev[:c.data_bytes]
        direct = stmat.reads_pageable(torch.cuda.current_device())

        def load(fl, r):
            fplan.load_files(fl, ddata, c.outs.ptrs, r, threads=args.io_threads, copy_stream=copy,
                             compute_stream=c.stream)
            if fplan.check(c.stream) != 0:
                raise RuntimeError("st_load_files flagged a bad destination")

        def first_load(r):
            fl = stmat.Files(parts)
            load(fl, r)
            fl.close()

        steps = max(3, min(args.steps, 5))

        def timed(step):
            for _ in range(2):
                step()
            if dist:
                dist.barrier()
            reps = []
            for _ in range(3):
                t0 = time.perf_counter()
                for _ in range(steps):
                    step()
                reps.append((time.perf_counter() - t0) / steps)
            return max_over_ranks(statistics.median(reps), dist, torch), reps

        main_ring = None if direct else ring
        es, reps = timed(lambda: load(files, main_ring))
        other, _ = timed(lambda: load(files, ring if direct else None))
        first, _ = timed(lambda: first_load(main_ring))
        gbs = lambda t: round(c.gb_dst_all / t, 1)
        return {"value": round(c.gb_dst_all / es, 3), "unit": "GB/s", "ms_per_step": round(es * 1e3, 3),
                "repeats_gbs": [gbs(r) for r in reps], "files": len(paths),
                "file_bytes_per_step": fplan.copy_bytes()[0],
                "chunk_bytes": chunk,
                "mode": "ring-less: copies from the files' mappings" if direct else
                        f"pinned ring of {3 * chunk} bytes, {args.io_threads} pread threads",
                "gpu_reads_pageable": direct,
                ("ring_gbs" if direct else "ringless_gbs"): gbs(other),
                "first_load_gbs": gbs(first),
                "source": "shard files in the page cache (written just before); first_load opens, loads and "
                          "closes the files inside each step"}
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


def max_over_ranks(x, dist, torch):
    if not dist:
        return x
    t = torch.tensor([x], device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, dist, torch):
    if not dist:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


class Case:
    """One workload resident on this GPU: the source bytes in pinned host
    memory (the end-to-end source) and on the device, the plan of this
    rank's outputs (all of them, or its part under --split partition) and
    their destination arena."""

    def __init__(self, args, name, rank, world, dist, stmat, torch):
        self.args, self.stmat, self.torch = args, stmat, torch
        self.w = w = build_workload(name, args.dst if name == args.workload else None)
        self.root, self.host, self.data_start = host_image(w, stmat, torch)
        self.ix = w.view(self.root)
        self.data_bytes = self.root.sizes()[1]
        part = args.split == "partition" and world > 1
        self.plan_kw = dict(workers=args.workers, blocks_per_sm=args.blocks_per_sm, unit_bytes=args.unit_bytes,
                            kernel=args.kernel, order=args.order, **w.selection(self.ix))
        if part:
            self.plan_kw.update(part=rank, n_parts=world)
        self.dev = torch.empty(self.host.numel() + 256, dtype=torch.uint8, device="cuda")
        if w.whole_file_on_device:
            self.dev[:self.host.numel()].copy_(self.host)
            self.data_ptr = self.dev.data_ptr() + self.data_start
        else:
            self.dev[:self.data_bytes].copy_(self.host[self.data_start:self.data_start + self.data_bytes])
            self.data_ptr = self.dev.data_ptr()
        self.stream = torch.cuda.current_stream()
        self.dist = dist
        self.replan(w)

    def replan(self, w):
        """Plans workload `w` over the resident bytes (the same checkpoint,
        another selection or output dtype) with fresh destinations."""
        torch, stmat = self.torch, self.stmat
        self.w, self.outs, self.flush = w, None, None
        self.plan = self.ix.plan(dst=w.dst[0], scale_suffix=w.scale_suffix, **self.plan_kw)
        self.outs = stmat.Outputs(self.plan)
        self.infos = self.plan.outputs()
        self.dst_bytes = sum(o["bytes"] for o in self.infos)
        self.src_bytes = source_bytes(self.ix, self.infos)
        self.gb_dst_all = sum_over_ranks(self.dst_bytes, self.dist, torch) / 1e9
        l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
        self.flush = None
        if self.src_bytes + self.dst_bytes < 4 * l2:
            self.flush = torch.empty(4 * l2, dtype=torch.uint8, device="cuda")
        self.l2_note = (f"L2 flushed before each timed launch ({4 * l2 / 1e6:.0f} MB written)"
                        if self.flush is not None else
                        f"inputs exceed L2 (no flush): {(self.src_bytes + self.dst_bytes) / 1e9:.2f} GB per step "
                        f"vs {l2 / 1e9:.3f} GB L2")

    def warm(self, n):
        for _ in range(max(3, n)):
            self.plan.materialize(self.data_ptr, self.outs.ptrs, stream=self.stream)
        self.torch.cuda.synchronize()
        if self.plan.check() != 0:
            raise RuntimeError(f"{self.w.name}: materialize flagged a bad destination")

    def time_launches(self, steps):
        """Per-launch device times (ms) of `steps` launches, CUDA events on the
        launching stream: back to back when the bytes exceed L2, else each
        after writing a buffer of 4x L2."""
        torch, plan, st = self.torch, self.plan, self.stream
        if self.flush is None:
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
            evs[0].record(st)
            for k in range(steps):
                plan.materialize(self.data_ptr, self.outs.ptrs, stream=st)
                evs[k + 1].record(st)
            pairs = list(zip(evs[:-1], evs[1:]))
        else:
            pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                     for _ in range(steps)]
            for k in range(steps):
                self.flush.fill_(k & 0xFF)
                pairs[k][0].record(st)
                plan.materialize(self.data_ptr, self.outs.ptrs, stream=st)
                pairs[k][1].record(st)
        torch.cuda.synchronize()
        if plan.check() != 0:
            raise RuntimeError(f"{self.w.name}: materialize flagged a bad destination")
        return [a.elapsed_time(b) for a, b in pairs]

    def roofline(self, per):
        peak, peak_src = measured_peak()
        kernel_ms = statistics.mean(per)
        achieved = (self.src_bytes + self.dst_bytes) / 1e9 / (kernel_ms / 1e3)
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": profiled_traffic(self.w.name),
                "peak_source": peak_src, "kernel": "materialize_" + self.plan.stats()["kernel"],
                "kernel_ms_mean": round(kernel_ms, 4), "kernel_ms_min": round(min(per), 4),
                "kernel_ms_median": round(statistics.median(per), 4),
                "frac_of_nominal_7900": round(achieved / 7900.0, 4),
                "algorithmic_bytes_per_launch": self.src_bytes + self.dst_bytes}

    def e2e(self, dist, repeats=3, steps=None):
        """Same metric through st_load: pinned host -> device chunk copies
        overlapped with per-chunk kernels, then a device->host read of the
        status word (st_plan_check), every step."""
        args, torch, stmat = self.args, self.torch, self.stmat
        chunk = args.e2e_chunk_mb << 20
        eplan = self.ix.plan(dst=self.w.dst[0], scale_suffix=self.w.scale_suffix, chunk_bytes=chunk,
                             **self.plan_kw)
        copy = torch.cuda.Stream()
        hdata = self.host[self.data_start:self.data_start + self.data_bytes]
        ddata = self.dev[:self.data_bytes]
        for _ in range(2):
            eplan.load(hdata, ddata, self.outs.ptrs, copy_stream=copy, compute_stream=self.stream)
            eplan.check(self.stream)
        if dist:
            dist.barrier()
        # `repeats` repeats of esteps loads each; the median repeat is reported (the shared host
        # occasionally slows a whole repeat: all are listed)
        esteps = steps or max(3, min(args.steps, 10))
        reps = []
        for _ in range(repeats):
            t0 = time.perf_counter()
            for _ in range(esteps):
                eplan.load(hdata, ddata, self.outs.ptrs, copy_stream=copy, compute_stream=self.stream)
                if eplan.check(self.stream) != 0:
                    raise RuntimeError("st_load flagged a bad destination")
            reps.append((time.perf_counter() - t0) / esteps)
        es = max_over_ranks(statistics.median(reps), dist, torch)
        # the host link alone: st_stage_h2d of the data section, chunked like st_load
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        stmat.stage_h2d(ddata, hdata, self.data_bytes, chunk, stream=copy)
        copy.synchronize()
        ev0.record(copy)
        for _ in range(3):
            stmat.stage_h2d(ddata, hdata, self.data_bytes, chunk, stream=copy)
        ev1.record(copy)
        copy.synchronize()
        h2d_gbs = 3 * self.data_bytes / (ev0.elapsed_time(ev1) / 1e3) / 1e9
        copied, n_ranges = eplan.copy_bytes()   # a sparse plan copies only the ranges it reads
        return {"value": round(self.gb_dst_all / es, 3), "unit": "GB/s", "h2d_bytes_per_step": copied,
                "copy_ranges": n_ranges, "stage_h2d_gbs": round(h2d_gbs, 1),
                "d2h_bytes_per_step": 4, "ms_per_step": round(es * 1e3, 3),
                "repeats_gbs": [round(self.gb_dst_all / r, 1) for r in reps],
                "chunk_bytes": chunk, "chunks": eplan.stats()["chunks"]}

    def config(self):
        st = self.plan.stats()
        return {"workload": self.w.name, "src_bytes": self.src_bytes, "dst_bytes": self.dst_bytes,
                "tensors": len(self.infos), "src_dtypes": sorted({o["src_dtype"] for o in self.infos}),
                "dst_dtype": self.w.dst[0], "l2": self.l2_note, "shard_files": len(self.w.files),
                "workers": st["workers"], "pieces": st["pieces"], "kernel_build": st["kernel"],
                "launches_per_step": 1}

    def close(self):
        for k in ("outs", "dev", "flush", "plan", "host"):
            setattr(self, k, None)
        self.torch.cuda.synchronize()
        self.torch.cuda.empty_cache()


# rows that are another selection or output dtype of the row before them: the
# checkpoint stays resident and is planned again
SAME_CHECKPOINT = {"llm8b_f16": "llm8b"}


def measure_row(args, c, name, world, dist, steps):
    """One entry of "configs": kernel timing, roofline and the end-to-end
    rate of the workload resident in case `c`, plus the file and lazy paths
    for the UNet checkpoint."""
    torch = c.torch
    c.warm(args.warmup)
    if dist:
        dist.barrier()
    per = c.time_launches(steps)
    ms = max_over_ranks(sum(per) / steps, dist, torch)
    row = {"workload": c.w.name, "value": round(c.gb_dst_all / (ms / 1e3), 3), "unit": "GB/s",
           "ms_per_step": round(ms, 4), "steps": steps, "config": c.config(), "roofline": c.roofline(per),
           "gpu_launches": steps}
    if not args.no_e2e:
        row["e2e"] = c.e2e(dist, repeats=2, steps=max(3, min(steps, 5)))
        if args.e2e_files == "on" or (args.e2e_files == "auto" and name == "unet"):
            row["e2e_files"] = time_load_files(args, c, dist, world)
        if args.lazy == "on" or (args.lazy == "auto" and name == "unet"):
            row["lazy"] = time_lazy(args, c.w, c.host, c.data_start, c.stmat, torch)
    return row


def run_ours(args, rank, world, local):
    import torch
    from safetensors_materialization_gb300 import stmat
    stmat.lib()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    # pinned memory and reader threads on the GPU's own CPU socket
    try:
        host_cpus = stmat.host_affinity(local, apply=True)
    except stmat.StmatError as e:
        host_cpus = f"not bound: {e}"

    c = Case(args, args.workload, rank, world, dist, stmat, torch)
    c.warm(args.warmup)

    # ---- device-timed region: K launches, per-launch events on the launching stream
    clocks = ClockSampler(local)
    clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    per = c.time_launches(args.steps)
    if dist:
        dist.barrier()
    clk = clocks.stop()
    ms = max_over_ranks(sum(per) / args.steps, dist, torch)
    value = c.gb_dst_all / (ms / 1e3)

    # ---- end to end through the C ABI: pinned host -> device copies overlapped
    # with per-chunk kernels (st_load), then a device->host read of the status word
    e2e = None if args.no_e2e else c.e2e(dist)
    e2e_files = lazy = None
    if not args.no_e2e and (args.e2e_files == "on" or (args.e2e_files == "auto" and c.data_bytes < 8e9)):
        e2e_files = time_load_files(args, c, dist, world)
    if args.lazy == "on" or (args.lazy == "auto" and len(c.infos) <= 2000 and c.data_bytes < 8e9
                             and not args.no_e2e):
        lazy = time_lazy(args, c.w, c.host, c.data_start, stmat, torch)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        data = c.host.numpy()[c.data_start:c.data_start + c.w.files[0].data_bytes]   # the first shard's
        v, desc, nbytes, dt, k, sizes = oracle_sample(c.w, args.cpu_seconds, data)
        cpu = {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc,
               "seconds": round(dt, 2), "host_cores": os.cpu_count(), "host_cpu": host_cpu_model()}
        # the same oracle code over the same outputs on every host core (a second, labelled row)
        cores = len(os.sched_getaffinity(0))
        if cores > 1:
            sel, _ = oracle_selection(c.w)
            op = OracleThreads(sel, data, cores)
            try:
                nb, dta = op.run(k)
            finally:
                op.close()
            where = c.w.name if len(c.w.files) == 1 else f"shard 0 of {c.w.name}"
            cpu["all_cores"] = {"value": round(nb / dta / 1e9, 4), "unit": "GB/s", "cores": cores,
                                "kind": "oracle",
                                "sample": f"the same first {k} outputs ({nb / 1e6:.1f} MB dst) of {where}, "
                                          f"{cores} threads"}
        del data
    headline_cfg = c.config()
    roof = c.roofline(per)
    c.close()
    del c

    # ---- the other configurations, each timed in this process (one GPU only)
    rows = None
    if args.configs == "all" or (args.configs == "auto" and args.workload == HEADLINE and world == 1):
        rows, case = [], None
        cclk = ClockSampler(local)
        cclk.start()
        try:
            for name in CONFIG_ROWS:
                if name == args.workload:
                    continue
                if case is not None and SAME_CHECKPOINT.get(name) == case_name:
                    case.replan(build_workload(name))
                else:
                    if case is not None:
                        case.close()
                    case, case_name = Case(args, name, rank, world, dist, stmat, torch), name
                rows.append(measure_row(args, case, name, world, dist, args.steps))
        finally:
            if case is not None:
                case.close()
        configs_clocks = cclk.stop()
    if rank == 0:
        headline_cfg.update({"parallelism": f"{args.split} x{world}", "host_cpus": host_cpus})
        line = {
            "metric": "materialized GB/s (dst bytes)", "value": round(value, 3), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak" if args.split == "replica" else "strong",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": headline_cfg,
            "roofline": roof,
            "gpu_launches": args.steps,
            "clocks": clk,
            "e2e": e2e,
            "e2e_files": e2e_files,
            "lazy": lazy,
            "cpu_baseline": cpu,
        }
        if rows is not None:
            line["configs"] = rows
            line["configs_clocks"] = configs_clocks
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    argv = sys.argv[1:]
    args = parse_args(argv)
    rank, world, local = dist_env()
    cmd = launch_command(args, world, argv)
    if cmd is not None:
        sys.exit(subprocess.call(cmd))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
