"""Decode-step benchmark of the paged KV-cache library on GB300.

One step = the whole hot path for one decode-attention layer: the paged
cache write of one new token per sequence (reshape_and_cache), then paged
decode attention over every sequence grown by that token.  The default
workload is the Llama-3-70B-shaped layer (128 sequences, 64 query / 8 KV
heads, head_dim 128, 16-token blocks, bf16 KV, lognormal lengths with median
2048).  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config NAME] [--kernel auto|simt|mma] [--partition P]
                    [--unfused] [--eager]

The timed steps replay the step captured once as a CUDA graph (``--eager``
launches each step from Python instead); ``--unfused`` runs the cache write
and the decode as two launches.

``--impl reference`` times the fp64 CPU oracle on this host's cores on a
bounded sample of the same workload (the reference arm of this repository).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from paged_kv_cache_225_gb300 import workloads as W  # noqa: E402
from paged_kv_cache_225_gb300.metrics import algorithmic_bytes, prefill_algorithmic  # noqa: E402

METRIC = "decode-attn KV GB/s & tokens/s on 1 GB300, % of HBM peak (70B-shape layer)"
FALLBACK_HBM_GBS = 6800.0
DTYPE_NAME = {W.F32: "f32", W.BF16: "bf16", W.FP8_E5M2: "fp8_e5m2", W.FP8_E4M3: "fp8_e4m3",
              W.INT4: "int4"}
CONFIG_TEXT = {
    "tiny_fp32": "tiny fp32 decode: 4 seqs, 4 q/4 kv heads, D=64, lengths U[1,64]",
    "llama3_8b": "Llama-3-8B-shaped decode layer: 64 seqs, 32 q/8 kv heads, D=128, bf16 KV, "
                 "lengths U[512,4096]",
    "llama3_70b": "Llama-3-70B-shaped decode layer: 128 seqs, 64 q/8 kv heads, D=128, bf16 KV, "
                  "lognormal lengths (median 2048, sigma 0.8)",
    "long_split": "long-context split-KV: 8 seqs x 32768 tokens, 64 q/8 kv heads, D=128, bf16 KV",
    "fp8_chat": "fp8-e5m2 KV chat mix: 128 seqs, 64 q/8 kv heads, D=128, lengths U[256,512], "
                "8-block shared prefixes",
    "e4m3_70b": "Llama-3-70B-shaped decode layer with an fp8-e4m3 KV cache (per-tensor scale "
                "1/8): 128 seqs, 64 q/8 kv heads, D=128, lognormal lengths (median 2048)",
    "int4_70b": "Llama-3-70B-shaped decode layer with an INT4 KV cache (scale 1/2, two tokens "
                "per byte): 128 seqs, 64 q/8 kv heads, D=128, lognormal lengths (median 2048)",
    "prefill_tiny": "several causal queries per sequence, tiny mix: 7 seqs, 8 q/2 kv heads, "
                    "D=64, bf16 KV",
    "spec_verify_70b": "speculative verification on the Llama-3-70B-shaped layer: 128 seqs x 5 "
                       "causal queries, 64 q/8 kv heads, D=128, bf16 KV, lognormal lengths "
                       "(median 2048, sigma 0.8)",
    "cow_copy_70b": "copy-on-write page copies on the Llama-3-70B-shaped pool: 2048 (src, dst) "
                    "block pairs, 8 kv heads x 128 x 16 bf16 per block and cache; plus the host "
                    "block manager's append of 128 forked sequences",
    "chunked_prefill_8b": "chunked prefill on the Llama-3-8B-shaped layer: 4 seqs with a "
                          "256-token prompt chunk (context U[1024,4096]) + 60 decoding seqs "
                          "(U[512,4096]), 32 q/8 kv heads, D=128, bf16 KV",
    "spec_verify_70b_fp8": "speculative verification on the Llama-3-70B-shaped layer with an "
                           "fp8-e5m2 KV cache (scale 1): 128 seqs x 5 causal queries, 64 q/8 kv "
                           "heads, D=128, lognormal lengths (median 2048, sigma 0.8)",
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="llama3_70b",
                    choices=W.CONFIG_ORDER + list(W.PREFILL_CONFIGS) + ["cow_copy_70b"])
    ap.add_argument("--kernel", default="auto", choices=["auto", "simt", "mma"])
    ap.add_argument("--partition", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--unfused", action="store_true",
                    help="cache write and decode as two launches instead of one")
    ap.add_argument("--eager", action="store_true",
                    help="launch every step from Python instead of replaying a CUDA graph")
    ap.add_argument("--layers", type=int, default=1,
                    help="decode this many layers of the workload (shared tables and lengths, "
                         "own caches) in one launch, against as many separate launches")
    return ap.parse_args(argv)


# Sources that do not define or launch the decode kernels.
_NOT_DECODE = {"pkv_cache.cu", "pkv_noalloc.cu", "pkv_prefill.cu", "pkv_prefill_tc.cu",
               "pkv_prefill.cuh"}


def source_hash() -> str:
    """Hash of the decode-kernel sources; ties a stored ncu traffic figure to them."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_225_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")) and f not in _NOT_DECODE:
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def stored_traffic(config: str, kernel: str):
    """Per-launch DRAM bytes from a committed ncu summary, if it matches the sources."""
    path = os.path.join(ROOT, "profiles", f"decode_{config}_{kernel}_traffic.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("source_hash") != source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def workload_text(name: str) -> str:
    return CONFIG_TEXT[name]


def max_over_ranks(x: float) -> float:
    """Max of a host float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    dev = torch.device("cuda", torch.cuda.current_device()) \
        if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, elapsed_s: float) -> float:
    """Units all ranks processed per second of the slowest rank (weak scaling)."""
    return units_per_rank * world / elapsed_s


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running.

    Started before the warm-up; each sample carries nvidia-smi's own
    timestamp, so the summary covers exactly the window asked for (the
    soak before the timed steps through their end) even if the tool's output
    reaches us late."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int, enabled: bool = True, interval_ms: int = 100):
        import threading
        self.proc = None
        self.gpu = gpu_index
        self.rows = []
        self.lock = threading.Lock()
        self.thread = None
        if enabled:
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                     "--format=csv,noheader,nounits", "-lms", str(interval_ms)],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
            except OSError:
                self.proc = None
        if self.proc is not None:
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()

    @staticmethod
    def now() -> float:
        return time.time()

    def _read(self):
        import datetime
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != 8:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                row = (ts, float(parts[1]), float(parts[2]), parts[4:])
            except ValueError:
                continue
            with self.lock:
                self.rows.append(row)

    def count_since(self, t0: float) -> int:
        with self.lock:
            return sum(1 for r in self.rows if r[0] >= t0)

    def stop(self, since: float = 0.0, until: float = float("inf")):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        import signal
        self.proc.send_signal(signal.SIGINT)
        try:
            self.proc.wait(timeout=3)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self.thread.join(timeout=3)
        with self.lock:
            rows = [r for r in self.rows if since <= r[0] <= until]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({self.REASONS[i] for r in rows for i, v in enumerate(r[3])
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": rows[0][2],
                "reasons": reasons, "samples": len(rows),
                "window_s": round(min(until, self.now()) - since, 3)}


def soak(run, sampler: ClockSampler, min_s: float = 1.0, min_samples: int = 5,
         max_s: float = 6.0) -> float:
    """Replays `run` (one step, no sync) for at least min_s seconds and until the
    sampler holds min_samples clock samples (at most max_s seconds), so that
    the clocks are read under the same load the timed steps see.  Returns the
    soak's start time; the clock window runs from there to the timed end."""
    import torch
    t0 = ClockSampler.now()
    while True:
        for _ in range(16):
            run()
        torch.cuda.synchronize()
        el = ClockSampler.now() - t0
        if el >= max_s or (el >= min_s and (sampler.proc is None or
                                             sampler.count_since(t0) >= min_samples)):
            return t0


# --------------------------------------------------------------- GPU arm

def run_ours(args):
    import torch
    import torch.distributed as dist

    import paged_kv_cache_225_gb300 as pkv

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    w = W.make_workload(args.config)
    cfg = w.cfg
    S, Hq, Hkv, D = cfg.num_seqs, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim
    lens = (w.seq_lens + 1).astype(np.int32)           # each step appends one token
    max_len = int(lens.max())
    ab = algorithmic_bytes(w, lens)
    # The fused launch also reads the new K/V rows and writes them to the cache.
    new_rows = cfg.num_seqs * cfg.num_kv_heads * cfg.head_dim * 2
    append_bytes = 0 if args.unfused else \
        new_rows * (W.ELEM_BYTES[cfg.q_dtype] + W.ELEM_BYTES[cfg.kv_dtype])

    def t(a, dt):
        a = np.ascontiguousarray(a)
        if dt == W.F32:
            return torch.from_numpy(a)
        if dt == W.BF16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
        if dt == W.FP8_E4M3:
            return torch.from_numpy(a).view(torch.float8_e4m3fn)
        if dt == W.INT4:
            return torch.from_numpy(a)                  # packed nibbles as uint8
        return torch.from_numpy(a).view(torch.float8_e5m2)

    host = {
        "q": t(w.q, cfg.q_dtype), "new_k": t(w.new_k, cfg.q_dtype),
        "new_v": t(w.new_v, cfg.q_dtype),
        "tables": torch.from_numpy(w.block_tables), "lens": torch.from_numpy(lens),
    }
    if args.unfused:
        host["slots"] = torch.from_numpy(w.slot_mapping)
    kc = t(w.k_cache, cfg.kv_dtype).to(dev)
    vc = t(w.v_cache, cfg.kv_dtype).to(dev)
    d = {k: v.to(dev) for k, v in host.items()}
    out = torch.empty((S, Hq, D), dtype=torch.float32, device=dev)
    part = pkv.partition_tokens(S, Hq, Hkv, D, max_len, args.partition)
    ws = torch.empty(pkv.workspace_size(S, Hq, Hkv, D, max_len, args.partition),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    ks = vs = cfg.kv_scale

    def step(dd, ev=None, o=None):
        o = out if o is None else o
        if args.unfused:
            pkv.reshape_and_cache(dd["new_k"], dd["new_v"], dd["slots"], kc, vc, k_scale=ks,
                                  v_scale=vs)
        if ev is not None:
            ev[0].record(stream)
        if args.unfused:
            pkv.paged_attn_decode(dd["q"], kc, vc, dd["tables"], dd["lens"], w.scale, o,
                                  k_scale=ks, v_scale=vs, max_seq_len=max_len,
                                  partition_tokens=args.partition, impl=args.kernel,
                                  workspace=ws)
        else:
            pkv.paged_attn_decode_append(dd["q"], dd["new_k"], dd["new_v"], kc, vc,
                                         dd["tables"], dd["lens"], w.scale, o, k_scale=ks,
                                         v_scale=vs, max_seq_len=max_len,
                                         partition_tokens=args.partition, impl=args.kernel,
                                         workspace=ws)
        if ev is not None:
            ev[1].record(stream)

    sampler = ClockSampler(local, enabled=not args.no_clocks)
    for _ in range(max(args.warmup, 3)):
        step(d)
    torch.cuda.synchronize()
    status = pkv.read_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {pkv.STATUS.get(status, status)} during warm-up")

    K = args.steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if args.eager:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
    else:
        # The step (workspace memset + kernel launches) captured once as a
        # CUDA graph and replayed K times: no CPU launch gaps on small layers.
        graph_stream = torch.cuda.Stream(dev)
        graph_stream.wait_stream(stream)
        g_step = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step, stream=graph_stream):
            step(d)
        g_call = None
        if args.unfused:  # the decode call alone, for the roofline timing
            g_call = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_call, stream=graph_stream):
                pkv.paged_attn_decode(d["q"], kc, vc, d["tables"], d["lens"], w.scale, out,
                                      k_scale=ks, v_scale=vs, max_seq_len=max_len,
                                      partition_tokens=args.partition, impl=args.kernel,
                                      workspace=ws)
        stream.wait_stream(graph_stream)
        for _ in range(3):
            g_step.replay()
        torch.cuda.synchronize()
    clock_t0 = soak((lambda: step(d)) if args.eager else g_step.replay, sampler)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(K):
        if args.eager:
            step(d, evs[i])
        else:
            g_step.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop(since=clock_t0)
    elapsed_ms = t0.elapsed_time(t1)
    if args.eager:
        decode_ms = [a.elapsed_time(b) for a, b in evs]
    elif g_call is None:
        decode_ms = [elapsed_ms / K]  # the step is the one decode launch
    else:
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(K):
            g_call.replay()
        c1.record(stream)
        torch.cuda.synchronize()
        decode_ms = [c0.elapsed_time(c1) / K]
    elapsed_ms = max_over_ranks(elapsed_ms)
    status = pkv.read_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {pkv.STATUS.get(status, status)} in the timed run")

    # End to end through the public API with host buffers: every step copies
    # its pinned inputs in and its output back inside the timed region.  The
    # copies run on a second stream with double-buffered device inputs and
    # outputs, so step i+1's inputs and step i's output move while step i /
    # i+1 compute (the usual serving pipeline); each step's kernel waits for
    # its own inputs, and each input buffer is refilled only after the step
    # that read it has finished.
    e2e = None
    if not args.no_e2e:
        pinned = {k: v.pin_memory() for k, v in host.items()}
        h2d = sum(v.numel() * v.element_size() for v in pinned.values())
        d2h = out.numel() * out.element_size()
        bufs = [d, {k: torch.empty_like(v) for k, v in d.items()}]
        outs = [out, torch.empty_like(out)]
        outs_host = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        copy_stream = torch.cuda.Stream(dev)
        Ke = max(1, min(K, 500))

        def pipelined(n):
            ready = [torch.cuda.Event() for _ in range(2)]
            done = [None, None]
            out_free = [None, None]   # the output buffer's copy to the host has finished
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(copy_stream)

            def h2d_step(i):
                b = i % 2
                if done[b] is not None:
                    copy_stream.wait_event(done[b])
                with torch.cuda.stream(copy_stream):
                    for k, v in pinned.items():
                        bufs[b][k].copy_(v, non_blocking=True)
                ready[b].record(copy_stream)

            h2d_step(0)
            for i in range(n):
                b = i % 2
                stream.wait_event(ready[b])
                if out_free[b] is not None:
                    stream.wait_event(out_free[b])
                step(bufs[b], o=outs[b])
                done[b] = torch.cuda.Event()
                done[b].record(stream)
                if i + 1 < n:
                    h2d_step(i + 1)
                copy_stream.wait_event(done[b])
                with torch.cuda.stream(copy_stream):
                    outs_host[b].copy_(outs[b], non_blocking=True)
                out_free[b] = torch.cuda.Event()
                out_free[b].record(copy_stream)
            e1.record(copy_stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / n

        pipelined(3)
        e_ms = pipelined(Ke)
        # Every step computes the same output: the two host copies agree
        # bit for bit unless the pipeline raced.
        if not torch.equal(outs_host[0], outs_host[1]):
            raise RuntimeError("pipelined end-to-end steps disagree")
        e2e = {"value": ab["kv"] * world / (e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e_ms, "steps": Ke,
               "pipeline": "copies on a second stream, double-buffered inputs and outputs"}

    ms_step = elapsed_ms / K
    kv_gbs = whole_job_rate(ab["kv"], world, ms_step * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    dec_ms = statistics.mean(decode_ms)
    launch_bytes = ab["total"] + append_bytes
    achieved = launch_bytes / (dec_ms * 1e-3) / 1e9
    kernel_impl = args.kernel
    if kernel_impl == "auto":
        kernel_impl = "mma" if (cfg.kv_dtype != W.F32 and cfg.q_dtype == W.BF16) else "simt"
    traffic = stored_traffic(args.config, kernel_impl)
    # One fused launch (or cache write + decode when --unfused).
    launches_per_step = 2 if args.unfused else 1
    line = {
        "metric": METRIC, "value": kv_gbs, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_NAME[cfg.kv_dtype],
        "data": "synthetic: seeded N(0,1) q/K/V, shuffled physical blocks (no dataset)",
        "config": {"workload": workload_text(args.config), "name": args.config,
                   "num_seqs": S, "num_q_heads": Hq, "num_kv_heads": Hkv, "head_dim": D,
                   "block_size": cfg.block_size, "tokens_per_step": ab["tokens"],
                   "kv_bytes_per_step": ab["kv"],
                   "schedule": ("stream-K (equal page ranges per CTA)"
                                if part == pkv.SCHEDULE_STREAMK else
                                f"{part}-token partitions" if part > 0 else
                                "one CTA per (sequence, KV head)"),
                   "kernel": kernel_impl,
                   "l2": f"no flush: KV read per step ({ab['kv'] / 1e9:.2f} GB) exceeds L2 "
                         "(129 MB)" if ab["kv"] > 256e6 else
                         "no flush: KV per step smaller than 2x L2 (reported, not corrected)",
                   "step": ("reshape_and_cache of 1 token/seq, then paged decode over L+1"
                            if args.unfused else
                            "one launch: cache write of 1 token/seq fused into paged decode "
                            "over L+1"),
                   "launch": "eager from Python" if args.eager else
                             "step captured once as a CUDA graph, replayed per step"},
        "tokens_per_s": whole_job_rate(S, world, ms_step * 1e-3),
        "pct_hbm_peak": 100.0 * ab["total"] / (ms_step * 1e-3) / 1e9 / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": (f"paged_attn_decode{'' if args.unfused else '_append'} call "
                                f"({kernel_impl}; mean of {K} launches, CUDA events on the "
                                "launch stream" + (")" if args.eager else
                                                   ", CUDA-graph replays)")),
                     "algorithmic_bytes_per_launch": launch_bytes,
                     "peak_source": f"{peak_kind} hbm_gbs"},
        "gpu_launches": K * launches_per_step,
        "clocks": clocks,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, lens, budget_s=10.0)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------- CPU arm

def _oracle_step(w, lens, seqs, threads):
    """The oracle's decode step restricted to sequences ``seqs``: cache write + attention."""
    import oracle
    cfg = w.cfg
    idx = np.asarray(seqs)
    kc, vc = w.k_cache, w.v_cache
    sub_new_k = np.ascontiguousarray(w.new_k[idx])
    sub_new_v = np.ascontiguousarray(w.new_v[idx])
    sub_slots = np.ascontiguousarray(w.slot_mapping[idx])
    # Writing into the workload's own host caches is idempotent across steps
    # (the same token lands in the same slot every time).
    oracle.reshape_and_cache(sub_new_k, sub_new_v, cfg.q_dtype, sub_slots, kc, vc, cfg.kv_dtype,
                             cfg.kv_scale, cfg.kv_scale)
    return oracle.paged_decode_seqs(w.q, cfg.q_dtype, kc, vc, cfg.kv_dtype, w.block_tables, lens,
                                    w.scale, seqs=idx, k_scale=cfg.kv_scale, v_scale=cfg.kv_scale,
                                    num_threads=threads)


def _timed_oracle(run, budget_s):
    """Calls run() (returns the KV bytes it attended) until budget_s seconds of
    oracle time have passed (bounded at 3x in wall time); (bytes, seconds, calls)."""
    kv, t_total, calls = 0, 0.0, 0
    t_start = time.perf_counter()
    while t_total < budget_s and time.perf_counter() - t_start < 3 * budget_s:
        t0 = time.perf_counter()
        kv += run(calls)
        t_total += time.perf_counter() - t0
        calls += 1
    return kv, t_total, calls


def cpu_baseline(w, lens, budget_s=10.0):
    """The oracle on this host's cores, on bounded samples of the workload.

    All cores: whole decode steps (the cache write and attention of every
    sequence of the batch in one oracle call, OpenMP over its (sequence, KV
    head) units).  One thread: chunks of 16 sequences in a seeded random
    order.  Each leg runs for about budget_s seconds."""
    import oracle
    threads = oracle.max_threads()
    cfg = w.cfg
    S = cfg.num_seqs
    row = cfg.num_kv_heads * 2 * cfg.head_dim * W.ELEM_BYTES[cfg.kv_dtype]
    every = list(range(S))
    step_kv = int(lens.sum()) * row

    def whole(_):
        _oracle_step(w, lens, every, threads)
        return step_kv

    kv_all, t_all, n_all = _timed_oracle(whole, budget_s)
    order = np.random.default_rng(1234).permutation(S)
    chunk = min(16, S)

    def one_thread(i):
        seqs = [int(order[(i * chunk + j) % S]) for j in range(chunk)]
        _oracle_step(w, lens, seqs, 1)
        return sum(int(lens[x]) for x in seqs) * row

    kv_one, t_one, n_one = _timed_oracle(one_thread, budget_s)
    return {"value": kv_all / t_all / 1e9, "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{n_all} whole decode steps ({S} sequences each, cache write + "
                      f"attention, {kv_all / 1e9:.2f} GB of KV) in {t_all:.1f} s, fp64 C "
                      f"oracle with OpenMP over (sequence, KV head) on {threads} threads",
            "tokens_per_s": n_all * S / t_all,
            "single_thread": {"value": kv_one / t_one / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": f"{n_one} chunks of {chunk} sequences (random order, "
                                        f"{kv_one / 1e9:.2f} GB of KV) in {t_one:.1f} s on "
                                        "one thread"}}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    w = W.make_workload(args.config)
    cfg = w.cfg
    lens = (w.seq_lens + 1).astype(np.int32)
    threads = oracle.max_threads()
    row = cfg.num_kv_heads * 2 * cfg.head_dim * W.ELEM_BYTES[cfg.kv_dtype]
    # Size each step's sample so the whole run stays near two minutes.
    order = np.random.default_rng(99).permutation(cfg.num_seqs)
    probe = [int(x) for x in order[:min(16, cfg.num_seqs)]]
    t0 = time.perf_counter()
    _oracle_step(w, lens, probe, threads)
    per_seq = max((time.perf_counter() - t0) / len(probe), 1e-5)
    total_steps = args.steps + max(args.warmup, 0)
    per_step_budget = 120.0 / max(total_steps, 1)
    n_seq = int(max(1, min(cfg.num_seqs, per_step_budget / per_seq)))
    cursor = 0

    def one_step():
        nonlocal cursor
        seqs = [int(order[(cursor + i) % cfg.num_seqs]) for i in range(n_seq)]
        cursor += n_seq
        _oracle_step(w, lens, seqs, threads)
        return sum(int(lens[s]) for s in seqs)

    for _ in range(args.warmup):
        one_step()
    tok = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        tok += one_step()
    el = time.perf_counter() - t0
    kv = tok * row
    value = kv / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic: seeded N(0,1) q/K/V, shuffled physical blocks",
        "config": {"workload": workload_text(args.config), "name": args.config,
                   "sample_seqs_per_step": n_seq},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{n_seq} of {cfg.num_seqs} sequences per step "
                                   "(cache write + attention), fp64 C oracle"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------- several queries per sequence

def _query_rows(w):
    """Slots of every query token and the K/V rows the pool holds there, as
    bf16 bits: the stored values (codes times the dequant scale for fp8 /
    INT4 caches, exact in bf16), so writing them back stores the same codes."""
    base = w.cfg.base
    B = base.block_size
    kf = W.storage_to_float32(w.k_cache, base.kv_dtype)
    vf = W.storage_to_float32(w.v_cache, base.kv_dtype)
    if base.kv_dtype in W.SCALED:
        kf = kf * np.float32(base.kv_scale)
        vf = vf * np.float32(base.kv_scale)
    slots, ks, vs = [], [], []
    for s in range(w.seq_lens.size):
        L = int(w.seq_lens[s])
        n = int(w.q_start[s + 1] - w.q_start[s])
        for pos in range(L - n, L):
            blk = int(w.block_tables[s, pos // B])
            slots.append(blk * B + pos % B)
            ks.append(kf[blk, :, :, pos % B])
            vs.append(vf[blk, :, :, pos % B])
    return (np.asarray(slots, dtype=np.int64),
            W.round_to_storage(np.ascontiguousarray(np.stack(ks)), W.BF16),
            W.round_to_storage(np.ascontiguousarray(np.stack(vs)), W.BF16))


def run_prefill(args):
    """One step = the cache write of every query token's K/V, then causal paged
    attention of all queries (chunked prefill / speculative verification)."""
    import torch
    import torch.distributed as dist

    import paged_kv_cache_225_gb300 as pkv

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    w = W.make_prefill_workload(args.config)
    base = w.cfg.base
    S, Hq, Hkv, D = base.num_seqs, base.num_q_heads, base.num_kv_heads, base.head_dim
    T, max_q, max_len = w.num_tokens, w.max_q_len, int(w.seq_lens.max())
    ab = prefill_algorithmic(w)
    slots, new_k, new_v = _query_rows(w)
    write_bytes = T * Hkv * D * 2 * (2 + W.ELEM_BYTES[base.kv_dtype])
    ks = vs = base.kv_scale

    def t(a, dt):
        a = np.ascontiguousarray(a)
        if dt == W.BF16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
        if dt == W.FP8_E5M2:
            return torch.from_numpy(a).view(torch.float8_e5m2)
        if dt == W.FP8_E4M3:
            return torch.from_numpy(a).view(torch.float8_e4m3fn)
        return torch.from_numpy(a)

    host = {"q": t(w.q, base.q_dtype), "q_start": torch.from_numpy(w.q_start),
            "tables": torch.from_numpy(w.block_tables), "lens": torch.from_numpy(w.seq_lens),
            "new_k": t(new_k, W.BF16), "new_v": t(new_v, W.BF16),
            "slots": torch.from_numpy(slots)}
    kc = t(w.k_cache, base.kv_dtype).to(dev)
    vc = t(w.v_cache, base.kv_dtype).to(dev)
    d = {k: v.to(dev) for k, v in host.items()}
    out = torch.empty((T, Hq, D), dtype=torch.float32, device=dev)
    part = pkv.prefill_partition_tokens(S, T, Hq, Hkv, D, max_q, max_len, args.partition)
    ws = torch.empty(pkv.prefill_workspace_size(S, T, Hq, Hkv, D, max_q, max_len,
                                                args.partition), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def attend(dd):
        pkv.paged_attn_prefill(dd["q"], dd["q_start"], kc, vc, dd["tables"], dd["lens"],
                               w.scale, out, max_q_len=max_q, max_seq_len=max_len,
                               partition_tokens=args.partition, workspace=ws,
                               k_scale=ks, v_scale=vs)

    def step(dd):
        pkv.reshape_and_cache(dd["new_k"], dd["new_v"], dd["slots"], kc, vc, k_scale=ks,
                              v_scale=vs)
        attend(dd)

    sampler = ClockSampler(local, enabled=not args.no_clocks)
    for _ in range(max(args.warmup, 3)):
        step(d)
    torch.cuda.synchronize()
    status = pkv.read_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {pkv.STATUS.get(status, status)} during warm-up")
    K = args.steps
    graph_stream = torch.cuda.Stream(dev)
    graph_stream.wait_stream(stream)
    g_step, g_call = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=graph_stream):
        step(d)
    with torch.cuda.graph(g_call, stream=graph_stream):
        attend(d)
    stream.wait_stream(graph_stream)
    for _ in range(3):
        g_step.replay()
    torch.cuda.synchronize()
    clock_t0 = soak(g_step.replay, sampler)
    if world > 1:
        dist.barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(K):
        g_step.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop(since=clock_t0)
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1))
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for _ in range(K):
        g_call.replay()
    c1.record(stream)
    torch.cuda.synchronize()
    call_ms = c0.elapsed_time(c1) / K
    status = pkv.read_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {pkv.STATUS.get(status, status)} in the timed run")

    e2e = None
    if not args.no_e2e:
        pinned = {k: v.pin_memory() for k, v in host.items()}
        out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in pinned.values())
        d2h = out_host.numel() * out_host.element_size()
        Ke = max(1, min(K, 200))
        for _ in range(3):
            for k, v in pinned.items():
                d[k].copy_(v, non_blocking=True)
            step(d)
            out_host.copy_(out, non_blocking=True)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(Ke):
            for k, v in pinned.items():
                d[k].copy_(v, non_blocking=True)
            step(d)
            out_host.copy_(out, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = e0.elapsed_time(e1) / Ke
        e2e = {"value": ab["kv"] * world / (e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e_ms, "steps": Ke}

    ms_step = elapsed_ms / K
    peak, peak_kind = hbm_peak()
    achieved = ab["total"] / (call_ms * 1e-3) / 1e9
    tflops = ab["flops"] / (call_ms * 1e-3) / 1e12
    bf16_peak = None
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            bf16_peak = float(json.load(f)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        bf16_peak = 1900.0
    launches = 2 + (1 if part > 0 and max_len > part else 0)
    line = {
        "metric": METRIC, "value": whole_job_rate(ab["kv"], world, ms_step * 1e-3) / 1e9,
        "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE_NAME[base.kv_dtype],
        "data": "synthetic: seeded N(0,1) q/K/V, shuffled physical blocks (no dataset)",
        "config": {"workload": workload_text(args.config), "name": args.config,
                   "num_seqs": S, "num_queries": T, "num_q_heads": Hq, "num_kv_heads": Hkv,
                   "head_dim": D, "block_size": base.block_size, "tokens": ab["tokens"],
                   "kv_bytes_per_step": ab["kv"], "flops_per_step": ab["flops"],
                   "partition": part,
                   "l2": "no flush: KV read per step exceeds L2 (129 MB)",
                   "step": "reshape_and_cache of every query token, then causal paged "
                           "attention of all queries",
                   "launch": "step captured once as a CUDA graph, replayed per step"},
        "queries_per_s": whole_job_rate(T, world, ms_step * 1e-3),
        "pct_hbm_peak": 100.0 * ab["total"] / (ms_step * 1e-3) / 1e9 / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": f"paged_attn_prefill call (mean of {K} CUDA-graph replays, "
                               "CUDA events on the launch stream)",
                     "algorithmic_bytes_per_launch": ab["total"],
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "tensor": {"achieved_tflops": tflops, "bf16_peak_tflops": bf16_peak,
                                "frac": tflops / bf16_peak,
                                "note": ("tcgen05.mma kind::f16 (M = 128 rows, padded); "
                                         "P.V issued twice (bf16 high part + residual)"
                                         if base.kv_dtype == W.BF16 else
                                         "mma.sync m16n8k16 f16 (cache codes widened in "
                                         "registers), 16-row warp tiles")}},
        "gpu_launches": K * launches,
        "clocks": clocks,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = prefill_cpu_baseline(w, budget_s=10.0)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def _oracle_prefill_seqs(w, seqs, threads):
    """The oracle's several-queries attention for the listed sequences only."""
    import oracle
    base = w.cfg.base
    idx = list(seqs)
    lens = w.seq_lens[idx]
    qs = [w.q[w.q_start[s]:w.q_start[s + 1]] for s in idx]
    q_start = np.zeros(len(idx) + 1, dtype=np.int32)
    q_start[1:] = np.cumsum([x.shape[0] for x in qs])
    return oracle.paged_prefill(np.ascontiguousarray(np.concatenate(qs)), base.q_dtype,
                                q_start, w.k_cache, w.v_cache, base.kv_dtype,
                                np.ascontiguousarray(w.block_tables[idx]), lens, w.scale,
                                k_scale=base.kv_scale, v_scale=base.kv_scale,
                                num_threads=threads)


def prefill_cpu_baseline(w, budget_s=10.0):
    """The oracle's several-queries attention on this host: whole steps (every
    sequence in one call) on all cores, and chunks of 16 sequences on one
    thread, about budget_s seconds each."""
    import oracle
    threads = oracle.max_threads()
    base = w.cfg.base
    S = w.seq_lens.size
    row = base.num_kv_heads * 2 * base.head_dim * W.ELEM_BYTES[base.kv_dtype]
    every = list(range(S))
    step_kv = int(w.seq_lens.sum()) * row

    def whole(_):
        _oracle_prefill_seqs(w, every, threads)
        return step_kv

    kv_all, t_all, n_all = _timed_oracle(whole, budget_s)
    order = np.random.default_rng(1234).permutation(S)
    chunk = min(16, S)

    def one_thread(i):
        seqs = [int(order[(i * chunk + j) % S]) for j in range(chunk)]
        _oracle_prefill_seqs(w, seqs, 1)
        return sum(int(w.seq_lens[x]) for x in seqs) * row

    kv_one, t_one, n_one = _timed_oracle(one_thread, budget_s)
    return {"value": kv_all / t_all / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{n_all} whole steps ({S} sequences each, {kv_all / 1e9:.2f} GB of KV) "
                      f"in {t_all:.1f} s, fp64 C oracle with OpenMP over (sequence, KV head) "
                      f"on {threads} threads",
            "single_thread": {"value": kv_one / t_one / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": f"{n_one} chunks of {chunk} sequences "
                                        f"({kv_one / 1e9:.2f} GB of KV) in {t_one:.1f} s on "
                                        "one thread"}}


def run_reference_prefill(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    w = W.make_prefill_workload(args.config)
    base = w.cfg.base
    threads = oracle.max_threads()
    row = base.num_kv_heads * 2 * base.head_dim * W.ELEM_BYTES[base.kv_dtype]
    S = w.seq_lens.size
    order = np.random.default_rng(99).permutation(S)
    probe = [int(x) for x in order[:min(16, S)]]
    t0 = time.perf_counter()
    _oracle_prefill_seqs(w, probe, threads)
    per_seq = max((time.perf_counter() - t0) / len(probe), 1e-5)
    total_steps = args.steps + max(args.warmup, 0)
    n_seq = int(max(1, min(S, (120.0 / max(total_steps, 1)) / per_seq)))
    cursor = 0

    def one_step():
        nonlocal cursor
        seqs = [int(order[(cursor + i) % S]) for i in range(n_seq)]
        cursor += n_seq
        _oracle_prefill_seqs(w, seqs, threads)
        return sum(int(w.seq_lens[s]) for s in seqs)

    for _ in range(args.warmup):
        one_step()
    tok = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        tok += one_step()
    el = time.perf_counter() - t0
    value = tok * row / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded N(0,1) q/K/V, shuffled physical blocks",
        "config": {"workload": workload_text(args.config), "name": args.config,
                   "sample_seqs_per_step": n_seq},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{n_seq} of {S} sequences per step, fp64 C oracle"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------- copy-on-write copies

def run_copy(args):
    """One step = pkv_copy_blocks of 2048 disjoint page pairs on the 70B-shaped
    pool (both caches); the host block manager's per-step append is timed
    alongside (128 sequences forked from one prompt)."""
    import torch
    import torch.distributed as dist

    import paged_kv_cache_225_gb300 as pkv

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    N, Hkv, D, npairs = 8192, 8, 128, 2048
    block_bytes = Hkv * D * 16 * 2
    rng = np.random.default_rng(2024)
    ids = rng.permutation(N)[:2 * npairs].astype(np.int32)
    pairs_h = torch.from_numpy(ids.reshape(npairs, 2).copy())
    kc = torch.randn((N, Hkv, D, 16), device=dev).to(torch.bfloat16)
    vc = torch.randn((N, Hkv, D, 16), device=dev).to(torch.bfloat16)
    pairs = pairs_h.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(local, enabled=not args.no_clocks)
    for _ in range(max(args.warmup, 3)):
        pkv.copy_blocks(kc, vc, pairs, status=status)
    torch.cuda.synchronize()
    K = args.steps
    gs = torch.cuda.Stream(dev)
    gs.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=gs):
        pkv.copy_blocks(kc, vc, pairs, status=status)
    stream.wait_stream(gs)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    clock_t0 = soak(g.replay, sampler)
    if world > 1:
        dist.barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(K):
        g.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop(since=clock_t0)
    ms = max_over_ranks(t0.elapsed_time(t1)) / K
    if int(status.item()) != 0:
        raise RuntimeError("copy_blocks reported a bad pair")
    moved = npairs * 2 * block_bytes * 2          # read + write, K and V
    peak, peak_kind = hbm_peak()
    achieved = moved / (ms * 1e-3) / 1e9

    e2e = None
    if not args.no_e2e:
        pinned = pairs_h.pin_memory()
        Ke = max(1, min(K, 500))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(Ke):
            pairs.copy_(pinned, non_blocking=True)
            pkv.copy_blocks(kc, vc, pairs, status=status)
        st_host = status.to("cpu", non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = e0.elapsed_time(e1) / Ke
        e2e = {"value": moved * world / (e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": int(pairs_h.numel() * 4), "d2h_bytes_per_step": 4,
               "ms_per_step": e_ms, "steps": Ke, "status": int(st_host.item())}

    # Host block manager: 128 sequences forked from a 1000-token prompt, one
    # append each per step (slots + copy pairs for the step).
    bm = pkv.BlockManager(N, 16, 4096)
    bm.add(0, 1000)
    seqs = list(range(1, 129))
    for sq in seqs:
        bm.fork(0, sq)
    steps_h = 200
    h0 = time.perf_counter()
    per_step = []
    for _ in range(steps_h):
        _, pr = bm.append(seqs)
        per_step.append(len(pr))
    host_us = (time.perf_counter() - h0) / steps_h * 1e6

    line = {
        "metric": METRIC, "value": whole_job_rate(moved, world, ms * 1e-3) / 1e9, "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: random bf16 pool, seeded disjoint block pairs (no dataset)",
        "config": {"workload": workload_text("cow_copy_70b"), "name": "cow_copy_70b",
                   "num_blocks": N, "pairs": npairs, "block_bytes_per_cache": block_bytes,
                   "bytes_moved_per_step": moved,
                   "l2": "no flush: 268 MB moved per step exceeds L2 (129 MB)",
                   "launch": "copy captured once as a CUDA graph, replayed per step"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": f"copy_blocks_kernel (mean of {K} CUDA-graph replays)",
                     "algorithmic_bytes_per_launch": moved,
                     "peak_source": f"{peak_kind} hbm_gbs"},
        "host_block_manager": {"append_us_per_step": host_us, "sequences": len(seqs),
                               "copies_first_step": per_step[0], "copies_total": sum(per_step),
                               "note": "ctypes call from Python included"},
        "gpu_launches": K,
        "clocks": clocks,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if rank == 0 and not args.no_cpu_baseline:
        # The plain copy on the host (numpy), on a sample of the pairs.
        kh = np.random.default_rng(1).standard_normal((4096, Hkv, D, 16)).astype(np.float16)
        sub = np.random.default_rng(2).permutation(4096)[:512].reshape(256, 2)
        c0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - c0 < 5.0:
            kh[sub[:, 1]] = kh[sub[:, 0]]
            reps += 1
        el = time.perf_counter() - c0
        line["cpu_baseline"] = {"value": reps * 256 * block_bytes * 2 / el / 1e9, "unit": "GB/s",
                                "cores": 1, "kind": "numpy page copy",
                                "sample": f"{reps} x 256 page copies of one 16-bit cache in "
                                          f"{el:.1f} s"}
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------ several layers per launch

def run_layers(args):
    """One step = the decode of args.layers layers of one batch (shared block
    tables and lengths, each layer with its own caches, query, new token rows
    and output) in one pkv_paged_attn_decode_layers launch, the cache write of
    every layer's new token fused in.  The same work as args.layers separate
    fused launches (one CUDA graph holding them back to back) is timed beside
    it."""
    import torch
    import torch.distributed as dist

    import paged_kv_cache_225_gb300 as pkv

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    NL = args.layers
    ws = W.make_layers(args.config, NL)
    w0 = ws[0]
    cfg = w0.cfg
    S, Hq, Hkv, D = cfg.num_seqs, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim
    lens = (w0.seq_lens + 1).astype(np.int32)
    max_len = int(lens.max())
    ab = algorithmic_bytes(w0, lens)                     # per layer
    new_rows = S * Hkv * D * 2
    append_bytes = new_rows * (W.ELEM_BYTES[cfg.q_dtype] + W.ELEM_BYTES[cfg.kv_dtype])
    launch_bytes = NL * (ab["total"] + append_bytes)

    def t(a, dt):
        a = np.ascontiguousarray(a)
        if dt == W.F32:
            return torch.from_numpy(a)
        if dt == W.BF16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
        if dt == W.FP8_E4M3:
            return torch.from_numpy(a).view(torch.float8_e4m3fn)
        if dt == W.INT4:
            return torch.from_numpy(a)
        return torch.from_numpy(a).view(torch.float8_e5m2)

    layers = []
    for w in ws:
        layers.append({"q": t(w.q, cfg.q_dtype).to(dev), "new_k": t(w.new_k, cfg.q_dtype).to(dev),
                       "new_v": t(w.new_v, cfg.q_dtype).to(dev),
                       "k_cache": t(w.k_cache, cfg.kv_dtype).to(dev),
                       "v_cache": t(w.v_cache, cfg.kv_dtype).to(dev),
                       "out": torch.empty((S, Hq, D), dtype=torch.float32, device=dev)})
    table = pkv.layer_table(layers)
    tables = torch.from_numpy(w0.block_tables).to(dev)
    lens_dev = torch.from_numpy(lens).to(dev)
    part = pkv.layers_partition_tokens(NL, S, Hq, Hkv, D, max_len, args.partition)
    wsp = torch.empty(pkv.layers_workspace_size(NL, S, Hq, Hkv, D, max_len, args.partition),
                      dtype=torch.uint8, device=dev)
    single_part = pkv.partition_tokens(S, Hq, Hkv, D, max_len, args.partition)
    ws1 = [torch.empty(pkv.workspace_size(S, Hq, Hkv, D, max_len, args.partition),
                       dtype=torch.uint8, device=dev) for _ in range(NL)]
    stream = torch.cuda.current_stream(dev)
    ks = cfg.kv_scale

    def fused():
        pkv.paged_attn_decode_layers(layers, tables, lens_dev, w0.scale, k_scale=ks, v_scale=ks,
                                     max_seq_len=max_len, partition_tokens=args.partition,
                                     impl=args.kernel, workspace=wsp, table=table)

    def separate():
        for lay, wsx in zip(layers, ws1):
            pkv.paged_attn_decode_append(lay["q"], lay["new_k"], lay["new_v"], lay["k_cache"],
                                         lay["v_cache"], tables, lens_dev, w0.scale, lay["out"],
                                         k_scale=ks, v_scale=ks, max_seq_len=max_len,
                                         partition_tokens=args.partition, impl=args.kernel,
                                         workspace=wsx)

    sampler = ClockSampler(local, enabled=not args.no_clocks)
    for _ in range(max(args.warmup, 3)):
        fused()
        separate()
    torch.cuda.synchronize()
    for x in [wsp] + ws1:
        status = pkv.read_status(x)
        if status != 0:
            raise RuntimeError(f"device status {pkv.STATUS.get(status, status)} during warm-up")
    gs = torch.cuda.Stream(dev)
    gs.wait_stream(stream)
    g_fused, g_sep = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_fused, stream=gs):
        fused()
    with torch.cuda.graph(g_sep, stream=gs):
        separate()
    stream.wait_stream(gs)
    for _ in range(3):
        g_fused.replay()
        g_sep.replay()
    torch.cuda.synchronize()
    K = args.steps
    clock_t0 = soak(g_fused.replay, sampler)
    if world > 1:
        dist.barrier()

    def timed(g):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(K):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / K

    ms_fused = timed(g_fused)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop(since=clock_t0)
    ms_sep = timed(g_sep)
    ms_fused = max_over_ranks(ms_fused)
    for x in [wsp] + ws1:
        status = pkv.read_status(x)
        if status != 0:
            raise RuntimeError(f"device status {pkv.STATUS.get(status, status)} in the timed run")

    # End to end: every layer's q and new rows and the shared tables and
    # lengths copied in from pinned host memory, every output copied back,
    # serialised on the launch stream.
    e2e = None
    if not args.no_e2e:
        pins = [{k: layers[i][k].cpu().pin_memory() for k in ("q", "new_k", "new_v")}
                for i in range(NL)]
        pin_tab = torch.from_numpy(w0.block_tables).pin_memory()
        pin_len = torch.from_numpy(lens).pin_memory()
        outs_h = [torch.empty((S, Hq, D), dtype=torch.float32).pin_memory() for _ in range(NL)]
        h2d = sum(v.numel() * v.element_size() for p_ in pins for v in p_.values()) + \
            pin_tab.numel() * 4 + pin_len.numel() * 4
        d2h = NL * S * Hq * D * 4
        Ke = max(1, min(K, 200))

        def e2e_step():
            for i in range(NL):
                for k, v in pins[i].items():
                    layers[i][k].copy_(v, non_blocking=True)
            tables.copy_(pin_tab, non_blocking=True)
            lens_dev.copy_(pin_len, non_blocking=True)
            fused()
            for i in range(NL):
                outs_h[i].copy_(layers[i]["out"], non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(Ke):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = e0.elapsed_time(e1) / Ke
        e2e = {"value": NL * ab["kv"] * world / (e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e_ms, "steps": Ke, "pipeline": "copies serialised on one stream"}

    peak, peak_kind = hbm_peak()
    achieved = launch_bytes / (ms_fused * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": whole_job_rate(NL * ab["kv"], world, ms_fused * 1e-3) / 1e9,
        "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_fused, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE_NAME[cfg.kv_dtype],
        "data": "synthetic: seeded N(0,1) q/K/V per layer, shuffled physical blocks (no dataset)",
        "config": {"workload": f"{NL} layers of: " + workload_text(args.config),
                   "name": args.config, "layers": NL, "num_seqs": S, "num_q_heads": Hq,
                   "num_kv_heads": Hkv, "head_dim": D, "tokens_per_layer": ab["tokens"],
                   "kv_bytes_per_step": NL * ab["kv"],
                   "schedule": ("stream-K (equal page ranges per CTA)"
                                if part == pkv.SCHEDULE_STREAMK else
                                f"{part}-token partitions" if part > 0 else
                                "one CTA per (layer, sequence, KV head)"),
                   "l2": f"no flush: {NL} layers' caches ({NL * (w0.k_cache.nbytes * 2) / 1e9:.2f}"
                         " GB) cycle through L2 (129 MB)",
                   "step": "one launch: every layer's cache write fused into its paged decode "
                           "over L+1",
                   "launch": "step captured once as a CUDA graph, replayed per step"},
        "ms_per_layer": ms_fused / NL,
        "tokens_per_s": whole_job_rate(NL * S, world, ms_fused * 1e-3),
        "separate_launches": {
            "ms_per_step": ms_sep, "ms_per_layer": ms_sep / NL,
            "value": NL * ab["kv"] / (ms_sep * 1e-3) / 1e9,
            "schedule": (f"{single_part}-token partitions" if single_part > 0 else
                         "stream-K" if single_part == pkv.SCHEDULE_STREAMK else
                         "one CTA per (sequence, KV head)"),
            "note": f"{NL} pkv_paged_attn_decode_append launches back to back in one CUDA graph"},
        "pct_hbm_peak": 100.0 * NL * ab["total"] / (ms_fused * 1e-3) / 1e9 / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": f"paged_attn_decode_layers call (mean of {K} CUDA-graph replays, "
                               "CUDA events on the launch stream)",
                     "algorithmic_bytes_per_launch": launch_bytes,
                     "peak_source": f"{peak_kind} hbm_gbs"},
        "gpu_launches": K,
        "clocks": clocks,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    prefill = args.config in W.PREFILL_CONFIGS
    if args.layers > 1 and not prefill and args.config != "cow_copy_70b":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the "
                              "oracle on one layer (run without --layers)"}))
            return
        run_layers(args)
        return
    if args.config == "cow_copy_70b":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "no oracle arm for page copies: "
                              "the copy is its own definition (numpy cpu_baseline reported)"}))
            return
        run_copy(args)
        return
    if args.impl == "reference":
        (run_reference_prefill if prefill else run_reference)(args)
    else:
        (run_prefill if prefill else run_ours)(args)


if __name__ == "__main__":
    main()
