#!/usr/bin/env python3
"""Benchmark of the TurboQuant store + fused decode path on GB300.

Default workload (c4): the turboquant_4bit_nc preset at head_dim 256, with
16 query heads over 4 KV heads and 4 layers (seeds 42 + 1337 * layer).  Every
layer's cache uses the hybrid-model page: lcm(4 * 262 B, 4096 B) = 536576 B,
i.e. 512 tokens per block.  One step is, per layer, a bulk tq_store_kv of
65536 new tokens followed by tq_decode_attention over 256 sequences x 2048
cached tokens.

Reported:
  value      decode packed-KV GB/s: bytes of packed slots read by decode /
             decode time (CUDA events on the launch stream)
  store      tq_store_kv Mtok/s
  e2e        the same GB/s through the public API with host buffers: per step
             the H2D copy of new K/V, slots, queries and tables from pinned
             memory, the step, and the D2H copy of the outputs
  roofline   decode algorithmic bytes / time against the measured HBM peak
  cpu_baseline  the CPU oracle timed on a bounded sample of the same workload

``--impl reference`` times the CPU oracle itself on the same metric; its
steps are bounded samples.  Under torchrun each rank runs its own replica on
its own GPU ("weak" scaling); rank 0 prints one JSON line.
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
import tempfile
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
METRIC = "fused TQ decode attn packed-KV HBM GB/s (% of peak); tq_store Mtok/s"
FALLBACK_HBM_GBS = 6800.0
#: seconds of untimed steps run under the clock sampler before the timed region
PREROLL_S = 0.5


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="c4", help="c1 | c2 | c3 | c4 (c4 is the reported configuration)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--layers", type=int, default=None, help="use only the first N layers (profiling)")
    ap.add_argument("--seqs", type=int, default=None, help="decode only the first N sequences (profiling)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU oracle baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sub-workloads", default="c2,c3",
                    help="with the c4 workload: other configurations timed in the same run ('' to skip)")
    ap.add_argument("--preroll-s", type=float, default=PREROLL_S,
                    help="seconds of untimed steps under the clock sampler before the timed region")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the dequant, ring and comparator fields (profiling runs)")
    ap.add_argument("--oracle-child", default=None, help=argparse.SUPPRESS)
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# multi-rank helpers (timing only; the data path has no collective)
# ---------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(backend: str):
    import torch.distributed as dist

    _, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return world


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def reduce_scalar(x: float, op: str, device=None) -> float:
    """max / sum of a per-rank scalar over all ranks (identity on one rank)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def weak_scaling_value(units: float, seconds: float, device=None) -> float:
    """Whole-job throughput: the units all ranks processed / the slowest
    rank's time (max over ranks), as the launch contract defines it."""
    total = reduce_scalar(units, "sum", device)
    slowest = reduce_scalar(seconds, "max", device)
    return total / slowest


# ---------------------------------------------------------------------------
# accounting
# ---------------------------------------------------------------------------

def slot_bytes_cfg(head_dim: int, kb: int, vb: int) -> int:
    key = head_dim if kb == 8 else -(-head_dim * kb // 8) + 2
    val = -(-head_dim * vb // 8) + 4
    s = key + val
    return s + (s & 1)


def decode_bytes(wl, slot_al: int):
    """(packed-KV bytes, all algorithmic bytes) of one decode call: per
    sequence L*H*slot packed bytes, plus q (Hq*d bf16), out (Hq*d fp32),
    the block-table entries read and the sequence length."""
    lens = wl.seq_lens.astype(np.int64)
    packed = int(np.sum(lens) * wl.num_kv_heads * slot_al)
    blocks = int(np.sum((lens + wl.block_size - 1) // wl.block_size))
    other = wl.num_seqs * (wl.num_q_heads * wl.head_dim * (2 + 4) + 4) + 4 * blocks
    return packed, packed + other


def store_bytes_per_token(wl, slot_al: int) -> int:
    """bf16 K and V read, the packed token row written, the int64 slot id."""
    return 2 * wl.num_kv_heads * wl.head_dim * 2 + wl.num_kv_heads * slot_al + 8


def measured_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            d = json.loads(p.read_text())
            return float(d["hbm_gbs"]), "measured"
        except (KeyError, ValueError):
            pass
    return FALLBACK_HBM_GBS, "fallback"


def decode_source_digest() -> str:
    """sha256 (16 hex digits) over the code of the decode kernel sources, in
    name order: comments are dropped and whitespace runs collapsed, so that
    editing a comment does not void a traffic record of unchanged code."""
    import re

    csrc = ROOT / "kv_cache_quantization_store_gb300" / "csrc"
    h = hashlib.sha256()
    for f in sorted(csrc.glob("tq_decode*")):
        text = f.read_text()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(f.name.encode())
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def decode_traffic_record():
    """DRAM bytes per decode launch from the committed ncu summary, used only
    while the decode source is unchanged since the capture (else None)."""
    f = ROOT / "profiles" / "decode_traffic.txt"
    if not f.exists():
        return None
    vals = {}
    for line in f.read_text().splitlines():
        if "=" in line and not line.lstrip().startswith("#"):
            key, val = line.split("=", 1)
            vals[key.strip()] = val.strip()
    if vals.get("source_sha256_16") != decode_source_digest():
        return None
    try:
        return float(vals["dram_bytes_per_launch_c4"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 25

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        if self.proc is not None:
            # the timed region starts once samples are flowing (at most 3 s)
            import time
            t0 = time.monotonic()
            while time.monotonic() - t0 < 3.0 and self.proc.poll() is None:
                if Path(self.file.name).stat().st_size > 0:
                    break
                time.sleep(0.02)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, load_start=None, timed=None):
        """Median SM clock, maximum clock and throttle reasons over the samples
        taken while the GPU was loaded (host wall-clock window ``load_start``
        .. end of the timed region); ``timed`` = (t0, t1) also counts the
        samples inside the timed region itself."""
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        rows = []
        for line in Path(self.file.name).read_text().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 10:
                rows.append(f)
        os.unlink(self.file.name)
        return summarize_clock_rows(rows, load_start, timed, self.PERIOD_MS)


def _smi_time(stamp: str):
    """nvidia-smi's local timestamp ('YYYY/MM/DD HH:MM:SS.mmm') -> epoch seconds."""
    import datetime

    try:
        return datetime.datetime.strptime(stamp, "%Y/%m/%d %H:%M:%S.%f").timestamp()
    except ValueError:
        return None


def summarize_clock_rows(rows, load_start=None, timed=None, period_ms=25):
    """Clock summary over nvidia-smi CSV rows (timestamp, index, sm, max sm,
    power, active, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap)."""
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
    end = timed[1] if timed else None
    window = []
    for r in rows:
        t = _smi_time(r[0])
        if t is None or load_start is None or end is None or load_start <= t <= end + period_ms * 1e-3:
            window.append((t, r))
    if not window:  # clock skew between host and sampler: keep every row
        window = [(_smi_time(r[0]), r) for r in rows]
    sel = [r for _, r in window]
    sm = [float(r[2]) for r in sel if r[2].replace(".", "").isdigit()]
    mx = [float(r[3]) for r in sel if r[3].replace(".", "").isdigit()]
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({n for r in sel for n, v in zip(names, r[6:10]) if v.lower() == "active"})
    out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
           "reasons": reasons, "samples": len(sel), "period_ms": period_ms,
           "window": "untimed steps just before the timed region, and the timed region"}
    if timed:
        out["samples_in_timed_region"] = sum(1 for t, _ in window if t is not None and timed[0] <= t <= timed[1])
    return out


# ---------------------------------------------------------------------------
# the CUDA path
# ---------------------------------------------------------------------------

def run_ours(args):
    import torch

    import kv_cache_quantization_store_gb300 as tq
    from kv_cache_quantization_store_gb300 import build as tq_build
    from kv_cache_quantization_store_gb300 import workloads as W

    rank, world, local_rank = dist_env()
    dist_init("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0:
        tq_build.build()
    barrier()
    wl = shrink(W.named(args.workload), args)
    cfg = tq.tq_config_init(wl.head_dim, wl.key_bits, wl.value_bits, wl.norm_correction, wl.seed)
    slot_al = cfg.slot_size_aligned
    table_np, nblk = wl.layout()
    sm_np = wl.slot_mapping()
    n_tok = wl.num_tokens
    store_n = wl.store_tokens or n_tok
    layers = list(wl.layers)
    h, d = wl.num_kv_heads, wl.head_dim

    # ---- inputs resident in HBM ------------------------------------------------
    k_all = torch.empty((n_tok, h, d), dtype=torch.bfloat16, device=dev)
    v_all = torch.empty_like(k_all)
    piece = 65536
    for a in range(0, n_tok, piece):
        kc, vc = wl.kv(a, min(n_tok, a + piece))
        k_all[a:a + kc.shape[0]].copy_(torch.from_numpy(kc).to(torch.bfloat16))
        v_all[a:a + vc.shape[0]].copy_(torch.from_numpy(vc).to(torch.bfloat16))
    slots_all = torch.from_numpy(sm_np).to(dev)
    q = torch.from_numpy(wl.q()).to(torch.bfloat16).to(dev)
    table = torch.from_numpy(table_np).to(dev)
    lens = torch.from_numpy(wl.seq_lens.astype(np.int32)).to(dev)
    max_len = int(wl.seq_lens.max())
    caches = [tq.new_paged_cache(cfg, nblk, wl.block_size, h, l, block_stride=wl.block_stride, device=dev)
              for l in layers]
    for c in caches:  # prefill every layer's history (untimed)
        tq.tq_store_kv(cfg, k_all, v_all, slots_all, c)
    k_new, v_new, slots_new = k_all[:store_n], v_all[:store_n], slots_all[:store_n]
    ws_bytes = tq.tq_decode_workspace_size(cfg, wl.num_seqs, wl.num_q_heads, h, wl.block_size, max_len)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    outs = [torch.empty((wl.num_seqs, wl.num_q_heads, d), dtype=torch.float32, device=dev) for _ in layers]
    torch.cuda.synchronize()
    for c in caches:
        if c.error_flags():
            raise RuntimeError(f"cache error flags {c.error_flags()} after prefill")

    stream = torch.cuda.current_stream()
    n_ev = max(1, args.steps) * len(layers)
    ev = {k: [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for k in ("s0", "s1", "d0", "d1")}

    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if needs_l2_flush(wl, slot_al) else None

    def step(i=None):
        for j, (c, o) in enumerate(zip(caches, outs)):
            if flush is not None:
                flush.fill_(j & 0xFF)
            if i is not None:
                ev["s0"][i * len(layers) + j].record(stream)
            tq.tq_store_kv(cfg, k_new, v_new, slots_new, c, stream=stream)
            if i is not None:
                ev["s1"][i * len(layers) + j].record(stream)
            if flush is not None:
                flush.fill_((j + 1) & 0xFF)
            if i is not None:
                ev["d0"][i * len(layers) + j].record(stream)
            tq.tq_decode_attention(cfg, q, c, table, lens, max_len, o, ws, stream=stream)
            if i is not None:
                ev["d1"][i * len(layers) + j].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    props = torch.cuda.get_device_properties(dev)
    gpu_id = f"GPU-{props.uuid}" if getattr(props, "uuid", None) else str(torch.cuda.current_device())
    with ClockSampler(gpu_id) as clocks:
        # untimed steps under the sampler for at least PREROLL_S, so that the
        # clock record covers the GPU under this load even when the timed
        # region is shorter than a sampling period
        load_start = time.time()
        while time.time() - load_start < args.preroll_s:
            step()
            torch.cuda.synchronize()
        barrier()
        host_t0 = time.time()
        t0.record(stream)
        for i in range(args.steps):
            step(i)
        t1.record(stream)
        torch.cuda.synchronize()
        host_t1 = time.time()
    barrier()
    total_ms = t0.elapsed_time(t1)
    store_ms = sum(a.elapsed_time(b) for a, b in zip(ev["s0"], ev["s1"]))
    dec_ms = sum(a.elapsed_time(b) for a, b in zip(ev["d0"], ev["d1"]))
    for c in caches:
        if c.error_flags():
            raise RuntimeError(f"cache error flags {c.error_flags()} after the timed steps")

    packed, algo = decode_bytes(wl, slot_al)
    n_calls = args.steps * len(layers)
    total_ms_max = reduce_scalar(total_ms, "max", dev)
    value = weak_scaling_value(packed * n_calls, dec_ms * 1e-3, dev) / 1e9
    store_mtok = weak_scaling_value(store_n * n_calls, store_ms * 1e-3, dev) / 1e6
    peak, peak_kind = measured_peaks()
    dec_avg_s = dec_ms / n_calls * 1e-3
    achieved = algo / dec_avg_s / 1e9
    store_gbs = store_bytes_per_token(wl, slot_al) * store_n / (store_ms / n_calls * 1e-3) / 1e9

    # ---- end to end through host buffers ---------------------------------------
    e2e = run_e2e(args, tq, wl, cfg, caches, k_new, v_new, slots_new, q, table, lens, max_len, ws, outs, stream,
                  packed, dev)
    dq = ring = comparator = None
    if not args.no_extras:
        dq = measure_dequant(tq, wl, cfg, caches[0], table, max_len, dev, stream, peak)
        ring = measure_ring(tq, wl, cfg, caches[0], table, k_all, v_all, q, max_len, dev, stream)
        comparator = measure_comparator(tq, wl, cfg, caches[0], table, q, max_len, dev, stream, dec_avg_s * 1e6)
    subs = {}
    if wl.name == "c4" and args.sub_workloads:
        for name in [x for x in args.sub_workloads.split(",") if x]:
            subs[name] = measure_workload(name, tq, dev, stream, peak, comparator=not args.no_extras)

    clk = clocks.summary(load_start, (host_t0, host_t1))
    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms_max / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": workload_config(wl, cfg, slot_al, world),
        "store": {"value": round(store_mtok, 2), "unit": "Mtok/s", "tokens_per_call": store_n,
                  "hbm_gbs": round(store_gbs, 1), "frac": round(store_gbs / peak, 4),
                  "peak_kind": f"{peak_kind} copy bandwidth"},
        "decode_frac_of_peak": round(packed / dec_avg_s / 1e9 / peak, 4),
        "roofline": {"kernel": "tq_decode_attention", "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_kind": peak_kind, "traffic": decode_traffic_record(),
                     "algorithmic_bytes_per_launch": algo, "avg_launch_us": round(dec_avg_s * 1e6, 2)},
        "e2e": e2e,
        "gpu_launches": n_calls * 3,
        "clocks": clk,
    }
    if dq is not None:
        result["dequant"] = dq
    if ring is not None:
        result["ring"] = ring
    if comparator is not None:
        result["comparator"] = comparator
    if subs:
        result["workloads"] = subs
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        result["cpu_baseline"] = cpu_baseline(args)
    if rank == 0:
        print(json.dumps(result), flush=True)


def shrink(wl, args):
    """A reduced copy of the workload for profiling runs (fewer layers and
    decode sequences); the full configuration is the default."""
    if args.layers:
        wl.layers = tuple(wl.layers[: args.layers])
    if args.seqs:
        wl.seq_lens = wl.seq_lens[: args.seqs]
        if wl.store_tokens:
            wl.store_tokens = min(wl.store_tokens, int(wl.seq_lens.sum()))
        wl.description += f" [reduced: {len(wl.layers)} layer(s), {args.seqs} sequences]"
    elif args.layers:
        wl.description += f" [reduced: {len(wl.layers)} layer(s)]"
    return wl


def measure_workload(name, tq, dev, stream, peak, store_reps=5, decode_reps=20, comparator=True):
    """Another configuration timed in the same run: its bulk store of every
    cached token and its decode of every sequence, device-resident inputs,
    CUDA events on the launch stream around each call.  K and V are drawn on
    the device (Workload.kv_device: the configuration's distribution, not the
    values of Workload.kv); the caches and K/V are larger than the L2."""
    import torch

    from kv_cache_quantization_store_gb300 import workloads as W

    wl = W.named(name)
    cfg = tq.tq_config_init(wl.head_dim, wl.key_bits, wl.value_bits, wl.norm_correction, wl.seed)
    slot_al = cfg.slot_size_aligned
    table_np, nblk = wl.layout()
    k, v = wl.kv_device(dev)
    slots = torch.from_numpy(wl.slot_mapping()).to(dev)
    q = torch.from_numpy(wl.q()).to(torch.bfloat16).to(dev)
    table = torch.from_numpy(table_np).to(dev)
    lens = torch.from_numpy(wl.seq_lens.astype(np.int32)).to(dev)
    max_len = int(wl.seq_lens.max())
    cache = tq.new_paged_cache(cfg, nblk, wl.block_size, wl.num_kv_heads, 0, block_stride=wl.block_stride,
                               device=dev)
    ws = torch.zeros(tq.tq_decode_workspace_size(cfg, wl.num_seqs, wl.num_q_heads, wl.num_kv_heads,
                                                 wl.block_size, max_len), dtype=torch.uint8, device=dev)
    out = torch.empty((wl.num_seqs, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device=dev)

    def timed(fn, n, warm=2):
        for _ in range(warm):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        torch.cuda.synchronize()
        for a, b in ev:
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e-3

    st = timed(lambda: tq.tq_store_kv(cfg, k, v, slots, cache, stream=stream), store_reps)
    dt = timed(lambda: tq.tq_decode_attention(cfg, q, cache, table, lens, max_len, out, ws, stream=stream),
               decode_reps)
    if cache.error_flags():
        raise RuntimeError(f"{name}: cache error flags {cache.error_flags()}")
    packed, algo = decode_bytes(wl, slot_al)
    n_tok = wl.num_tokens
    store_gbs = store_bytes_per_token(wl, slot_al) * n_tok / st / 1e9
    res = {
        "workload": f"{wl.name}: {wl.description}",
        "decode": {"value": round(packed / dt / 1e9, 1), "unit": "GB/s packed-KV",
                   "roofline": {"achieved": round(algo / dt / 1e9, 1), "frac": round(algo / dt / 1e9 / peak, 4),
                                "algorithmic_bytes_per_launch": algo, "avg_launch_us": round(dt * 1e6, 2)}},
        "store": {"value": round(n_tok / st / 1e6, 2), "unit": "Mtok/s", "tokens_per_call": n_tok,
                  "hbm_gbs": round(store_gbs, 1), "frac": round(store_gbs / peak, 4),
                  "avg_launch_us": round(st * 1e6, 2)},
        "inputs": "K/V drawn on the device with the configuration's distribution; caches and K/V larger than L2",
        "calls": {"store": store_reps, "decode": decode_reps},
    }
    del k, v
    if comparator:
        res["comparator"] = measure_comparator(tq, wl, cfg, cache, table, q, max_len, dev, stream, dt * 1e6)
    del cache, ws, out
    torch.cuda.empty_cache()
    return res


def measure_comparator(tq, wl, cfg, cache, table, q, max_len, dev, stream, fused_us, reps=5):
    """The dequant-then-dense path ([ART] article, "Obstacle 1"), outside
    the timed step: tq_dequant of every decode sequence's history to bf16 K
    and V, then tq_dense_decode_attention over them; mean CUDA-event time of
    each over `reps` calls, against the fused decode's time per call."""
    import torch

    lens = wl.seq_lens.astype(np.int64)
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)).to(dev)
    n = int(lens.sum())
    h, d = wl.num_kv_heads, wl.head_dim
    k_rows = torch.empty((n, h, d), dtype=torch.bfloat16, device=dev)
    v_rows = torch.empty_like(k_rows)
    ws = torch.zeros(tq.tq_dense_decode_workspace_size(d, wl.num_seqs, wl.num_q_heads, h, max_len),
                     dtype=torch.uint8, device=dev)
    out = torch.empty((wl.num_seqs, wl.num_q_heads, d), dtype=torch.float32, device=dev)

    def deq():
        tq.tq_dequant(cfg, cache, table, cu, max_len, k_rows, v_rows, stream=stream)

    def dense():
        tq.tq_dense_decode_attention(q, k_rows, v_rows, cu, max_len, out, ws, stream=stream)

    for _ in range(2):
        deq()
        dense()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps)]
    torch.cuda.synchronize()
    for a, b, c in ev:
        a.record(stream)
        deq()
        b.record(stream)
        dense()
        c.record(stream)
    torch.cuda.synchronize()
    dq_us = statistics.mean(a.elapsed_time(b) for a, b, _ in ev) * 1e3
    dn_us = statistics.mean(b.elapsed_time(c) for _, b, c in ev) * 1e3
    bf16_bytes = n * h * d * 2 * 2  # K and V rows, written by the dequant and read by the dense decode
    del k_rows, v_rows, ws, out
    torch.cuda.empty_cache()
    return {"dequant_us": round(dq_us, 2), "dense_decode_us": round(dn_us, 2), "total_us": round(dq_us + dn_us, 2),
            "fused_decode_us": round(fused_us, 2), "fused_speedup": round((dq_us + dn_us) / fused_us, 2),
            "dense_decode_gbs_bf16": round(bf16_bytes / dn_us / 1e3, 1),
            "note": "dequant of every decode sequence to bf16 K/V rows, then dense split-KV decode over them; "
                    "not part of the timed step"}


def measure_dequant(tq, wl, cfg, cache, table, max_len, dev, stream, peak, reps=10):
    """tq_dequant of the workload's decode sequences (continuation prefill),
    outside the timed step: packed bytes read + bf16 K and V written, per
    call, over the median CUDA-event time of `reps` calls."""
    import torch

    lens = wl.seq_lens.astype(np.int64)
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)).to(dev)
    n = int(lens.sum())
    h, d = wl.num_kv_heads, wl.head_dim
    k_out = torch.empty((n, h, d), dtype=torch.bfloat16, device=dev)
    v_out = torch.empty_like(k_out)
    for _ in range(3):
        tq.tq_dequant(cfg, cache, table, cu, max_len, k_out, v_out, stream=stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    torch.cuda.synchronize()
    for a, b in ev:
        a.record(stream)
        tq.tq_dequant(cfg, cache, table, cu, max_len, k_out, v_out, stream=stream)
        b.record(stream)
    torch.cuda.synchronize()
    us = statistics.median(a.elapsed_time(b) for a, b in ev) * 1e3
    bytes_ = n * h * (cfg.slot_size_aligned + 4 * d)
    del k_out, v_out
    return {"value": round(bytes_ / us / 1e3, 1), "unit": "GB/s", "frac": round(bytes_ / us / 1e3 / peak, 4),
            "us_per_call": round(us, 2), "tokens": n,
            "bytes_per_call": bytes_, "note": "packed slots read + bf16 K and V written; not part of the timed step"}


def measure_ring(tq, wl, cfg, cache, table, k_all, v_all, q, max_len, dev, stream, cycles=2):
    """Ring-buffered store ([ART] article, full_tq write path), outside the
    timed step.  Every sequence replays its last R positions as R
    single-token decode steps through tq_ring_append (the ring's flush
    rewrites the same packed bytes), against tq_store_kv of the same token
    per sequence and step; then the ring decode with R/2 exact tokens per
    sequence against the plain decode of the same lengths."""
    import torch

    r_len = tq.TQ_RING_TOKENS
    lens = wl.seq_lens.astype(np.int64)
    if (lens < r_len).any():
        return {"skipped": f"sequences shorter than the {r_len}-token ring"}
    s_n, h, d = wl.num_seqs, wl.num_kv_heads, wl.head_dim
    cu = np.concatenate([[0], np.cumsum(lens)])
    start = lens - r_len
    ring_k, ring_v = tq.new_ring(cfg, s_n, h, r_len, device=dev)
    ws = torch.empty(tq.tq_ring_workspace_size(s_n), dtype=torch.uint8, device=dev)
    one_each = torch.arange(s_n + 1, dtype=torch.int32, device=dev)
    rows = torch.from_numpy(cu[:-1][None, :] + start[None, :] + np.arange(r_len)[:, None]).to(dev)  # [R, S]
    k_steps, v_steps = k_all[rows], v_all[rows]  # [R, S, H, d]
    lens_steps = torch.from_numpy((start[None, :] + np.arange(r_len)[:, None]).astype(np.int32)).to(dev)
    pos = start[None, :] + np.arange(r_len)[:, None]
    slots_steps = torch.from_numpy(table.cpu().numpy()[np.arange(s_n)[None, :], pos // wl.block_size].astype(np.int64)
                                   * wl.block_size + pos % wl.block_size).to(dev)
    # the ring state of a sequence of `start` tokens: positions R floor(start/R) .. start - 1
    head = start - start % r_len
    pre_rows = [np.arange(cu[s] + head[s], cu[s] + start[s]) for s in range(s_n)]
    pre_cu = torch.from_numpy(np.concatenate([[0], np.cumsum([len(r) for r in pre_rows])]).astype(np.int32)).to(dev)
    pre_idx = torch.from_numpy(np.concatenate(pre_rows).astype(np.int64)).to(dev)
    pre_k, pre_v = k_all[pre_idx].contiguous(), v_all[pre_idx].contiguous()
    pre_lens = torch.from_numpy(head.astype(np.int32)).to(dev)

    def refill():
        tq.tq_ring_append(cfg, pre_k, pre_v, pre_cu, pre_lens, ring_k, ring_v, cache, table, ws, stream=stream)

    def timed(fn, n):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for i, (a, b) in enumerate(ev):
            a.record(stream)
            fn(i)
            b.record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) * 1e3 for a, b in ev]

    def append(i, st=stream):
        tq.tq_ring_append(cfg, k_steps[i], v_steps[i], one_each, lens_steps[i], ring_k, ring_v, cache, table, ws,
                          stream=st)

    def direct(i, st=stream):
        tq.tq_store_kv(cfg, k_steps[i], v_steps[i], slots_steps[i], cache, stream=st)

    def one_kernel(i, st=stream):
        tq.tq_ring_step(cfg, k_steps[i], v_steps[i], lens_steps[i], ring_k, ring_v, cache, table, stream=st)

    # per-call latency, host launch included (the device work of one step is small)
    refill()
    latency_ring = timed(append, r_len)
    latency_direct = timed(direct, r_len)
    # device time per step: the R steps of a cycle captured in one CUDA graph
    graphs = {}
    try:
        for name, fn in (("ring", append), ("step", one_kernel), ("direct", direct)):
            refill()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for i in range(r_len):
                    fn(i, None)  # the capture stream
            graphs[name] = g
    except RuntimeError as exc:  # report the latency figures alone
        torch.cuda.synchronize()
        graphs = {}
        graph_error = str(exc).splitlines()[0]
    else:
        graph_error = None
    per_step = {"ring": float("nan"), "step": float("nan"), "direct": float("nan")}
    for name, g in graphs.items():
        t = []
        for _ in range(cycles + 1):
            refill()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            t.append(a.elapsed_time(b) * 1e3 / r_len)
        per_step[name] = statistics.median(t[1:])
    if cache.error_flags():
        raise RuntimeError(f"cache error flags {cache.error_flags()} after the ring cycles")
    # decode with half a ring of exact tokens
    half = r_len // 2
    refill()
    for i in range(half):
        append(i)
    mid_lens = lens_steps[half]  # start + R/2 tokens per sequence
    out = torch.empty((s_n, wl.num_q_heads, d), dtype=torch.float32, device=dev)
    ws_r = torch.zeros(tq.tq_decode_ring_workspace_size(cfg, s_n, wl.num_q_heads, h, wl.block_size, max_len),
                       dtype=torch.uint8, device=dev)
    ws_p = torch.zeros(tq.tq_decode_workspace_size(cfg, s_n, wl.num_q_heads, h, wl.block_size, max_len),
                       dtype=torch.uint8, device=dev)
    ring_dec = timed(lambda i: tq.tq_decode_attention_ring(cfg, q, cache, table, mid_lens, max_len, ring_k, ring_v,
                                                           out, ws_r, stream=stream), 12)[2:]
    plain_dec = timed(lambda i: tq.tq_decode_attention(cfg, q, cache, table, mid_lens, max_len, out, ws_p,
                                                       stream=stream), 12)[2:]
    res = {"ring_tokens": r_len, "cycle_steps": r_len,
            "append_device_us_per_step": round(per_step["ring"], 2),
            "ring_step_device_us_per_step": round(per_step["step"], 2),
            "store_direct_device_us_per_step": round(per_step["direct"], 2),
            "append_mtok_s": round(s_n / per_step["ring"], 2),
            "ring_step_mtok_s": round(s_n / per_step["step"], 2),
            "store_direct_mtok_s": round(s_n / per_step["direct"], 2),
            "append_latency_us_median": round(statistics.median(latency_ring), 2),
            "store_direct_latency_us_median": round(statistics.median(latency_direct), 2),
            "decode_ring_us": round(statistics.median(ring_dec), 2),
            "decode_plain_us": round(statistics.median(plain_dec), 2), "ring_rows_in_decode": half,
            "note": "one token per sequence per step, device time from a CUDA graph of one ring cycle; "
                    "not part of the timed step"}
    if graph_error:
        res["graph_error"] = graph_error
    return res


def run_e2e(args, tq, wl, cfg, caches, k_new, v_new, slots_new, q, table, lens, max_len, ws, outs, stream,
            packed, dev):
    """The step through the public API from pinned host buffers: every step
    copies its inputs to the device, runs the store and decode of every
    layer, and reads the outputs back.  Inputs and outputs are double
    buffered, so step i + 1's host-to-device copy (copy stream) and step
    i - 1's read-back (read-back stream) overlap step i's kernels (compute
    stream); events order each buffer's reuse.  The timed region starts
    before the first step's copy and ends after the last step's read-back."""
    import torch

    # every layer gets its own upload of new keys and values (a model's layers
    # each produce their own K/V): one pinned host copy per layer
    kv_host = [(k_new.cpu().pin_memory(), v_new.cpu().pin_memory())]
    for _ in range(1, len(caches)):
        kv_host.append((kv_host[0][0].clone().pin_memory(), kv_host[0][1].clone().pin_memory()))
    host = {name: t.cpu().pin_memory() for name, t in
            (("slots", slots_new), ("q", q), ("table", table), ("lens", lens))}
    for j, (hk, hv) in enumerate(kv_host):
        host[f"k{j}"] = hk
        host[f"v{j}"] = hv
    nbuf = 2
    dev_in = [{name: torch.empty_like(t, device=dev) for name, t in host.items()} for _ in range(nbuf)]
    dev_out = [[torch.empty_like(o) for o in outs] for _ in range(nbuf)]
    host_out = [[torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs] for _ in range(nbuf)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    copy_s = torch.cuda.Stream(dev)
    back_s = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in range(nbuf)]
    computed = [torch.cuda.Event() for _ in range(nbuf)]
    drained = [torch.cuda.Event() for _ in range(nbuf)]
    state = {"i": 0}

    def e2e_step():
        bi = state["i"] % nbuf
        state["i"] += 1
        copy_s.wait_event(computed[bi])  # step i - 2 has finished reading these inputs
        with torch.cuda.stream(copy_s):
            for name, t in host.items():
                dev_in[bi][name].copy_(t, non_blocking=True)
        copied[bi].record(copy_s)
        stream.wait_event(copied[bi])
        stream.wait_event(drained[bi])  # step i - 2's outputs have been read back
        din = dev_in[bi]
        for j, (c, o) in enumerate(zip(caches, dev_out[bi])):
            tq.tq_store_kv(cfg, din[f"k{j}"], din[f"v{j}"], din["slots"], c, stream=stream)
            tq.tq_decode_attention(cfg, din["q"], c, din["table"], din["lens"], max_len, o, ws, stream=stream)
        computed[bi].record(stream)
        back_s.wait_event(computed[bi])
        with torch.cuda.stream(back_s):
            for o, ho in zip(dev_out[bi], host_out[bi]):
                ho.copy_(o, non_blocking=True)
        drained[bi].record(back_s)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    copy_s.wait_event(a)
    back_s.wait_event(a)
    for _ in range(args.e2e_steps):
        e2e_step()
    for ev in drained:
        stream.wait_event(ev)
    b.record(stream)
    torch.cuda.synchronize()
    ms = reduce_scalar(a.elapsed_time(b), "max", dev)
    _, world, _ = dist_env()
    value = world * packed * len(caches) * args.e2e_steps / (ms * 1e-3) / 1e9
    return {"value": round(value, 2), "unit": "GB/s", "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": args.e2e_steps, "ms_per_step": round(ms / args.e2e_steps, 4),
            "api": "kv_cache_quantization_store_gb300.tq_store_kv / tq_decode_attention (C ABI via ctypes); "
                   "inputs and outputs double buffered, copies on their own streams",
            "inputs": f"per step: new K and V uploaded once per layer ({len(caches)} uploads), slot ids, queries, "
                      "block table and lengths once; every layer's output read back"}


#: GB300 L2 (129 MB): working sets that fit are flushed between timed kernels
L2_BYTES = 129 * 1024 * 1024
FLUSH_BYTES = 256 * 1024 * 1024


def needs_l2_flush(wl, slot_al) -> bool:
    """True when a layer's decode cache or the store's bf16 K/V fits in the
    L2, so that a timed kernel could find its input cached."""
    page = wl.block_stride or wl.block_size * wl.num_kv_heads * slot_al
    cache = page * wl.layout()[1]
    store_kv = (wl.store_tokens or wl.num_tokens) * wl.num_kv_heads * wl.head_dim * 4
    return min(cache, store_kv) <= L2_BYTES


def workload_config(wl, cfg, slot_al, world):
    page = wl.block_stride or wl.block_size * wl.num_kv_heads * slot_al
    return {
        "workload": f"{wl.name}: {wl.description}",
        "preset": wl.preset,
        "head_dim": wl.head_dim,
        "key_bits": wl.key_bits,
        "value_bits": wl.value_bits,
        "norm_correction": bool(wl.norm_correction),
        "num_q_heads": wl.num_q_heads,
        "num_kv_heads": wl.num_kv_heads,
        "layers": len(wl.layers),
        "decode_batch": wl.num_seqs,
        "seq_len": int(wl.seq_lens.max()) if len(set(wl.seq_lens.tolist())) == 1 else "ragged",
        "store_tokens": wl.store_tokens or wl.num_tokens,
        "block_size": wl.block_size,
        "block_bytes": page,
        "slot_bytes": slot_al,
        "cache_bytes_per_layer": page * wl.layout()[1],
        "l2": ("flushed: a 256 MB buffer is written before every timed store and decode (outside their events)"
               if needs_l2_flush(wl, slot_al) else
               "no flush: each layer's decode reads its own cache and the store its K/V, both larger than the "
               "129 MB L2"),
        "parallelism": f"replicas x{world}",
        "kv": "one K/V draw shared by the layers; layers differ by seed (random signs)",
    }


# ---------------------------------------------------------------------------
# the CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(wl_name: str, budget_s: float, layer_idx: int = 0, max_seqs: int | None = None):
    """Times the oracle on whole sequences of the workload until the budget is
    spent: its store of each sequence's tokens, then its decode of them."""
    import oracle as O
    from kv_cache_quantization_store_gb300 import workloads as W

    wl = W.named(wl_name)
    ocfg = O.Config(head_dim=wl.head_dim, key_quant_bits=wl.key_bits, value_quant_bits=wl.value_bits,
                    seed=wl.seed, norm_correction=wl.norm_correction)
    layer = O.make_layer(ocfg, layer_idx)
    table, nblk = wl.layout()
    cache = O.new_cache(ocfg, nblk, wl.block_size, wl.num_kv_heads, wl.block_stride)
    q_all = wl.q()
    cu = wl.cu_seqlens()
    sm = wl.slot_mapping()
    t_store = t_dec = 0.0
    toks = packed = 0
    seqs = 0
    per_seq = []
    start = time.perf_counter()
    for s in range(wl.num_seqs):
        a, b = int(cu[s]), int(cu[s + 1])
        k, v = wl.kv(a, b, threads=1)
        t = time.perf_counter()
        O.store_kv(layer, k, v, sm[a:b], cache)
        ts = time.perf_counter() - t
        t = time.perf_counter()
        O.decode_attention(layer, q_all[s:s + 1], cache, table[s:s + 1], wl.seq_lens[s:s + 1])
        td = time.perf_counter() - t
        t_store += ts
        t_dec += td
        per_seq.append((b - a, ts, td))
        toks += b - a
        packed += (b - a) * wl.num_kv_heads * ocfg.slot_size_aligned
        seqs += 1
        if time.perf_counter() - start > budget_s or (max_seqs and seqs >= max_seqs):
            break
    return {"decode_gbs": packed / t_dec / 1e9, "store_mtok_s": toks / t_store / 1e6, "seqs": seqs,
            "tokens": toks, "decode_s": t_dec, "store_s": t_store, "per_seq": per_seq,
            "slot_bytes": ocfg.slot_size_aligned, "num_kv_heads": wl.num_kv_heads}


def _oracle_worker(spec, seqs, barrier_, out_q):
    """One process of the all-cores oracle baseline: prepares its share of
    the sequences (inputs drawn and the layer built before timing), then
    stores them all and decodes them all, each phase started at a barrier
    shared by every worker; reports its phase times."""
    sys.path.insert(0, str(ROOT))
    import oracle as O
    from kv_cache_quantization_store_gb300 import workloads as W

    wl = W.named(spec["workload"])
    ocfg = O.Config(head_dim=wl.head_dim, key_quant_bits=wl.key_bits, value_quant_bits=wl.value_bits,
                    seed=wl.seed, norm_correction=wl.norm_correction)
    layer = O.make_layer(ocfg, 0)
    table, nblk = wl.layout()
    q_all = wl.q()
    cu = wl.cu_seqlens()
    sm = wl.slot_mapping()
    inputs = [(s, wl.kv(int(cu[s]), int(cu[s + 1]), threads=1)) for s in seqs]
    cache = O.new_cache(ocfg, nblk, wl.block_size, wl.num_kv_heads, wl.block_stride)
    barrier_.wait()
    t = time.perf_counter()
    for s, (k, v) in inputs:
        O.store_kv(layer, k, v, sm[int(cu[s]):int(cu[s + 1])], cache)
    t_store = time.perf_counter() - t
    barrier_.wait()
    t = time.perf_counter()
    for s, _ in inputs:
        O.decode_attention(layer, q_all[s:s + 1], cache, table[s:s + 1], wl.seq_lens[s:s + 1])
    t_dec = time.perf_counter() - t
    out_q.put((t_store, t_dec))


def oracle_all_cores(wl_name: str, seq_seconds: float, budget_s: float):
    """The oracle on every host core: one spawned process per core, each with
    single-threaded BLAS and its own share of whole sequences.  The sequence
    count is sized from the single-thread time per sequence to about
    ``budget_s`` of work per process; the store and decode phases each run
    from a common barrier, and a phase's time is its slowest process's."""
    import multiprocessing as mp

    from kv_cache_quantization_store_gb300 import workloads as W

    wl = W.named(wl_name)
    procs = len(os.sched_getaffinity(0))
    per_proc = max(1, int(budget_s / max(seq_seconds, 1e-6)))
    n = min(wl.num_seqs, procs * per_proc)
    procs = min(procs, n)
    shares = [list(range(i, n, procs)) for i in range(procs)]
    ctx = mp.get_context("spawn")
    barrier_ = ctx.Barrier(procs)
    out_q = ctx.Queue()
    spec = {"workload": wl_name}
    workers = [ctx.Process(target=_oracle_worker, args=(spec, sh, barrier_, out_q)) for sh in shares]
    for w in workers:
        w.start()
    res = [out_q.get(timeout=1800) for _ in workers]
    for w in workers:
        w.join()
    toks = int(sum(wl.seq_lens[:n]))
    ocfg_slot = slot_bytes_cfg(wl.head_dim, wl.key_bits, wl.value_bits)
    packed = toks * wl.num_kv_heads * ocfg_slot
    t_store = max(r[0] for r in res)
    t_dec = max(r[1] for r in res)
    return {"decode_gbs": packed / t_dec / 1e9, "store_mtok_s": toks / t_store / 1e6, "seqs": n,
            "tokens": toks, "procs": procs, "decode_s": t_dec, "store_s": t_store}


def oracle_child_env():
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "NUMEXPR_NUM_THREADS"):
        env[var] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    return env


def run_oracle_child(wl_name: str, budget: float, max_seqs: int | None = None, all_cores_seq_s=None):
    """The oracle runs in a child process with no GPU and single-threaded
    BLAS (its spawned workers inherit that environment)."""
    cmd = [sys.executable, str(Path(__file__).resolve()), "--oracle-child",
           json.dumps({"workload": wl_name, "budget": budget, "max_seqs": max_seqs,
                       "all_cores_seq_s": all_cores_seq_s})]
    res = subprocess.run(cmd, env=oracle_child_env(), capture_output=True, text=True, timeout=1800)
    if res.returncode != 0:
        raise RuntimeError(f"oracle child failed: {res.stderr[-2000:]}")
    return json.loads(res.stdout.strip().splitlines()[-1])


def cpu_baseline(args):
    """The oracle timed single-threaded (the reported value) and on every
    host core (``all_cores``), on bounded samples of the workload."""
    r = run_oracle_child(args.workload, args.cpu_seconds)
    out = {"value": round(r["decode_gbs"], 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": (f"{r['seqs']} whole sequences of {args.workload} (layer 0): oracle store of their "
                      f"{r['tokens']} tokens then oracle decode of all query heads; single thread "
                      "(BLAS pinned to 1)"),
           "store_mtok_s": round(r["store_mtok_s"], 6), "host_cores_available": len(os.sched_getaffinity(0))}
    seq_s = (r["store_s"] + r["decode_s"]) / max(1, r["seqs"])
    try:
        a = run_oracle_child(args.workload, args.cpu_seconds, all_cores_seq_s=seq_s)
    except Exception as exc:  # report the single-thread figure alone
        out["all_cores"] = {"error": str(exc).splitlines()[0] if str(exc) else type(exc).__name__}
    else:
        out["all_cores"] = {
            "value": round(a["decode_gbs"], 6), "unit": "GB/s", "cores": a["procs"],
            "store_mtok_s": round(a["store_mtok_s"], 6),
            "sample": (f"{a['seqs']} whole sequences of {args.workload} (layer 0) shared by {a['procs']} "
                       "spawned processes (one per host core, BLAS pinned to 1): oracle store of every "
                       "sequence, then oracle decode; each phase timed from a common barrier to the "
                       "slowest process")}
    return out


def run_reference(args):
    """The CPU oracle as the reference arm: one step = one whole sequence of
    the workload (layer 0): the oracle's store of its tokens, then its decode
    of every query head.  Rank 0 alone runs; other ranks exit."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    r = run_oracle_child(args.workload, float("inf"), max_seqs=args.warmup + args.steps)
    timed = r["per_seq"][args.warmup:]
    if not timed:
        raise RuntimeError("no timed reference steps")
    dec_s = sum(td for _, _, td in timed)
    store_s = sum(ts for _, ts, _ in timed)
    toks = sum(n for n, _, _ in timed)
    value = toks * r["num_kv_heads"] * r["slot_bytes"] / dec_s / 1e9
    sample = (f"each step: one whole sequence of {args.workload} (layer 0, {timed[0][0]} tokens): "
              "oracle store then oracle decode of every query head, single thread (BLAS pinned to 1)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s", "n_gpus": world,
        "steps": len(timed), "warmup": args.warmup, "ms_per_step": round((dec_s + store_s) / len(timed) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "impl": "CPU oracle (NumPy fp64)"},
        "store": {"value": round(toks / store_s / 1e6, 6), "unit": "Mtok/s"},
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "kind": "oracle", "cores": 1, "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.oracle_child:
        spec = json.loads(args.oracle_child)
        sys.path.insert(0, str(ROOT))
        budget = spec["budget"] if spec["budget"] is not None else float("inf")
        if spec.get("all_cores_seq_s"):
            r = oracle_all_cores(spec["workload"], spec["all_cores_seq_s"], budget)
        else:
            r = oracle_sample(spec["workload"], budget, max_seqs=spec.get("max_seqs"))
        print(json.dumps(r))
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
