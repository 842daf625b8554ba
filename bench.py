#!/usr/bin/env python3
"""Benchmark of the GPULZ coder on GB300: one step = encode + decode of the
512x512x512 uint32 Lorenzo-code volume (536.9 MB, chunk_size 4096, word_size 4,
match level 1), the largest of the five workloads, inputs resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config ID] [--no-per-config] [--window W] [--split]

Prints ONE JSON line (rank 0). `value` is the round-trip throughput (input
bytes / (encode time + decode time)); the line also carries encode and decode
GB/s, the ratio, the HBM roofline fraction of the encode kernel (headline) and
of the decode kernel, and a `per_config` table in which each of the five
workloads is timed the same way and checked against the oracle in this run.
L2 is flushed (a 256 MB write) before every timed encode and every timed
decode. With N > 1 (torchrun), every rank codes its own copy of the workload
(weak scaling, no data-path collective); the timed region is bracketed by a
barrier + synchronize and the max over ranks is taken.

--impl reference times the CPU oracle (the plain sequential C coder, spread
over the host's cores by chunk range) on the same workload and metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GPULZ encode/decode GB/s (uncompressed), ratio; fraction of GB300 HBM roofline"
VALUE_IS = ("round trip: uncompressed bytes / (encode + decode time), decimal GB/s; "
            "encode_gbs, decode_gbs, ratio and roofline fractions alongside")
UNIT = "GB/s"
CFG_ID = 4
PER_CONFIG = (1, 2, 3, 4, 5)
L2_FLUSH_BYTES = 256 << 20  # > 129 MB L2
FALLBACK_HBM_GBS = 6800.0


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", type=int, default=CFG_ID)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-per-config", action="store_true",
                   help="skip the per-workload table (configs 1-5)")
    p.add_argument("--per-config-steps", type=int, default=10)
    p.add_argument("--max-bytes", type=int, default=0,
                   help="code only the first N bytes of the workload (smaller profiling cases)")
    p.add_argument("--window", type=int, default=32,
                   help="exact near window in elements (32..64; above 32 on level-0 workloads)")
    p.add_argument("--split", action="store_true",
                   help="time split mode (four ports) instead of the single stream; one GPU")
    return p.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def workload_config(cfg, window=32, n_bytes=None):
    extra = {} if window == 32 else {"near_window": window}
    if n_bytes is not None and n_bytes != cfg.n_bytes:
        extra["first_bytes_only"] = n_bytes
    return extra | {
        "workload": cfg.name,
        "field": "x".join(str(s) for s in cfg.shape) + " float32 sinusoids+noise, " + cfg.codes,
        "n_bytes": cfg.n_bytes if n_bytes is None else n_bytes,
        "word_size": cfg.word_size,
        "chunk_size": cfg.chunk_size,
        "match_level": cfg.match_level,
        "seed": cfg.seed,
        "l2": "flushed before every timed encode and every timed decode (256 MB write)",
    }


# ----------------------------------------------------------------------------
# clocks sampler
# ----------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------
def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def alu_peak_tops(dev):
    """Integer-ALU issue peak: 4 SMSPs x 32 lanes per SM per cycle (one warp
    instruction per SMSP per cycle) x SMs x the maximum SM clock."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz, src = 2070.0, "nominal max SM clock 2070 MHz"
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f)["sm_max_mhz"])
            src = "MEASURED_PEAKS.json sm_max_mhz %.0f MHz" % mhz
    except (OSError, KeyError, ValueError):
        pass
    return sms * 128 * mhz * 1e6 / 1e12, "%d SMs x 128 lane-ops/cycle x %s" % (sms, src)


KERNEL_SOURCES = {"encode_kernel": ("gpulz_encode.cu", "gpulz_internal.cuh"),
                  "decode_kernel": ("gpulz_decode.cu", "gpulz_internal.cuh")}


def kernel_source_sha(kernel: str) -> str:
    """Hash of the sources a kernel is built from (a recorded ncu figure is
    only reported while it matches)."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "lz77_family_coder_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel
    sources are unchanged since it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    r = rec.get(kernel, {})
    if r.get("workload") != workload or r.get("source_sha") != kernel_source_sha(kernel):
        return None
    return r.get("dram_bytes_per_launch")


def max_over_ranks(value: float, dist, device) -> float:
    """Max of a per-rank scalar over the process group (the timed region of the
    slowest rank defines the job's time)."""
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_baseline(x, cfg, reps=3, window=32):
    import oracle
    threads = os.cpu_count() or 1
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        s = oracle.compress_threads(x, cfg.word_size, cfg.chunk_size, cfg.match_level, threads,
                                    window=window)
        y = oracle.decompress_threads(s, x.size, threads)
        times.append(time.perf_counter() - t0)
    assert (y == x).all()
    t = statistics.median(times)
    return {"value": round(x.size / t / 1e9, 4), "unit": UNIT, "cores": threads,
            "kind": "oracle",
            "sample": "whole workload (%d bytes), encode+decode round trip, median of %d"
                      % (x.size, reps)}


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
class Workload:
    """Device buffers of one workload and its timed encode/decode calls."""

    def __init__(self, g, cfg, x, dev, stream, window=32):
        import torch
        self.g, self.cfg, self.x, self.window = g, cfg, x, window
        self.n = x.size
        self.stream = stream
        self.sh = stream.cuda_stream
        self.d_in = torch.from_numpy(x).to(dev)
        self.cap = g.gpulz_compress_bound(self.n, cfg.word_size, cfg.chunk_size)
        self.out = torch.empty(self.cap, dtype=torch.uint8, device=dev)
        self.nb = torch.zeros(1, dtype=torch.int64, device=dev)
        self.y = torch.empty(max(self.n, 1), dtype=torch.uint8, device=dev)

    def compress(self):
        g, c = self.g, self.cfg
        if self.window == 32:
            st = g.gpulz_compress(self.d_in, self.n, c.word_size, c.chunk_size, c.match_level,
                                  self.out, self.cap, self.nb, self.sh)
        else:
            st = g.gpulz_compress_window(self.d_in, self.n, c.word_size, c.chunk_size,
                                         c.match_level, self.window, self.out, self.cap, self.nb,
                                         self.sh)
        assert st == g.GPULZ_OK, st

    def decompress(self):
        assert self.g.gpulz_decompress(self.out, self.y, self.n, self.sh) == self.g.GPULZ_OK

    def timed(self, K, flush, kernel_events=False):
        """K encode + decode calls, L2 flushed (outside the events) before each
        call. Per call, CUDA events on the launching stream bracket either the
        whole library call or, with kernel_events, only its encode or decode
        kernel (events the library records around that launch)."""
        import torch
        g, stream = self.g, self.stream
        ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(K)]
        for q in ev:
            for e in q:
                e.record(stream)  # creates the event
        torch.cuda.synchronize()
        for k in range(K):
            flush.fill_(k & 0xFF)
            if kernel_events:
                g.gpulz_set_kernel_events(ev[k][0], ev[k][1])
            else:
                ev[k][0].record(stream)
            self.compress()
            if not kernel_events:
                ev[k][1].record(stream)
            flush.fill_((k + 1) & 0xFF)
            if kernel_events:
                g.gpulz_set_kernel_events(ev[k][2], ev[k][3])
            else:
                ev[k][2].record(stream)
            self.decompress()
            if not kernel_events:
                ev[k][3].record(stream)
        g.gpulz_set_kernel_events(None, None)
        torch.cuda.synchronize()
        return ([q[0].elapsed_time(q[1]) for q in ev], [q[2].elapsed_time(q[3]) for q in ev])

    def parity(self, threads):
        """The stream and the decoded bytes of the last call against the oracle."""
        import numpy as np
        import oracle
        c = self.cfg
        S = int(self.nb.item())
        got = self.out[:S].cpu().numpy()
        ref = oracle.compress_threads(self.x, c.word_size, c.chunk_size, c.match_level, threads,
                                      window=self.window)
        ok = np.array_equal(got, ref) and np.array_equal(self.y[:self.n].cpu().numpy(), self.x)
        return ok, S


def hbm_fraction(alg_bytes, ms, peak):
    gbs = alg_bytes / (ms * 1e-3) / 1e9
    return round(gbs, 2), round(gbs / peak, 4)


def per_config_table(g, dev, stream, flush, steps, threads, peak, have=None):
    """Every workload of PER_CONFIG timed like the headline one (L2 flushed
    before each call; whole calls and kernels alone) and checked against the
    oracle; `have` maps a config id to an already measured row."""
    import synth
    rows = {}
    for cid in PER_CONFIG:
        if have and cid in have:
            rows[str(cid)] = have[cid]
            continue
        cfg = synth.CONFIGS[cid]
        x = synth.generate(cid)
        w = Workload(g, cfg, x, dev, stream)
        for _ in range(3):
            w.compress()
            w.decompress()
        t_enc, t_dec = w.timed(steps, flush)
        k_enc, k_dec = w.timed(steps, flush, kernel_events=True)
        status = g.gpulz_device_status(w.sh)
        ok, S = w.parity(threads)
        rows[str(cid)] = config_row(cfg, w.n, S, t_enc, t_dec, k_enc, k_dec, peak,
                                    ok and status == 0)
        del w
    return rows


def config_row(cfg, n, S, t_enc, t_dec, k_enc, k_dec, peak, ok):
    enc_ms, dec_ms = statistics.mean(t_enc), statistics.mean(t_dec)
    ek, dk = statistics.mean(k_enc), statistics.mean(k_dec)
    return {
        "workload": cfg.name, "n_bytes": n, "word_size": cfg.word_size,
        "chunk_size": cfg.chunk_size, "match_level": cfg.match_level,
        "ratio": round(n / S, 4), "stream_bytes": S,
        "encode_gbs": round(n / (enc_ms * 1e-3) / 1e9, 2),
        "decode_gbs": round(n / (dec_ms * 1e-3) / 1e9, 2),
        "round_trip_gbs": round(n / ((enc_ms + dec_ms) * 1e-3) / 1e9, 2),
        "encode_kernel_ms": round(ek, 5), "decode_kernel_ms": round(dk, 5),
        "encode_kernel_hbm_frac": hbm_fraction(n + S, ek, peak)[1],
        "decode_kernel_hbm_frac": hbm_fraction(S + n, dk, peak)[1],
        "parity": "bit-exact vs oracle" if ok else "MISMATCH",
        "steps": len(t_enc),
    }


def run_ours(args):
    import torch
    import torch.distributed as dist

    import lz77_family_coder_gb300 as g
    import synth

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    g.load()  # raises if the CUDA library is missing: no fallback
    cfg = synth.CONFIGS[args.config]
    x = synth.generate(cfg)
    if args.max_bytes:
        x = x[: args.max_bytes].copy()
    stream = torch.cuda.current_stream(dev)
    W = args.window
    wl = Workload(g, cfg, x, dev, stream, window=W)
    n, sh = wl.n, wl.sh
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    threads = os.cpu_count() or 1

    for _ in range(max(args.warmup, 3)):
        flush.fill_(1)
        wl.compress()
        flush.fill_(2)
        wl.decompress()
    assert g.gpulz_device_status(sh) == g.GPULZ_OK
    torch.cuda.synchronize()

    K = args.steps
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t_enc, t_dec = wl.timed(K, flush)
    if world > 1:
        dist.barrier()
    # the main kernels alone: a second run of K steps in which the library
    # records events right around its encode and decode kernels (kept out of
    # the run above so that the extra records cannot perturb `value`)
    k_enc, k_dec = wl.timed(K, flush, kernel_events=True)
    total_ms = sum(t_enc) + sum(t_dec)
    if world > 1:
        total_ms = max_over_ranks(total_ms, dist, dev)
    status = g.gpulz_device_status(sh)

    # parity after timing, on the same buffers
    parity = "unchecked"
    S = int(wl.nb.item())
    if rank == 0:
        ok, S = wl.parity(threads)
        parity = "bit-exact vs oracle" if ok and status == 0 else "MISMATCH"

    # end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        h_x = torch.from_numpy(x).pin_memory()
        h_nb = torch.zeros(1, dtype=torch.int64).pin_memory()
        h_s = torch.empty(wl.cap, dtype=torch.uint8).pin_memory()
        h_y = torch.empty(n, dtype=torch.uint8).pin_memory()
        d_s = torch.empty(wl.cap, dtype=torch.uint8, device=dev)

        def e2e_step():
            wl.d_in.copy_(h_x, non_blocking=True)
            wl.compress()
            h_nb.copy_(wl.nb, non_blocking=True)
            stream.synchronize()
            s_len = int(h_nb[0])
            h_s[:s_len].copy_(wl.out[:s_len], non_blocking=True)
            d_s[:s_len].copy_(h_s[:s_len], non_blocking=True)
            assert g.gpulz_decompress(d_s, wl.y, n, sh) == g.GPULZ_OK
            h_y.copy_(wl.y[:n], non_blocking=True)
            stream.synchronize()
            return s_len

        for _ in range(3):
            e2e_step()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        s_len = 0
        for _ in range(K):
            s_len = e2e_step()
        torch.cuda.synchronize()
        t_e2e = time.perf_counter() - t0
        if world > 1:
            t_e2e = max_over_ranks(t_e2e, dist, dev)
        assert torch.equal(h_y, h_x)
        e2e = {"value": round(world * n * K / t_e2e / 1e9, 3), "unit": UNIT,
               "h2d_bytes_per_step": n + s_len, "d2h_bytes_per_step": 8 + s_len + n,
               "path": "pinned host -> gpulz_compress -> host stream -> gpulz_decompress -> host"}
        del h_x, h_s, h_y, d_s

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peak, peak_kind = measured_peak()
    alu_peak, alu_src = alu_peak_tops(dev)
    enc_ms, dec_ms = statistics.mean(t_enc), statistics.mean(t_dec)
    enc_k_ms, dec_k_ms = statistics.mean(k_enc), statistics.mean(k_dec)
    enc_alg = n + S       # bytes: input read + stream written
    dec_alg = S + n       # bytes: stream read + output written
    enc_ach, enc_frac = hbm_fraction(enc_alg, enc_k_ms, peak)
    dec_ach, dec_frac = hbm_fraction(dec_alg, dec_k_ms, peak)
    enc_ops = W * (n // cfg.word_size)  # near-window equality compares
    traffic = recorded_traffic("encode_kernel", cfg.name)
    roofline = {
        "kernel": "encode_kernel (timed alone: events the library records around its launch)",
        "bound": "hbm",
        "achieved": enc_ach,
        "peak": peak,
        "unit": "GB/s",
        "frac": enc_frac,
        "peak_source": peak_kind + " (MEASURED_PEAKS.json hbm_gbs, burst copy)",
        "alg_bytes_per_launch": enc_alg,
        "alg_bytes_rule": "input bytes read + stream bytes written",
        "kernel_ms": round(enc_k_ms, 5),
        "traffic": traffic,
        "traffic_source": ("recorded: ncu dram__bytes_read.sum + dram__bytes_write.sum of this "
                           "kernel source on this workload (profiles/traffic.json)"
                           if traffic is not None else None),
        "alu_issue": {"achieved": round(enc_ops / (enc_k_ms * 1e-3) / 1e12, 4),
                      "peak": round(alu_peak, 3), "unit": "T compares/s",
                      "frac": round(enc_ops / (enc_k_ms * 1e-3) / 1e12 / alu_peak, 4),
                      "peak_source": "warp-instruction issue rate: " + alu_src,
                      "ops_per_launch": enc_ops,
                      "ops_rule": "%d equality compares per element" % W},
        "decode": {"kernel": "decode_kernel (timed alone, same way)",
                   "bound": "hbm", "kernel_ms": round(dec_k_ms, 5), "alg_bytes": dec_alg,
                   "achieved": dec_ach, "peak": peak, "unit": "GB/s", "frac": dec_frac,
                   "traffic": recorded_traffic("decode_kernel", cfg.name)},
        "encode_pass_ms": round(enc_ms, 5),
        "decode_pass_ms": round(dec_ms, 5),
    }
    line = {
        "metric": METRIC,
        "value_is": VALUE_IS,
        "value": round(world * n * K / (total_ms * 1e-3) / 1e9, 3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": max(args.warmup, 3),
        "ms_per_step": round(total_ms / K, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": cfg.dtype,
        "data": "synthetic (seeded stand-in for Lorenzo-quantized CLDHGH residuals)",
        "config": workload_config(cfg, W, n),
        "encode_gbs": round(n / (enc_ms * 1e-3) / 1e9, 2),
        "decode_gbs": round(n / (dec_ms * 1e-3) / 1e9, 2),
        "ratio": round(n / S, 4),
        "stream_bytes": S,
        "parity": parity,
        "device_status": status,
        "roofline": roofline,
        "gpu_launches": 5 * K,  # per step: encode, tile scan, copy; offset scan, decode
        "clocks": clocks.summary(),
        "e2e": e2e,
    }
    if not args.no_per_config and world == 1 and W == 32 and not args.max_bytes:
        have = {args.config: config_row(cfg, n, S, t_enc, t_dec, k_enc, k_dec, peak,
                                        parity == "bit-exact vs oracle")}
        del wl
        line["per_config"] = per_config_table(g, dev, stream, flush, args.per_config_steps,
                                              threads, peak, have)
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(x, cfg, window=W)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------
# reference arm: the CPU oracle on the host cores
# ----------------------------------------------------------------------------
def run_reference(args):
    world, rank, local = dist_env()
    if rank != 0:
        return
    import oracle
    import synth
    cfg = synth.CONFIGS[args.config]
    x = synth.generate(cfg)
    threads = os.cpu_count() or 1

    def step():
        s = oracle.compress_threads(x, cfg.word_size, cfg.chunk_size, cfg.match_level, threads,
                                    window=args.window)
        y = oracle.decompress_threads(s, x.size, threads)
        return s, y

    for _ in range(max(args.warmup, 3)):
        s, y = step()
    assert (y == x).all()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        s, y = step()
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = round(x.size * args.steps / total / 1e9, 4)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value_is": VALUE_IS,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": round(total * 1e3 / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": cfg.dtype,
        "data": "synthetic (seeded stand-in for Lorenzo-quantized CLDHGH residuals)",
        "config": workload_config(cfg, args.window),
        "ratio": round(x.size / s.size, 4),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": "whole workload per step (%d bytes), encode+decode round trip"
                                   % x.size},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_split(args):
    """Split mode (four ports) on one GPU: encode + decode per step, device
    timed with CUDA events, L2 flushed between steps, ports checked against
    the oracle's after timing."""
    import numpy as np
    import torch
    import synth
    import lz77_family_coder_gb300 as g
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    g.load()
    cfg = synth.CONFIGS[args.config]
    ws, cs, lvl = cfg.word_size, cfg.chunk_size, cfg.match_level
    x = synth.generate(cfg)
    n = x.size
    d_in = torch.from_numpy(x).to(dev)
    st, bounds = g.gpulz_split_bounds(n, ws, cs)
    assert st == g.GPULZ_OK
    ports = [torch.empty(max(b, 4), dtype=torch.uint8, device=dev) for b in bounds]
    caps = [p.numel() for p in ports]
    pb = torch.zeros(4, dtype=torch.int64, device=dev)
    y = torch.empty(n, dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    assert g.gpulz_compress_split(d_in, n, ws, cs, lvl, *ports, caps, pb, sh) == g.GPULZ_OK
    plen = [int(v) for v in pb.cpu().numpy()]
    for _ in range(max(args.warmup, 3)):
        flush.fill_(1)
        assert g.gpulz_compress_split(d_in, n, ws, cs, lvl, *ports, caps, pb, sh) == g.GPULZ_OK
        assert g.gpulz_decompress_split(*ports, plen, y, n, sh) == g.GPULZ_OK
    assert g.gpulz_device_status(sh) == g.GPULZ_OK
    K = args.steps
    torch.cuda.synchronize()
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(K)]
    with ClockSampler(0) as clocks:
        for k in range(K):
            flush.fill_(k & 0xFF)
            ev[k][0].record(stream)
            assert g.gpulz_compress_split(d_in, n, ws, cs, lvl, *ports, caps, pb, sh) == g.GPULZ_OK
            ev[k][1].record(stream)
            flush.fill_((k + 1) & 0xFF)
            ev[k][2].record(stream)
            assert g.gpulz_decompress_split(*ports, plen, y, n, sh) == g.GPULZ_OK
            ev[k][3].record(stream)
        torch.cuda.synchronize()
    t_enc = [q[0].elapsed_time(q[1]) for q in ev]
    t_dec = [q[2].elapsed_time(q[3]) for q in ev]
    status = g.gpulz_device_status(sh)
    import oracle
    ref = oracle.compress_split(x, ws, cs, lvl)
    got = [p[:k].cpu().numpy() for p, k in zip(ports, plen)]
    ok = all(np.array_equal(a, b) for a, b in zip(got, ref)) and np.array_equal(y.cpu().numpy(), x)
    enc_ms, dec_ms = statistics.mean(t_enc), statistics.mean(t_dec)
    total = sum(plen)
    line = {
        "metric": "GPULZ split-mode encode+decode round-trip throughput (uncompressed GB/s)",
        "value": round(n * K / ((sum(t_enc) + sum(t_dec)) * 1e-3) / 1e9, 3),
        "unit": UNIT, "n_gpus": 1, "steps": K, "warmup": max(args.warmup, 3),
        "ms_per_step": round((sum(t_enc) + sum(t_dec)) / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype,
        "data": "synthetic (seeded stand-in for Lorenzo-quantized CLDHGH residuals)",
        "config": dict(workload_config(cfg), format="split (meta, literals, lengths, offsets)"),
        "encode_gbs": round(n / (enc_ms * 1e-3) / 1e9, 2),
        "decode_gbs": round(n / (dec_ms * 1e-3) / 1e9, 2),
        "port_bytes": dict(zip(("meta", "literals", "lengths", "offsets"), plen)),
        "ratio": round(n / total, 4),
        "parity": "bit-exact vs oracle" if ok and status == 0 else "MISMATCH",
        "device_status": status,
        "gpu_launches": 5 * K,
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)


def synth_level(cfg_id):
    import synth
    return synth.CONFIGS[cfg_id].match_level


def main():
    args = parse_args()
    if args.window != 32 and (args.window < 32 or args.window > 64 or args.split or
                              synth_level(args.config) != 0):
        raise SystemExit("--window: 32..64, single-stream level-0 workloads only")
    if args.impl == "reference":
        run_reference(args)
    elif args.split:
        run_split(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
