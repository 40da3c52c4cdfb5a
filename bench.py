"""Benchmark of the GB300 KV codec: one step = the whole hot path on one
batch of synthetic KV cache --
  1. kvpool_encode_ex   (int8 K, per-tensor scale or --k-format q8_0 blocks;
                         V FWHT + Lloyd-Max 3 bit)
  2. kvpool_decode_into (fan-out of every layer into N agent caches)
  3. cachecard_pack     (per-token {2,4,8,16}-bit groups + metadata)
  4. cachecard_unpack   (back to bf16 past_key_values)
Metric: bf16-equivalent GB/s of the step (bytes of bf16 KV consumed or
produced: encode raw + decode N*raw + pack raw + unpack raw) and its
fraction of the GB300 HBM roofline.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload NAME] [--agents N] [--tokens T] [--layers L]
                       [--k-format per_tensor|q8_0] [--mode step|attend|realign]
Under torchrun (N > 1) every rank runs its own replica (independent pools:
weak scaling, no collective on the data path); rank 0 prints one JSON line.
"""
import argparse
import ctypes
import hashlib
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

import agent_shared_compressed_gb300 as kv  # noqa: E402
from agent_shared_compressed_gb300 import synth  # noqa: E402

METRIC = "KV codec encode/decode GB/s (bf16-equivalent) and % of GB300 HBM peak"
DEFAULT_WORKLOAD = "llama3-8b-4k-15agents"
L2_BYTES = 129 * 1024 * 1024
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
DECODE_SOURCES = ["agent_shared_compressed_gb300/csrc/kvpool_decode.cu",
                  "agent_shared_compressed_gb300/csrc/kvp_vec.cuh",
                  "agent_shared_compressed_gb300/csrc/kvp_internal.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_fanout_traffic.json")


# ----------------------------------------------------------------------------
# environment helpers
# ----------------------------------------------------------------------------

def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload, agents, tokens, layers):
    """DRAM bytes (read + write) of one decode launch, from the committed ncu
    capture of a small case scaled to this workload's launch, if the capture
    is of the current decode kernel source and its scaling names this
    workload; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("source_hash") != source_hash(DECODE_SOURCES):
        return None
    sc = rec.get("scale", {})
    if (sc.get("workload"), sc.get("agents"), sc.get("tokens"), sc.get("layers")) != (workload, agents, tokens, layers):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (driver library,
    read-only queries) on a background thread."""
    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}

    def __init__(self, index, period=0.005):
        self.period = period
        self.samples = []
        self.reasons = 0
        self.max_mhz = None
        self.ok = False
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
                return
            m = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.h, ctypes.c_int(1), ctypes.byref(m)) == 0:
                self.max_mhz = m.value
            self.ok = True
        except OSError:
            self.ok = False

    def _run(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self.stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.h, ctypes.c_int(1), ctypes.byref(clk)) == 0:
                self.samples.append(clk.value)
            if fn(self.h, ctypes.byref(rs)) == 0:
                self.reasons |= rs.value
            time.sleep(self.period)

    def __enter__(self):
        if self.ok:
            self.stop = threading.Event()
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self.stop.set()
            self.t.join()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unavailable"]}
        return {"sm_mhz": float(statistics.median(self.samples)), "sm_max_mhz": self.max_mhz,
                "reasons": [n for b, n in sorted(self.REASONS.items()) if self.reasons & b],
                "samples": len(self.samples)}


# ----------------------------------------------------------------------------
# workload
# ----------------------------------------------------------------------------

def workload(args):
    w = dict(synth.WORKLOADS[args.workload])
    if args.agents:
        w["N"] = args.agents
    if args.tokens:
        w["T"] = args.tokens
    if args.layers:
        w["L"] = args.layers
    return w


K_FORMATS = {"per_tensor": 0, "q8_0": 1}  # KVP_K_PER_TENSOR, KVP_K_Q8_0


def step_bytes(w, pool_bytes, card_bytes):
    raw = 2 * w["L"] * w["H"] * w["T"] * w["d"] * 2
    return {
        "raw": raw,
        "bf16_equiv": raw * (w["N"] + 3),
        "encode_alg": raw + pool_bytes,
        "decode_alg": pool_bytes + w["N"] * raw,
        "pack_alg": raw + card_bytes,
        "unpack_alg": card_bytes + raw,
    }


class Codec:
    """Device buffers for one replica of the step and the calls that run it."""

    def __init__(self, w, device, seed=0, outputs=True, k_mode=0):
        L, H, d, T, N = w["L"], w["H"], w["d"], w["T"], w["N"]
        self.w = w
        self.k_mode = k_mode
        self.shape = kv.Shape(L, H, d, T)
        self.k, self.v = synth.kv_layers(L, H, T, d, seed=seed, device=device)
        self.bits_host = synth.card_bits(T, seed=seed).numpy()
        self.bits = torch.from_numpy(self.bits_host).to(device)
        self.pool_bytes = kv.kvpool_pool_bytes_ex(self.shape, k_mode)
        self.ws_bytes = kv.kvpool_workspace_bytes(self.shape)
        self.card_bytes = kv.cachecard_bytes(self.shape, self.bits_host)
        self.pool = torch.empty(self.pool_bytes, dtype=torch.uint8, device=device)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
        self.card = torch.empty(self.card_bytes, dtype=torch.uint8, device=device)
        # agent caches and card output (skipped when only the pool is needed)
        n_out = N * L if outputs else 0
        self.caches_k = [torch.empty((H, T, d), dtype=torch.bfloat16, device=device) for _ in range(n_out)]
        self.caches_v = [torch.empty((H, T, d), dtype=torch.bfloat16, device=device) for _ in range(n_out)]
        self.out_k = [torch.empty((H, T, d), dtype=torch.bfloat16, device=device) for _ in range(L if outputs else 0)]
        self.out_v = [torch.empty((H, T, d), dtype=torch.bfloat16, device=device) for _ in range(L if outputs else 0)]
        self.hdr = None

    def encode(self, st):
        kv.check(kv.kvpool_encode_ex(self.shape, self.k_mode, self.k, self.v, self.pool, self.pool_bytes,
                                     self.ws, self.ws_bytes, st), "encode")

    def decode(self, st):
        kv.check(kv.kvpool_decode_into(self.pool, self.shape, 0, self.w["L"], self.w["N"], self.caches_k,
                                       self.caches_v, st), "decode")

    def pack(self, st):
        kv.check(kv.cachecard_pack(self.shape, 0x8B, 0, self.bits, self.k, self.v, self.card, self.card_bytes,
                                   st), "pack")

    def unpack(self, st):
        if self.hdr is None:
            self.hdr = kv.CardHeader()
            kv.check(kv.cachecard_read_header(self.card, self.hdr, st), "read_header")
        kv.check(kv.cachecard_unpack(self.card, self.hdr, self.out_k, self.out_v, st), "unpack")


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

def aggregate_ranks(local_ms, steps, bytes_per_step, world, device):
    """Whole-job throughput of N independent replicas: the slowest rank's
    time (max over ranks) and the bytes all ranks processed.  Returns
    (ms per step, GB/s)."""
    total_ms = float(local_ms)
    if world > 1:
        t = torch.tensor([total_ms], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_per_step = total_ms / steps
    return ms_per_step, world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


MIN_TIMED_S = 0.5          # the timed blocks together last at least this long
MAX_BLOCKS = 60
EXTRA_WORKLOADS = ["llama3-8b-32k-4agents"]  # timed beside the headline one in the default run


def phase_stats(ms, alg_bytes, peak):
    """Best / median / mean of one phase's per-step CUDA-event times (ms)."""
    best, med = float(np.min(ms)), float(np.median(ms))
    gbs = alg_bytes / (med * 1e-3) / 1e9
    return {"ms": round(med, 4), "ms_best": round(best, 4), "ms_mean": round(float(np.mean(ms)), 4),
            "alg_bytes": int(alg_bytes), "alg_GBps": round(gbs, 1),
            "alg_GBps_best": round(alg_bytes / (best * 1e-3) / 1e9, 1),
            "frac_of_measured_peak": round(gbs / peak, 4), "frac_of_8TBps": round(gbs / NOMINAL_HBM_GBS, 4)}


def time_blocks(c, st, flush, steps, world, device, est_step_ms, local_rank):
    """Time blocks of exactly `steps` steps, each bracketed by a barrier and a
    device synchronisation on both sides, until the blocks together last at
    least MIN_TIMED_S (so the clock sampler sees the GPU under load).
    Returns (per-phase ms [blocks, steps, 4], launches, clocks summary)."""
    blocks = int(min(MAX_BLOCKS, max(1, math.ceil(MIN_TIMED_S * 1e3 / max(1e-3, steps * est_step_ms)))))
    if world > 1:  # every rank runs the same number of blocks
        t = torch.tensor([blocks], dtype=torch.int64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        blocks = int(t.item())
    phases = []
    launches0 = kv.kvp_launch_count()
    sampler = ClockSampler(local_rank)
    with sampler:
        for _ in range(blocks):
            ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
            if world > 1:
                torch.distributed.barrier()
            torch.cuda.synchronize(device)
            for i in range(steps):
                if flush is not None:
                    flush.zero_()
                e = ev[i]
                e[0].record(st)
                c.encode(st)
                e[1].record(st)
                c.decode(st)
                e[2].record(st)
                c.pack(st)
                e[3].record(st)
                c.unpack(st)
                e[4].record(st)
            torch.cuda.synchronize(device)
            if world > 1:
                torch.distributed.barrier()
            phases.append([[e[j].elapsed_time(e[j + 1]) for j in range(4)] for e in ev])
    launches = kv.kvp_launch_count() - launches0
    return np.array(phases), launches, sampler.summary()


def measure_workload(name, w, args, rank, world, device, local_rank, k_mode, e2e=True):
    """Set up one workload's replica, warm up, time it (median block) and
    return (result dict, Codec, step bytes)."""
    c = Codec(w, device, seed=rank, k_mode=k_mode)
    st = torch.cuda.current_stream(device)
    sb = step_bytes(w, c.pool_bytes, c.card_bytes)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device) if sb["raw"] < 4 * L2_BYTES else None

    # warm-up (also reads the card header once: the unpack's host metadata);
    # the last warm-up steps' times size the timed blocks
    wev = [torch.cuda.Event(enable_timing=True) for _ in range(args.warmup + 1)]
    wev[0].record(st)
    for i in range(args.warmup):
        c.encode(st); c.decode(st); c.pack(st); c.unpack(st)
        wev[i + 1].record(st)
    torch.cuda.synchronize(device)
    for rc, what in ((kv.kvpool_status(c.pool, st), "pool"), (kv.cachecard_status(c.card, st), "card")):
        if rc != kv.KVP_OK:
            raise RuntimeError("%s status after warm-up: %s" % (what, kv.kvp_strerror(rc)))
    est_step_ms = min(wev[i].elapsed_time(wev[i + 1]) for i in range(1, args.warmup)) if args.warmup > 1 else 5.0

    phase, launches, clocks = time_blocks(c, st, flush, args.steps, world, device, est_step_ms, local_rank)
    block_ms = phase.sum(axis=(1, 2))                 # [blocks]
    med_block = float(np.median(block_ms))
    ms_per_step, value = aggregate_ranks(med_block, args.steps, sb["bf16_equiv"], world, device)

    peak, peak_kind = hbm_peak()
    flat = phase.reshape(-1, 4)
    names = ("encode", "decode", "pack", "unpack")
    algs = (sb["encode_alg"], sb["decode_alg"], sb["pack_alg"], sb["unpack_alg"])
    breakdown = {n: phase_stats(flat[:, j], b, peak) for j, (n, b) in enumerate(zip(names, algs))}
    if k_mode == 0:
        breakdown["encode"]["implemented_bytes"] = int(sb["encode_alg"] + sb["raw"] // 2)  # K is read twice
    dec_ms = breakdown["decode"]["ms"]
    achieved = sb["decode_alg"] / (dec_ms * 1e-3) / 1e9
    traffic = recorded_traffic(name, w["N"], w["T"], w["L"]) if k_mode == 0 else None
    out = {
        "value": round(value, 2), "unit": "GB/s", "ms_per_step": round(ms_per_step, 4),
        "steps": args.steps, "blocks": int(phase.shape[0]),
        "timed_s": round(float(block_ms.sum()) * 1e-3, 3),
        "block_GBps": {"median": round(value, 2),
                       "best": round(sb["bf16_equiv"] * args.steps / (float(block_ms.min()) * 1e-3) / 1e9 * world, 2),
                       "worst": round(sb["bf16_equiv"] * args.steps / (float(block_ms.max()) * 1e-3) / 1e9 * world,
                                      2)},
        "config": {"workload": name, "layers": w["L"], "kv_heads": w["H"], "head_dim": w["d"],
                   "tokens": w["T"], "agents": w["N"], "k_format": args.k_format,
                   "card_bits": "iid {2,4,8,16} p={.25,.40,.25,.10}",
                   "l2": ("flushed between steps (2x L2 write)" if flush is not None
                          else "inputs larger than L2 (%d MB K/V per step)" % (sb["raw"] // 10 ** 6)),
                   "parallelism": "replicas" if world > 1 else "single"},
        "roofline": {"kernel": "decode_fanout", "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "frac_nominal_8000": round(achieved / NOMINAL_HBM_GBS, 4),
                     "alg_bytes_per_launch": int(sb["decode_alg"]), "traffic": traffic},
        "gpu_launches": int(launches),
        "clocks": clocks,
        "breakdown": breakdown,
    }
    if e2e:
        # end to end through the C ABI with host buffers: H2D of the step's
        # K/V (and bitwidths) from pinned memory, the four calls, D2H of the
        # pool and the card (the two shareable artefacts) and their status
        out["e2e"] = run_e2e(c, st, device, args, sb)
    return out, c, sb


def store_ceilings(device, nbytes=8 << 30, reps=10):
    """HBM ceilings of the codec's store patterns, measured by the library's
    probe kernels over `nbytes` (far beyond L2): best and median GB/s of
    `reps` launches each, CUDA events on the launching stream."""
    st = torch.cuda.current_stream(device)
    dst = torch.empty(nbytes, dtype=torch.uint8, device=device)
    src = torch.empty(nbytes, dtype=torch.uint8, device=device)
    out = {}
    for name, mode, moved in (("store_v4", kv.KVP_PROBE_STORE, nbytes),
                              ("bulk_store_4k", kv.KVP_PROBE_BULK_STORE, nbytes),
                              ("copy_v4", kv.KVP_PROBE_COPY, 2 * nbytes)):
        for _ in range(3):
            kv.check(kv.kvp_bandwidth_probe(mode, dst, src, nbytes, st), name)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
        ev[0].record(st)
        for i in range(reps):
            kv.check(kv.kvp_bandwidth_probe(mode, dst, src, nbytes, st), name)
            ev[i + 1].record(st)
        torch.cuda.synchronize(device)
        ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(reps)]
        out[name] = {"GBps_best": round(moved / (min(ms) * 1e-3) / 1e9, 1),
                     "GBps_median": round(moved / (float(np.median(ms)) * 1e-3) / 1e9, 1)}
    del dst, src
    torch.cuda.empty_cache()
    out["bytes"] = int(nbytes)
    return out


def run_ours(args, rank, world, local_rank):
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    kv.load()
    k_mode = K_FORMATS[args.k_format]
    w = workload(args)
    res, c, sb = measure_workload(args.workload, w, args, rank, world, device, local_rank, k_mode)
    out = {
        "metric": METRIC, "value": res["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": "bf16", "data": "synthetic",
        "config": res["config"], "roofline": res["roofline"], "e2e": res["e2e"],
        "gpu_launches": res["gpu_launches"], "clocks": res["clocks"], "breakdown": res["breakdown"],
        "timing": {"blocks": res["blocks"], "steps_per_block": args.steps, "timed_s": res["timed_s"],
                   "value_from": "median block", "block_GBps": res["block_GBps"],
                   "phase_ms": "median over every timed step (ms_best: best)"},
    }
    ks, vs = c.k, c.v  # the headline inputs stay for the CPU baseline; the rest is freed
    host = {"oracle_inputs": (lambda i: (synth.bits16(ks[i]), synth.bits16(vs[i]))), "w": c.w}
    del c
    torch.cuda.empty_cache()
    extra = EXTRA_WORKLOADS if (args.extra_workloads and args.workload == DEFAULT_WORKLOAD and
                                not (args.agents or args.tokens or args.layers)) else []
    if extra:
        out["per_workload"] = {}
        for name in extra:
            r, c2, _ = measure_workload(name, dict(synth.WORKLOADS[name]), args, rank, world, device, local_rank,
                                        k_mode)
            out["per_workload"][name] = r
            del c2
            torch.cuda.empty_cache()
    if args.ceilings and rank == 0:
        out["store_ceilings"] = store_ceilings(device)
        dec = out["breakdown"]["decode"]["alg_GBps"]
        bulk = out["store_ceilings"]["bulk_store_4k"]["GBps_best"]
        out["roofline"]["frac_of_bulk_store_ceiling"] = round(dec / bulk, 4)
    return out, host, sb


def run_e2e(c, st, device, args, sb):
    """The same step end to end through the C ABI with host buffers: every
    step copies its K/V (and bitwidths) from pinned host memory to the device,
    runs the four calls, and reads the pool and the card (the two shareable
    artefacts) back to pinned host memory.  Steps are pipelined the way a
    serving loop would run them: step i+1's inputs are copied (one stream)
    while step i computes, and step i's results are read back (another
    stream) while step i+1 computes; device inputs and outputs are
    double-buffered and ordered with events."""
    L, H, d, T = c.w["L"], c.w["H"], c.w["d"], c.w["T"]
    steps = max(2, min(args.steps, 20))
    hK = torch.stack([t.cpu() for t in c.k]).pin_memory()
    hV = torch.stack([t.cpu() for t in c.v]).pin_memory()
    hbits = torch.from_numpy(c.bits_host).pin_memory()
    dK = [torch.empty_like(hK, device=device) for _ in range(2)]
    dV = [torch.empty_like(hV, device=device) for _ in range(2)]
    dbits = [torch.empty_like(hbits, device=device) for _ in range(2)]
    pools = [c.pool, torch.empty_like(c.pool)]
    cards = [c.card, torch.empty_like(c.card)]
    hpool = [torch.empty(c.pool_bytes, dtype=torch.uint8).pin_memory() for _ in range(2)]
    hcard = [torch.empty(c.card_bytes, dtype=torch.uint8).pin_memory() for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event()
    ev_in, ev_comp, ev_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for e in ev_comp + ev_out:
        e.record(st)

    def h2d(b):
        s_in.wait_event(ev_comp[b])               # the step that last used buffer b is done
        with torch.cuda.stream(s_in):
            dK[b].copy_(hK, non_blocking=True)
            dV[b].copy_(hV, non_blocking=True)
            dbits[b].copy_(hbits, non_blocking=True)
        ev_in[b].record(s_in)

    def compute(b):
        st.wait_event(ev_in[b])
        st.wait_event(ev_out[b])                  # buffer b's previous results have been read
        kl, vl = list(dK[b].unbind(0)), list(dV[b].unbind(0))
        kv.check(kv.kvpool_encode_ex(c.shape, c.k_mode, kl, vl, pools[b], c.pool_bytes, c.ws, c.ws_bytes, st),
                 "encode")
        kv.check(kv.kvpool_decode_into(pools[b], c.shape, 0, L, c.w["N"], c.caches_k, c.caches_v, st), "decode")
        kv.check(kv.cachecard_pack(c.shape, 0x8B, 0, dbits[b], kl, vl, cards[b], c.card_bytes, st), "pack")
        kv.check(kv.cachecard_unpack(cards[b], c.hdr, c.out_k, c.out_v, st), "unpack")
        ev_comp[b].record(st)

    def d2h(b):
        s_out.wait_event(ev_comp[b])
        with torch.cuda.stream(s_out):
            hpool[b].copy_(pools[b], non_blocking=True)
            hcard[b].copy_(cards[b], non_blocking=True)
        ev_out[b].record(s_out)

    def run(n):
        h2d(0)
        for i in range(n):
            b = i % 2
            compute(b)
            if i + 1 < n:
                h2d(1 - b)
            d2h(b)

    run(2)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    s_in.wait_event(e0)
    run(steps)
    st.wait_event(ev_out[(steps - 1) % 2])
    st.wait_event(ev_out[steps % 2])
    e1.record(st)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / steps
    for b in range(2):
        if kv.kvpool_status(pools[b], st) != kv.KVP_OK or kv.cachecard_status(cards[b], st) != kv.KVP_OK:
            raise RuntimeError("e2e status")
    # the read-back artefacts are the device's own bytes
    if not (torch.equal(hpool[0], pools[0].cpu()) and torch.equal(hcard[0], cards[0].cpu())):
        raise RuntimeError("e2e read-back mismatch")
    return {"value": round(sb["bf16_equiv"] / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "steps": steps, "pipelined": True,
            "h2d_bytes_per_step": int(hK.numel() * 2 + hV.numel() * 2 + hbits.numel()),
            "d2h_bytes_per_step": int(c.pool_bytes + c.card_bytes)}


# ----------------------------------------------------------------------------
# the fp64 oracle on the host: CPU baseline and reference arm
# ----------------------------------------------------------------------------

def oracle_step(layers_k, layers_v, bits, n_agents):
    """The whole step on the oracle for the given layers; returns seconds."""
    import oracle as O
    t0 = time.perf_counter()
    pool, _, _ = O.pool_encode(layers_k, layers_v)
    O.pool_decode_into(pool, 0, len(layers_k), n_agents)
    card, _, _ = O.card_pack(layers_k, layers_v, bits)
    O.card_unpack(card)
    return time.perf_counter() - t0


def oracle_sample(w, seed, budget_s, layer_fn):
    """Time the oracle on the first n layers of the workload, n grown until
    about budget_s of work (and at most 4 GB of decoded agent caches on the
    host), the n-layer step repeated until budget_s seconds have passed;
    layer_fn(i) gives layer i's (K, V) bf16 bits.  Returns (GB/s, cores,
    description, seconds)."""
    import oracle as O
    L, H, d, T, N = w["L"], w["H"], w["d"], w["T"], w["N"]
    bits = synth.card_bits(T, seed=seed).numpy()
    k0, v0 = layer_fn(0)
    t1 = oracle_step([k0], [v0], bits, N)
    raw1 = 2 * H * T * d * 2
    n_mem = max(1, int(4e9 // (N * raw1)))
    n = int(max(1, min(L, n_mem, budget_s / max(t1, 1e-3))))
    ks, vs = [k0], [v0]
    for i in range(1, n):
        k, v = layer_fn(i)
        ks.append(k)
        vs.append(v)
    t, reps = 0.0, 0
    while reps == 0 or (t < budget_s and reps < 200):
        t += oracle_step(ks, vs, bits, N)
        reps += 1
    gbs = raw1 * n * (N + 3) * reps / t / 1e9
    desc = ("layers 0..%d of %d, all %d agents, whole step (encode, fan-out decode, card pack, unpack), "
            "%d repetitions" % (n - 1, L, N, reps))
    return gbs, O.get_threads(), desc, t


def oracle_phases(w, seed, layer_fn, reps=3):
    """Each phase of the step on the oracle (encode, fan-out decode into N,
    card pack, card unpack) for layer 0 of the workload, on every host core
    (OpenMP) and on one thread: best and median of `reps` runs, as seconds
    and bf16-equivalent GB/s (encode and pack consume the layer's raw K/V,
    decode produces N copies of it, unpack one)."""
    import oracle as O
    H, d, T, N = w["H"], w["d"], w["T"], w["N"]
    raw1 = 2 * H * T * d * 2
    bits = synth.card_bits(T, seed=seed).numpy()
    k0, v0 = layer_fn(0)
    pool, _, _ = O.pool_encode([k0], [v0])
    card, _, _ = O.card_pack([k0], [v0], bits)
    calls = {"encode": (lambda: O.pool_encode([k0], [v0]), raw1),
             "decode": (lambda: O.pool_decode_into(pool, 0, 1, N), N * raw1),
             "pack": (lambda: O.card_pack([k0], [v0], bits), raw1),
             "unpack": (lambda: O.card_unpack(card), raw1)}
    all_cores = O.get_threads()
    out = {"sample": "layer 0 of %d (H=%d d=%d T=%d), %d agents; best and median of %d" % (w["L"], H, d, T, N, reps),
           "threads_all": all_cores}
    try:
        for label, th in (("all_cores", all_cores), ("one_thread", 1)):
            O.set_threads(th)
            res = {}
            for name, (fn, nbytes) in calls.items():
                secs = []
                for _ in range(reps):
                    t0 = time.perf_counter()
                    fn()
                    secs.append(time.perf_counter() - t0)
                best, med = min(secs), float(np.median(secs))
                res[name] = {"s_best": round(best, 4), "s_median": round(med, 4),
                             "GBps_best": round(nbytes / best / 1e9, 4), "GBps_median": round(nbytes / med / 1e9, 4)}
            out[label] = res
    finally:
        O.set_threads(all_cores)
    return out


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is a bounded sample (one
    layer of the workload) timed on the host cores."""
    import oracle as O
    w = workload(args)
    H, d, T, N = w["H"], w["d"], w["T"], w["N"]
    ks, vs = synth.kv_layers(1, H, T, d, seed=0, device="cpu")
    k1, v1 = [synth.bits16(ks[0])], [synth.bits16(vs[0])]
    bits = synth.card_bits(T, seed=0).numpy()
    for _ in range(args.warmup):
        oracle_step(k1, v1, bits, N)
    secs = [oracle_step(k1, v1, bits, N) for _ in range(args.steps)]
    raw1 = 2 * H * T * d * 2
    tot = sum(secs)
    value = raw1 * (N + 3) * args.steps / tot / 1e9
    sample = "one layer of %d per step (L=%d H=%d d=%d T=%d), all %d agents" % (w["L"], w["L"], H, d, T, N)
    return {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * tot / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "io_dtype": "bf16", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": args.workload, "layers": w["L"], "kv_heads": H, "head_dim": d, "tokens": T,
                   "agents": N, "card_bits": "iid {2,4,8,16} p={.25,.40,.25,.10}", "l2": "host (CPU)",
                   "parallelism": "single"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": O.get_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------

def run_attend(args):
    """Pool attention for one decode step of every agent over every layer
    (a forward pass's worth of attention over the shared context), straight
    from the compressed pool.  Llama-3-8B has 32 query heads over 8 KV heads;
    SmolLM2-1.7B 32 over 32."""
    torch.cuda.set_device(0)
    kv.load()
    w = workload(args)
    L, H, d, T, N = w["L"], w["H"], w["d"], w["T"], w["N"]
    nq = 32
    c = Codec(w, torch.device("cuda", 0), seed=0, outputs=False, k_mode=K_FORMATS[args.k_format])
    st = torch.cuda.current_stream()
    c.encode(st)
    kv.check(kv.kvpool_status(c.pool, st), "encode")
    g = torch.Generator(device="cuda").manual_seed(1)
    q = torch.randn(N, nq, d, generator=g, device="cuda").to(torch.bfloat16)
    out = torch.empty(N, nq, d, dtype=torch.float32, device="cuda")
    lse = torch.empty(N, nq, dtype=torch.float32, device="cuda")
    R = args.lora_rank
    wsb = (kv.kvpool_attend_lora_workspace_bytes(c.shape, N, nq, R) if R
           else kv.kvpool_attend_workspace_bytes(c.shape, N, nq))
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    scale = 1.0 / math.sqrt(d)
    if R:  # one shared low-rank cache and per-agent up-projections per layer
        lora = [synth.lora_inputs(T, H, d, N, R, seed=100 + l, device="cuda") for l in range(L)]

    def step():
        cur = torch.cuda.current_stream()
        for l in range(L):
            if R:
                kv.check(kv.kvpool_attend_lora(c.pool, c.shape, l, N, nq, q, scale, R, lora[l][0], lora[l][1], out,
                                               lse, ws, wsb, cur), "attend_lora")
            else:
                kv.check(kv.kvpool_attend(c.pool, c.shape, l, N, nq, q, scale, out, lse, ws, wsb, cur), "attend")
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    # the 2*L launches of a step are replayed from a CUDA graph, so the host's
    # per-call cost does not pace the GPU
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = kv.kvp_launch_count()
    e0.record(st)
    for _ in range(args.steps):
        graph.replay()
    e1.record(st)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    launches = 2 * L * args.steps  # replayed graph nodes (the counter sees only direct launches)
    pool_bytes = c.pool_bytes
    io = N * nq * d * 2 + N * nq * (d + 1) * 4
    flops = 2.0 * N * nq * T * (2 * d + R) * L + (2.0 * N * nq * R * d * L if R else 0.0)
    peak, kind = hbm_peak()
    gbs = (pool_bytes + L * io) / (ms * 1e-3) / 1e9
    # what the agents would otherwise read: N bf16 caches of every layer
    caches = N * 2 * L * H * T * d * 2
    return {
        "metric": "pool attention: agents' decode-step attention over all layers from the compressed pool",
        "value": round(ms * 1e3 / L, 2), "unit": "us per layer", "higher_is_better": False,
        "ms_per_step": round(ms, 4), "steps": args.steps, "warmup": args.warmup, "n_gpus": 1,
        "dtype": "bf16 q / int8 k / 3-bit v", "data": "synthetic",
        "config": {"workload": args.workload, "k_format": args.k_format, "lora_rank": R, "layers": L, "kv_heads": H,
                   "q_heads": nq, "head_dim": d,
                   "tokens": T, "agents": N},
        "pool_GBps": round(gbs, 1), "frac_of_measured_peak": round(gbs / peak, 4), "peak_kind": kind,
        "tensor_TFLOPs": round(flops / (ms * 1e-3) / 1e12, 2),
        "bytes_read_vs_bf16_caches": round((pool_bytes + L * io) / caches, 4),
        "gpu_launches": int(launches),
        "graph": True,
    }


def run_realign(args):
    """CacheCard unpack with every key moved to new positions (rotary
    realignment) against the plain unpack of the same card, on the
    Llama-3.1-8B-shaped card.  Card and outputs exceed L2, so repetitions
    need no flush."""
    torch.cuda.set_device(0)
    kv.load()
    if args.workload == DEFAULT_WORKLOAD:
        args.workload = "llama31-8b-cachecard-8k"
    w = workload(args)
    L, d = w["L"], w["d"]
    c = Codec(w, torch.device("cuda", 0), seed=0, outputs=True)
    st = torch.cuda.current_stream()
    c.pack(st)
    kv.check(kv.cachecard_status(c.card, st), "pack")
    hdr = kv.CardHeader()
    kv.check(kv.cachecard_read_header(c.card, hdr, st), "read_header")
    inv_freq = [1.0 / 500000.0 ** (i / d) for i in range(0, d, 2)]  # Llama-3 rotary base
    shift = 4096

    def realign():
        kv.check(kv.cachecard_unpack_at(c.card, hdr, hdr.pos_offset + shift, inv_freq, c.out_k, c.out_v, st),
                 "unpack_at")

    def plain():
        kv.check(kv.cachecard_unpack(c.card, hdr, c.out_k, c.out_v, st), "unpack")

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(args.steps):
            fn()
        e1.record(st)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    launches0 = kv.kvp_launch_count()
    clocks = ClockSampler(0)
    with clocks:
        ms = timed(realign)
    launches = kv.kvp_launch_count() - launches0 - args.warmup
    ms_plain = timed(plain)
    sb = step_bytes(w, c.pool_bytes, c.card_bytes)
    alg = sb["unpack_alg"]
    peak, kind = hbm_peak()
    gbs = alg / (ms * 1e-3) / 1e9
    return {
        "metric": "CacheCard unpack with keys re-aligned to new positions, GB/s (card read + bf16 K/V written)",
        "value": round(gbs, 1), "unit": "GB/s", "higher_is_better": True,
        "ms_per_step": round(ms, 4), "steps": args.steps, "warmup": args.warmup, "n_gpus": 1,
        "dtype": "f32 (bf16 out)", "data": "synthetic",
        "config": {"workload": args.workload, "layers": L, "kv_heads": w["H"], "head_dim": d, "tokens": w["T"],
                   "shift": shift, "rotary_base": 500000.0, "l2": "card and outputs exceed L2"},
        "roofline": {"kernel": "card_unpack_rope", "bound": "hbm", "achieved": round(gbs, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(gbs / peak, 4), "peak_kind": kind, "traffic": None},
        "plain_unpack": {"ms": round(ms_plain, 4), "GBps": round(alg / (ms_plain * 1e-3) / 1e9, 1)},
        "gpu_launches": int(launches),
        "clocks": clocks.summary(),
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--agents", type=int, default=0)
    ap.add_argument("--tokens", type=int, default=0)
    ap.add_argument("--layers", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-workloads", dest="extra_workloads", action="store_false",
                    help="time only the selected workload (default: also the 32K-token / 4-agent pool)")
    ap.add_argument("--no-ceilings", dest="ceilings", action="store_false",
                    help="skip the store / copy ceiling probes")
    ap.add_argument("--lora-rank", type=int, default=0, choices=[0, 16, 32],
                    help="attend mode: agents' values carry a LoRA term from a shared low-rank cache of this rank")
    ap.add_argument("--k-format", choices=sorted(K_FORMATS), default="per_tensor",
                    help="pool key format: one scale per layer tensor (default) or q8_0 blocks")
    ap.add_argument("--mode", choices=["step", "attend", "realign"], default="step",
                    help="step: the whole codec path (default); attend: attention over the pool; "
                         "realign: card unpack with keys moved to new positions")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.mode in ("attend", "realign"):
        if rank == 0:
            print(json.dumps(run_attend(args) if args.mode == "attend" else run_realign(args)), flush=True)
        return

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return

    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    out, host, sb = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if args.no_cpu_baseline:
            out["cpu_baseline"] = None
        else:
            gbs, cores, desc, secs = oracle_sample(host["w"], 0, args.cpu_budget, host["oracle_inputs"])
            out["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                   "sample": desc, "seconds": round(secs, 2),
                                   "nproc": os.cpu_count(),
                                   "per_phase": oracle_phases(host["w"], 0, host["oracle_inputs"])}
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
