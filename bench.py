"""Benchmark: decode steps of paged attention on the Llama-3-8B-shaped layer.

One step = the whole hot path over one batch: kv_append of the 16 new K/V
rows and paged_decode_attention of 16 sequences x 32 query heads over
4097..4160 cached tokens (bf16 K/V, 8 KV heads, d 128, block size 16).
Steps cycle through the workload's 64 consecutive decode steps.  In the
device-timed loop the slot mapping of every step is computed on the host
before the timed region (it is host bookkeeping, not device work); the
end-to-end loop computes it on the host inside every step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pkv|reference]
    python bench.py --profile NAME      # a few calls of one kernel, for ncu

Prints one JSON line.  `value` is achieved GB/s of algorithmic bytes over
the whole step with inputs resident in HBM; the device is kept busy (a GPU
sleep) while the host queues the timed steps, so host launch latency is not
part of the device time.  `roofline` times the attention kernel alone in its
own loop of back-to-back launches.  `e2e` repeats the measurement through the
C ABI with host buffers: every step computes its slot mapping on the host,
copies its inputs from one pinned buffer to the device in one copy and its
output back, and the host reads the result (two steps in flight).  The
reference arm (--impl reference) times the fp64 CPU oracle.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_273_gb300 import workloads as W  # noqa: E402

WORKLOAD = "llama3_8b"
METRIC = "paged decode-attn achieved HBM GB/s (% of GB300 peak) and decode tokens/s/layer"
KERNEL_SOURCES = [os.path.join(ROOT, "paged_kv_cache_273_gb300", "csrc", f)
                  for f in ("decode_kernel.cuh", "device_common.cuh")]


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def eb(code):
    return {W.F32: 4, W.F16: 2, W.BF16: 2, W.I8: 1}[code]


def row_bytes(code, head_dim):
    """Bytes of one cached row (4-bit codes: two per byte)."""
    return head_dim // 2 if code == W.I4 else head_dim * eb(code)


def attention_bytes(wl: W.Workload, lens: np.ndarray) -> int:
    """Algorithmic bytes of one attention call: every cached K and V row once
    (+ int8 scales), q, the fp32 output, the block-table entries and lengths."""
    L = lens.astype(np.int64)
    kv = int(L.sum()) * wl.num_kv_heads * row_bytes(wl.kv_dtype, wl.head_dim) * 2
    if wl.kv_dtype in (W.I8, W.I4):
        kv += int(L.sum()) * wl.num_kv_heads * 2 * 2
    q = wl.batch * wl.num_q_heads * wl.head_dim * eb(wl.q_dtype)
    out = wl.batch * wl.num_q_heads * wl.head_dim * 4
    table = int((-(-L // wl.block_size)).sum()) * 4
    return kv + q + out + table + wl.batch * 4


def attention_bytes_window(wl: W.Workload, lens: np.ndarray, window: int) -> int:
    """attention_bytes for a sliding window: the last min(L, window) rows of each
    sequence and the table entries of the blocks that hold them."""
    L = lens.astype(np.int64)
    lo = np.maximum(L - window, 0)
    rows = int((L - lo).sum())
    kv = rows * wl.num_kv_heads * row_bytes(wl.kv_dtype, wl.head_dim) * 2
    if wl.kv_dtype in (W.I8, W.I4):
        kv += rows * wl.num_kv_heads * 2 * 2
    q = wl.batch * wl.num_q_heads * wl.head_dim * eb(wl.q_dtype)
    out = wl.batch * wl.num_q_heads * wl.head_dim * 4
    table = int((-(-L // wl.block_size) - lo // wl.block_size).sum()) * 4
    return kv + q + out + table + wl.batch * 4


def attention_bytes_unique(wl: W.Workload, lens: np.ndarray, tables: np.ndarray) -> int:
    """attention_bytes with every cached row counted once, however many
    sequences' tables point at its block (shared prefix blocks)."""
    L = lens.astype(np.int64)
    bs = wl.block_size
    rows_of = {}                        # block id -> rows read from it (the most any sequence reads)
    for b in range(len(L)):
        n = int(-(-L[b] // bs))
        for j in range(n):
            r = int(min(bs, L[b] - j * bs))
            bid = int(tables[b, j])
            if r > rows_of.get(bid, 0):
                rows_of[bid] = r
    rows = sum(rows_of.values())
    kv = rows * wl.num_kv_heads * row_bytes(wl.kv_dtype, wl.head_dim) * 2
    if wl.kv_dtype in (W.I8, W.I4):
        kv += rows * wl.num_kv_heads * 2 * 2
    return attention_bytes(wl, lens) - attention_kv_bytes(wl, lens) + kv


def attention_kv_bytes(wl: W.Workload, lens: np.ndarray) -> int:
    """The K/V (and scale) part of attention_bytes."""
    L = int(lens.astype(np.int64).sum())
    kv = L * wl.num_kv_heads * row_bytes(wl.kv_dtype, wl.head_dim) * 2
    if wl.kv_dtype in (W.I8, W.I4):
        kv += L * wl.num_kv_heads * 2 * 2
    return kv


def append_bytes(wl: W.Workload, ntok: int) -> int:
    """New K/V rows read and written once, plus the slot mapping."""
    row = wl.num_kv_heads * wl.head_dim
    return ntok * row * (eb(wl.src_dtype) + eb(wl.kv_dtype)) * 2 + ntok * 4


# ------------------------------------------------------------------ device timing helpers
SLEEP_CYCLES_PER_US = 2000        # the GPU sleep counts SM clocks (about 2 GHz)


def sleep_ahead(us: float) -> None:
    """Queue a GPU sleep of about `us` microseconds on the current stream, so
    that the host can queue the launches of a timed loop before the device
    reaches them (the loop's device time then holds no host launch latency)."""
    import torch
    torch.cuda._sleep(int(max(us, 10.0) * SLEEP_CYCLES_PER_US))


def timed_loop(stream, body, n: int, host_us: float, repeats: int = 3) -> list:
    """Device time (ms) of n back-to-back calls of body(i), `repeats` times,
    each timed by one event pair on `stream` after a sleep that covers the
    host's queueing of the n calls."""
    import torch
    out = []
    for _ in range(repeats):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sleep_ahead(min(n * host_us * 1.5 + 100.0, 500e3))
        e0.record(stream)
        for i in range(n):
            body(i)
        e1.record(stream)
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1))
    return out


def host_queue_us(body, n: int = 20) -> float:
    """Host microseconds to queue one call of body(i) (measured over n calls,
    then drained)."""
    import torch
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(n):
        body(i)
    t = (time.perf_counter() - t0) / n * 1e6
    torch.cuda.synchronize()
    return t


def traffic_record(name: str):
    """DRAM bytes per launch of a kernel from profiles/, while the kernel
    source it was taken on is unchanged; else None."""
    path = os.path.join(ROOT, "profiles", "decode_%s_traffic.json" % name)
    try:
        with open(path) as f:
            tr = json.load(f)
        if tr.get("kernel_source_sha256") == kernel_source_hash():
            return tr.get("traffic_bytes_per_launch")
    except Exception:
        pass
    return None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        # raw samples (the JSON line carries their summary); PKV_CLOCKS_DIR
        # keeps them somewhere else than the temporary directory
        out_dir = os.environ.get("PKV_CLOCKS_DIR", tempfile.gettempdir())
        self.path = os.path.join(out_dir, "clocks_bench_%d.csv" % os.getpid())

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ oracle (CPU) timing
def oracle_state(inp: W.Inputs):
    """Oracle cache for the workload (host), built by the oracle's own append."""
    from oracle import oracle as O
    wl = inp.workload
    shape = (inp.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
    raw = {W.F32: np.float32, W.F16: np.uint16, W.BF16: np.uint16}[wl.kv_dtype]
    ok, ov = np.zeros(shape, raw), np.zeros(shape, raw)
    B = wl.batch
    slots = O.slot_mapping(inp.block_tables, wl.block_size, np.zeros(B, np.int32), inp.prefix_lens)
    O.append(inp.hist_k, inp.hist_v, wl.kv_dtype, slots, wl.block_size, ok, ov)
    for s in range(wl.decode_steps):
        sl = O.slot_mapping(inp.block_tables, wl.block_size, (inp.prefix_lens + s).astype(np.int32),
                            np.ones(B, np.int32))
        O.append(inp.step_k[s], inp.step_v[s], wl.kv_dtype, sl, wl.block_size, ok, ov)
    return ok, ov


def time_oracle(inp: W.Inputs, ok, ov, seqs, step: int, budget_s: float, max_reps=None,
                nthreads: int = 0):
    """Run the oracle's decode attention for the given sequences until the
    budget is used; returns (seconds per call, algorithmic bytes per call).
    nthreads > 0 sets the oracle's thread count (it stays set)."""
    from oracle import oracle as O
    wl = inp.workload
    lens = inp.lens_after_step(step)[seqs]
    q = inp.step_q[step][seqs]
    tables = inp.block_tables[seqs]
    sub = dataclasses.replace(wl, batch=len(seqs))
    nbytes = attention_bytes(sub, lens)
    reps, t0 = 0, time.perf_counter()
    while True:
        O.paged_decode_attention(q, wl.q_dtype, ok, ov, wl.kv_dtype, tables, lens,
                                 1.0 / np.sqrt(wl.head_dim), nthreads=nthreads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_reps is not None and reps >= max_reps):
            break
    return el / reps, nbytes


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from oracle import oracle as O
    O.build()
    inp = W.make_inputs(WORKLOAD)
    wl = inp.workload
    ok, ov = oracle_state(inp)
    cores = O.max_threads()
    # per-step sample: the first n sequences of one decode step, n sized so
    # the whole run stays within about two minutes
    t_one, _ = time_oracle(inp, ok, ov, [0], 0, 0.0, max_reps=1)
    total_budget = 120.0
    per_step = total_budget / max(1, args.steps + args.warmup)
    n = int(max(1, min(wl.batch, per_step / max(t_one, 1e-6))))
    seqs = list(range(n))
    for w in range(args.warmup):
        time_oracle(inp, ok, ov, seqs, w % wl.decode_steps, 0.0, max_reps=1)
    total_t, total_b = 0.0, 0
    for k in range(args.steps):
        t, b = time_oracle(inp, ok, ov, seqs, k % wl.decode_steps, 0.0, max_reps=1)
        total_t += t
        total_b += b
    gbs = total_b / total_t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_t / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_block(wl, L2_NOTE),
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": "attention of %d of %d sequences per step (all KV heads), "
                                   "fp64 C oracle, OpenMP" % (n, wl.batch)},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# the timing rule this workload meets (the same config on both arms)
L2_NOTE = "inputs larger than L2 (268 MB of K/V read per step vs 126 MB L2), no flush"


def config_block(wl, l2_note):
    return {"workload": "%s: %d q / %d KV heads, head_dim %d, block_size %d, batch %d x %d..%d "
                        "tokens, %s K/V, %d decode steps" % (
                            wl.name, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size,
                            wl.batch, wl.len_lo + 1, wl.len_lo + wl.decode_steps,
                            {0: "fp32", 1: "fp16", 2: "bf16", 3: "int8"}[wl.kv_dtype],
                            wl.decode_steps),
            "kv_dtype": {0: "fp32", 1: "fp16", 2: "bf16", 3: "int8"}[wl.kv_dtype],
            "global_batch": wl.batch, "seq_len": wl.len_lo + wl.decode_steps,
            "l2": l2_note}


# ------------------------------------------------------------------ other workload shapes
def build_device_workload(name: str, dev):
    """Pool, caches and call arguments of a workload's decode attention, with
    the caches filled with random codes / values on the device (timing only;
    parity is the tests' job)."""
    import torch
    from paged_kv_cache_273_gb300 import pkv
    inp = W.make_inputs(name, values=False)
    wl = inp.workload
    B, Hq, Hkv, D, bs = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size
    pool = pkv.kv_block_pool_init(inp.num_blocks, bs, Hkv, D, wl.kv_dtype)
    kc, vc, ks, vs = pool.alloc_cache(dev)
    for c in (kc, vc):
        if c.dtype == torch.int8:
            c.random_(-127, 128)
        elif c.dtype == torch.uint8:
            c.random_(0, 256)
        else:
            c.normal_()
    for c in (ks, vs):
        if c is not None:
            c.uniform_(0.001, 0.05)
    qdt = {W.F16: torch.float16, W.BF16: torch.bfloat16, W.F32: torch.float32}[wl.q_dtype]
    q = torch.randn((B, Hq, D), device=dev).to(qdt)
    lens_h = inp.lens_after_step(0)
    lens = torch.from_numpy(lens_h).to(dev)
    tables = torch.from_numpy(inp.block_tables).to(dev)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    ws = pkv.alloc_workspace(pool, B, Hq, dev)
    max_len = int(lens_h.max())
    return dict(inp=inp, wl=wl, pool=pool, kc=kc, vc=vc, ks=ks, vs=vs, q=q, lens=lens,
                lens_h=lens_h, tables=tables, out=out, ws=ws, max_len=max_len)


def kernel_name(wl) -> str:
    return "paged_decode_kernel<%d,%d,%s>" % (wl.head_dim, wl.group,
                                               {W.F32: "f32", W.F16: "f16", W.BF16: "bf16",
                                                W.I8: "i8", W.I4: "i4"}[wl.kv_dtype])


def time_workload(name: str, dev, stream, peak: float, reps: int = 20) -> dict:
    """Attention on another workload's shape (lengths, tables, dtypes), on
    device-filled caches: `reps` back-to-back calls, three times, median."""
    from paged_kv_cache_273_gb300 import pkv
    d = build_device_workload(name, dev)
    wl = d["wl"]

    def call(i=0):
        pkv.paged_decode_attention(d["pool"], d["q"], d["kc"], d["vc"], d["tables"], d["lens"],
                                   1.0 / np.sqrt(wl.head_dim), d["out"], d["ws"], d["max_len"],
                                   d["ks"], d["vs"], stream=stream)

    for _ in range(3):
        call()
    host_us = host_queue_us(call, 5)
    ms = statistics.median(timed_loop(stream, call, reps, host_us))
    if pkv.pkv_check_error(d["pool"]) != pkv.PKV_OK:
        raise RuntimeError("device error timing workload %s" % name)
    us = ms / reps * 1e3
    nbytes = attention_bytes(wl, d["lens_h"])
    res = {"value": nbytes / (us / 1e6) / 1e9, "unit": "GB/s",
           "frac": nbytes / (us / 1e6) / 1e9 / peak, "launch_us": us,
           "bytes_per_launch": nbytes,
           "cache_mb": 2 * d["kc"].numel() * d["kc"].element_size() / 1e6,
           "kernel": kernel_name(wl), "traffic": traffic_record(name),
           "note": "back to back, %d calls, median of 3; logical bytes (a shared prefix row "
                   "counted once per sequence that reads it)" % reps}
    if wl.shared_prefix_tokens > 0:
        # a shared prefix: the line's GB/s counts every cached row once (the
        # shared blocks once for all sequences that read them), the logical
        # figure beside it
        ub = attention_bytes_unique(wl, d["lens_h"], d["inp"].block_tables)
        res["logical"] = {"value": res["value"], "unit": "GB/s", "frac": res["frac"],
                          "bytes_per_launch": nbytes,
                          "note": "a shared prefix row counted once per sequence that reads it"}
        res.update({"value": ub / (us / 1e6) / 1e9, "frac": ub / (us / 1e6) / 1e9 / peak,
                    "bytes_per_launch": ub,
                    "note": "back to back, %d calls, median of 3; unique bytes (every cached "
                            "row once: the shared prefix blocks once for all sequences that "
                            "share them)" % reps})
        # the same call with the shared prefix scored once per group
        g = pkv.kv_prefix_groups(d["inp"].block_tables, d["lens_h"], wl.block_size)
        gd = pkv.prefix_groups_to_device(g, dev)
        cws = pkv.alloc_cascade_workspace(d["pool"], wl.batch, wl.num_q_heads,
                                          g["max_prefix_len"], dev)

        def ccall(i=0):
            pkv.paged_decode_attention_cascade(d["pool"], d["q"], d["kc"], d["vc"], d["tables"],
                                               d["lens"], 1.0 / np.sqrt(wl.head_dim), d["out"],
                                               cws, d["max_len"], gd, stream=stream)

        for _ in range(3):
            ccall()
        cms = statistics.median(timed_loop(stream, ccall, reps, host_queue_us(ccall, 5)))
        if pkv.pkv_check_error(d["pool"]) != pkv.PKV_OK:
            raise RuntimeError("device error timing the cascade on %s" % name)
        cus = cms / reps * 1e3
        res["cascade"] = {
            "value": ub / (cus / 1e6) / 1e9, "unit": "GB/s", "frac": ub / (cus / 1e6) / 1e9 / peak,
            "launch_us": cus, "bytes_per_launch": ub, "logical_value": nbytes / (cus / 1e6) / 1e9,
            "groups": g["num_groups"], "max_group_size": g["max_group_size"],
            "prefix_tokens": g["max_prefix_len"],
            "note": "paged_decode_attention_cascade (prefix pass on tcgen05 + decode over each "
                    "sequence's own rows), unique bytes; %d calls back to back, median of 3; "
                    "logical_value counts shared rows once per sequence" % reps}
    del d
    return res


def time_shared_prompt(dev, stream, peak: float | None, B=64, P=8192, reps=10, profile=False):
    """Decode attention where all B sequences share a P-token prompt (one
    copy of its blocks) and add private suffixes of 64..1024 tokens (seeded),
    on the Llama-2-70B head shape (64 q / 8 KV heads, d 128, fp16, block
    size 16): the plain call, which scores the prompt once per sequence,
    against paged_decode_attention_cascade, which scores it once."""
    import torch
    from paged_kv_cache_273_gb300 import pkv
    rng = np.random.default_rng(12)
    Hq, Hkv, D, bs = 64, 8, 128, 16
    suf = rng.integers(64, 1025, size=B)
    lens = (P + suf).astype(np.int32)
    pb = P // bs
    nb = -(-lens // bs)
    NB = pb + int((nb - pb).sum()) + 16
    perm = rng.permutation(NB).astype(np.int32)
    tables = np.zeros((B, int(nb.max())), np.int32)
    tables[:, :pb] = perm[:pb]
    cur = pb
    for b in range(B):
        n = int(nb[b]) - pb
        tables[b, pb:pb + n] = perm[cur:cur + n]
        cur += n
    pool = pkv.kv_block_pool_init(NB, bs, Hkv, D, pkv.PKV_F16)
    kc, vc, _, _ = pool.alloc_cache(dev)
    kc.normal_()
    vc.normal_()
    q = torch.randn((B, Hq, D), device=dev).to(torch.float16)
    td = torch.from_numpy(tables).to(dev)
    ld = torch.from_numpy(lens).to(dev)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    ws = pkv.alloc_workspace(pool, B, Hq, dev)
    g = pkv.kv_prefix_groups(tables, lens, bs)
    gd = pkv.prefix_groups_to_device(g, dev)
    cws = pkv.alloc_cascade_workspace(pool, B, Hq, g["max_prefix_len"], dev)
    ml = int(lens.max())

    def plain(i=0):
        pkv.paged_decode_attention(pool, q, kc, vc, td, ld, D ** -0.5, out, ws, ml, stream=stream)

    def casc(i=0):
        pkv.paged_decode_attention_cascade(pool, q, kc, vc, td, ld, D ** -0.5, out, cws, ml, gd,
                                           stream=stream)

    if profile:            # a few calls for a profiler, no timing
        for _ in range(4):
            casc()
        torch.cuda.synchronize()
        if pkv.pkv_check_error(pool) != pkv.PKV_OK:
            raise RuntimeError("device error profiling the shared-prompt cascade")
        return None

    us = {}
    for name, f in (("plain", plain), ("cascade", casc)):
        for _ in range(3):
            f()
        us[name] = statistics.median(timed_loop(stream, f, reps, host_queue_us(f, 3))) / reps * 1e3
    if pkv.pkv_check_error(pool) != pkv.PKV_OK:
        raise RuntimeError("device error in the shared-prompt measurement")
    wl = W.Workload("shared_prompt", Hq, Hkv, D, bs, B, W.F16, W.F16, W.F16, 12, "fixed", P, P, 1)
    logical = attention_bytes(wl, lens)
    unique = attention_bytes_unique(wl, lens, tables)
    return {"config": "%d sequences sharing a %d-token prompt + 64..1024 own tokens, 64 q / 8 "
                      "KV heads, d 128, fp16, block size 16" % (B, P),
            "plain_us": us["plain"], "cascade_us": us["cascade"],
            "unique_bytes": unique, "logical_bytes": logical,
            "plain": {"value": unique / (us["plain"] / 1e6) / 1e9, "unit": "GB/s",
                      "frac": unique / (us["plain"] / 1e6) / 1e9 / peak},
            "cascade": {"value": unique / (us["cascade"] / 1e6) / 1e9, "unit": "GB/s",
                        "frac": unique / (us["cascade"] / 1e6) / 1e9 / peak},
            "note": "unique bytes (the prompt's rows once); %d calls back to back, median of 3"
                    % reps}


def time_prefill(dev, stream, peak_tflops: float, B=4, n=4096, reps=10) -> dict:
    """Causal prefill of B prompts of n tokens on the Llama-3-8B head shape
    (32 q / 8 KV heads, d 128, bf16, block size 16), device-filled caches."""
    import torch
    from paged_kv_cache_273_gb300 import pkv
    Hq, Hkv, D, bs = 32, 8, 128, 16
    nb = n // bs
    pool = pkv.kv_block_pool_init(B * nb, bs, Hkv, D, pkv.PKV_BF16)
    kc, vc, _, _ = pool.alloc_cache(dev)
    kc.normal_()
    vc.normal_()
    g = torch.Generator(device=dev)
    g.manual_seed(6)
    tables = torch.randperm(B * nb, device=dev, generator=g).to(torch.int32).reshape(B, nb)
    qs = torch.arange(0, (B + 1) * n, n, device=dev, dtype=torch.int32)
    lens = torch.full((B,), n, device=dev, dtype=torch.int32)
    q = torch.randn((B * n, Hq, D), device=dev).to(torch.bfloat16)
    out = torch.empty((B * n, Hq, D), device=dev, dtype=torch.float32)

    def call():
        pkv.paged_prefill_attention(pool, q, kc, vc, tables, qs, lens, D ** -0.5, out, n,
                                    stream=stream)

    for _ in range(3):
        call()
    host_us = host_queue_us(lambda i: call(), 3)
    ms = statistics.median(timed_loop(stream, lambda i: call(), reps, host_us))
    if pkv.pkv_check_error(pool) != pkv.PKV_OK:
        raise RuntimeError("device error in the prefill measurement")
    us = ms / reps * 1e3
    flops = 4.0 * B * (n * (n + 1) / 2) * D * Hq          # QK^T and PV over the causal half
    tf = flops / (us / 1e6) / 1e12
    return {"value": tf, "unit": "TFLOP/s", "bound": "tensor", "frac": tf / peak_tflops,
            "launch_us": us, "flops_per_launch": flops,
            "config": "%d prompts x %d tokens, causal, 32 q / 8 KV heads, d 128, bf16, "
                      "block size 16" % (B, n),
            "note": "tcgen05.mma kind::f16, bf16 in, fp32 accumulators in tensor memory; "
                    "%d calls back to back, median of 3; peak = measured bf16 burst" % reps}


# ------------------------------------------------------------------ ranks
def whole_job(units_per_rank: float, seconds: float, world: int, reduce_max=None):
    """Whole-job throughput of a weak-scaling run: every rank processed
    units_per_rank in `seconds` of its own; the job lasted as long as the
    slowest rank, and all ranks' units count.  reduce_max(x) returns the
    maximum of x over the ranks (needed when world > 1).  Returns (units per
    second, the job's seconds)."""
    t = reduce_max(seconds) if world > 1 else seconds
    return units_per_rank * world / t, t


def dist_max(dist, device):
    """reduce_max for whole_job over a torch.distributed process group (NCCL
    with a CUDA device, gloo with the CPU)."""
    def reduce_max(x: float) -> float:
        import torch
        tt = torch.tensor([x], dtype=torch.float64, device=device)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        return float(tt.item())
    return reduce_max


# ------------------------------------------------------------------ GPU arm
ROOF_LAUNCHES = 256       # attention launches per repeat of the roofline loop
E2E_MIN_STEPS = 256       # end-to-end steps timed whatever --steps is


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except Exception:
        return {}


def run_e2e(pool, inp, kc, vc, tables, ws, scale, max_len, steps, dev, stream, bytes_attn,
            bytes_app, world, rmax):
    """The metric end to end through the C ABI with host buffers.  Every
    step: the host computes the step's slot mapping into a pinned staging
    buffer that already holds the step's k, v, q and lengths; one
    paged_decode_step call copies the buffer to the device, appends, attends
    and copies the output back to pinned memory; the host reads it.  Two
    steps are in flight: the host prepares step k while the device runs step
    k - 1, and reads step k - 2's output."""
    import torch
    from paged_kv_cache_273_gb300 import pkv
    wl = inp.workload
    B, Hq, Hkv, D, bs = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size
    S = wl.decode_steps
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    nk, nq = B * Hkv * D * 2, B * Hq * D * 2
    o_k, o_v, o_q = 0, al(nk), 2 * al(nk)
    o_slot = o_q + al(nq)
    o_len = o_slot + al(B * 4)
    total = o_len + al(B * 4)
    stage = []
    for st in range(S):
        h = torch.empty(total, dtype=torch.uint8).pin_memory()
        hn = h.numpy()
        hn[o_k:o_k + nk] = inp.step_k[st].view(np.uint8).reshape(-1)
        hn[o_v:o_v + nk] = inp.step_v[st].view(np.uint8).reshape(-1)
        hn[o_q:o_q + nq] = inp.step_q[st].view(np.uint8).reshape(-1)
        hn[o_len:o_len + B * 4] = inp.lens_after_step(st).view(np.uint8)
        stage.append(h)
    d_stage = torch.empty(total, dtype=torch.uint8, device=dev)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    step = pkv.DecodeStep(pool, d_stage, pkv.StepLayout(o_k, o_v, o_q, o_slot, o_len),
                          torch.bfloat16, torch.bfloat16, Hq, kc, vc, tables, B, max_len, scale,
                          out, ws, stream=stream)
    h_out = [torch.empty((B, Hq, D), dtype=torch.float32).pin_memory() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    tables_h = np.ascontiguousarray(inp.block_tables, dtype=np.int32)
    start = np.zeros(B, np.int32)
    checksum = [0.0]

    def host_read(k):
        done[k % 2].synchronize()
        checksum[0] += float(h_out[k % 2].numpy()[0, 0, 0])

    def e2e_step(k):
        s = k % S
        if k >= 2:
            host_read(k - 2)
        start[:] = inp.prefix_lens + s
        pkv.kv_slot_mapping(tables_h, bs, start,
                            out=stage[s].numpy()[o_slot:o_slot + B * 4].view(np.int32))
        step(stage[s], h_out[k % 2])
        done[k % 2].record(stream)

    for w in range(4):
        e2e_step(w)
    host_read(2)
    host_read(3)
    torch.cuda.synchronize()
    n = max(E2E_MIN_STEPS, min(steps, 2000))
    t0 = time.perf_counter()
    for k in range(n):
        e2e_step(k)
    host_read(n - 2)
    host_read(n - 1)
    e2e_s = time.perf_counter() - t0
    e2e_bytes = sum(bytes_attn[k % S] + bytes_app for k in range(n))
    value = whole_job(e2e_bytes, e2e_s, world, rmax)[0] / 1e9
    return {"value": value, "unit": "GB/s", "h2d_bytes_per_step": total,
            "d2h_bytes_per_step": out.numel() * 4, "steps": n,
            "note": "paged_decode_step per step: one pinned-to-device copy of the step's inputs "
                    "(k, v, q, slot mapping, lengths), kv_append, attention writing its output "
                    "to pinned host memory, which the host reads; slot mapping on the host in "
                    "the step; two steps in flight"}


def run_gpu(args):
    import torch
    import torch.distributed as dist
    from paged_kv_cache_273_gb300 import pkv

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    # Weak scaling: every rank runs its own replica of the workload (the
    # sequences of a batch are independent; no data-path collective).
    inp = W.make_inputs(WORKLOAD)
    wl = inp.workload
    B, Hq, Hkv, D, bs = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size
    pool = pkv.kv_block_pool_init(inp.num_blocks, bs, Hkv, D, wl.kv_dtype)
    kc, vc, _, _ = pool.alloc_cache(dev)

    def dev16(raw):
        return torch.from_numpy(np.ascontiguousarray(raw).view(np.int16)).to(dev).view(
            torch.bfloat16)

    zeros = np.zeros(B, np.int32)
    hslots = pkv.kv_slot_mapping(inp.block_tables, bs, zeros, inp.prefix_lens)
    pkv.kv_append(pool, dev16(inp.hist_k), dev16(inp.hist_v), torch.from_numpy(hslots).to(dev),
                  kc, vc)
    tables = torch.from_numpy(inp.block_tables).to(dev)
    ws = pkv.alloc_workspace(pool, B, Hq, dev)
    S = wl.decode_steps
    step_slots = [pkv.kv_slot_mapping(inp.block_tables, bs, (inp.prefix_lens + s).astype(np.int32))
                  for s in range(S)]
    d_k = [dev16(inp.step_k[s]) for s in range(S)]
    d_v = [dev16(inp.step_v[s]) for s in range(S)]
    d_q = [dev16(inp.step_q[s]) for s in range(S)]
    d_slots = [torch.from_numpy(step_slots[s]).to(dev) for s in range(S)]
    lens_h = [inp.lens_after_step(s) for s in range(S)]
    d_lens = [torch.from_numpy(lens_h[s]).to(dev) for s in range(S)]
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    scale = 1.0 / np.sqrt(D)
    max_len = int(inp.final_lens.max())
    torch.cuda.synchronize()

    def attend(s):
        pkv.paged_decode_attention(pool, d_q[s], kc, vc, tables, d_lens[s], scale, out, ws,
                                   max_len, stream=stream)

    def step(k):
        s = k % S
        pkv.kv_append(pool, d_k[s], d_v[s], d_slots[s], kc, vc, stream=stream)
        attend(s)

    for w in range(args.warmup):
        step(w)
    torch.cuda.synchronize()
    if pkv.pkv_check_error(pool) != pkv.PKV_OK:
        raise RuntimeError("device error during warm-up")
    host_us = host_queue_us(step, 20)

    bytes_attn = [attention_bytes(wl, lens_h[s]) for s in range(S)]
    bytes_app = append_bytes(wl, B)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)                     # let the sampler take its first reading
    # The device sleeps while the host queues the first steps (up to the
    # launch queue's depth), so the timed region holds device work only.
    sleep_ahead(min(args.steps, 2000) * host_us * 1.5 + 100.0)
    t_start.record(stream)
    for k in range(args.steps):
        step(k)
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    status = pkv.pkv_check_error(pool)
    if status != pkv.PKV_OK:
        raise RuntimeError("device error in timed region: %s" % pkv.status_string(status))

    step_bytes = sum(bytes_attn[k % S] + bytes_app for k in range(args.steps))
    rmax = dist_max(dist, dev) if world > 1 else None
    rate, t_max_s = whole_job(step_bytes, total_ms / 1e3, world, rmax)
    t_max = t_max_s * 1e3
    value = rate / 1e9
    tok_s = B * args.steps * world / (t_max / 1e3)

    # ---- the attention kernel alone: ROOF_LAUNCHES back-to-back launches
    # over the 64 decode steps' inputs (same caches), one event pair around
    # the loop, three repeats, median
    attn_host_us = host_queue_us(attend, 20)
    roof_ms = timed_loop(stream, lambda i: attend(i % S), ROOF_LAUNCHES, attn_host_us)
    launch_ms = statistics.median(roof_ms) / ROOF_LAUNCHES
    roof_bytes = sum(bytes_attn[i % S] for i in range(ROOF_LAUNCHES)) / ROOF_LAUNCHES
    achieved = roof_bytes / (launch_ms / 1e3) / 1e9
    # secondary: the attention launch between appends, events around it (an
    # event between the two launches ends their overlap, so this is longer)
    pairs = []
    for k in range(64):
        s = k % S
        pkv.kv_append(pool, d_k[s], d_v[s], d_slots[s], kc, vc, stream=stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        attend(s)
        e1.record(stream)
        pairs.append((e0, e1))
    torch.cuda.synchronize()
    in_step_us = statistics.median(a.elapsed_time(b) for a, b in pairs) * 1e3
    if pkv.pkv_check_error(pool) != pkv.PKV_OK:
        raise RuntimeError("device error in the attention loop")

    # ---- end to end through the C ABI with host buffers
    e2e = run_e2e(pool, inp, kc, vc, tables, ws, scale, max_len, args.steps, dev, stream,
                  bytes_attn, bytes_app, world, rmax)

    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    peak_note = "measured"
    if not peak:
        peak, peak_note = 6800.0, "fallback"

    # ---- copy-on-write block copy (kv_block_copy) on a pool of the same shape:
    # 4096 block pairs per launch, 268 MB read + 268 MB written (twice L2)
    cow_blocks = 8192
    cow_pool = pkv.kv_block_pool_init(cow_blocks, bs, Hkv, D, wl.kv_dtype)
    ck, cv, _, _ = cow_pool.alloc_cache(dev)
    perm = np.random.default_rng(5).permutation(cow_blocks).astype(np.int32)
    c_src = torch.from_numpy(perm[:cow_blocks // 2].copy()).to(dev)
    c_dst = torch.from_numpy(perm[cow_blocks // 2:].copy()).to(dev)
    cow_bytes = (cow_blocks // 2) * Hkv * bs * D * eb(wl.kv_dtype) * 2 * 2   # K+V, read+write

    def cow(i=0):
        pkv.kv_block_copy(cow_pool, c_src, c_dst, ck, cv, stream=stream)

    for _ in range(3):
        cow()
    cow_reps = 50
    cow_ms = statistics.median(timed_loop(stream, cow, cow_reps, host_queue_us(cow, 5))) / cow_reps
    if pkv.pkv_check_error(cow_pool) != pkv.PKV_OK:
        raise RuntimeError("device error in the block-copy measurement")
    del ck, cv

    # ---- sliding-window attention (window 1024) on the same caches.  The
    # window's 67 MB fit in L2, so before every call L2 is refilled with
    # other data (a 256 MB read, clean lines: nothing to write back).  The
    # refills and calls run back to back with no host wait in between, and
    # the time of the refills alone is subtracted, so neither host launch
    # latency nor the refill counts.
    win = 1024
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev).fill_(1.0)
    win_bytes = attention_bytes_window(wl, lens_h[0], win)

    def win_call():
        pkv.paged_decode_attention_window(pool, d_q[0], kc, vc, tables, d_lens[0], scale, out, ws,
                                          max_len, win, stream=stream)

    for _ in range(3):
        flush.sum()
        win_call()
    win_reps = 50
    t_with = statistics.median(timed_loop(stream, lambda i: (flush.sum(), win_call()), win_reps,
                                          60.0))
    t_flush = statistics.median(timed_loop(stream, lambda i: flush.sum(), win_reps, 30.0))
    win_ms = (t_with - t_flush) / win_reps
    if pkv.pkv_check_error(pool) != pkv.PKV_OK:
        raise RuntimeError("device error in the sliding-window measurement")
    del flush

    # ---- the other workload shapes (rank 0 at N = 1 only; not part of `value`)
    others = {}
    if world == 1:
        for name in ("gpt2", "llama2_70b", "int8", "int4"):
            others[name] = time_workload(name, dev, stream, peak)
        others["shared_prompt_8k"] = time_shared_prompt(dev, stream, peak)
    bf16_peak = peaks.get("bf16_tflops") or 1900.0
    prefill = time_prefill(dev, stream, bf16_peak) if world == 1 else None

    if rank == 0:
        cpu = None
        if world == 1:
            from oracle import oracle as O
            O.build()
            ok, ov = oracle_state(inp)
            cores = O.max_threads()
            t_call, b_call = time_oracle(inp, ok, ov, list(range(B)), 0, 10.0, nthreads=cores)
            t1, b1 = time_oracle(inp, ok, ov, [0], 0, 8.0, nthreads=1)
            time_oracle(inp, ok, ov, [0], 0, 0.0, max_reps=1, nthreads=cores)   # restore
            cpu = {"value": b_call / t_call / 1e9, "unit": "GB/s", "cores": cores,
                   "kind": "oracle",
                   "sample": "full decode-step attention (16 seq x 32 heads, 4097 tokens) "
                             "repeated for ~10 s, fp64 C oracle, OpenMP",
                   "one_core": {"value": b1 / t1 / 1e9, "unit": "GB/s", "cores": 1,
                                "sample": "attention of 1 of the 16 sequences (32 heads, "
                                          "4097 tokens) repeated for ~8 s on one thread"}}
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": config_block(wl, L2_NOTE),
            "tokens_per_s_per_layer": tok_s,
            "pct_of_hbm_peak": 100.0 * value / peak,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic_record(WORKLOAD),
                         "kernel": kernel_name(wl), "launch_us": launch_ms * 1e3,
                         "launches_timed": ROOF_LAUNCHES, "repeats": len(roof_ms),
                         "bytes_per_launch": roof_bytes, "in_step_launch_us": in_step_us,
                         "peak_source": peak_note,
                         "note": "%d back-to-back launches over the 64 decode steps' inputs, "
                                 "one event pair, median of %d; in_step_launch_us: events "
                                 "around the launch between appends (median of 64)"
                                 % (ROOF_LAUNCHES, len(roof_ms))},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": 2 * args.steps,
            "extra_kernels": {
                "kv_block_copy": {"value": cow_bytes / (cow_ms / 1e3) / 1e9, "unit": "GB/s",
                                  "frac": cow_bytes / (cow_ms / 1e3) / 1e9 / peak,
                                  "launch_us": cow_ms * 1e3, "bytes_per_launch": cow_bytes,
                                  "pairs": cow_blocks // 2,
                                  "note": "copy-on-write block copy, bf16 blocks of the "
                                          "same shape, read + write bytes"},
                "paged_decode_attention_window": {
                    "value": win_bytes / (win_ms / 1e3) / 1e9, "unit": "GB/s",
                    "frac": win_bytes / (win_ms / 1e3) / 1e9 / peak, "launch_us": win_ms * 1e3,
                    "bytes_per_launch": win_bytes, "window": win,
                    "note": "same workload, last 1024 rows of each sequence; L2 refilled "
                            "by a 256 MB read before each call, 50 calls back to back, "
                            "the reads' own time subtracted (median of 3)"}},
            "other_workloads": others,
            "prefill": prefill,
            "clocks": clk,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_profile(name: str) -> int:
    """A few calls of one kernel on its timing workload, for ncu captures
    (no timing, no JSON line): NAME is a workload (its decode attention) or
    'prefill'."""
    import torch
    from paged_kv_cache_273_gb300 import pkv
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    if name == "prefill":
        time_prefill(dev, stream, 1900.0, reps=1)
        return 0
    if name == "llama2_70b_cascade":
        d = build_device_workload("llama2_70b", dev)
        wl = d["wl"]
        g = pkv.kv_prefix_groups(d["inp"].block_tables, d["lens_h"], wl.block_size)
        gd = pkv.prefix_groups_to_device(g, dev)
        cws = pkv.alloc_cascade_workspace(d["pool"], wl.batch, wl.num_q_heads,
                                          g["max_prefix_len"], dev)
        for _ in range(4):
            pkv.paged_decode_attention_cascade(d["pool"], d["q"], d["kc"], d["vc"], d["tables"],
                                               d["lens"], 1.0 / np.sqrt(wl.head_dim), d["out"],
                                               cws, d["max_len"], gd, stream=stream)
        torch.cuda.synchronize()
        if pkv.pkv_check_error(d["pool"]) != pkv.PKV_OK:
            raise RuntimeError("device error profiling the cascade")
        print("profiled the cascade on llama2_70b: 4 calls")
        return 0
    if name == "shared_prompt_cascade":
        time_shared_prompt(dev, stream, None, profile=True)
        print("profiled the cascade on the shared 8192-token prompt: 4 calls")
        return 0
    d = build_device_workload(name, dev)
    wl = d["wl"]
    for _ in range(4):
        pkv.paged_decode_attention(d["pool"], d["q"], d["kc"], d["vc"], d["tables"], d["lens"],
                                   1.0 / np.sqrt(wl.head_dim), d["out"], d["ws"], d["max_len"],
                                   d["ks"], d["vs"], stream=stream)
    torch.cuda.synchronize()
    if pkv.pkv_check_error(d["pool"]) != pkv.PKV_OK:
        raise RuntimeError("device error profiling %s" % name)
    print("profiled %s: 4 calls of %s" % (name, kernel_name(wl)))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--profile", default=None,
                    choices=["gpt2", "llama3_8b", "llama2_70b", "int8", "int4", "prefill",
                             "llama2_70b_cascade", "shared_prompt_cascade"])
    args = ap.parse_args()
    if args.profile:
        return run_profile(args.profile)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
