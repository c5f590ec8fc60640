"""Benchmark: INT2 paged decode-attention step on one GB300.

Headline workload (the one the metric is quoted on): Qwen3-4B-shaped
single-layer decode, batch 1, 32 q / 8 KV heads, head_dim 128, context
100,000 tokens = 64 BF16 sink + 99,680 INT2 history + 256 BF16 recent, page 16
with a shuffled page table, group 128.  Inputs are seeded synthetic data
(``bit_kv_cache_12_gb300.synth``, the generator the parity tests use); the pool
is filled by the library's own append kernel.

The default run also measures, in the same JSON line under ``workloads``,
every other workload of the study (``bit_kv_cache_12_gb300.workloads``:
seeded device generators with the same shapes and value structure):
  tiny      batch 1, 8 q / 2 KV heads, context 1,024, page 16, group 128
  batch64   Qwen3-8B shape, batch 64, context U[8192, 32768] per sequence,
            page 16, 4 outlier channels per head x10, Haar R, group 128
  long16    Qwen3-32B shape, batch 16, 64 q / 8 KV heads (GQA 8), context
            131,072, page 32, 0.1% token positions x20, Haar R, group 128
  append    64 sequences x 8 KV heads x 4096 tokens evicted in one call,
            Student-t(4) K/V, separate R_k / R_v, clip 0.9, group 64, page 16
and the online step a server runs (``online_step``): one ``kv_append_step``
(the new token enters the recent ring and the oldest recent token is rotated,
quantized and packed into history) followed by the decode, at batch 1 (the
headline workload) and at batch 64.  ``--workload`` runs one of them alone.

One step = one ``kv_decode_attention`` call (whole batch, one layer), or one
``kv_append_quantize`` call for ``append``.  No step finds its data in L2:
  * the headline workload (60 MB) lives in a pool of 8 layers and step i
    decodes layer i mod 8, as a server decodes the layers of one token in
    turn: every step reads its own 60 MB of history, tiers and rotations from
    HBM, while the kernel's code and the page table (shared by the layers, as
    in a paged server) stay warm; the same decode after an L2 flush (256 MiB
    write + 256 MiB read outside the timed events) is reported beside it;
  * batch64, long16, append and the BF16 comparison pools are each larger
    than L2 (0.4 to 8.6 GB), so consecutive steps run back to back;
  * tiny (0.7 MB) is flushed before every step.
Timing: CUDA events on the launching stream around each step, device
synchronised before and after, max over ranks (one replica of the workload
per GPU).

``--impl reference`` times the CPU oracle on the headline workload instead:
W untimed and K timed whole decode steps on the host cores.

Prints exactly one JSON line on rank 0.
"""

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "INT2 paged decode-attention us/step (HBM GB/s, % of roofline) vs BF16 path"
APPEND_METRIC = "INT2 append (rotate, clip, quantize, pack) us/call (HBM GB/s, % of roofline)"
L2_FLUSH = "flushed between steps (256 MiB write + 256 MiB read outside the timed events)"
L2_LARGER = "inputs larger than L2: consecutive steps read disjoint data (no flush)"
L2_LAYERS = ("inputs larger than L2: the pool holds {n} layers of the workload ({mb:.0f} MB of history) "
             "and step i decodes layer i mod {n} (no flush; the page table is shared by all layers)")
HEADLINE_LAYERS = 8
WORKLOADS = ["all", "qwen3_4b", "tiny", "batch64", "long16", "append"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="all", choices=WORKLOADS)
    ap.add_argument("--ctx", type=int, default=100_000)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


# DRAM traffic of the decode kernel from an ncu capture (profiles/), valid only
# while the sources it was taken from are unchanged.
TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "decode_int2_traffic.json")
KERNEL_SOURCES = ["bit_kv_cache_12_gb300/csrc/kv_decode.cu", "bit_kv_cache_12_gb300/csrc/kv_device.cuh",
                  "bit_kv_cache_12_gb300/csrc/kv_internal.h"]


def kernel_source_digest():
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(workload):
    """dram read + write bytes per launch, or None if absent or stale."""
    try:
        rec = json.load(open(TRAFFIC_RECORD))
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != kernel_source_digest() or rec.get("workload") != workload:
        return None
    return int(rec["dram_bytes_read"]) + int(rec["dram_bytes_write"])


# --------------------------------------------------------------------------
# algorithmic bytes
# --------------------------------------------------------------------------

def algorithmic_bytes(c):
    """Bytes the method must move per decode step: 72 B (group 128) or 80 B
    (group 64) per history token per KV head, 512 B per BF16 tier token per KV
    head, R_k and R_v^T (128 KB per KV head), the page ids, q and out."""
    ng = 128 // c.GS
    per_hist_token = 32 + 32 + 8 * ng                 # K codes, V codes, K and V (s, z)
    hist = int(np.sum(c.hist_len)) * c.Hkv * per_hist_token
    tiers = int(np.sum(c.sink_len + c.rec_len)) * c.Hkv * 2 * 256
    rot = c.Hkv * 2 * 128 * 128 * 4
    pages = int(np.sum((c.hist_len + c.P - 1) // c.P))
    pt = pages * 4 * c.Hkv                            # each KV head reads its page ids
    qo = c.B * c.Hq * 128 * (2 + 4)
    return hist + tiers + rot + pt + qo, dict(hist=hist, tiers=tiers, rot=rot, page_table=pt, q_out=qo)


def bf16_bytes(c):
    lens = c.sink_len + c.hist_len + c.rec_len
    pages = int(np.sum((lens + c.P - 1) // c.P))
    return int(np.sum(lens)) * c.Hkv * 512 + pages * 4 * c.Hkv + c.B * c.Hq * 128 * 6


def append_bytes_flops(n_rows, GS):
    """Append: bf16 K and V rows in; codes and (s, z) out; x R for K and V."""
    alg = n_rows * 256 * 2 + n_rows * (32 + 4 * (128 // GS)) * 2
    flops = 2.0 * 128 * 128 * n_rows * 2
    return alg, flops


# --------------------------------------------------------------------------
# clocks
# --------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, dev):
        self.dev = dev
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.p is not None:
            self.p.terminate()
            try:
                out, _ = self.p.communicate(timeout=5)
            except Exception:
                self.p.kill()
                out = ""
            self.lines = [l for l in out.strip().splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(f[0])); mx = float(f[1])
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# the oracle on the host (CPU baseline and reference arm)
# --------------------------------------------------------------------------

def _oracle_step_fn(wl):
    from oracle import attention as att
    from oracle import kvquant as kq
    tb = kq.tile_bytes(wl.group_size) * (wl.page_size // 16)
    pages = np.zeros((wl.num_pages, wl.Hkv, tb), np.uint8)
    for b in range(wl.B):                      # packing is setup, not timed
        if wl.hist_len[b]:
            kq.pack_history_full(wl.hist_k[b], wl.hist_v[b], wl.Rk, wl.Rv, wl.clip_k, wl.clip_v,
                                 wl.page_table[b], wl.num_pages, wl.Hkv, wl.page_size,
                                 wl.group_size, pages)
    hist = lambda b, g: kq.read_history(pages, wl.page_table[b], int(wl.hist_len[b]), g,
                                        wl.page_size, wl.group_size)

    def step():
        att.decode_three_tier(wl.q, wl.Rk, wl.Rv, wl.sink_k, wl.sink_v, wl.sink_len, hist,
                              wl.hist_len, wl.rec_k, wl.rec_v, wl.rec_len, wl.rec_start, wl.Hkv,
                              wl.group_size, wl.scale)
    return step


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def cpu_baseline(wl, min_seconds=10.0, max_seconds=30.0):
    """Time the oracle on the host cores: whole decode steps (every KV head and
    query head, full context) repeated until about ``min_seconds`` of CPU work
    has run; the value is the mean time of one step."""
    step = _oracle_step_fn(wl)
    steps = 0
    t0 = time.perf_counter()
    while True:
        step()
        steps += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or dt + dt / steps > max_seconds:
            break
    return {"value": dt / steps * 1e6, "unit": "us", "cores": _cores(), "kind": "oracle",
            "sample": f"{steps} whole decode steps of the bench workload (all {wl.Hkv} KV heads, "
                      f"{wl.Hq} query heads, full context) with the numpy fp64 oracle "
                      f"(unpack, dequantize, three-tier attention) in {dt:.1f} s"}


_SINGLE_CORE_CHILD = r"""
import json, os, sys, time
sys.path.insert(0, sys.argv[1])
os.sched_setaffinity(0, {min(os.sched_getaffinity(0))})
import bench
from bit_kv_cache_12_gb300 import synth
wl = synth.qwen3_4b_decode(ctx=int(sys.argv[2]))
step = bench._oracle_step_fn(wl)
t0 = time.perf_counter(); step(); dt = time.perf_counter() - t0
print(json.dumps({"seconds": dt, "cores": len(os.sched_getaffinity(0))}))
"""


def cpu_baseline_single_core(ctx):
    """One whole oracle decode step of the headline workload on one host core
    (a child process pinned to one core, every thread pool of numpy's BLAS
    limited to one thread before numpy loads)."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = "1"
    try:
        r = subprocess.run([sys.executable, "-c", _SINGLE_CORE_CHILD, ROOT, str(ctx)], env=env,
                           capture_output=True, text=True, timeout=300)
        res = json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:                       # a host without the affinity call, a timeout
        return {"value": None, "error": str(e)[:200]}
    return {"value": res["seconds"] * 1e6, "unit": "us", "cores": res["cores"],
            "sample": "one whole decode step of the bench workload with the numpy fp64 oracle, "
                      "one process pinned to one core, BLAS threads 1"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    if args.workload not in ("all", "qwen3_4b"):
        print(json.dumps({"impl": "reference", "unavailable":
                          f"the oracle reference arm covers the headline workload only, not {args.workload}"}))
        return
    from bit_kv_cache_12_gb300 import synth
    wl = synth.qwen3_4b_decode(ctx=args.ctx)
    step = _oracle_step_fn(wl)
    for _ in range(args.warmup):
        step()
    ts = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        ts.append(time.perf_counter() - t0)
    us = float(np.mean(ts) * 1e6)
    cb = {"value": us, "unit": "us", "cores": _cores(), "kind": "oracle",
          "sample": f"{args.steps} timed whole decode steps (after {args.warmup} untimed) of the bench "
                    f"workload with the numpy fp64 oracle, {float(np.sum(ts)):.1f} s"}
    line = {"impl": "reference", "metric": METRIC, "value": us, "unit": "us",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "config": headline_config(wl), "cpu_baseline": cb,
            "e2e": {"value": us, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def headline_config(wl):
    hist_mb = HEADLINE_LAYERS * int(np.sum(wl.hist_len)) * wl.Hkv * (64 + 8 * 128 // wl.group_size) / 1e6
    return {"workload": wl.name, "batch": wl.B, "q_heads": wl.Hq, "kv_heads": wl.Hkv, "head_dim": 128,
            "context": int(wl.meta["ctx"][0]), "sink": int(wl.sink_len[0]),
            "int2_history": int(wl.hist_len[0]), "recent": int(wl.rec_len[0]),
            "page_size": wl.page_size, "group_size": wl.group_size,
            "l2": L2_LAYERS.format(n=HEADLINE_LAYERS, mb=hist_mb), "layers_in_pool": HEADLINE_LAYERS}


# --------------------------------------------------------------------------
# timing helpers
# --------------------------------------------------------------------------

def make_timer(torch, dev, stream, kvdist):
    # L2 flush between steps: write a 256 MiB buffer (evicts the pool), then
    # read another 256 MiB buffer so the write-back of the dirty lines happens
    # here and not inside the timed kernel.  Both are outside the events.
    flush_w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(64 << 20, dtype=torch.float32, device=dev)

    def flush():
        flush_w.zero_()
        flush_r.sum()

    def timed(fn, steps, warmup, flush_l2=False, per_step_pass=True):
        """fn(i) is step i; warm-up steps are -warmup .. -1.  With a flush each
        step is timed alone between its own events.  Without one the K steps run
        back to back between two region events, every step queued before the
        first starts (the mean is region / K: launch latency overlapped as in a
        serving loop); a second pass of the same steps with per-step events
        gives the distribution (skipped for steps that change the pool)."""
        t0 = time.perf_counter()
        for i in range(-warmup, 0):
            if flush_l2:
                flush()
            fn(i)
        host_per_step = (time.perf_counter() - t0) / max(warmup, 1)
        torch.cuda.synchronize()
        kvdist.barrier()

        def per_step():
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(steps)]
            for i, (s0, s1) in enumerate(ev):
                if flush_l2:
                    flush()
                s0.record(stream); fn(i); s1.record(stream)
            torch.cuda.synchronize()
            return np.array([s0.elapsed_time(s1) for s0, s1 in ev])   # ms

        if flush_l2:
            per = per_step()
            kvdist.barrier()
            return Timing(per, None)
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        # hold the stream (a bounded spin kernel) while the host queues every step
        hold_s = max(0.02, 3.0 * host_per_step * steps)
        torch.cuda._sleep(int(hold_s * SPIN_CYCLES_PER_S))
        r0.record(stream)
        t1 = time.perf_counter()
        for i in range(steps):
            fn(i)
        r1.record(stream)
        queued_s = time.perf_counter() - t1
        torch.cuda.synchronize()
        region = r0.elapsed_time(r1)
        per = per_step() if per_step_pass else None
        kvdist.barrier()
        if queued_s >= hold_s and per is not None:   # the GPU may have waited for the host
            return Timing(per, None)
        return Timing(per, region, steps, host_bound=queued_s >= hold_s)
    return timed


class Timing:
    """Per-step event times (ms) and, for back-to-back steps, the region time."""

    def __init__(self, per_step_ms, region_ms, steps=None, host_bound=False):
        self.per_step = per_step_ms
        self.region_ms = region_ms
        self.steps = steps if steps is not None else len(per_step_ms)
        self.host_bound = host_bound   # the region may include waits for the host

    @property
    def mean_ms(self):
        if self.region_ms is not None:
            return self.region_ms / self.steps
        return float(np.mean(self.per_step))


# cycles of torch's spin kernel per second (the SM clock is at most 2.07 GHz,
# so the hold lasts at least the time asked for)
SPIN_CYCLES_PER_S = 2.1e9


def peak_hbm():
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(peaks_path):
        return float(json.load(open(peaks_path))["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    return 6800.0, "fallback 6.8 TB/s"


def us_stats(t):
    out = {"us": float(t.mean_ms * 1e3)}
    if t.per_step is not None:
        out["us_p10_p50_p90"] = [float(np.percentile(t.per_step, p) * 1e3) for p in (10, 50, 90)]
    if t.region_ms is not None:
        out["timing"] = ("region of the back-to-back steps (all queued before the first starts) / steps; "
                         "percentiles from a second pass with per-step events")
        if t.per_step is not None:
            out["us_per_step_events"] = float(np.mean(t.per_step) * 1e3)
        if t.host_bound:
            out["timing"] += " (the host queued slower than the hold: an upper bound)"
    else:
        out["timing"] = "mean of per-step events"
    return out


class Env:
    """What every measurement needs: torch, device, stream, timer, ranks."""

    def __init__(self, args, torch, dev, rank, world, local, kvdist):
        self.args, self.torch, self.dev = args, torch, dev
        self.rank, self.world, self.local, self.kvdist = rank, world, local, kvdist
        self.stream = torch.cuda.current_stream()
        self.timed = make_timer(torch, dev, self.stream, kvdist)
        self.peak, self.peak_src = peak_hbm()

    def i32(self, a):
        return self.torch.as_tensor(np.ascontiguousarray(np.asarray(a, np.int32))).to(self.dev)

    def max_ranks(self, vals):
        return self.kvdist.max_over_ranks(vals, device=self.dev)


# --------------------------------------------------------------------------
# decode measurements
# --------------------------------------------------------------------------

class DecodeRig:
    """An INT2 pool holding case c in each of ``layers`` layers (the library's
    append), the decode step over a layer, and the BF16 pool of the same tokens
    with its decode step.  With ``spare_steps`` > 0 every sequence gets that
    many spare history positions (page ids past the case's pages, in the
    extended table ``pt_ext``) for per-step placement; the decode itself uses
    the case's own page table."""

    def __init__(self, env, c, spare_steps=0, layers=1):
        from bit_kv_cache_12_gb300 import native
        torch, dev, i32 = env.torch, env.dev, env.i32
        self.env, self.c, self.native = env, c, native
        B, Hq, Hkv = c.B, c.Hq, c.Hkv
        spare_pages = (spare_steps + c.P - 1) // c.P + 1 if spare_steps else 0
        pt_np = c.page_table
        if spare_pages:
            pages_per = (c.hist_len + c.P - 1) // c.P
            pt_np = np.full((B, c.page_table.shape[1] + spare_pages), -1, np.int32)
            for b in range(B):
                n = int(pages_per[b])
                pt_np[b, :n] = c.page_table[b, :n]
                pt_np[b, n:n + spare_pages] = c.num_pages + b * spare_pages + np.arange(spare_pages)
        self.pt_np, self.pt_ext_np = c.page_table, pt_np
        self.layers = layers
        self.small = False                    # set for workloads that fit in L2
        self.pool = native.KVPool(native.KV_POOL_INT2_3TIER, layers, Hq, Hkv, c.P,
                                  c.num_pages + B * spare_pages, B, group_size=c.GS)
        self.Rk = torch.as_tensor(c.Rk).to(dev); self.Rv = torch.as_tensor(c.Rv).to(dev)
        self.ck = torch.as_tensor(c.clip_k).to(dev); self.cv = torch.as_tensor(c.clip_v).to(dev)
        cu = np.zeros(B + 1, np.int32); cu[1:] = np.cumsum(c.hist_len)
        self.cu = cu
        self.pt = i32(c.page_table)
        self.pt_ext = i32(pt_np)
        for l in range(layers):
            native.kv_pool_set_rotation(self.pool.handle, l, self.Rk, self.Rv, self.ck, self.cv)
            sk, sv, rk, rv = self.pool.tier_views(l)
            sk[:B].copy_(c.sink_k); sv[:B].copy_(c.sink_v)
            rk[:B].copy_(c.rec_k); rv[:B].copy_(c.rec_v)
            native.kv_append_quantize(self.pool.handle, l, B, c.hist_k, c.hist_v, i32(cu), i32(np.zeros(B)),
                                      self.pt, c.page_table.shape[1], int(max(1, c.hist_len.max())))
        torch.cuda.synchronize()
        if self.pool.error():
            raise RuntimeError("device error while filling the pool")
        self.lens = [i32(c.sink_len), i32(c.hist_len), i32(c.rec_len), i32(c.rec_start)]
        self.max_hist = int(c.hist_len.max())
        self.ws_bytes = native.kv_decode_workspace_bytes(self.pool.handle, B, self.max_hist + spare_steps)
        self.ws = torch.zeros(self.ws_bytes // 4 + 4, dtype=torch.float32, device=dev)
        self.out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
        self.bpool = None

    def decode(self, i=0, q=None, lens=None, out=None, max_hist=None, extended=False):
        """The decode of step i: layer i mod layers."""
        c, n = self.c, self.native
        pt, pt_np = (self.pt_ext, self.pt_ext_np) if extended else (self.pt, self.pt_np)
        n.kv_decode_attention(self.pool.handle, i % self.layers, c.B, c.q if q is None else q,
                              *(self.lens if lens is None else lens), pt, pt_np.shape[1],
                              self.max_hist if max_hist is None else max_hist, c.scale,
                              self.out if out is None else out, self.ws, self.ws_bytes, self.env.stream)

    def build_bf16(self):
        """The BF16 pool with the same tokens in logical order (sink, history,
        ring from its start), shuffled pages."""
        torch, dev, c, n, i32 = self.env.torch, self.env.dev, self.c, self.native, self.env.i32
        B = c.B
        lens = (c.sink_len + c.hist_len + c.rec_len).astype(np.int32)
        bpages = (lens + c.P - 1) // c.P
        brng = np.random.default_rng(77)
        btotal = int(bpages.sum()) + 1
        bperm = brng.permutation(btotal).astype(np.int32)
        bpt_np = np.full((B, int(bpages.max())), -1, np.int32)
        o = 0
        for b in range(B):
            bpt_np[b, :bpages[b]] = bperm[o:o + bpages[b]]; o += bpages[b]
        self.bpool = n.KVPool(n.KV_POOL_BF16, 1, c.Hq, c.Hkv, c.P, btotal, B)
        W_cap = c.rec_k.shape[2]
        for b in range(B):
            s_, r_ = int(c.sink_len[b]), int(c.rec_len[b])
            ring = torch.as_tensor((c.rec_start[b] + np.arange(r_)) % W_cap, device=dev)
            kk = torch.cat([c.sink_k[b, :, :s_].transpose(0, 1), c.hist_k[self.cu[b]:self.cu[b + 1]],
                            c.rec_k[b][:, ring].transpose(0, 1)]).contiguous()
            vv = torch.cat([c.sink_v[b, :, :s_].transpose(0, 1), c.hist_v[self.cu[b]:self.cu[b + 1]],
                            c.rec_v[b][:, ring].transpose(0, 1)]).contiguous()
            n.kv_append_bf16(self.bpool.handle, 0, 1, kk, vv, i32([0, kk.shape[0]]), i32([0]),
                             i32(bpt_np[b:b + 1]), bpt_np.shape[1], kk.shape[0])
            del kk, vv
        torch.cuda.synchronize()
        self.bpt_np, self.bpt, self.blens = bpt_np, i32(bpt_np), i32(lens)
        self.bmax = int(lens.max())
        self.bws_bytes = n.kv_decode_workspace_bytes(self.bpool.handle, B, self.bmax)
        self.bws = torch.zeros(self.bws_bytes // 4 + 4, dtype=torch.float32, device=dev)
        self.bout = torch.empty_like(self.out)

    def decode_bf16(self, i=0):
        c = self.c
        self.native.kv_decode_attention_bf16(self.bpool.handle, 0, c.B, c.q, self.blens, self.bpt,
                                             self.bpt_np.shape[1], self.bmax, c.scale, self.bout,
                                             self.bws, self.bws_bytes, self.env.stream)

    def errors(self):
        return (self.pool.error() if self.pool else 0) or (self.bpool.error() if self.bpool else 0)

    def close(self):
        for p in (self.pool, self.bpool):
            if p is not None:
                p.close()
        self.pool = self.bpool = None


def decode_summary(env, rig, steps, warmup, with_bf16=True, flush_l2=False):
    """INT2 and BF16 decode of a rig: times, algorithmic bytes, GB/s, roofline.
    The INT2 steps are flushed only with flush_l2; the BF16 pools are larger
    than L2 except for the tiny workload, which is flushed too."""
    c = rig.c
    t = env.timed(rig.decode, steps, max(3, warmup), flush_l2=flush_l2)
    res = us_stats(t)
    res["us"] = env.max_ranks([res["us"]])[0]
    alg, parts = algorithmic_bytes(c)
    gbs = alg / (res["us"] * 1e-6) / 1e9
    res.update({"algorithmic_bytes": alg, "gbs": gbs, "frac_of_measured_peak": gbs / env.peak,
                "frac_of_8tbs": gbs / 8000.0})
    if with_bf16:
        rig.build_bf16()
        tb = env.timed(rig.decode_bf16, max(5, steps // 2), 3, flush_l2=flush_l2)
        us_b = env.max_ranks([float(tb.mean_ms * 1e3)])[0]
        bb = bf16_bytes(c)
        res["bf16_path"] = {"us": us_b, "bytes": bb, "gbs": bb / (us_b * 1e-6) / 1e9,
                            "frac_of_measured_peak": bb / (us_b * 1e-6) / 1e9 / env.peak,
                            "speedup_int2_vs_bf16": us_b / res["us"]}
    if rig.errors():
        raise RuntimeError(f"device error during the {c.name} steps")
    return res, t, parts


def online_step(env, rig, steps, warmup, decode_us):
    """The step a server runs: kv_append_step (every sequence's new token
    enters its recent ring; the full ring's oldest token is rotated, clipped,
    quantized and packed into history) then the decode reading the
    device-updated lengths.  Every timed step grows each history by one."""
    torch, c, n = env.torch, rig.c, rig.native
    gen = torch.Generator(device=env.dev)
    gen.manual_seed(11)
    new = torch.randn(2, c.B, c.Hkv, 128, generator=gen, device=env.dev).to(torch.bfloat16)
    L = rig.layers
    lens = [[env.i32(c.sink_len), env.i32(c.hist_len), env.i32(c.rec_len), env.i32(c.rec_start)]
            for _ in range(L)]                    # each layer's own lengths
    total = max(3, warmup) + steps
    max_hist = rig.max_hist + total

    def step(i):                                  # step i places into and decodes layer i mod L
        l = i % L
        n.kv_append_step(rig.pool.handle, l, c.B, new[0], new[1], *lens[l], rig.pt_ext,
                         rig.pt_ext_np.shape[1], env.stream)
        rig.decode(i, lens=lens[l], max_hist=max_hist, extended=True)
    t = env.timed(step, steps, max(3, warmup), flush_l2=(L == 1 and rig.small), per_step_pass=False)
    if rig.pool.error():
        raise RuntimeError("device error during the online steps")
    placed = sum(int((lens[l][1].cpu().numpy() - c.hist_len).sum()) for l in range(L))
    if placed != total * c.B:
        raise RuntimeError("the placement did not evict one token per step")
    us = env.max_ranks([float(t.mean_ms * 1e3)])[0]
    return {"us": us, "timing": us_stats(t)["timing"], "decode_alone_us": decode_us,
            "ratio_to_decode_alone": us / decode_us,
            "batch": c.B, "launches_per_step": 2,
            "what": "kv_append_step (new token into the recent ring, the oldest recent token rotated, "
                    "clipped, quantized and packed into INT2 history) then kv_decode_attention "
                    "over the updated cache, in one timed region"}


def run_headline(env, wl):
    """The headline workload: decode, BF16 path, end-to-end calls, several
    queries per sequence, the online step and the oracle on the host."""
    from bit_kv_cache_12_gb300 import workloads
    args, torch, dev = env.args, env.torch, env.dev
    c = workloads.case_from_synth(wl, torch, dev, "")
    rig = DecodeRig(env, c, spare_steps=max(3, args.warmup) + args.steps + 8, layers=HEADLINE_LAYERS)
    B, Hq = c.B, c.Hq
    with ClockSampler(env.local) as clk:
        res, t_int2, parts = decode_summary(env, rig, args.steps, args.warmup)
    us = res["us"]
    # the same decode (layer 0) after an L2 flush before every step: code, page
    # table and rotations are cold as well
    t_fl = env.timed(lambda i: rig.decode(0), args.steps, max(3, args.warmup), flush_l2=True)
    flushed = us_stats(t_fl)
    flushed["what"] = ("the same decode of layer 0 with " + L2_FLUSH + "; the kernel's code, the page "
                       "table and R come from HBM too")

    # ---- end to end through the C ABI with host buffers: the step's inputs
    # (q and the four length arrays) in one pinned staging buffer, one copy in,
    # the output copied back ----
    q_bytes = B * Hq * 128 * 2
    meta = np.stack([c.sink_len, c.hist_len, c.rec_len, c.rec_start]).astype(np.int32)
    stage_host = torch.empty(q_bytes + meta.nbytes, dtype=torch.uint8).pin_memory()
    stage_host[:q_bytes].copy_(torch.from_numpy(np.ascontiguousarray(c.q_np).view(np.uint8).reshape(-1)))
    stage_host[q_bytes:].copy_(torch.from_numpy(meta.view(np.uint8).reshape(-1)))
    stage_dev = torch.empty_like(stage_host, device=dev)
    q_dev = stage_dev[:q_bytes].view(torch.bfloat16).view(B, Hq, 128)
    meta_dev = stage_dev[q_bytes:].view(torch.int32).view(4, B)
    out_host = torch.empty((B, Hq, 128), dtype=torch.float32).pin_memory()

    def e2e_step(i):
        stage_dev.copy_(stage_host, non_blocking=True)
        rig.decode(i, q=q_dev, lens=[meta_dev[0], meta_dev[1], meta_dev[2], meta_dev[3]])
        out_host.copy_(rig.out, non_blocking=True)

    t_e2e = env.timed(e2e_step, args.steps, 3)
    h2d = stage_host.numel()
    d2h = out_host.numel() * 4

    # where the staged step's time goes: each copy alone, and the input copy
    # followed by the decode (every copy-engine <-> kernel hand-over on the
    # stream waits for the previous operation to finish)
    def h2d_then_decode(i):
        stage_dev.copy_(stage_host, non_blocking=True)
        rig.decode(i, q=q_dev, lens=[meta_dev[0], meta_dev[1], meta_dev[2], meta_dev[3]])

    t_parts = [env.timed(lambda i: stage_dev.copy_(stage_host, non_blocking=True), args.steps, 3,
                         per_step_pass=False),
               env.timed(lambda i: out_host.copy_(rig.out, non_blocking=True), args.steps, 3,
                         per_step_pass=False),
               env.timed(h2d_then_decode, args.steps, 3, per_step_pass=False)]

    # ---- the same call handed the pinned host buffers themselves ----
    q_host = stage_host[:q_bytes].view(torch.bfloat16).view(B, Hq, 128)
    meta_host = stage_host[q_bytes:].view(torch.int32).view(4, B)

    def mapped_step(i):
        rig.decode(i, q=q_host, lens=[meta_host[0], meta_host[1], meta_host[2], meta_host[3]], out=out_host)

    t_mapped = env.timed(mapped_step, args.steps, 3)

    # ---- several queries per sequence over the same cache ----
    from bit_kv_cache_12_gb300 import native
    TQ = 2
    qm = torch.randn(B, TQ, Hq, 128, generator=torch.Generator(device=dev).manual_seed(9),
                     device=dev).to(torch.bfloat16)
    m_ws_bytes = native.kv_decode_multi_workspace_bytes(rig.pool.handle, B, TQ, rig.max_hist)
    m_ws = torch.zeros(m_ws_bytes // 4 + 4, dtype=torch.float32, device=dev)
    m_out = torch.empty((B, TQ, Hq, 128), dtype=torch.float32, device=dev)
    m_lse = torch.empty((B, TQ, Hq), dtype=torch.float32, device=dev)

    def mstep(i):
        native.kv_decode_attention_multi(rig.pool.handle, i % rig.layers, B, TQ, qm, *rig.lens, rig.pt,
                                         rig.pt_np.shape[1], rig.max_hist, c.scale, m_out, m_lse, m_ws,
                                         m_ws_bytes, env.stream)

    t_multi = env.timed(mstep, max(5, args.steps // 2), 3) if TQ * (Hq // c.Hkv) <= 8 else None
    if rig.pool.error():
        raise RuntimeError("device error during the end-to-end and multi-query steps")
    us_e2e, us_mapped = env.max_ranks([float(t_e2e.mean_ms * 1e3), float(t_mapped.mean_ms * 1e3)])
    us_h2d, us_d2h, us_h2d_dec = env.max_ranks([float(t.mean_ms * 1e3) for t in t_parts])

    # ---- the online step at batch 1 (mutates the pool: last) ----
    online = online_step(env, rig, args.steps, args.warmup, us)
    rig.close()

    achieved = res["algorithmic_bytes"] / (us * 1e-6) / 1e9
    config = headline_config(wl)
    line = {
        "metric": METRIC, "value": us, "unit": "us", "n_gpus": env.world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "int2 codes, f16 MMA, f32 accumulate",
        "data": "synthetic (seeded; pool filled by kv_append_quantize)",
        "config": config,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": env.peak, "unit": "GB/s",
                     "frac": achieved / env.peak, "traffic": measured_traffic(c.name),
                     "peak_source": env.peak_src, "frac_of_8tbs": achieved / 8000.0,
                     "algorithmic_bytes": res["algorithmic_bytes"], "bytes_breakdown": parts},
        "us_p10_p50_p90": res["us_p10_p50_p90"],
        "flushed_l2": flushed,
        "bf16_path": res["bf16_path"],
        "online_step": {"batch1": online},
        "e2e": {"value": us_e2e, "unit": "us", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "what": "kv_decode_attention with host buffers: one pinned staging copy in (q and "
                        "the four length arrays), the output copied back, both inside the timed region",
                "breakdown_us": {"h2d_copy_alone": us_h2d, "d2h_copy_alone": us_d2h,
                                 "h2d_copy_then_decode": us_h2d_dec, "decode_alone": us,
                                 "what": "back-to-back steps of each part alone; the copies take about "
                                         "2 us each on their own, the rest of the staged step is the "
                                         "hand-over between the copy engine and the kernels on one "
                                         "stream (the decode cannot start its prologue under a copy)"}},
        "e2e_host_mapped": {"value": us_mapped, "unit": "us", "h2d_bytes_per_step": int(h2d),
                            "d2h_bytes_per_step": int(d2h),
                            "what": "the same call given the pinned host buffers directly: the kernel "
                                    "reads q and the lengths and writes the output across the CPU-GPU "
                                    "link inside the timed region (no staging copies)"},
        "multi_query": (None if t_multi is None else
                        {"us": float(t_multi.mean_ms * 1e3), "queries_per_sequence": TQ,
                         "what": "one kv_decode_attention_multi call over the same cache, "
                                 "output and log-sum-exp"}),
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    return line


def run_decode_workload(env, c, steps, warmup, online=False, small=False):
    """small: the workload fits in L2 and every step is flushed."""
    rig = DecodeRig(env, c, spare_steps=(max(3, warmup) + steps + 8) if online else 0)
    rig.small = small
    res, _, parts = decode_summary(env, rig, steps, warmup, flush_l2=small)
    c.config["l2"] = L2_FLUSH if small else L2_LARGER
    res["config"] = c.config
    res["bytes_breakdown"] = parts
    if online:
        res["online_step"] = online_step(env, rig, steps, warmup, res["us"])
    rig.close()
    return res


def run_append(env, steps, warmup):
    """64 sequences x 8 KV heads x 4096 tokens evicted in one kv_append_quantize."""
    from bit_kv_cache_12_gb300 import native, workloads
    torch, dev = env.torch, env.dev
    w = workloads.append_workload(torch, dev)
    n_seqs, Hkv, T, P, GS = w["n_seqs"], w["Hkv"], w["T"], w["page_size"], w["group_size"]
    k, v, Rk, Rv, ck, cv = w["k"], w["v"], w["Rk"], w["Rv"], w["clip_k"], w["clip_v"]
    pages_per, num_pages, pt_np = w["pages_per_seq"], w["num_pages"], w["page_table"]
    pool = native.KVPool(native.KV_POOL_INT2_3TIER, 1, Hkv, Hkv, P, num_pages, n_seqs, group_size=GS)
    native.kv_pool_set_rotation(pool.handle, 0, torch.as_tensor(Rk).to(dev), torch.as_tensor(Rv).to(dev),
                                torch.as_tensor(ck).to(dev), torch.as_tensor(cv).to(dev))
    cu = torch.as_tensor(np.arange(n_seqs + 1, dtype=np.int32) * T, device=dev)
    hs = torch.zeros(n_seqs, dtype=torch.int32, device=dev)
    pt = torch.as_tensor(pt_np, device=dev)

    def step(i):
        native.kv_append_quantize(pool.handle, 0, n_seqs, k, v, cu, hs, pt, pages_per, T, env.stream)

    t = env.timed(step, steps, max(3, warmup))
    if pool.error():
        raise RuntimeError("device error during the timed appends")
    pool.close()
    res = us_stats(t)
    res["us"] = env.max_ranks([res["us"]])[0]
    alg, flops = append_bytes_flops(n_seqs * T * Hkv, GS)
    gbs = alg / (res["us"] * 1e-6) / 1e9
    res.update({"algorithmic_bytes": alg, "gbs": gbs, "frac_of_measured_peak": gbs / env.peak,
                "frac_of_8tbs": gbs / 8000.0, "rotation_tflops": flops / (res["us"] * 1e-6) / 1e12,
                "launches": 2,
                "config": {"workload": "append_64x4096_h8_g64", "sequences": n_seqs, "tokens_per_seq": T,
                           "kv_heads": Hkv, "page_size": P, "group_size": GS, "l2": L2_LARGER}})
    return res


def main():
    args = parse()
    from bit_kv_cache_12_gb300 import dist as kvdist
    if args.impl == "reference":
        rank, world, _ = kvdist.rank_world()
        run_reference(args, rank, world)
        return
    # one replica of the workload per GPU (sequences are independent; no
    # collective on the data path), timings reduced by max over ranks
    rank, world, local = kvdist.init("nccl")
    import torch
    from bit_kv_cache_12_gb300 import synth, workloads
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    env = Env(args, torch, dev, rank, world, local, kvdist)
    w = args.workload
    if w in ("all", "qwen3_4b"):
        wl = synth.qwen3_4b_decode(ctx=args.ctx)
        line = run_headline(env, wl)
        if w == "all":
            sub_steps = min(args.steps, 20)
            nested = {}
            nested["tiny"] = run_decode_workload(env, workloads.case_from_synth(synth.tiny_decode(), torch,
                                                                                dev, L2_FLUSH),
                                                 sub_steps, args.warmup, small=True)
            c = workloads.batch64(torch, dev, L2_LARGER)
            nested["batch64"] = run_decode_workload(env, c, sub_steps, args.warmup, online=True)
            line["online_step"]["batch64"] = nested["batch64"].pop("online_step")
            del c
            torch.cuda.empty_cache()
            c = workloads.long16(torch, dev, L2_LARGER)
            nested["long16"] = run_decode_workload(env, c, sub_steps, args.warmup)
            del c
            torch.cuda.empty_cache()
            nested["append"] = run_append(env, sub_steps, args.warmup)
            line["workloads"] = nested
        if rank == 0:
            cb = None
            if not args.no_cpu_baseline:
                cb = cpu_baseline(wl)
                cb["single_core"] = cpu_baseline_single_core(args.ctx)
            line["cpu_baseline"] = cb
            print(json.dumps(line))
    else:
        if w == "append":
            res = run_append(env, args.steps, args.warmup)
            metric = APPEND_METRIC
        else:
            c = (workloads.case_from_synth(synth.tiny_decode(), torch, dev, L2_FLUSH) if w == "tiny"
                 else getattr(workloads, w)(torch, dev, L2_LARGER))
            res = run_decode_workload(env, c, args.steps, args.warmup, online=(w == "batch64"),
                                      small=(w == "tiny"))
            metric = METRIC
        if rank == 0:
            us = res.pop("us")
            line = {"metric": metric, "value": us, "unit": "us", "n_gpus": world, "steps": args.steps,
                    "warmup": max(3, args.warmup), "ms_per_step": us / 1e3, "higher_is_better": False,
                    "scaling": "weak", "vs_baseline": None, "data": "synthetic (seeded)",
                    "config": res.pop("config"),
                    "roofline": {"bound": "hbm", "achieved": res["gbs"], "peak": env.peak, "unit": "GB/s",
                                 "frac": res["frac_of_measured_peak"], "traffic": None,
                                 "peak_source": env.peak_src},
                    "gpu_launches": args.steps * (2 if w == "append" else 1), "cpu_baseline": None, **res}
            print(json.dumps(line))
    kvdist.shutdown()


if __name__ == "__main__":
    main()
