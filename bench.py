"""Benchmark: INT2 paged decode-attention step on one GB300.

Default workload (the one the headline number is quoted on): Qwen3-4B-shaped
single-layer decode, batch 1, 32 q / 8 KV heads, head_dim 128, context
100,000 tokens = 64 BF16 sink + 99,680 INT2 history + 256 BF16 recent, page 16
with a shuffled page table, group 128.  Inputs are seeded synthetic data
(``bit_kv_cache_12_gb300.synth``, the generator the parity tests use); the pool
is filled by the library's own append kernel.

``--workload`` selects the other workloads of the same study, generated on the
device from seeded torch generators with the same shapes and value structure:
  batch64   Qwen3-8B shape, batch 64, context U[8192, 32768] per sequence,
            page 16, 4 outlier channels per head x10, Haar R, group 128
  long16    Qwen3-32B shape, batch 16, 64 q / 8 KV heads (GQA 8), context
            131,072, page 32, 0.1% token positions x20, Haar R, group 128
  append    64 sequences x 8 KV heads x 4096 tokens evicted in one call,
            Student-t(4) K/V, separate R_k / R_v, clip 0.9, group 64, page 16

One step = one ``kv_decode_attention`` call (whole batch, one layer), or one
``kv_append_quantize`` call for ``append``.  Every timed step is preceded by
an L2 flush outside the timed events: a 256 MiB device write, then a 256 MiB
read so the dirty lines are written back before the step starts.  Timing:
CUDA events on the launching stream around each step, device synchronised
before and after, max over ranks (one replica of the workload per GPU).

``--impl reference`` times the CPU oracle on the default workload instead:
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
L2_NOTE = "flushed between steps (256 MiB write + 256 MiB read outside the timed events)"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen3_4b", choices=["qwen3_4b", "batch64", "long16", "append"])
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


def run_reference(args, rank, world):
    if rank != 0:
        return
    if args.workload != "qwen3_4b":
        print(json.dumps({"impl": "reference", "unavailable":
                          f"the oracle reference arm covers the default workload only, not {args.workload}"}))
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
            "data": "synthetic (seeded)", "config": config_of_wl(wl), "cpu_baseline": cb,
            "e2e": {"value": us, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def config_of_wl(wl):
    return {"workload": wl.name, "batch": wl.B, "q_heads": wl.Hq, "kv_heads": wl.Hkv, "head_dim": 128,
            "context": int(wl.meta["ctx"][0]), "sink": int(wl.sink_len[0]),
            "int2_history": int(wl.hist_len[0]), "recent": int(wl.rec_len[0]),
            "page_size": wl.page_size, "group_size": wl.group_size, "l2": L2_NOTE}


# --------------------------------------------------------------------------
# decode workloads resident on the device
# --------------------------------------------------------------------------

class Case:
    """A three-tier decode workload whose K/V live on the device."""


def case_from_synth(wl, torch, dev):
    def bf16(u16):
        return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).to(dev)
    c = Case()
    c.name, c.B, c.Hq, c.Hkv, c.P, c.GS, c.scale = (wl.name, wl.B, wl.Hq, wl.Hkv, wl.page_size,
                                                    wl.group_size, wl.scale)
    c.sink_len, c.hist_len = wl.sink_len.astype(np.int32), wl.hist_len.astype(np.int32)
    c.rec_len, c.rec_start = wl.rec_len.astype(np.int32), wl.rec_start.astype(np.int32)
    c.page_table, c.num_pages = wl.page_table, wl.num_pages
    c.Rk, c.Rv, c.clip_k, c.clip_v = wl.Rk, wl.Rv, wl.clip_k, wl.clip_v
    c.q_np = wl.q
    c.q = bf16(wl.q)
    c.hist_k = bf16(np.concatenate(wl.hist_k)); c.hist_v = bf16(np.concatenate(wl.hist_v))
    c.sink_k, c.sink_v = bf16(wl.sink_k), bf16(wl.sink_v)
    c.rec_k, c.rec_v = bf16(wl.rec_k), bf16(wl.rec_v)
    c.config = config_of_wl(wl)
    return c


def _haar(rng, n):
    from bit_kv_cache_12_gb300 import synth
    return np.stack([synth.haar_orthogonal(rng) for _ in range(n)]).astype(np.float32)


def _clip_from(x, R, ratio, torch):
    """ratio x per-channel absmax of the rotated rows x [T][Hkv][128] (device)."""
    Hkv = x.shape[1]
    out = np.zeros((Hkv, 128), np.float32)
    for g in range(Hkv):
        Rg = torch.as_tensor(R[g], device=x.device)
        m = torch.zeros(128, device=x.device)
        for s in range(0, x.shape[0], 1 << 18):
            m = torch.maximum(m, (x[s:s + (1 << 18), g].float() @ Rg).abs().amax(dim=0))
        out[g] = ratio * m.cpu().numpy()
    return out


def case_generated(kind, torch, dev):
    """batch64 / long16 workloads generated on the device (seeded)."""
    S_CAP, W_CAP = 64, 256
    if kind == "batch64":
        seed, B, Hq, Hkv, P = 4, 64, 32, 8, 16
        rng = np.random.default_rng(seed)
        ctx = rng.integers(8192, 32768 + 1, size=B)
        name = "qwen3_8b_b64_h32x8_ctx8192-32768"
    else:
        seed, B, Hq, Hkv, P = 5, 16, 64, 8, 32
        rng = np.random.default_rng(seed)
        ctx = np.full(B, 131072)
        name = "qwen3_32b_b16_h64x8_ctx131072"
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    c = Case()
    c.name, c.B, c.Hq, c.Hkv, c.P, c.GS, c.scale = name, B, Hq, Hkv, P, 128, 1.0 / np.sqrt(128.0)
    c.sink_len = np.minimum(ctx, S_CAP).astype(np.int32)
    c.rec_len = np.minimum(ctx - c.sink_len, W_CAP).astype(np.int32)
    c.hist_len = (ctx - c.sink_len - c.rec_len).astype(np.int32)
    c.rec_start = rng.integers(0, W_CAP, size=B).astype(np.int32)
    pages_per = (c.hist_len + P - 1) // P
    c.num_pages = int(pages_per.sum()) + 1
    perm = rng.permutation(c.num_pages).astype(np.int32)
    c.page_table = np.full((B, int(pages_per.max())), -1, np.int32)
    o = 0
    for b in range(B):
        c.page_table[b, :pages_per[b]] = perm[o:o + pages_per[b]]; o += pages_per[b]
    T = int(c.hist_len.sum())
    scale = torch.ones(Hkv, 128, device=dev)
    if kind == "batch64":                      # 4 outlier channels per KV head, x10
        for g in range(Hkv):
            scale[g, torch.as_tensor(rng.choice(128, 4, replace=False), device=dev)] = 10.0

    def kv(n_rows):
        return (torch.randn(n_rows, Hkv, 128, generator=gen, device=dev) * scale).to(torch.bfloat16)
    c.hist_k, c.hist_v = kv(T), kv(T)
    c.sink_k = kv(B * S_CAP).view(B, S_CAP, Hkv, 128).transpose(1, 2).contiguous()
    c.sink_v = kv(B * S_CAP).view(B, S_CAP, Hkv, 128).transpose(1, 2).contiguous()
    c.rec_k = kv(B * W_CAP).view(B, W_CAP, Hkv, 128).transpose(1, 2).contiguous()
    c.rec_v = kv(B * W_CAP).view(B, W_CAP, Hkv, 128).transpose(1, 2).contiguous()
    if kind == "long16":                       # 0.1% token positions per sequence, all heads, x20
        n_out = int(round(0.001 * 131072))
        cu = np.concatenate([[0], np.cumsum(c.hist_len)])
        for b in range(B):
            pos = rng.choice(int(c.hist_len[b]), n_out, replace=False) + cu[b]
            idx = torch.as_tensor(pos, device=dev)
            c.hist_k[idx] = (c.hist_k[idx].float() * 20).to(torch.bfloat16)
            c.hist_v[idx] = (c.hist_v[idx].float() * 20).to(torch.bfloat16)
    c.Rk, c.Rv = _haar(rng, Hkv), _haar(rng, Hkv)
    c.clip_k = _clip_from(c.hist_k, c.Rk, 0.95, torch)
    c.clip_v = _clip_from(c.hist_v, c.Rv, 0.95, torch)
    c.q = torch.randn(B, Hq, 128, generator=gen, device=dev).to(torch.bfloat16)
    c.q_np = c.q.view(torch.int16).cpu().numpy().view(np.uint16)
    c.config = {"workload": name, "batch": B, "q_heads": Hq, "kv_heads": Hkv, "head_dim": 128,
                "context": [int(ctx.min()), int(ctx.max())], "context_mean": float(ctx.mean()),
                "sink": S_CAP, "recent": W_CAP, "int2_history_tokens": T, "page_size": P,
                "group_size": 128, "l2": L2_NOTE,
                "generation": "seeded torch generator on the device"}
    return c


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

    def timed(fn, steps, warmup):
        for _ in range(warmup):
            flush(); fn()
        torch.cuda.synchronize()
        kvdist.barrier()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for s0, s1 in ev:
            flush()
            s0.record(stream); fn(); s1.record(stream)
        torch.cuda.synchronize()
        kvdist.barrier()
        return np.array([s0.elapsed_time(s1) for s0, s1 in ev])   # ms
    return timed


def peak_hbm():
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(peaks_path):
        return float(json.load(open(peaks_path))["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    return 6800.0, "fallback 6.8 TB/s"


# --------------------------------------------------------------------------
# decode benchmark
# --------------------------------------------------------------------------

def run_decode(args, c, wl, torch, dev, rank, world, local, kvdist):
    from bit_kv_cache_12_gb300 import native
    B, Hq, Hkv = c.B, c.Hq, c.Hkv
    stream = torch.cuda.current_stream()
    timed = make_timer(torch, dev, stream, kvdist)

    def i32(a):
        return torch.as_tensor(np.ascontiguousarray(np.asarray(a, np.int32))).to(dev)

    # ---- INT2 pool filled by the library's append kernel ----
    pool = native.KVPool(native.KV_POOL_INT2_3TIER, 1, Hq, Hkv, c.P, c.num_pages, B, group_size=c.GS)
    Rk = torch.as_tensor(c.Rk).to(dev); Rv = torch.as_tensor(c.Rv).to(dev)
    ck = torch.as_tensor(c.clip_k).to(dev); cv = torch.as_tensor(c.clip_v).to(dev)
    native.kv_pool_set_rotation(pool.handle, 0, Rk, Rv, ck, cv)
    sk, sv, rk, rv = pool.tier_views(0)
    sk[:B].copy_(c.sink_k); sv[:B].copy_(c.sink_v)
    rk[:B].copy_(c.rec_k); rv[:B].copy_(c.rec_v)
    cu = np.zeros(B + 1, np.int32); cu[1:] = np.cumsum(c.hist_len)
    pt = i32(c.page_table)
    native.kv_append_quantize(pool.handle, 0, B, c.hist_k, c.hist_v, i32(cu), i32(np.zeros(B)), pt,
                              c.page_table.shape[1], int(c.hist_len.max()))
    torch.cuda.synchronize()
    if pool.error():
        raise RuntimeError("device error while filling the pool")

    q = c.q
    sink_len, hist_len = i32(c.sink_len), i32(c.hist_len)
    rec_len, rec_start = i32(c.rec_len), i32(c.rec_start)
    max_hist = int(c.hist_len.max())
    ws_bytes = native.kv_decode_workspace_bytes(pool.handle, B, max_hist)
    ws = torch.zeros(ws_bytes // 4 + 4, dtype=torch.float32, device=dev)
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)

    def step():
        native.kv_decode_attention(pool.handle, 0, B, q, sink_len, hist_len, rec_len, rec_start, pt,
                                   c.page_table.shape[1], max_hist, c.scale, out, ws, ws_bytes, stream)

    # ---- BF16 pool with the same tokens in logical order ----
    lens = (c.sink_len + c.hist_len + c.rec_len).astype(np.int32)
    bpages = (lens + c.P - 1) // c.P
    brng = np.random.default_rng(77)
    btotal = int(bpages.sum()) + 1
    bperm = brng.permutation(btotal).astype(np.int32)
    bpt_np = np.full((B, int(bpages.max())), -1, np.int32)
    o = 0
    for b in range(B):
        bpt_np[b, :bpages[b]] = bperm[o:o + bpages[b]]; o += bpages[b]
    bpool = native.KVPool(native.KV_POOL_BF16, 1, Hq, Hkv, c.P, btotal, B)
    W_cap = c.rec_k.shape[2]
    for b in range(B):
        s_, r_ = int(c.sink_len[b]), int(c.rec_len[b])
        ring = torch.as_tensor((c.rec_start[b] + np.arange(r_)) % W_cap, device=dev)
        kk = torch.cat([c.sink_k[b, :, :s_].transpose(0, 1), c.hist_k[cu[b]:cu[b + 1]],
                        c.rec_k[b][:, ring].transpose(0, 1)]).contiguous()
        vv = torch.cat([c.sink_v[b, :, :s_].transpose(0, 1), c.hist_v[cu[b]:cu[b + 1]],
                        c.rec_v[b][:, ring].transpose(0, 1)]).contiguous()
        native.kv_append_bf16(bpool.handle, 0, 1, kk, vv, i32([0, kk.shape[0]]), i32([0]),
                              i32(bpt_np[b:b + 1]), bpt_np.shape[1], kk.shape[0])
        del kk, vv
    torch.cuda.synchronize()
    bpt = i32(bpt_np)
    blen = i32(lens)
    bws_bytes = native.kv_decode_workspace_bytes(bpool.handle, B, int(lens.max()))
    bws = torch.zeros(bws_bytes // 4 + 4, dtype=torch.float32, device=dev)
    bout = torch.empty_like(out)

    def bstep():
        native.kv_decode_attention_bf16(bpool.handle, 0, B, q, blen, bpt, bpt_np.shape[1],
                                        int(lens.max()), c.scale, bout, bws, bws_bytes, stream)

    with ClockSampler(local) as clk:
        t_int2 = timed(step, args.steps, max(3, args.warmup))
    t_bf16 = timed(bstep, max(5, args.steps // 2), 3)
    if pool.error() or bpool.error():
        raise RuntimeError("device error during the timed steps")

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

    def e2e_step():
        stage_dev.copy_(stage_host, non_blocking=True)
        native.kv_decode_attention(pool.handle, 0, B, q_dev, meta_dev[0], meta_dev[1], meta_dev[2],
                                   meta_dev[3], pt, c.page_table.shape[1], max_hist, c.scale, out,
                                   ws, ws_bytes, stream)
        out_host.copy_(out, non_blocking=True)

    t_e2e = timed(e2e_step, args.steps, 3)
    h2d = stage_host.numel()
    d2h = out_host.numel() * 4

    # ---- the same call handed the pinned host buffers themselves: the kernel
    # reads q and the lengths and writes out across the CPU-GPU link ----
    q_host = stage_host[:q_bytes].view(torch.bfloat16).view(B, Hq, 128)
    meta_host = stage_host[q_bytes:].view(torch.int32).view(4, B)

    def mapped_step():
        native.kv_decode_attention(pool.handle, 0, B, q_host, meta_host[0], meta_host[1], meta_host[2],
                                   meta_host[3], pt, c.page_table.shape[1], max_hist, c.scale, out_host,
                                   ws, ws_bytes, stream)

    t_mapped = timed(mapped_step, args.steps, 3)
    if pool.error():
        raise RuntimeError("device error during the end-to-end steps")

    # ---- several queries per sequence over the same cache (two positions of a
    # chunk, or a draft and its successor), with the log-sum-exp ----
    TQ = 2
    qm = torch.randn(B, TQ, Hq, 128, generator=torch.Generator(device=dev).manual_seed(9),
                     device=dev).to(torch.bfloat16)
    m_ws_bytes = native.kv_decode_multi_workspace_bytes(pool.handle, B, TQ, max_hist)
    m_ws = torch.zeros(m_ws_bytes // 4 + 4, dtype=torch.float32, device=dev)
    m_out = torch.empty((B, TQ, Hq, 128), dtype=torch.float32, device=dev)
    m_lse = torch.empty((B, TQ, Hq), dtype=torch.float32, device=dev)

    def mstep():
        native.kv_decode_attention_multi(pool.handle, 0, B, TQ, qm, sink_len, hist_len, rec_len, rec_start,
                                         pt, c.page_table.shape[1], max_hist, c.scale, m_out, m_lse, m_ws,
                                         m_ws_bytes, stream)

    t_multi = (timed(mstep, max(5, args.steps // 2), 3)
               if TQ * (Hq // Hkv) <= 8 else None)

    # ---- per-step token placement at batch 64 (every sequence evicts one
    # recent token into INT2 history per step) ----
    SB, SH, SP = 64, Hkv, 16
    spool = native.KVPool(native.KV_POOL_INT2_3TIER, 1, Hq, SH, SP, SB * 4, SB, group_size=c.GS)
    native.kv_pool_set_rotation(spool.handle, 0, Rk, Rv, ck, cv)
    s_rng = np.random.default_rng(5)
    s_pt = i32(s_rng.permutation(SB * 4).reshape(SB, 4))
    s_lens = [i32(np.full(SB, 64)), i32(np.zeros(SB)), i32(np.full(SB, 256)), i32(np.zeros(SB))]
    s_gen = torch.Generator(device=dev)
    s_gen.manual_seed(5)
    s_new = torch.randn(2, SB, SH, 128, generator=s_gen, device=dev).to(torch.bfloat16)

    def astep():
        native.kv_append_step(spool.handle, 0, SB, s_new[0], s_new[1], *s_lens, s_pt, 4, stream)

    t_step = timed(astep, 20, 3)
    if spool.error():
        raise RuntimeError("device error during the append steps")
    spool.close()

    us = float(np.mean(t_int2) * 1e3)
    us_bf16 = float(np.mean(t_bf16) * 1e3)
    us, us_bf16, us_e2e, us_mapped = kvdist.max_over_ranks(
        [us, us_bf16, float(np.mean(t_e2e) * 1e3), float(np.mean(t_mapped) * 1e3)], device=dev)

    alg, parts = algorithmic_bytes(c)
    peak, peak_src = peak_hbm()
    achieved = alg / (us * 1e-6) / 1e9
    if rank == 0:
        cb = None
        if wl is not None and not args.no_cpu_baseline:
            cb = cpu_baseline(wl)
        line = {
            "metric": METRIC, "value": us, "unit": "us", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": us / 1e3, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "int2 codes, f16 MMA, f32 accumulate",
            "data": "synthetic (seeded; pool filled by kv_append_quantize)",
            "config": c.config,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": measured_traffic(c.name),
                         "peak_source": peak_src, "algorithmic_bytes": alg, "bytes_breakdown": parts},
            "us_p10_p50_p90": [float(np.percentile(t_int2, p) * 1e3) for p in (10, 50, 90)],
            "bf16_path": {"us": us_bf16, "bytes": bf16_bytes(c),
                          "gbs": bf16_bytes(c) / (us_bf16 * 1e-6) / 1e9,
                          "speedup_int2_vs_bf16": us_bf16 / us},
            "append_step": {"us": float(np.mean(t_step) * 1e3), "batch": SB, "kv_heads": SH,
                            "what": "one kv_append_step call (eviction and placement launches): each sequence's new token enters the "
                                    "recent ring and its oldest recent token is rotated, clipped, "
                                    "quantized and packed into INT2 history"},
            "e2e": {"value": us_e2e, "unit": "us", "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h),
                    "what": "kv_decode_attention with host buffers: one pinned staging copy in (q and "
                            "the four length arrays), the output copied back, both inside the timed region"},
            "e2e_host_mapped": {"value": us_mapped, "unit": "us", "h2d_bytes_per_step": int(h2d),
                                "d2h_bytes_per_step": int(d2h),
                                "what": "the same call given the pinned host buffers directly: the kernel "
                                        "reads q and the lengths and writes the output across the CPU-GPU "
                                        "link inside the timed region (no staging copies)"},
            "multi_query": (None if t_multi is None else
                            {"us": float(np.mean(t_multi) * 1e3), "queries_per_sequence": TQ,
                             "what": "one kv_decode_attention_multi call over the same cache, "
                                     "output and log-sum-exp"}),
            "gpu_launches": args.steps,
            "clocks": clk.summary(),
            "cpu_baseline": cb,
        }
        print(json.dumps(line))
    pool.close(); bpool.close()


# --------------------------------------------------------------------------
# append benchmark
# --------------------------------------------------------------------------

def run_append(args, torch, dev, rank, world, local, kvdist):
    from bit_kv_cache_12_gb300 import native
    n_seqs, Hkv, T, P, GS = 64, 8, 4096, 16, 64
    seed = 3
    rng = np.random.default_rng(seed)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    stream = torch.cuda.current_stream()
    timed = make_timer(torch, dev, stream, kvdist)

    def student_t4(n):                         # N(0,1) / sqrt(chi2_4 / 4)
        z = torch.randn(n, Hkv, 128, generator=gen, device=dev)
        chi = (torch.randn(4, n, Hkv, 128, generator=gen, device=dev) ** 2).sum(0) / 4.0
        return (z / chi.sqrt()).to(torch.bfloat16)
    k, v = student_t4(n_seqs * T), student_t4(n_seqs * T)
    Rk, Rv = _haar(rng, Hkv), _haar(rng, Hkv)
    ck, cv = _clip_from(k, Rk, 0.9, torch), _clip_from(v, Rv, 0.9, torch)
    pages_per = T // P
    num_pages = n_seqs * pages_per
    pt_np = rng.permutation(num_pages).astype(np.int32).reshape(n_seqs, pages_per)
    pool = native.KVPool(native.KV_POOL_INT2_3TIER, 1, Hkv, Hkv, P, num_pages, n_seqs, group_size=GS)
    native.kv_pool_set_rotation(pool.handle, 0, torch.as_tensor(Rk).to(dev), torch.as_tensor(Rv).to(dev),
                                torch.as_tensor(ck).to(dev), torch.as_tensor(cv).to(dev))
    cu = torch.as_tensor(np.arange(n_seqs + 1, dtype=np.int32) * T, device=dev)
    hs = torch.zeros(n_seqs, dtype=torch.int32, device=dev)
    pt = torch.as_tensor(pt_np, device=dev)

    def step():
        native.kv_append_quantize(pool.handle, 0, n_seqs, k, v, cu, hs, pt, pages_per, T, stream)

    with ClockSampler(local) as clk:
        t = timed(step, args.steps, max(3, args.warmup))
    if pool.error():
        raise RuntimeError("device error during the timed appends")
    us = kvdist.max_over_ranks([float(np.mean(t) * 1e3)], device=dev)[0]
    rows = n_seqs * T * Hkv
    alg = rows * 256 * 2 + rows * (32 + 4 * (128 // GS)) * 2     # bf16 K+V in; codes + s/z out
    flops = 2.0 * 128 * 128 * rows * 2                           # x R for K and V
    peak, peak_src = peak_hbm()
    achieved = alg / (us * 1e-6) / 1e9
    if rank == 0:
        line = {
            "metric": APPEND_METRIC, "value": us, "unit": "us", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": us / 1e3, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in, bf16 hi+lo MMA rotation, f32",
            "data": "synthetic (seeded torch generator on the device, Student-t(4))",
            "config": {"workload": "append_64x4096_h8_g64", "sequences": n_seqs, "tokens_per_seq": T,
                       "kv_heads": Hkv, "page_size": P, "group_size": GS, "l2": L2_NOTE},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": None, "peak_source": peak_src,
                         "algorithmic_bytes": alg},
            "rotation_tflops": flops / (us * 1e-6) / 1e12,
            "us_p10_p50_p90": [float(np.percentile(t, p) * 1e3) for p in (10, 50, 90)],
            "gpu_launches": args.steps, "clocks": clk.summary(), "cpu_baseline": None,
        }
        print(json.dumps(line))
    pool.close()


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
    from bit_kv_cache_12_gb300 import synth
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.workload == "append":
        run_append(args, torch, dev, rank, world, local, kvdist)
    elif args.workload == "qwen3_4b":
        wl = synth.qwen3_4b_decode(ctx=args.ctx)
        run_decode(args, case_from_synth(wl, torch, dev), wl, torch, dev, rank, world, local, kvdist)
    else:
        run_decode(args, case_generated(args.workload, torch, dev), None, torch, dev, rank, world,
                   local, kvdist)
    kvdist.shutdown()


if __name__ == "__main__":
    main()
