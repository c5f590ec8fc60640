"""Benchmark: INT2 paged decode-attention step on one GB300.

Workload (default): Qwen3-4B-shaped single-layer decode, batch 1, 32 q / 8 KV
heads, head_dim 128, context 100,000 tokens = 64 BF16 sink + 99,680 INT2
history + 256 BF16 recent, page 16 with a shuffled page table, group 128.
Inputs are seeded synthetic data (``bit_kv_cache_12_gb300.synth``); the pool
is filled by the library's own append kernel.

One step = one ``kv_decode_attention`` call (whole batch, one layer).  Every
timed step is preceded by an L2 flush outside the timed events: a 256 MiB
device write, then a 256 MiB read so the dirty lines are written back before
the step starts.  Timing: CUDA events on the launching stream around each
step, device synchronised before and after, max over ranks.

``--impl reference`` times the CPU oracle on the same workload instead (a
bounded sample; see the ``cpu_baseline`` entry of the output line).

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


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
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


def algorithmic_bytes(wl):
    """Bytes the method must move per decode step."""
    ng = 128 // wl.group_size
    per_hist_token = 32 + 32 + 8 * ng                 # K codes, V codes, K and V (s, z)
    hist = int(np.sum(wl.hist_len)) * wl.Hkv * per_hist_token
    tiers = int(np.sum(wl.sink_len + wl.rec_len)) * wl.Hkv * 2 * 256
    rot = wl.Hkv * 2 * 128 * 128 * 4                  # R_k and R_v^T, fp32
    pages = int(np.sum((wl.hist_len + wl.page_size - 1) // wl.page_size))
    pt = pages * 4 * wl.Hkv                           # each KV head reads its page ids
    qo = wl.B * wl.Hq * 128 * (2 + 4)
    return hist + tiers + rot + pt + qo, dict(hist=hist, tiers=tiers, rot=rot, page_table=pt, q_out=qo)


def bf16_bytes(wl):
    n = int(np.sum(wl.sink_len + wl.hist_len + wl.rec_len))
    pages = int(np.sum((wl.sink_len + wl.hist_len + wl.rec_len + wl.page_size - 1) // wl.page_size))
    return n * wl.Hkv * 512 + pages * 4 * wl.Hkv + wl.B * wl.Hq * 128 * 6


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


def cpu_baseline(wl, min_seconds=10.0, max_seconds=30.0):
    """Time the oracle on the host cores: whole decode steps (every KV head and
    query head, full context) repeated until about ``min_seconds`` of CPU work
    has run; the value is the mean time of one step."""
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
    steps = 0
    t0 = time.perf_counter()
    while True:
        att.decode_three_tier(wl.q, wl.Rk, wl.Rv, wl.sink_k, wl.sink_v, wl.sink_len, hist,
                              wl.hist_len, wl.rec_k, wl.rec_v, wl.rec_len, wl.rec_start, wl.Hkv,
                              wl.group_size, wl.scale)
        steps += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or dt + dt / steps > max_seconds:
            break
    try:
        cores = len(os.sched_getaffinity(0))
    except Exception:
        cores = os.cpu_count()
    return {"value": dt / steps * 1e6, "unit": "us", "cores": cores, "kind": "oracle",
            "sample": f"{steps} whole decode steps of the bench workload (all {wl.Hkv} KV heads, "
                      f"{wl.Hq} query heads, full context) with the numpy fp64 oracle "
                      f"(unpack, dequantize, three-tier attention) in {dt:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    from bit_kv_cache_12_gb300 import synth
    wl = synth.qwen3_4b_decode(ctx=args.ctx)
    cb = cpu_baseline(wl, min_seconds=min(60.0, 10.0 * max(1, args.steps) / 10))
    vals = [cb["value"]]
    line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "us",
            "n_gpus": world, "steps": len(vals), "warmup": 0, "ms_per_step": cb["value"] / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "config": config_of(wl),
            "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


METRIC = "INT2 paged decode-attention us/step (HBM GB/s, % of roofline) vs BF16 path"


def config_of(wl):
    return {"workload": wl.name, "batch": wl.B, "q_heads": wl.Hq, "kv_heads": wl.Hkv, "head_dim": 128,
            "context": int(wl.meta["ctx"][0]), "sink": int(wl.sink_len[0]),
            "int2_history": int(wl.hist_len[0]), "recent": int(wl.rec_len[0]),
            "page_size": wl.page_size, "group_size": wl.group_size,
            "l2": "flushed between steps (256 MiB write + 256 MiB read outside the timed events)"}


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
    from bit_kv_cache_12_gb300 import native, synth
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    wl = synth.qwen3_4b_decode(ctx=args.ctx)
    B, Hq, Hkv = wl.B, wl.Hq, wl.Hkv

    def bf16(u16):
        return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).to(dev)

    def i32(a):
        return torch.as_tensor(np.ascontiguousarray(np.asarray(a, np.int32))).to(dev)

    # ---- INT2 pool filled by the library's append kernel ----
    pool = native.KVPool(native.KV_POOL_INT2_3TIER, 1, Hq, Hkv, wl.page_size, wl.num_pages, B,
                         group_size=wl.group_size)
    Rk = torch.as_tensor(wl.Rk).to(dev); Rv = torch.as_tensor(wl.Rv).to(dev)
    ck = torch.as_tensor(wl.clip_k).to(dev); cv = torch.as_tensor(wl.clip_v).to(dev)
    native.kv_pool_set_rotation(pool.handle, 0, Rk, Rv, ck, cv)
    sk, sv, rk, rv = pool.tier_views(0)
    sk[:B].copy_(bf16(wl.sink_k)); sv[:B].copy_(bf16(wl.sink_v))
    rk[:B].copy_(bf16(wl.rec_k)); rv[:B].copy_(bf16(wl.rec_v))
    hk = bf16(np.concatenate(wl.hist_k)); hv = bf16(np.concatenate(wl.hist_v))
    cu = np.zeros(B + 1, np.int32); cu[1:] = np.cumsum(wl.hist_len)
    pt = i32(wl.page_table)
    native.kv_append_quantize(pool.handle, 0, B, hk, hv, i32(cu), i32(np.zeros(B)), pt,
                              wl.page_table.shape[1], int(wl.hist_len.max()))
    torch.cuda.synchronize()
    if pool.error():
        raise RuntimeError("device error while filling the pool")
    del hk, hv

    q = bf16(wl.q)
    sink_len, hist_len = i32(wl.sink_len), i32(wl.hist_len)
    rec_len, rec_start = i32(wl.rec_len), i32(wl.rec_start)
    max_hist = int(wl.hist_len.max())
    ws_bytes = native.kv_decode_workspace_bytes(pool.handle, B, max_hist)
    ws = torch.zeros(ws_bytes // 4 + 4, dtype=torch.float32, device=dev)
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        native.kv_decode_attention(pool.handle, 0, B, q, sink_len, hist_len, rec_len, rec_start, pt,
                                   wl.page_table.shape[1], max_hist, wl.scale, out, ws, ws_bytes,
                                   stream)

    # ---- BF16 pool with the same tokens ----
    lens = (wl.sink_len + wl.hist_len + wl.rec_len).astype(np.int32)
    bpages = (lens + wl.page_size - 1) // wl.page_size
    brng = np.random.default_rng(77)
    btotal = int(bpages.sum()) + 1
    bperm = brng.permutation(btotal).astype(np.int32)
    bpt_np = np.full((B, int(bpages.max())), -1, np.int32)
    o = 0
    for b in range(B):
        bpt_np[b, :bpages[b]] = bperm[o:o + bpages[b]]; o += bpages[b]
    bpool = native.KVPool(native.KV_POOL_BF16, 1, Hq, Hkv, wl.page_size, btotal, B)
    for b in range(B):
        s_ = int(wl.sink_len[b]); r_ = int(wl.rec_len[b])
        ring = (wl.rec_start[b] + np.arange(r_)) % wl.rec_k.shape[2]
        kk = np.concatenate([wl.sink_k[b, :, :s_].transpose(1, 0, 2), wl.hist_k[b],
                             wl.rec_k[b][:, ring].transpose(1, 0, 2)])
        vv = np.concatenate([wl.sink_v[b, :, :s_].transpose(1, 0, 2), wl.hist_v[b],
                             wl.rec_v[b][:, ring].transpose(1, 0, 2)])
        native.kv_append_bf16(bpool.handle, 0, 1, bf16(kk), bf16(vv), i32([0, len(kk)]), i32([0]),
                              i32(bpt_np[b:b + 1]), bpt_np.shape[1], len(kk))
        del kk, vv
    torch.cuda.synchronize()
    bpt = i32(bpt_np)
    blen = i32(lens)
    bws_bytes = native.kv_decode_workspace_bytes(bpool.handle, B, int(lens.max()))
    bws = torch.zeros(bws_bytes // 4 + 4, dtype=torch.float32, device=dev)
    bout = torch.empty_like(out)

    def bstep():
        native.kv_decode_attention_bf16(bpool.handle, 0, B, q, blen, bpt, bpt_np.shape[1],
                                        int(lens.max()), wl.scale, bout, bws, bws_bytes, stream)

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
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for s0, s1 in ev:
            flush()
            s0.record(stream); fn(); s1.record(stream)
        torch.cuda.synchronize()
        kvdist.barrier()
        return np.array([s0.elapsed_time(s1) for s0, s1 in ev])   # ms

    with ClockSampler(local) as clk:
        t_int2 = timed(step, args.steps, max(3, args.warmup))
    t_bf16 = timed(bstep, max(5, args.steps // 2), 3)
    if pool.error() or bpool.error():
        raise RuntimeError("device error during the timed steps")

    # ---- end to end through the C ABI with host buffers ----
    q_host = torch.from_numpy(wl.q.view(np.int16)).view(torch.bfloat16).pin_memory()
    meta_host = torch.from_numpy(np.stack([wl.sink_len, wl.hist_len, wl.rec_len, wl.rec_start]).astype(np.int32)).pin_memory()
    meta_dev = torch.empty_like(meta_host, device=dev)
    out_host = torch.empty((B, Hq, 128), dtype=torch.float32).pin_memory()

    def e2e_step():
        q.copy_(q_host, non_blocking=True)
        meta_dev.copy_(meta_host, non_blocking=True)
        native.kv_decode_attention(pool.handle, 0, B, q, meta_dev[0], meta_dev[1], meta_dev[2],
                                   meta_dev[3], pt, wl.page_table.shape[1], max_hist, wl.scale, out,
                                   ws, ws_bytes, stream)
        out_host.copy_(out, non_blocking=True)

    t_e2e = timed(e2e_step, args.steps, 3)

    # ---- per-step token placement at batch 64 (every sequence evicts one
    # recent token into INT2 history per step) ----
    SB, SH, SP = 64, Hkv, 16
    spool = native.KVPool(native.KV_POOL_INT2_3TIER, 1, Hq, SH, SP, SB * 4, SB, group_size=wl.group_size)
    native.kv_pool_set_rotation(spool.handle, 0, Rk, Rv, ck, cv)
    s_rng = np.random.default_rng(5)
    s_pt = i32(s_rng.permutation(SB * 4).reshape(SB, 4))
    s_lens = [i32(np.full(SB, 64)), i32(np.zeros(SB)), i32(np.full(SB, 256)), i32(np.zeros(SB))]
    s_new = bf16(synth.f32_to_bf16_bits(s_rng.standard_normal((2, SB, SH, 128)).astype(np.float32)))

    def astep():
        native.kv_append_step(spool.handle, 0, SB, s_new[0], s_new[1], *s_lens, s_pt, 4, stream)

    t_step = timed(astep, 20, 3)
    if spool.error():
        raise RuntimeError("device error during the append steps")
    spool.close()
    h2d = q_host.numel() * 2 + meta_host.numel() * 4
    d2h = out_host.numel() * 4

    us = float(np.mean(t_int2) * 1e3)
    us_bf16 = float(np.mean(t_bf16) * 1e3)
    us, us_bf16, us_e2e = kvdist.max_over_ranks([us, us_bf16, float(np.mean(t_e2e) * 1e3)], device=dev)

    alg, parts = algorithmic_bytes(wl)
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(peaks_path):
        peak = float(json.load(open(peaks_path))["hbm_gbs"]); peak_src = "measured (MEASURED_PEAKS.json hbm_gbs)"
    else:
        peak = 6800.0; peak_src = "fallback 6.8 TB/s"
    achieved = alg / (us * 1e-6) / 1e9
    if rank == 0:
        cb = None
        if not args.no_cpu_baseline:
            cb = cpu_baseline(wl)
        line = {
            "metric": METRIC, "value": us, "unit": "us", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": us / 1e3, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "int2 codes, f16 MMA, f32 accumulate",
            "data": "synthetic (seeded numpy; pool filled by kv_append_quantize)",
            "config": config_of(wl),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": measured_traffic(wl.name), "peak_source": peak_src,
                         "algorithmic_bytes": alg, "bytes_breakdown": parts},
            "us_p10_p50_p90": [float(np.percentile(t_int2, p) * 1e3) for p in (10, 50, 90)],
            "bf16_path": {"us": us_bf16, "bytes": bf16_bytes(wl),
                          "gbs": bf16_bytes(wl) / (us_bf16 * 1e-6) / 1e9,
                          "speedup_int2_vs_bf16": us_bf16 / us},
            "append_step": {"us": float(np.mean(t_step) * 1e3), "batch": SB, "kv_heads": SH,
                            "what": "one kv_append_step launch: each sequence's new token enters the "
                                    "recent ring and its oldest recent token is rotated, clipped, "
                                    "quantized and packed into INT2 history"},
            "e2e": {"value": us_e2e, "unit": "us", "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h)},
            "gpu_launches": args.steps,
            "clocks": clk.summary(),
            "cpu_baseline": cb,
        }
        print(json.dumps(line))
    pool.close(); bpool.close()
    kvdist.shutdown()


if __name__ == "__main__":
    main()
