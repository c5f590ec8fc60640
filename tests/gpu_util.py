"""Helpers for the GPU parity tests: move seeded workloads into pools, run the
library through its C ABI, and run the oracle on the same inputs."""

import numpy as np
import torch

from bit_kv_cache_12_gb300 import native
from oracle import attention as att
from oracle import kvquant as kq


def bf16_dev(u16):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).cuda()


def i32_dev(a):
    return torch.as_tensor(np.ascontiguousarray(np.asarray(a, np.int32))).cuda()


def f32_dev(a):
    return torch.as_tensor(np.ascontiguousarray(np.asarray(a, np.float32))).cuda()


def metrics(out, ref):
    out = np.asarray(out, np.float64); ref = np.asarray(ref, np.float64)
    d = out - ref
    return float(np.abs(d).max()), float(np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-300))


# ---------------------------------------------------------------------------
# INT2 three-tier pool
# ---------------------------------------------------------------------------

def make_int2_pool(wl, num_pages=None, max_seqs=None):
    pool = native.KVPool(native.KV_POOL_INT2_3TIER, 1, wl.Hq, wl.Hkv, wl.page_size,
                         num_pages or wl.num_pages, max_seqs or wl.B, group_size=wl.group_size)
    Rk, Rv = f32_dev(wl.Rk), f32_dev(wl.Rv)
    ck, cv = f32_dev(wl.clip_k), f32_dev(wl.clip_v)
    native.kv_pool_set_rotation(pool.handle, 0, Rk, Rv, ck, cv)
    sk, sv, rk, rv = pool.tier_views(0)
    B = wl.B
    sk[:B].copy_(bf16_dev(wl.sink_k)); sv[:B].copy_(bf16_dev(wl.sink_v))
    rk[:B].copy_(bf16_dev(wl.rec_k)); rv[:B].copy_(bf16_dev(wl.rec_v))
    torch.cuda.synchronize()
    pool._keep = (Rk, Rv, ck, cv)
    return pool


def oracle_pages(wl, page_table=None, num_pages=None):
    """History pages quantized and packed by the oracle (fp64 rotation)."""
    pt = wl.page_table if page_table is None else page_table
    tb = kq.tile_bytes(wl.group_size) * (wl.page_size // 16)
    pages = np.zeros((num_pages or wl.num_pages, wl.Hkv, tb), np.uint8)
    for b in range(wl.B):
        if wl.hist_len[b] == 0:
            continue
        kq.pack_history_full(wl.hist_k[b], wl.hist_v[b], wl.Rk, wl.Rv, wl.clip_k, wl.clip_v,
                             pt[b], pages.shape[0], wl.Hkv, wl.page_size, wl.group_size, pages)
    return pages


def upload_pages(pool, pages):
    pool.hist_view(0).copy_(torch.from_numpy(pages))
    torch.cuda.synchronize()


def gpu_append_history(pool, wl, page_table=None):
    """All history tokens of every sequence through kv_append_quantize."""
    pt = wl.page_table if page_table is None else page_table
    k = np.concatenate([h for h in wl.hist_k]) if wl.B else np.zeros((0, wl.Hkv, 128), np.uint16)
    v = np.concatenate([h for h in wl.hist_v])
    cu = np.zeros(wl.B + 1, np.int32); cu[1:] = np.cumsum(wl.hist_len)
    kd, vd = bf16_dev(k), bf16_dev(v)
    cud, hs, ptd = i32_dev(cu), i32_dev(np.zeros(wl.B)), i32_dev(pt)
    native.kv_append_quantize(pool.handle, 0, wl.B, kd, vd, cud, hs, ptd, pt.shape[1],
                              int(max(1, wl.hist_len.max())))
    torch.cuda.synchronize()


def gpu_decode(pool, wl, page_table=None, max_hist=None, q=None, hist_len=None, sink_len=None,
               rec_len=None, rec_start=None, scale=None):
    pt = wl.page_table if page_table is None else page_table
    hist_len = wl.hist_len if hist_len is None else hist_len
    mh = int(max(hist_len.max(), 0)) if max_hist is None else max_hist
    ws_bytes = native.kv_decode_workspace_bytes(pool.handle, wl.B, mh)
    ws = torch.empty(max(ws_bytes, 16) // 4 + 4, dtype=torch.float32, device="cuda")
    out = torch.full((wl.B, wl.Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    args = [i32_dev(wl.sink_len if sink_len is None else sink_len), i32_dev(hist_len),
            i32_dev(wl.rec_len if rec_len is None else rec_len),
            i32_dev(wl.rec_start if rec_start is None else rec_start)]
    native.kv_decode_attention(pool.handle, 0, wl.B, bf16_dev(wl.q if q is None else q), *args,
                               i32_dev(pt), pt.shape[1], mh, wl.scale if scale is None else scale,
                               out, ws, ws_bytes)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def oracle_decode(wl, pages, page_table=None, hist_len=None, sink_len=None, rec_len=None,
                  rec_start=None, q=None, heads=None):
    pt = wl.page_table if page_table is None else page_table
    hist_len = wl.hist_len if hist_len is None else hist_len
    hist = lambda b, g: kq.read_history(pages, pt[b], int(hist_len[b]), g, wl.page_size,
                                        wl.group_size)
    return att.decode_three_tier(wl.q if q is None else q, wl.Rk, wl.Rv, wl.sink_k, wl.sink_v,
                                 wl.sink_len if sink_len is None else sink_len, hist, hist_len,
                                 wl.rec_k, wl.rec_v, wl.rec_len if rec_len is None else rec_len,
                                 wl.rec_start if rec_start is None else rec_start, wl.Hkv,
                                 wl.group_size, wl.scale)


# ---------------------------------------------------------------------------
# all-BF16 pool with the same logical tokens
# ---------------------------------------------------------------------------

def logical_tokens(wl, b):
    """Sink, history and recent rows of sequence b in order: [n, Hkv, 128] bf16 bits."""
    s = int(wl.sink_len[b]); r = int(wl.rec_len[b])
    ring = (wl.rec_start[b] + np.arange(r)) % wl.rec_k.shape[2]
    k = np.concatenate([wl.sink_k[b, :, :s].transpose(1, 0, 2), wl.hist_k[b],
                        wl.rec_k[b][:, ring].transpose(1, 0, 2)])
    v = np.concatenate([wl.sink_v[b, :, :s].transpose(1, 0, 2), wl.hist_v[b],
                        wl.rec_v[b][:, ring].transpose(1, 0, 2)])
    return k, v


def make_bf16_pool(wl, page_size=None):
    P = page_size or wl.page_size
    lens = np.array([int(wl.sink_len[b] + wl.hist_len[b] + wl.rec_len[b]) for b in range(wl.B)])
    pages_per = (lens + P - 1) // P
    rng = np.random.default_rng(1234)
    total = int(pages_per.sum()) + 3
    perm = rng.permutation(total).astype(np.int32)
    pt = np.full((wl.B, max(1, int(pages_per.max()))), -1, np.int32)
    o = 0
    for b in range(wl.B):
        pt[b, :pages_per[b]] = perm[o:o + pages_per[b]]; o += pages_per[b]
    pool = native.KVPool(native.KV_POOL_BF16, 1, wl.Hq, wl.Hkv, P, total, wl.B)
    ks, vs = zip(*[logical_tokens(wl, b) for b in range(wl.B)])
    k = np.concatenate(ks); v = np.concatenate(vs)
    cu = np.zeros(wl.B + 1, np.int32); cu[1:] = np.cumsum(lens)
    native.kv_append_bf16(pool.handle, 0, wl.B, bf16_dev(k), bf16_dev(v), i32_dev(cu),
                          i32_dev(np.zeros(wl.B)), i32_dev(pt), pt.shape[1], int(lens.max()))
    torch.cuda.synchronize()
    return pool, pt, lens


def gpu_decode_bf16(pool, wl, pt, lens, q=None):
    ml = int(lens.max())
    ws_bytes = native.kv_decode_workspace_bytes(pool.handle, wl.B, ml)
    ws = torch.empty(max(ws_bytes, 16) // 4 + 4, dtype=torch.float32, device="cuda")
    out = torch.full((wl.B, wl.Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    native.kv_decode_attention_bf16(pool.handle, 0, wl.B, bf16_dev(wl.q if q is None else q),
                                    i32_dev(lens), i32_dev(pt), pt.shape[1], ml, wl.scale, out, ws,
                                    ws_bytes)
    torch.cuda.synchronize()
    return out.cpu().numpy()


# ---------------------------------------------------------------------------
# device-resident workloads (bit_kv_cache_12_gb300.workloads): pool fill,
# one decode in the benchmark's launch configuration, oracle on sampled heads
# ---------------------------------------------------------------------------

def fill_pool_from_case(c):
    """An INT2 pool holding case c: tiers copied in, history through the
    library's own kv_append_quantize (as the benchmark fills it)."""
    pool = native.KVPool(native.KV_POOL_INT2_3TIER, 1, c.Hq, c.Hkv, c.P, c.num_pages, c.B,
                         group_size=c.GS)
    keep = (f32_dev(c.Rk), f32_dev(c.Rv), f32_dev(c.clip_k), f32_dev(c.clip_v))
    native.kv_pool_set_rotation(pool.handle, 0, *keep)
    pool._keep = keep
    sk, sv, rk, rv = pool.tier_views(0)
    sk[:c.B].copy_(c.sink_k); sv[:c.B].copy_(c.sink_v)
    rk[:c.B].copy_(c.rec_k); rv[:c.B].copy_(c.rec_v)
    cu = np.zeros(c.B + 1, np.int32); cu[1:] = np.cumsum(c.hist_len)
    native.kv_append_quantize(pool.handle, 0, c.B, c.hist_k, c.hist_v, i32_dev(cu),
                              i32_dev(np.zeros(c.B)), i32_dev(c.page_table), c.page_table.shape[1],
                              int(max(1, c.hist_len.max())))
    torch.cuda.synchronize()
    return pool


def decode_case(pool, c, hist_len=None, max_hist=None):
    """One kv_decode_attention over the whole batch of case c (the benchmark's call)."""
    hist_len = c.hist_len if hist_len is None else hist_len
    mh = int(c.hist_len.max()) if max_hist is None else max_hist
    ws_bytes = native.kv_decode_workspace_bytes(pool.handle, c.B, mh)
    ws = torch.empty(max(ws_bytes, 16) // 4 + 4, dtype=torch.float32, device="cuda")
    out = torch.full((c.B, c.Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    native.kv_decode_attention(pool.handle, 0, c.B, c.q, i32_dev(c.sink_len), i32_dev(hist_len),
                               i32_dev(c.rec_len), i32_dev(c.rec_start), i32_dev(c.page_table),
                               c.page_table.shape[1], mh, c.scale, out, ws, ws_bytes)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def oracle_kv_head(pool, c, b, g, hist_len=None):
    """Oracle outputs [G, 128] of every query head of KV head g of sequence b,
    from the codes the pool stores (only that sequence's pages are copied)."""
    h = int(c.hist_len[b] if hist_len is None else hist_len)
    npages = (h + c.P - 1) // c.P
    G = c.Hq // c.Hkv
    if npages:
        ids = torch.as_tensor(c.page_table[b, :npages].astype(np.int64), device="cuda")
        pages = pool.hist_view(0).index_select(0, ids).cpu().numpy()
        kc, vc, sk, zk, sv, zv = kq.read_history(pages, np.arange(npages), h, g, c.P, c.GS)
    else:
        kc = vc = np.zeros((0, 128), np.uint8)
        sk = zk = sv = zv = np.zeros((0, 128 // c.GS), np.float16)
    kd = kq.dequant(kc, sk, zk, c.GS)
    vd = kq.dequant(vc, sv, zv, c.GS)
    s, r = int(c.sink_len[b]), int(c.rec_len[b])
    sink_k = kq.bf16_bits_to_f64(_bits(c.sink_k[b, g, :s]))
    sink_v = kq.bf16_bits_to_f64(_bits(c.sink_v[b, g, :s]))
    cap = c.rec_k.shape[2]
    rec_k = kq.bf16_bits_to_f64(att.ring_order(_bits(c.rec_k[b, g]), int(c.rec_start[b]), r, cap))
    rec_v = kq.bf16_bits_to_f64(att.ring_order(_bits(c.rec_v[b, g]), int(c.rec_start[b]), r, cap))
    Rk = np.asarray(c.Rk[g], np.float64); Rv = np.asarray(c.Rv[g], np.float64)
    return np.stack([att.three_tier_head(kq.bf16_bits_to_f64(c.q_np[b, g * G + hh]), Rk, Rv, sink_k,
                                         sink_v, kd, vd, rec_k, rec_v, c.scale) for hh in range(G)])
