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
