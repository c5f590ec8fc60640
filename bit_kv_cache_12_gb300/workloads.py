"""Seeded synthetic decode workloads resident on the device.

Input generation only (no step of the hot path): K/V rows, queries, rotations,
clip thresholds, lengths and shuffled page tables, with the shapes and value
structure of the study's workloads.  The large workloads are generated on the
device from seeded torch generators (host generation of several GB of bf16
takes minutes); lengths, page permutations and outlier positions come from
numpy PCG64.  ``bench.py`` times these cases and the full-size parity tests
check the library on the very same inputs.

Workloads (head_dim 128, 64 sink + INT2 history + 256 recent tokens):
  batch64   Qwen3-8B shape: batch 64, 32 q / 8 KV heads, context U[8192,
            32768] per sequence, page 16, 4 outlier channels per KV head x10,
            Haar R, clip 0.95, group 128
  long16    Qwen3-32B shape: batch 16, 64 q / 8 KV heads (GQA 8), context
            131,072, page 32, 0.1% of token positions x20 (all heads, K and
            V), Haar R, clip 0.95, group 128
"""

import numpy as np

S_CAP, W_CAP = 64, 256


class Case:
    """A three-tier decode workload whose K/V live on the device.

    Attributes: name, B, Hq, Hkv, P (page size), GS (group size), scale;
    numpy int32 [B] sink_len, hist_len, rec_len, rec_start; page_table int32
    [B, max_pages], num_pages; Rk, Rv float32 [Hkv, 128, 128]; clip_k, clip_v
    float32 [Hkv, 128]; device bf16 q [B, Hq, 128], hist_k / hist_v [sum
    hist_len, Hkv, 128] (sequences back to back), sink_k / sink_v [B, Hkv,
    64, 128], rec_k / rec_v [B, Hkv, 256, 128] (ring order); q_np (bf16 bits
    of q on the host); config (a description for the benchmark line)."""

    @property
    def cu_hist(self):
        cu = np.zeros(self.B + 1, np.int64)
        cu[1:] = np.cumsum(self.hist_len)
        return cu


def case_from_synth(wl, torch, dev, l2_note=""):
    """A host-generated ``synth.Workload`` moved to the device."""
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
    ctx = wl.meta["ctx"]
    c.config = {"workload": wl.name, "batch": wl.B, "q_heads": wl.Hq, "kv_heads": wl.Hkv,
                "head_dim": 128, "context": int(ctx[0]) if wl.B == 1 else [int(ctx.min()), int(ctx.max())],
                "sink": int(wl.sink_len[0]), "int2_history": int(wl.hist_len[0]),
                "recent": int(wl.rec_len[0]), "page_size": wl.page_size, "group_size": wl.group_size,
                "l2": l2_note}
    return c


def append_workload(torch, dev, seed=3, n_seqs=64, Hkv=8, T=4096, P=16, GS=64, clip_ratio=0.9):
    """The bulk-append workload: n_seqs sequences x Hkv KV heads x T tokens of
    Student-t(4) K and V rows (bf16, on the device), per-head Haar R_k and R_v,
    clips at clip_ratio x the rotated per-channel absmax, a shuffled page
    table.  Returns a dict of the device inputs and their host copies."""
    rng = np.random.default_rng(seed)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)

    def student_t4(n):                         # N(0,1) / sqrt(chi2_4 / 4)
        z = torch.randn(n, Hkv, 128, generator=gen, device=dev)
        chi = (torch.randn(4, n, Hkv, 128, generator=gen, device=dev) ** 2).sum(0) / 4.0
        return (z / chi.sqrt()).to(torch.bfloat16)
    k, v = student_t4(n_seqs * T), student_t4(n_seqs * T)
    Rk, Rv = haar_stack(rng, Hkv), haar_stack(rng, Hkv)
    ck, cv = clip_from(k, Rk, clip_ratio, torch), clip_from(v, Rv, clip_ratio, torch)
    pages_per = T // P
    num_pages = n_seqs * pages_per
    pt_np = rng.permutation(num_pages).astype(np.int32).reshape(n_seqs, pages_per)
    return {"k": k, "v": v, "Rk": Rk, "Rv": Rv, "clip_k": ck, "clip_v": cv, "page_table": pt_np,
            "n_seqs": n_seqs, "Hkv": Hkv, "T": T, "page_size": P, "group_size": GS,
            "num_pages": num_pages, "pages_per_seq": pages_per}


def haar_stack(rng, n):
    from bit_kv_cache_12_gb300 import synth
    return np.stack([synth.haar_orthogonal(rng) for _ in range(n)]).astype(np.float32)


def clip_from(x, R, ratio, torch):
    """ratio x per-channel absmax of the rotated rows x [T][Hkv][128] (device):
    the calibration stand-in for the per-channel clip thresholds."""
    Hkv = x.shape[1]
    out = np.zeros((Hkv, 128), np.float32)
    for g in range(Hkv):
        Rg = torch.as_tensor(R[g], device=x.device)
        m = torch.zeros(128, device=x.device)
        for s in range(0, x.shape[0], 1 << 18):
            m = torch.maximum(m, (x[s:s + (1 << 18), g].float() @ Rg).abs().amax(dim=0))
        out[g] = ratio * m.cpu().numpy()
    out[out <= 0] = np.inf
    return out


def generate(torch, dev, name, seed, B, Hq, Hkv, P, ctx=None, ctx_range=None, outlier_channels=0,
             token_outlier_frac=0.0, clip_ratio=0.95, l2_note=""):
    """A seeded device-resident three-tier workload.

    ctx: int array [B] of total context lengths, or ctx_range (lo, hi): drawn
    uniformly (inclusive) from the workload's stream.  outlier_channels: that
    many seeded channels per KV head scaled x10 (K and V); token_outlier_frac:
    round(frac x context) of each sequence's history positions scaled x20 (all
    heads, K and V).  K/V ~ N(0,1) in bf16; separate seeded Haar R_k and R_v
    per head; clip thresholds clip_ratio x per-channel absmax of the rotated
    history."""
    rng = np.random.default_rng(seed)
    if ctx_range is not None:
        ctx = rng.integers(ctx_range[0], ctx_range[1] + 1, size=B)
    ctx = np.asarray(ctx, np.int64)
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
    c.page_table = np.full((B, max(1, int(pages_per.max()))), -1, np.int32)
    o = 0
    for b in range(B):
        c.page_table[b, :pages_per[b]] = perm[o:o + pages_per[b]]; o += pages_per[b]
    T = int(c.hist_len.sum())
    scale = torch.ones(Hkv, 128, device=dev)
    for g in range(Hkv if outlier_channels else 0):
        scale[g, torch.as_tensor(rng.choice(128, outlier_channels, replace=False), device=dev)] = 10.0

    def kv(n_rows):
        return (torch.randn(n_rows, Hkv, 128, generator=gen, device=dev) * scale).to(torch.bfloat16)
    c.hist_k, c.hist_v = kv(T), kv(T)
    c.sink_k = kv(B * S_CAP).view(B, S_CAP, Hkv, 128).transpose(1, 2).contiguous()
    c.sink_v = kv(B * S_CAP).view(B, S_CAP, Hkv, 128).transpose(1, 2).contiguous()
    c.rec_k = kv(B * W_CAP).view(B, W_CAP, Hkv, 128).transpose(1, 2).contiguous()
    c.rec_v = kv(B * W_CAP).view(B, W_CAP, Hkv, 128).transpose(1, 2).contiguous()
    if token_outlier_frac:
        cu = np.concatenate([[0], np.cumsum(c.hist_len)])
        for b in range(B):
            n_out = min(int(round(token_outlier_frac * int(ctx[b]))), int(c.hist_len[b]))
            pos = rng.choice(int(c.hist_len[b]), n_out, replace=False) + cu[b]
            idx = torch.as_tensor(pos, device=dev)
            c.hist_k[idx] = (c.hist_k[idx].float() * 20).to(torch.bfloat16)
            c.hist_v[idx] = (c.hist_v[idx].float() * 20).to(torch.bfloat16)
    c.Rk = haar_stack(rng, Hkv)
    c.Rv = haar_stack(rng, Hkv)
    c.clip_k = clip_from(c.hist_k, c.Rk, clip_ratio, torch)
    c.clip_v = clip_from(c.hist_v, c.Rv, clip_ratio, torch)
    c.q = torch.randn(B, Hq, 128, generator=gen, device=dev).to(torch.bfloat16)
    c.q_np = c.q.view(torch.int16).cpu().numpy().view(np.uint16)
    c.config = {"workload": name, "batch": B, "q_heads": Hq, "kv_heads": Hkv, "head_dim": 128,
                "context": [int(ctx.min()), int(ctx.max())], "context_mean": float(ctx.mean()),
                "sink": S_CAP, "recent": W_CAP, "int2_history_tokens": T, "page_size": P,
                "group_size": 128, "l2": l2_note, "generation": "seeded torch generator on the device"}
    return c


def batch64(torch, dev, l2_note=""):
    """Qwen3-8B shape, batch 64, context U[8192, 32768]."""
    return generate(torch, dev, "qwen3_8b_b64_h32x8_ctx8192-32768", 4, 64, 32, 8, 16,
                    ctx_range=(8192, 32768), outlier_channels=4, l2_note=l2_note)


def long16(torch, dev, l2_note=""):
    """Qwen3-32B shape, batch 16, GQA 8, context 131,072, page 32."""
    return generate(torch, dev, "qwen3_32b_b16_h64x8_ctx131072", 5, 16, 64, 8, 32,
                    np.full(16, 131072), token_outlier_frac=0.001, l2_note=l2_note)
