"""Seeded synthetic workloads for the 2-bit KV-cache hot path.

This module only draws inputs.  It holds none of the method's hot-path
arithmetic (no quantizer, packer or attention) and is shared by the tests,
``bench.py`` and the smoke check, on the CUDA side and on the oracle side.

It also plays the offline calibration that produces the rotation and clip
inputs.  On the OSCAR pages that step is an offline host-side procedure
(gist.science explainer, section 2.2 A "Offline-Kalibrierungsphase": target
covariance -> eigenbasis U, Hadamard H, bit-reversal permutation P_br,
R = U H P_br; per-layer clip thresholds from rotated calibration data).  Here
it runs on synthetic covariances, seeded.

Randomness: numpy PCG64, one ``SeedSequence`` per workload, spawning named
streams, so every array is reproducible on any machine.
"""

from dataclasses import dataclass, field
import numpy as np

HEAD_DIM = 128
SINK = 64
RECENT = 256


# --------------------------------------------------------------------------
# bf16 bit patterns (round-to-nearest-even from float32)
# --------------------------------------------------------------------------

def f32_to_bf16_bits(x):
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = x.view(np.uint32).astype(np.uint64)
    r = ((u >> 16) & 1) + 0x7FFF
    return ((u + r) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# Rotation inputs
# --------------------------------------------------------------------------

def haar_orthogonal(rng, d=HEAD_DIM):
    """Random orthogonal matrix: QR of a Gaussian, signs fixed (Haar measure)."""
    a = rng.standard_normal((d, d))
    q, r = np.linalg.qr(a)
    return q * np.sign(np.diag(r))[None, :]


def hadamard(d):
    """Normalised Sylvester Hadamard matrix (d a power of two)."""
    h = np.array([[1.0]])
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h / np.sqrt(d)


def bit_reversal_permutation(d):
    """Permutation matrix P with (x P)_j = x_{bitrev(j)}."""
    nb = int(np.log2(d))
    idx = np.array([int(format(i, f"0{nb}b")[::-1], 2) for i in range(d)])
    p = np.zeros((d, d))
    p[idx, np.arange(d)] = 1.0
    return p


def oscar_like_rotation(rng, d=HEAD_DIM):
    """R = U . H . P_br with U the eigenbasis (columns, descending eigenvalue)
    of a seeded covariance C = Q diag(1/i) Q^T."""
    q = haar_orthogonal(rng, d)
    c = (q * (1.0 / np.arange(1, d + 1))[None, :]) @ q.T
    w, u = np.linalg.eigh(c)
    u = u[:, np.argsort(w)[::-1]]
    return u @ hadamard(d) @ bit_reversal_permutation(d)


# --------------------------------------------------------------------------
# Workload container
# --------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    page_size: int
    group_size: int
    scale: float
    q: np.ndarray                  # uint16 bf16 bits [B, Hq, d]
    Rk: np.ndarray                 # float32 [Hkv, d, d]
    Rv: np.ndarray                 # float32 [Hkv, d, d]
    clip_k: np.ndarray             # float32 [Hkv, d]
    clip_v: np.ndarray             # float32 [Hkv, d]
    sink_len: np.ndarray           # int32 [B]
    hist_len: np.ndarray           # int32 [B]
    rec_len: np.ndarray            # int32 [B]
    rec_start: np.ndarray          # int32 [B]
    sink_k: np.ndarray             # uint16 [B, Hkv, SINK, d]
    sink_v: np.ndarray
    rec_k: np.ndarray              # uint16 [B, Hkv, RECENT, d] (ring order)
    rec_v: np.ndarray
    hist_k: list                   # per b: uint16 [hist_len[b], Hkv, d]
    hist_v: list
    page_table: np.ndarray         # int32 [B, max_pages]
    num_pages: int
    meta: dict = field(default_factory=dict)

    @property
    def G(self):
        return self.Hq // self.Hkv

    @property
    def max_pages(self):
        return self.page_table.shape[1]


def _kv_rows(rng, n, hkv, kind, outlier_ch=None, outlier_mul=1.0, token_outliers=None,
             token_mul=1.0, t_nu=4):
    """[n, hkv, d] float32 rows for K or V."""
    if kind == "t":
        x = rng.standard_t(t_nu, size=(n, hkv, HEAD_DIM)).astype(np.float32)
    else:
        x = rng.standard_normal((n, hkv, HEAD_DIM), dtype=np.float32)
    if outlier_ch is not None:
        for (h, c) in outlier_ch:
            x[:, h, c] *= outlier_mul
    if token_outliers is not None and len(token_outliers):
        x[token_outliers] *= token_mul
    return x


def _shuffled_page_table(rng, pages_per_seq, extra_pages=7):
    """Distinct physical page ids for every sequence, globally shuffled."""
    B = len(pages_per_seq)
    total = int(np.sum(pages_per_seq)) + extra_pages
    perm = rng.permutation(total).astype(np.int32)
    maxp = max(1, int(np.max(pages_per_seq)))
    pt = np.full((B, maxp), -1, np.int32)
    o = 0
    for b in range(B):
        n = int(pages_per_seq[b])
        pt[b, :n] = perm[o:o + n]
        o += n
    return pt, total


def _clip_from(rows_list, R, ratio, calib_tokens=4096):
    """ratio * per-channel absmax of rotated calibration rows, per head."""
    hkv = R.shape[0]
    out = np.zeros((hkv, HEAD_DIM), np.float32)
    for g in range(hkv):
        amax = np.zeros(HEAD_DIM)
        for rows in rows_list:
            if rows.shape[0] == 0:
                continue
            x = rows[:calib_tokens, g, :].astype(np.float64)
            amax = np.maximum(amax, np.abs(x @ R[g].astype(np.float64)).max(axis=0))
        out[g] = (ratio * amax).astype(np.float32)
        out[g][out[g] <= 0] = np.inf
    return out


def make_decode_workload(name, seed, B, Hq, Hkv, ctx, page_size=16, group_size=128,
                         kv_kind="normal", outliers_per_head=0, outlier_frac=None,
                         outlier_mul=10.0, token_outlier_frac=0.0, token_mul=20.0,
                         rotation="haar", clip_ratio=0.95, sink=SINK, recent=RECENT,
                         ring_random_start=True):
    """A three-tier decode workload.  ``ctx`` is an int or an array [B]."""
    ss = np.random.SeedSequence(seed)
    st = {n: np.random.default_rng(s) for n, s in
          zip(["rot", "kv", "q", "pt", "ch", "len", "ring", "tok"], ss.spawn(8))}
    ctx = np.broadcast_to(np.asarray(ctx, dtype=np.int64), (B,)).copy()
    sink_len = np.minimum(ctx, sink).astype(np.int32)
    rem = ctx - sink_len
    rec_len = np.minimum(rem, recent).astype(np.int32)
    hist_len = (rem - rec_len).astype(np.int32)
    rec_start = (st["ring"].integers(0, recent, size=B) if ring_random_start
                 else np.zeros(B)).astype(np.int32)

    # rotation
    if rotation == "identity":
        Rk = np.stack([np.eye(HEAD_DIM)] * Hkv)
        Rv = Rk.copy()
    elif rotation == "oscar":
        Rk = np.stack([oscar_like_rotation(st["rot"]) for _ in range(Hkv)])
        Rv = Rk.copy()
    else:
        Rk = np.stack([haar_orthogonal(st["rot"]) for _ in range(Hkv)])
        Rv = Rk.copy()

    # outlier channels
    outlier_ch = None
    if outliers_per_head:
        outlier_ch = [(h, int(c)) for h in range(Hkv)
                      for c in st["ch"].choice(HEAD_DIM, outliers_per_head, replace=False)]
    elif outlier_frac:
        n = int(round(outlier_frac * Hkv * HEAD_DIM))
        flat = st["ch"].choice(Hkv * HEAD_DIM, n, replace=False)
        outlier_ch = [(int(f) // HEAD_DIM, int(f) % HEAD_DIM) for f in flat]

    kind = "t" if kv_kind == "t" else "normal"
    sink_k = np.zeros((B, Hkv, sink, HEAD_DIM), np.uint16); sink_v = sink_k.copy()
    rec_k = np.zeros((B, Hkv, recent, HEAD_DIM), np.uint16); rec_v = rec_k.copy()
    hist_k, hist_v = [], []
    for b in range(B):
        n = int(ctx[b])
        tok = None
        if token_outlier_frac:
            tok = st["tok"].choice(n, int(round(token_outlier_frac * n)), replace=False)
        k = _kv_rows(st["kv"], n, Hkv, kind, outlier_ch, outlier_mul, tok, token_mul)
        v = _kv_rows(st["kv"], n, Hkv, kind, outlier_ch, outlier_mul, tok, token_mul)
        kb = f32_to_bf16_bits(k); vb = f32_to_bf16_bits(v)
        s_, h_, r_ = int(sink_len[b]), int(hist_len[b]), int(rec_len[b])
        sink_k[b, :, :s_] = kb[:s_].transpose(1, 0, 2)
        sink_v[b, :, :s_] = vb[:s_].transpose(1, 0, 2)
        hist_k.append(kb[s_:s_ + h_]); hist_v.append(vb[s_:s_ + h_])
        ring_idx = (rec_start[b] + np.arange(r_)) % recent
        rec_k[b][:, ring_idx] = kb[s_ + h_:].transpose(1, 0, 2)
        rec_v[b][:, ring_idx] = vb[s_ + h_:].transpose(1, 0, 2)

    hist_f32_k = [bf16_bits_to_f32(h) for h in hist_k]
    hist_f32_v = [bf16_bits_to_f32(h) for h in hist_v]
    if clip_ratio is None:
        clip_k = np.full((Hkv, HEAD_DIM), np.inf, np.float32); clip_v = clip_k.copy()
    else:
        clip_k = _clip_from(hist_f32_k, Rk, clip_ratio)
        clip_v = _clip_from(hist_f32_v, Rv, clip_ratio)

    pages_per_seq = (hist_len + page_size - 1) // page_size
    pt, num_pages = _shuffled_page_table(st["pt"], pages_per_seq)
    q = f32_to_bf16_bits(st["q"].standard_normal((B, Hq, HEAD_DIM), dtype=np.float32))
    return Workload(name=name, B=B, Hq=Hq, Hkv=Hkv, page_size=page_size, group_size=group_size,
                    scale=1.0 / np.sqrt(HEAD_DIM), q=q, Rk=Rk.astype(np.float32),
                    Rv=Rv.astype(np.float32), clip_k=clip_k, clip_v=clip_v, sink_len=sink_len,
                    hist_len=hist_len, rec_len=rec_len, rec_start=rec_start, sink_k=sink_k,
                    sink_v=sink_v, rec_k=rec_k, rec_v=rec_v, hist_k=hist_k, hist_v=hist_v,
                    page_table=pt, num_pages=num_pages, meta=dict(seed=seed, ctx=ctx))


# --------------------------------------------------------------------------
# The five named workloads (full size) and scaled-down variants for tests
# --------------------------------------------------------------------------

def tiny_decode(seed=1):
    """Batch 1, 8 q / 2 KV heads, context 1024 = 64 sink + 704 INT2 + 256 recent,
    page 16, N(0,1) K/V with 4 outlier channels per head x10, Haar R, clip 0.95,
    group 128."""
    return make_decode_workload("tiny_b1_h8x2_ctx1024", seed, B=1, Hq=8, Hkv=2, ctx=1024,
                                outliers_per_head=4, outlier_mul=10.0, rotation="haar")


def qwen3_4b_decode(seed=2, ctx=100_000):
    """Batch 1, 32 q / 8 KV heads, context 100,000, page 16 with shuffled page
    table, N(0,1) K/V with 1% of (head, channel) pairs x8, R from the eigenbasis
    of a synthetic covariance with 1/i spectrum (U H P_br), clip 0.95, group 128."""
    return make_decode_workload(f"qwen3_4b_b1_h32x8_ctx{ctx}", seed, B=1, Hq=32, Hkv=8,
                                ctx=ctx, outlier_frac=0.01, outlier_mul=8.0, rotation="oscar")


def qwen3_8b_batch_decode(seed=4, B=64, ctx_lo=8192, ctx_hi=32768):
    """Batch 64, 32 q / 8 KV heads, per-sequence context uniform in
    [8192, 32768], page 16, shuffled pages, outlier channels x10, group 128."""
    rng = np.random.default_rng(np.random.SeedSequence(seed).spawn(9)[8])
    ctx = rng.integers(ctx_lo, ctx_hi + 1, size=B)
    return make_decode_workload(f"qwen3_8b_b{B}_h32x8_ctx{ctx_lo}-{ctx_hi}", seed, B=B, Hq=32,
                                Hkv=8, ctx=ctx, outliers_per_head=4, outlier_mul=10.0)


def qwen3_32b_long_decode(seed=5, B=16, ctx=131_072):
    """Batch 16, 64 q / 8 KV heads (GQA 8), context 131,072 each, page 32,
    N(0,1) K/V plus 0.1% token-norm outliers x20, Haar R, group 128."""
    return make_decode_workload(f"qwen3_32b_b{B}_h64x8_ctx{ctx}", seed, B=B, Hq=64, Hkv=8,
                                ctx=ctx, page_size=32, token_outlier_frac=0.001, token_mul=20.0)


@dataclass
class AppendWorkload:
    name: str
    n_seqs: int
    Hkv: int
    tokens_per_seq: np.ndarray     # int32 [n]
    hist_start: np.ndarray         # int32 [n]
    page_size: int
    group_size: int
    k: np.ndarray                  # uint16 [T, Hkv, d]
    v: np.ndarray
    cu_tokens: np.ndarray          # int32 [n+1]
    Rk: np.ndarray
    Rv: np.ndarray
    clip_k: np.ndarray
    clip_v: np.ndarray
    page_table: np.ndarray         # int32 [n, max_pages]
    num_pages: int


def make_append_workload(name, seed, n_seqs, Hkv, tokens_per_seq, hist_start=0, page_size=16,
                         group_size=64, kv_kind="t", clip_ratio=0.9):
    """Bulk eviction: each sequence moves ``tokens_per_seq`` tokens from the
    recent window into INT2 history starting at history position ``hist_start``."""
    ss = np.random.SeedSequence(seed)
    r_rot, r_kv, r_pt = [np.random.default_rng(s) for s in ss.spawn(3)]
    tps = np.broadcast_to(np.asarray(tokens_per_seq, np.int64), (n_seqs,)).astype(np.int32)
    hs = np.broadcast_to(np.asarray(hist_start, np.int64), (n_seqs,)).astype(np.int32)
    T = int(tps.sum())
    kind = "t" if kv_kind == "t" else "normal"
    k = _kv_rows(r_kv, T, Hkv, kind)
    v = _kv_rows(r_kv, T, Hkv, kind)
    Rk = np.stack([haar_orthogonal(r_rot) for _ in range(Hkv)])
    Rv = np.stack([haar_orthogonal(r_rot) for _ in range(Hkv)])
    kb, vb = f32_to_bf16_bits(k), f32_to_bf16_bits(v)
    clip_k = _clip_from([bf16_bits_to_f32(kb)], Rk, clip_ratio, calib_tokens=T)
    clip_v = _clip_from([bf16_bits_to_f32(vb)], Rv, clip_ratio, calib_tokens=T)
    cu = np.zeros(n_seqs + 1, np.int32); cu[1:] = np.cumsum(tps)
    pages_per_seq = (hs + tps + page_size - 1) // page_size
    pt, num_pages = _shuffled_page_table(r_pt, pages_per_seq)
    return AppendWorkload(name=name, n_seqs=n_seqs, Hkv=Hkv, tokens_per_seq=tps, hist_start=hs,
                          page_size=page_size, group_size=group_size, k=kb, v=vb, cu_tokens=cu,
                          Rk=Rk.astype(np.float32), Rv=Rv.astype(np.float32), clip_k=clip_k,
                          clip_v=clip_v, page_table=pt, num_pages=num_pages)


def append_64x4096(seed=3):
    """64 sequences x 8 KV heads, 4096 tokens each evicted in one call,
    Student-t(4) K/V, per-head Haar R (separate for K and V), clip 0.9,
    group 64, page 16."""
    return make_append_workload("append_s64_h8_t4096_g64", seed, 64, 8, 4096)
