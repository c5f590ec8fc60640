"""Oracle: fp64 decode attention over the three-tier token pool (CPU, numpy).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Three tiers per sequence and KV head (yunpan.plus OSCAR write-up,
"1. 三段式 Token 池"; gist.science OSCAR explainer, section 2.2 B):
  sink    first 64 tokens, BF16, unrotated
  history middle tokens, INT2 codes of the rotated + clipped values
  recent  last 256 tokens, BF16, unrotated, kept in a ring buffer

One decode step for query head h of sequence b, KV head g = h // (Hq/Hkv):
  q'      = q . R_k[g]                       (history keys live in rotated space)
  l_t     = tau * q . k_t        for sink and recent tokens
  l_t     = tau * q' . deq(k'_t) for history tokens
  w_t     = exp(l_t - max l)
  o       = ( sum_{sink,recent} w_t v_t + (sum_hist w_t deq(v'_t)) . R_v[g]^T )
            / sum_t w_t
The inverse rotation of the value accumulator is the "inverse Rotation" the
explainer puts inside the attention kernel (section 2.2 B, Kernel-Integration).
tau is the caller's softmax scale (1/sqrt(d) by default; the pages are silent).

Several queries per sequence (a chunk continuing on the cached prefix, or
draft tokens being verified) each attend over the same cache independently;
with ``return_lse`` the natural log of sum_t exp(l_t) is returned as well, so
that a caller can merge the cache part with attention over the chunk's own
tokens by the log-sum-exp rule.
"""

import numpy as np

from . import kvquant as kq


def _softmax_combine(scores, values):
    m = np.max(scores)
    w = np.exp(scores - m)
    return (w[:, None] * values).sum(axis=0) / w.sum(), w


def three_tier_head(q, Rk, Rv, sink_k, sink_v, hist_k_deq, hist_v_deq, rec_k, rec_v, scale,
                    return_lse=False):
    """Attention for one query head.

    q [d]; Rk, Rv [d, d]; sink_k/v [S, d]; hist_*_deq [H, d] (rotated space,
    already dequantized); rec_k/v [W, d] in logical order (oldest first).
    All fp64.  Returns o [d] (and ln sum_t exp(l_t) with ``return_lse``)."""
    q = np.asarray(q, np.float64)
    qr = q @ Rk
    parts_l = []
    if sink_k.shape[0]:
        parts_l.append(scale * (sink_k @ q))
    if hist_k_deq.shape[0]:
        parts_l.append(scale * (hist_k_deq @ qr))
    if rec_k.shape[0]:
        parts_l.append(scale * (rec_k @ q))
    scores = np.concatenate(parts_l)
    m = scores.max()
    w = np.exp(scores - m)
    ns, nh = sink_k.shape[0], hist_k_deq.shape[0]
    ws, wh, wr = w[:ns], w[ns:ns + nh], w[ns + nh:]
    o = np.zeros(q.shape[0])
    if ns:
        o += ws @ sink_v
    if nh:
        o += (wh @ hist_v_deq) @ Rv.T
    if rec_k.shape[0]:
        o += wr @ rec_v
    if return_lse:
        return o / w.sum(), m + np.log(w.sum())
    return o / w.sum()


def ring_order(ring, start, length, capacity):
    """Logical (oldest-first) rows of a ring buffer [capacity, d]."""
    idx = (start + np.arange(length)) % capacity
    return ring[idx]


def decode_three_tier(q_bits, Rk, Rv, sink_k_bits, sink_v_bits, sink_len, hist, hist_len,
                      rec_k_bits, rec_v_bits, rec_len, rec_start, num_kv_heads, group_size,
                      scale):
    """Whole batch, one layer.

    q_bits [B, Hq, d] bf16 bits; Rk/Rv [Hkv, d, d] float; sink_*_bits
    [B, Hkv, S_cap, d]; rec_*_bits [B, Hkv, W_cap, d]; hist: callable
    (b, g) -> (kc, vc, sk, zk, sv, zv) for the hist_len[b] history tokens.
    Returns out [B, Hq, d] fp64."""
    B, Hq, d = q_bits.shape
    G = Hq // num_kv_heads
    W_cap = rec_k_bits.shape[2]
    out = np.zeros((B, Hq, d))
    for b in range(B):
        for g in range(num_kv_heads):
            kc, vc, sk, zk, sv, zv = hist(b, g)
            kd = kq.dequant(kc, sk, zk, group_size)
            vd = kq.dequant(vc, sv, zv, group_size)
            sk_ = kq.bf16_bits_to_f64(sink_k_bits[b, g, :sink_len[b]])
            sv_ = kq.bf16_bits_to_f64(sink_v_bits[b, g, :sink_len[b]])
            rk = kq.bf16_bits_to_f64(ring_order(rec_k_bits[b, g], rec_start[b], rec_len[b], W_cap))
            rv = kq.bf16_bits_to_f64(ring_order(rec_v_bits[b, g], rec_start[b], rec_len[b], W_cap))
            Rk64 = np.asarray(Rk[g], np.float64); Rv64 = np.asarray(Rv[g], np.float64)
            for hh in range(G):
                h = g * G + hh
                qf = kq.bf16_bits_to_f64(q_bits[b, h])
                out[b, h] = three_tier_head(qf, Rk64, Rv64, sk_, sv_, kd[:hist_len[b]],
                                            vd[:hist_len[b]], rk, rv, scale)
    return out


def decode_three_tier_multi(q_bits, Rk, Rv, sink_k_bits, sink_v_bits, sink_len, hist, hist_len,
                            rec_k_bits, rec_v_bits, rec_len, rec_start, num_kv_heads, group_size,
                            scale):
    """T queries per sequence over the same cache: q_bits [B, T, Hq, d].
    Returns out [B, T, Hq, d] and lse [B, T, Hq] (natural log), fp64."""
    B, T, Hq, d = q_bits.shape
    G = Hq // num_kv_heads
    W_cap = rec_k_bits.shape[2]
    out = np.zeros((B, T, Hq, d))
    lse = np.zeros((B, T, Hq))
    for b in range(B):
        for g in range(num_kv_heads):
            kc, vc, sk, zk, sv, zv = hist(b, g)
            kd = kq.dequant(kc, sk, zk, group_size)
            vd = kq.dequant(vc, sv, zv, group_size)
            sk_ = kq.bf16_bits_to_f64(sink_k_bits[b, g, :sink_len[b]])
            sv_ = kq.bf16_bits_to_f64(sink_v_bits[b, g, :sink_len[b]])
            rk = kq.bf16_bits_to_f64(ring_order(rec_k_bits[b, g], rec_start[b], rec_len[b], W_cap))
            rv = kq.bf16_bits_to_f64(ring_order(rec_v_bits[b, g], rec_start[b], rec_len[b], W_cap))
            Rk64 = np.asarray(Rk[g], np.float64); Rv64 = np.asarray(Rv[g], np.float64)
            for t in range(T):
                for hh in range(G):
                    h = g * G + hh
                    qf = kq.bf16_bits_to_f64(q_bits[b, t, h])
                    out[b, t, h], lse[b, t, h] = three_tier_head(
                        qf, Rk64, Rv64, sk_, sv_, kd[:hist_len[b]], vd[:hist_len[b]], rk, rv, scale,
                        return_lse=True)
    return out, lse


def decode_bf16_paged(q_bits, k_pages_bits, v_pages_bits, page_table, seq_len, num_kv_heads,
                      page_size, scale):
    """Plain softmax attention over an all-BF16 paged cache.

    k/v_pages_bits [num_pages, Hkv, page_size, d]; page_table [B, max_pages];
    seq_len [B].  Returns [B, Hq, d] fp64."""
    B, Hq, d = q_bits.shape
    G = Hq // num_kv_heads
    out = np.zeros((B, Hq, d))
    for b in range(B):
        n = int(seq_len[b])
        pos = np.arange(n)
        pages = np.asarray(page_table[b])[pos // page_size]
        for g in range(num_kv_heads):
            K = kq.bf16_bits_to_f64(k_pages_bits[pages, g, pos % page_size])
            V = kq.bf16_bits_to_f64(v_pages_bits[pages, g, pos % page_size])
            for hh in range(G):
                h = g * G + hh
                qf = kq.bf16_bits_to_f64(q_bits[b, h])
                o, _ = _softmax_combine(scale * (K @ qf), V)
                out[b, h] = o
    return out
