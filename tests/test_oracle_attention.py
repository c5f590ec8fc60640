"""Pins for the oracle's attention and for the generated rotations (CPU only)."""

import numpy as np
import pytest

from oracle import attention as att
from oracle import kvquant as kq
from bit_kv_cache_12_gb300 import synth


def plain_attention(q, K, V, scale):
    l = scale * (K @ q)
    w = np.exp(l - l.max())
    return (w @ V) / w.sum()


@pytest.mark.parametrize("kind", ["haar", "oscar"])
def test_rotations_are_orthogonal(kind):
    rng = np.random.default_rng(3)
    R = synth.haar_orthogonal(rng) if kind == "haar" else synth.oscar_like_rotation(rng)
    assert np.abs(R @ R.T - np.eye(128)).max() <= 1e-12
    assert np.abs(R.astype(np.float32).astype(np.float64) @ R.astype(np.float32).astype(np.float64).T
                  - np.eye(128)).max() <= 2e-6


def test_oscar_rotation_components():
    """H is orthogonal and +-1/sqrt(d); the bit-reversal permutation is an
    involution; U H P_br is orthogonal (section 2.2 A composite)."""
    H = synth.hadamard(128)
    assert np.allclose(H @ H.T, np.eye(128), atol=1e-13)
    assert np.allclose(np.abs(H), 1 / np.sqrt(128))
    P = synth.bit_reversal_permutation(128)
    assert np.array_equal(P @ P, np.eye(128))
    x = np.arange(128.0)
    assert (x @ P)[1] == 64.0 and (x @ P)[2] == 32.0


def _rand_tiers(rng, ns, nh, nr, scale_k=1.0):
    d = 128
    return (rng.standard_normal((ns, d)) * scale_k, rng.standard_normal((ns, d)),
            rng.standard_normal((nh, d)) * scale_k, rng.standard_normal((nh, d)),
            rng.standard_normal((nr, d)) * scale_k, rng.standard_normal((nr, d)))


@pytest.mark.parametrize("ns,nh,nr", [(5, 17, 9), (0, 30, 0), (3, 0, 4), (64, 700, 256)])
def test_rotation_invariance_without_quantization(ns, nh, nr):
    """History stored rotated but not quantized (k' = k R_k, v' = v R_v):
    the three-tier attention must equal plain attention on the original
    tokens.  Fails if R and R^T are swapped anywhere."""
    rng = np.random.default_rng(ns * 1000 + nh + nr)
    sk, sv, hk, hv, rk, rv = _rand_tiers(rng, ns, nh, nr)
    Rk = synth.haar_orthogonal(rng); Rv = synth.haar_orthogonal(rng)
    q = rng.standard_normal(128)
    got = att.three_tier_head(q, Rk, Rv, sk, sv, hk @ Rk, hv @ Rv, rk, rv, 0.088)
    want = plain_attention(q, np.concatenate([sk, hk, rk]), np.concatenate([sv, hv, rv]), 0.088)
    assert np.abs(got - want).max() <= 1e-12 * max(1.0, np.abs(want).max())


def _brute_force_longdouble(q, Rk, Rv, sk, sv, hk_rot, hv_rot, rk, rv, scale):
    """Independent formulation: history keys and values rotated back to the
    original basis first (k = k' R^T), no max subtraction, long double."""
    ld = np.longdouble
    q = q.astype(ld)
    keys = [sk.astype(ld), hk_rot.astype(ld) @ Rk.T.astype(ld), rk.astype(ld)]
    vals = [sv.astype(ld), hv_rot.astype(ld) @ Rv.T.astype(ld), rv.astype(ld)]
    num = np.zeros(128, ld); den = ld(0)
    for K, V in zip(keys, vals):
        for t in range(K.shape[0]):
            w = np.exp(ld(scale) * np.dot(K[t], q))
            num += w * V[t]; den += w
    return (num / den).astype(np.float64)


def test_brute_force_small_quantized():
    """<= 64 tokens with real INT2 history: oracle vs independent brute force."""
    rng = np.random.default_rng(21)
    Rk = synth.haar_orthogonal(rng); Rv = synth.haar_orthogonal(rng)
    sk, sv, hk, hv, rk, rv = _rand_tiers(rng, 8, 40, 16)
    qk = kq.quantize_rows((hk @ Rk).astype(np.float32), np.full(128, np.inf, np.float32), 128)
    qv = kq.quantize_rows((hv @ Rv).astype(np.float32), np.full(128, np.inf, np.float32), 128)
    kd = kq.dequant(*qk, 128); vd = kq.dequant(*qv, 128)
    q = rng.standard_normal(128)
    got = att.three_tier_head(q, Rk, Rv, sk, sv, kd, vd, rk, rv, 0.088)
    want = _brute_force_longdouble(q, Rk, Rv, sk, sv, kd, vd, rk, rv, 0.088)
    assert np.abs(got - want).max() <= 1e-12 * np.abs(want).max()


def test_closed_forms():
    rng = np.random.default_rng(8)
    Rk = synth.haar_orthogonal(rng); Rv = synth.haar_orthogonal(rng)
    sk, sv, hk, hv, rk, rv = _rand_tiers(rng, 4, 12, 6)
    # q = 0 -> uniform weights -> mean of all values (history rotated back)
    got = att.three_tier_head(np.zeros(128), Rk, Rv, sk, sv, hk, hv, rk, rv, 0.1)
    want = np.concatenate([sv, hv @ Rv.T, rv]).mean(0)
    assert np.abs(got - want).max() <= 1e-12
    # a single token -> its value
    got = att.three_tier_head(rng.standard_normal(128), Rk, Rv, sk[:0], sv[:0], hk[:1], hv[:1],
                              rk[:0], rv[:0], 0.1)
    assert np.abs(got - hv[0] @ Rv.T).max() <= 1e-12
    got = att.three_tier_head(rng.standard_normal(128), Rk, Rv, sk[:1], sv[:1], hk[:0], hv[:0],
                              rk[:0], rv[:0], 0.1)
    assert np.abs(got - sv[0]).max() <= 1e-12
    # all keys equal (history key stored rotated) -> mean of values
    k0 = rng.standard_normal(128)
    K = np.tile(k0, (4, 1))
    got = att.three_tier_head(rng.standard_normal(128), Rk, Rv, K[:2], sv[:2], K[:1] @ Rk,
                              hv[:1], K[:1], rv[:1], 0.3)
    want = np.concatenate([sv[:2], hv[:1] @ Rv.T, rv[:1]]).mean(0)
    assert np.abs(got - want).max() <= 1e-12


def test_grid_exact_int2_equals_plain_attention():
    """R = I, no clip, history values on the quantization grid: the INT2
    history is lossless, so three-tier attention = plain fp64 attention."""
    rng = np.random.default_rng(4)
    n = 50
    z = np.float32(-2.0); s = np.float32(1.25)
    k = rng.integers(0, 4, (n, 128)); k[:, 0] = 0; k[:, 1] = 3
    v = rng.integers(0, 4, (n, 128)); v[:, 0] = 0; v[:, 1] = 3
    hk = (z + k * s).astype(np.float32); hv = (z + v * s).astype(np.float32)
    I = np.eye(128); inf = np.full(128, np.inf, np.float32)
    kd = kq.dequant(*kq.quantize_rows(hk, inf, 128), 128)
    vd = kq.dequant(*kq.quantize_rows(hv, inf, 128), 128)
    sk, sv, _, _, rk, rv = _rand_tiers(rng, 3, 0, 5)
    q = rng.standard_normal(128)
    got = att.three_tier_head(q, I, I, sk, sv, kd, vd, rk, rv, 0.05)
    want = plain_attention(q, np.concatenate([sk, hk, rk]), np.concatenate([sv, hv, rv]), 0.05)
    assert np.abs(got - want).max() <= 1e-12


def test_ring_order():
    ring = np.arange(10)[:, None] * np.ones((1, 2))
    got = att.ring_order(ring, 7, 5, 10)[:, 0]
    assert got.tolist() == [7, 8, 9, 0, 1]


def test_bf16_paged_oracle_matches_plain():
    rng = np.random.default_rng(12)
    P, Hkv, Hq = 16, 2, 4
    n = 37
    pages = rng.permutation(8)[:3]
    kp = np.zeros((8, Hkv, P, 128), np.uint16); vp = kp.copy()
    K = synth.f32_to_bf16_bits(rng.standard_normal((n, Hkv, 128)).astype(np.float32))
    V = synth.f32_to_bf16_bits(rng.standard_normal((n, Hkv, 128)).astype(np.float32))
    for t in range(n):
        kp[pages[t // P], :, t % P] = K[t]; vp[pages[t // P], :, t % P] = V[t]
    q = synth.f32_to_bf16_bits(rng.standard_normal((1, Hq, 128)).astype(np.float32))
    out = att.decode_bf16_paged(q, kp, vp, pages[None, :], [n], Hkv, P, 0.088)
    for h in range(Hq):
        want = plain_attention(kq.bf16_bits_to_f64(q[0, h]), kq.bf16_bits_to_f64(K[:, h // 2]),
                               kq.bf16_bits_to_f64(V[:, h // 2]), 0.088)
        assert np.abs(out[0, h] - want).max() <= 1e-12


def test_three_tier_decode_on_tiny_workload_is_sane():
    """The batch entry reproduces the per-head function and the output lies in
    the convex hull bound of the values."""
    wl = synth.tiny_decode()
    pages = np.zeros((wl.num_pages, wl.Hkv, kq.tile_bytes(128)), np.uint8)
    for g in range(wl.Hkv):
        qq = kq.quantize_tokens(wl.hist_k[0][:, g], wl.hist_v[0][:, g], wl.Rk[g], wl.Rv[g],
                                wl.clip_k[g], wl.clip_v[g], 128)
        kq.pack_history(pages, wl.page_table[0], 0, qq, g, wl.Hkv, 16, 128)
    hist = lambda b, g: kq.read_history(pages, wl.page_table[b], int(wl.hist_len[b]), g, 16, 128)
    out = att.decode_three_tier(wl.q, wl.Rk, wl.Rv, wl.sink_k, wl.sink_v, wl.sink_len, hist,
                                wl.hist_len, wl.rec_k, wl.rec_v, wl.rec_len, wl.rec_start,
                                wl.Hkv, 128, wl.scale)
    assert out.shape == (1, 8, 128) and np.all(np.isfinite(out))
    assert np.abs(out).max() < 20


def test_log_sum_exp_closed_forms_and_library():
    """ln sum_t exp(l_t): a single token gives its scaled score; N equal keys
    give that score + ln N; a small random case equals scipy's logsumexp of
    scores formed independently (keys rotated back, q not rotated)."""
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(31)
    d, tau = 128, 0.11
    R = synth.haar_orthogonal(rng)
    e = np.zeros((0, d))
    q = rng.standard_normal(d)
    k1 = rng.standard_normal((1, d)); v1 = rng.standard_normal((1, d))
    _, lse = att.three_tier_head(q, R, R, k1, v1, e, e, e, e, tau, return_lse=True)
    assert abs(lse - tau * float(q @ k1[0])) <= 1e-12 * max(1.0, abs(lse))
    kN = np.repeat(k1, 7, axis=0); vN = rng.standard_normal((7, d))
    _, lse7 = att.three_tier_head(q, R, R, kN, vN, e, e, e, e, tau, return_lse=True)
    assert abs(lse7 - (tau * float(q @ k1[0]) + np.log(7.0))) <= 1e-12 * max(1.0, abs(lse7))
    sink = rng.standard_normal((3, d)); hist = rng.standard_normal((5, d)); rec = rng.standard_normal((4, d))
    vals = rng.standard_normal((12, d))
    _, lse_r = att.three_tier_head(q, R, R, sink, vals[:3], hist, vals[3:8], rec, vals[8:], tau,
                                   return_lse=True)
    keys_orig = np.concatenate([sink, hist @ R.T, rec])       # history keys back in the original basis
    assert abs(lse_r - scipy_special.logsumexp(tau * keys_orig @ q)) <= 1e-12 * abs(lse_r)


def test_multi_query_is_independent_single_queries():
    wl = synth.make_decode_workload("mq", 32, B=2, Hq=4, Hkv=2, ctx=[400, 700], page_size=16)
    pages = np.zeros((wl.num_pages, wl.Hkv, kq.tile_bytes(wl.group_size)), np.uint8)
    for b in range(wl.B):
        kq.pack_history_full(wl.hist_k[b], wl.hist_v[b], wl.Rk, wl.Rv, wl.clip_k, wl.clip_v, wl.page_table[b],
                             wl.num_pages, wl.Hkv, wl.page_size, wl.group_size, pages)
    hist = lambda b, g: kq.read_history(pages, wl.page_table[b], int(wl.hist_len[b]), g, wl.page_size,
                                        wl.group_size)
    rng = np.random.default_rng(33)
    T = 3
    qm = synth.f32_to_bf16_bits(rng.standard_normal((wl.B, T, wl.Hq, 128)).astype(np.float32))
    out, lse = att.decode_three_tier_multi(qm, wl.Rk, wl.Rv, wl.sink_k, wl.sink_v, wl.sink_len, hist,
                                           wl.hist_len, wl.rec_k, wl.rec_v, wl.rec_len, wl.rec_start,
                                           wl.Hkv, wl.group_size, wl.scale)
    assert out.shape == (wl.B, T, wl.Hq, 128) and lse.shape == (wl.B, T, wl.Hq)
    for t in range(T):
        one = att.decode_three_tier(qm[:, t], wl.Rk, wl.Rv, wl.sink_k, wl.sink_v, wl.sink_len, hist,
                                    wl.hist_len, wl.rec_k, wl.rec_v, wl.rec_len, wl.rec_start, wl.Hkv,
                                    wl.group_size, wl.scale)
        assert np.array_equal(out[:, t], one)


# ---------------------------------------------------------------------------
# the batch wrapper (decode_three_tier): GQA mapping, per-sequence lengths and
# ring starts, checked per (sequence, query head) against formulations that
# share none of its indexing
# ---------------------------------------------------------------------------

def _ragged_workload(seed, ctx, sink=8, recent=16):
    return synth.make_decode_workload(f"ragged{seed}", seed, B=len(ctx), Hq=8, Hkv=2, ctx=ctx,
                                      page_size=16, group_size=64, sink=sink, recent=recent,
                                      outliers_per_head=2)


def _oracle_pages(wl):
    pages = np.zeros((wl.num_pages, wl.Hkv, kq.tile_bytes(wl.group_size)), np.uint8)
    for b in range(wl.B):
        if wl.hist_len[b]:
            kq.pack_history_full(wl.hist_k[b], wl.hist_v[b], wl.Rk, wl.Rv, wl.clip_k, wl.clip_v,
                                 wl.page_table[b], wl.num_pages, wl.Hkv, wl.page_size, wl.group_size,
                                 pages)
    return pages


def test_batch_wrapper_each_head_equals_hand_assembled_brute_force():
    """Ragged batch (history 0, a partial tile, several tiles; short sink and
    partly filled rings starting mid-ring): output (b, h) equals the long-double
    brute force of KV head h // G of sequence b, its tokens gathered here with
    explicit loops (ring slot (start + t) mod capacity)."""
    wl = _ragged_workload(41, [5, 30, 61, 19])
    assert list(wl.hist_len) == [0, 6, 37, 0] and list(wl.rec_len) == [0, 16, 16, 11]
    pages = _oracle_pages(wl)
    hist = lambda b, g: kq.read_history(pages, wl.page_table[b], int(wl.hist_len[b]), g,
                                        wl.page_size, wl.group_size)
    out = att.decode_three_tier(wl.q, wl.Rk, wl.Rv, wl.sink_k, wl.sink_v, wl.sink_len, hist,
                                wl.hist_len, wl.rec_k, wl.rec_v, wl.rec_len, wl.rec_start, wl.Hkv,
                                wl.group_size, wl.scale)
    G = wl.Hq // wl.Hkv
    cap = wl.rec_k.shape[2]
    for b in range(wl.B):
        for h in range(wl.Hq):
            g = h // G
            sk = kq.bf16_bits_to_f64(wl.sink_k[b, g, :wl.sink_len[b]])
            sv = kq.bf16_bits_to_f64(wl.sink_v[b, g, :wl.sink_len[b]])
            slots = [(int(wl.rec_start[b]) + t) % cap for t in range(int(wl.rec_len[b]))]
            rk = kq.bf16_bits_to_f64(np.array([wl.rec_k[b, g, s] for s in slots]).reshape(-1, 128))
            rv = kq.bf16_bits_to_f64(np.array([wl.rec_v[b, g, s] for s in slots]).reshape(-1, 128))
            kc, vc, skk, zk, svv, zv = kq.read_history(pages, wl.page_table[b], int(wl.hist_len[b]), g,
                                                        wl.page_size, wl.group_size)
            kd = kq.dequant(kc, skk, zk, wl.group_size)
            vd = kq.dequant(vc, svv, zv, wl.group_size)
            want = _brute_force_longdouble(kq.bf16_bits_to_f64(wl.q[b, h]), wl.Rk[g].astype(np.float64),
                                           wl.Rv[g].astype(np.float64), sk, sv, kd, vd, rk, rv, wl.scale)
            assert np.abs(out[b, h] - want).max() <= 1e-12 * max(1.0, np.abs(want).max()), (b, h)


def test_batch_wrapper_without_history_equals_bf16_paged():
    """History 0 for every sequence: the three-tier wrapper equals the all-BF16
    paged decode of the same tokens (sink, then the ring from its start) placed
    in shuffled pages, and each head equals plain attention over the tokens of
    KV head h // G."""
    wl = _ragged_workload(42, [3, 8, 20, 24])
    assert int(wl.hist_len.max()) == 0
    rng = np.random.default_rng(42)
    P, cap = 16, wl.rec_k.shape[2]
    lens = (wl.sink_len + wl.rec_len).astype(int)
    npg = (lens + P - 1) // P
    perm = rng.permutation(int(npg.sum()) + 2)
    kp = np.zeros((len(perm), wl.Hkv, P, 128), np.uint16); vp = kp.copy()
    pt = np.full((wl.B, int(npg.max())), -1, np.int32)
    o = 0
    toks = []
    for b in range(wl.B):
        pt[b, :npg[b]] = perm[o:o + npg[b]]; o += npg[b]
        order = [wl.sink_k[b, :, t] for t in range(wl.sink_len[b])]
        vorder = [wl.sink_v[b, :, t] for t in range(wl.sink_len[b])]
        for t in range(int(wl.rec_len[b])):
            s = (int(wl.rec_start[b]) + t) % cap
            order.append(wl.rec_k[b, :, s]); vorder.append(wl.rec_v[b, :, s])
        K = np.array(order).reshape(-1, wl.Hkv, 128); V = np.array(vorder).reshape(-1, wl.Hkv, 128)
        for t in range(lens[b]):
            kp[pt[b, t // P], :, t % P] = K[t]; vp[pt[b, t // P], :, t % P] = V[t]
        toks.append((K, V))
    empty = lambda b, g: kq.read_history(np.zeros((1, wl.Hkv, kq.tile_bytes(64)), np.uint8),
                                         np.zeros(1, np.int32), 0, g, P, 64)
    got = att.decode_three_tier(wl.q, wl.Rk, wl.Rv, wl.sink_k, wl.sink_v, wl.sink_len, empty,
                                wl.hist_len, wl.rec_k, wl.rec_v, wl.rec_len, wl.rec_start, wl.Hkv,
                                64, wl.scale)
    ref = att.decode_bf16_paged(wl.q, kp, vp, pt, lens, wl.Hkv, P, wl.scale)
    assert np.abs(got - ref).max() <= 1e-13
    G = wl.Hq // wl.Hkv
    for b in range(wl.B):
        K, V = toks[b]
        for h in range(wl.Hq):
            want = plain_attention(kq.bf16_bits_to_f64(wl.q[b, h]), kq.bf16_bits_to_f64(K[:, h // G]),
                                   kq.bf16_bits_to_f64(V[:, h // G]), wl.scale)
            assert np.abs(got[b, h] - want).max() <= 1e-12, (b, h)
