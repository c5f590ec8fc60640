"""Pins for ``oracle.tiers.append_step`` (CPU).

The yunpan.plus OSCAR write-up, "1. 三段式 Token 池" and "2. 在线量化与反量化":
the sink keeps the first tokens, the recent tier keeps the latest ones, the
rest is INT2 history; a new token enters the recent tier and, when that is
full, the oldest recent token is rotated, clipped, quantized, packed and moved
into history.  Streaming tokens one by one into an empty pool must therefore
leave exactly: the first S tokens in the sink, the last W tokens in the recent
ring (oldest first from the start index), and every token in between in
history, quantized exactly as the bulk append path quantizes them."""

import copy

import numpy as np
import pytest

from bit_kv_cache_12_gb300 import synth
from oracle import attention as att
from oracle import kvquant as kq
from oracle import tiers


def _state(B, Hkv, S, W, num_pages, page_size, group_size):
    tb = kq.tile_bytes(group_size) * (page_size // 16)
    return dict(sink_k=np.zeros((B, Hkv, S, 128), np.uint16), sink_v=np.zeros((B, Hkv, S, 128), np.uint16),
                rec_k=np.zeros((B, Hkv, W, 128), np.uint16), rec_v=np.zeros((B, Hkv, W, 128), np.uint16),
                sink_len=np.zeros(B, np.int64), hist_len=np.zeros(B, np.int64),
                rec_len=np.zeros(B, np.int64), rec_start=np.zeros(B, np.int64),
                pages=np.zeros((num_pages, Hkv, tb), np.uint8))


def _tokens(rng, n, B, Hkv):
    x = rng.standard_normal((n, B, Hkv, 128)).astype(np.float32)
    x[..., 7] *= 6.0
    return synth.f32_to_bf16_bits(x)


@pytest.mark.parametrize("page_size,group_size", [(16, 128), (32, 64)])
def test_stream_from_empty_follows_the_tier_rule(page_size, group_size):
    rng = np.random.default_rng(11)
    B, Hkv, S, W = 2, 2, 4, 8
    n_hist = 45                                   # crosses tiles and pages
    N = S + W + n_hist
    pages_per = (n_hist + page_size - 1) // page_size
    num_pages = B * pages_per + 2
    perm = rng.permutation(num_pages).astype(np.int32)
    pt = perm[:B * pages_per].reshape(B, pages_per)
    Rk = np.stack([synth.haar_orthogonal(rng) for _ in range(Hkv)])
    Rv = np.stack([synth.haar_orthogonal(rng) for _ in range(Hkv)])
    ck = np.full((Hkv, 128), 2.5, np.float32); cv = np.full((Hkv, 128), np.inf, np.float32)
    toks_k, toks_v = _tokens(rng, N, B, Hkv), _tokens(rng, N, B, Hkv)
    st = _state(B, Hkv, S, W, num_pages, page_size, group_size)
    for i in range(N):
        assert tiers.append_step(st, toks_k[i], toks_v[i], pt, Rk, Rv, ck, cv, page_size,
                                 group_size) == []
    assert list(st["sink_len"]) == [S] * B
    assert list(st["rec_len"]) == [W] * B
    assert list(st["hist_len"]) == [n_hist] * B
    bulk = np.zeros_like(st["pages"])
    for b in range(B):
        for g in range(Hkv):
            assert np.array_equal(st["sink_k"][b, g], toks_k[:S, b, g])
            assert np.array_equal(st["sink_v"][b, g], toks_v[:S, b, g])
            assert np.array_equal(att.ring_order(st["rec_k"][b, g], st["rec_start"][b], W, W),
                                  toks_k[N - W:, b, g])
            assert np.array_equal(att.ring_order(st["rec_v"][b, g], st["rec_start"][b], W, W),
                                  toks_v[N - W:, b, g])
        kq.pack_history_full(toks_k[S:S + n_hist, b], toks_v[S:S + n_hist, b], Rk, Rv, ck, cv, pt[b],
                             num_pages, Hkv, page_size, group_size, bulk)
        for g in range(Hkv):
            got = kq.read_history(st["pages"], pt[b], n_hist, g, page_size, group_size)
            ref = kq.read_history(bulk, pt[b], n_hist, g, page_size, group_size)
            for a, r in zip(got, ref):
                assert np.array_equal(a, r)


def test_partial_tiers_take_the_token_without_eviction():
    rng = np.random.default_rng(12)
    B, Hkv, S, W = 3, 1, 4, 8
    st = _state(B, Hkv, S, W, 4, 16, 128)
    st["sink_len"][:] = [2, 4, 4]
    st["rec_len"][:] = [0, 3, 8]
    st["rec_start"][:] = [0, 6, 5]
    pt = np.array([[0], [1], [2]], np.int32)
    R = np.eye(128)[None]
    k, v = _tokens(rng, 1, B, Hkv)[0], _tokens(rng, 1, B, Hkv)[0]
    before = copy.deepcopy(st)
    tiers.append_step(st, k, v, pt, R, R, np.full((1, 128), np.inf), np.full((1, 128), np.inf), 16, 128)
    assert np.array_equal(st["sink_k"][0, 0, 2], k[0, 0]) and st["sink_len"][0] == 3
    assert np.array_equal(st["rec_k"][1, 0, (6 + 3) % 8], k[1, 0]) and st["rec_len"][1] == 4
    # sequence 2: ring full -> oldest (slot 5) leaves for history position 0
    assert st["hist_len"][2] == 1 and st["rec_start"][2] == 6
    assert np.array_equal(st["rec_k"][2, 0, 5], k[2, 0])
    kc = kq.read_history(st["pages"], pt[2], 1, 0, 16, 128)[0]
    q = kq.quantize_tokens(before["rec_k"][2, 0, 5][None], before["rec_v"][2, 0, 5][None], R[0], R[0],
                           np.full(128, np.inf), np.full(128, np.inf), 128)
    assert np.array_equal(kc, q["kc"])


def test_missing_page_refuses_the_step_and_changes_nothing():
    rng = np.random.default_rng(13)
    B, Hkv, S, W = 2, 2, 4, 8
    st = _state(B, Hkv, S, W, 2, 16, 128)
    st["sink_len"][:] = S
    st["rec_len"][:] = W
    st["rec_start"][:] = [3, 0]
    st["hist_len"][:] = [16, 5]                       # sequence 0 needs page index 1
    st["rec_k"][:] = _tokens(rng, 1, B * Hkv * W, 1)[0].reshape(B, Hkv, W, 128)
    pt = np.array([[0, -1], [1, -1]], np.int32)
    R = np.stack([np.eye(128)] * Hkv)
    inf = np.full((Hkv, 128), np.inf)
    before = copy.deepcopy(st)
    k, v = _tokens(rng, 1, B, Hkv)[0], _tokens(rng, 1, B, Hkv)[0]
    assert tiers.append_step(st, k, v, pt, R, R, inf, inf, 16, 128) == [0]
    for key in ("sink_k", "rec_k", "rec_v"):
        assert np.array_equal(st[key][0], before[key][0])
    assert st["hist_len"][0] == 16 and st["rec_start"][0] == 3
    assert st["hist_len"][1] == 6 and st["rec_start"][1] == 1   # the other sequence stepped
