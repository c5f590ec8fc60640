"""GPU parity of the per-step token placement (``kv_append_step``).

The yunpan.plus OSCAR write-up ("1. 三段式 Token 池", "2. 在线量化与反量化"):
a new token enters the recent tier; when that is full, the oldest recent token
is rotated, clipped, quantized and packed into the INT2 history.  The library
runs this on the device and updates the length arrays in place.  Checked
against ``oracle.tiers.append_step``: lengths and BF16 tiers exactly, history
codes up to rounding-boundary flips of the rotation (as in the append tests);
against the library's own bulk append of the same tokens bit-exactly (both
paths rotate and quantize with the same tensor-core product and epilogue); and
the decode that follows, reading the device-updated lengths, against the oracle
on the stored codes."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from bit_kv_cache_12_gb300 import native, synth
from oracle import attention as att
from oracle import kvquant as kq
from oracle import tiers
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 1e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    native.lib()


def _setup(rng, B, Hkv, Hq, P, GS, S, W, num_pages, clip=2.5):
    Rk = np.stack([synth.haar_orthogonal(rng) for _ in range(Hkv)])
    Rv = np.stack([synth.haar_orthogonal(rng) for _ in range(Hkv)])
    ck = np.full((Hkv, 128), clip, np.float32)
    cv = np.full((Hkv, 128), np.inf, np.float32)

    def make():
        pool = native.KVPool(native.KV_POOL_INT2_3TIER, 1, Hq, Hkv, P, num_pages, B, group_size=GS,
                             sink_tokens=S, recent_tokens=W)
        keep = (gu.f32_dev(Rk), gu.f32_dev(Rv), gu.f32_dev(ck), gu.f32_dev(cv))
        native.kv_pool_set_rotation(pool.handle, 0, *keep)
        pool._keep = keep
        return pool
    return make, Rk, Rv, ck, cv


def _tokens(rng, n, B, Hkv):
    x = rng.standard_normal((n, B, Hkv, 128)).astype(np.float32)
    x[..., 7] *= 6.0
    return synth.f32_to_bf16_bits(x)


def _empty_state(B, Hkv, S, W, num_pages, P, GS):
    tb = kq.tile_bytes(GS) * (P // 16)
    return dict(sink_k=np.zeros((B, Hkv, S, 128), np.uint16), sink_v=np.zeros((B, Hkv, S, 128), np.uint16),
                rec_k=np.zeros((B, Hkv, W, 128), np.uint16), rec_v=np.zeros((B, Hkv, W, 128), np.uint16),
                sink_len=np.zeros(B, np.int64), hist_len=np.zeros(B, np.int64),
                rec_len=np.zeros(B, np.int64), rec_start=np.zeros(B, np.int64),
                pages=np.zeros((num_pages, Hkv, tb), np.uint8))


def _u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _gpu_tiers(pool, B):
    sk, sv, rk, rv = pool.tier_views(0)
    return _u16(sk[:B]), _u16(sv[:B]), _u16(rk[:B]), _u16(rv[:B])


def _history_close(gpu_pages, ref_pages, pt, hist_len, Hkv, P, GS):
    """Codes equal up to a few rounding-boundary flips; s/z within one fp16 ulp."""
    bad = tot = 0
    for b in range(pt.shape[0]):
        for g in range(Hkv):
            got = kq.read_history(gpu_pages, pt[b], int(hist_len[b]), g, P, GS)
            ref = kq.read_history(ref_pages, pt[b], int(hist_len[b]), g, P, GS)
            for a, r in zip(got[:2], ref[:2]):
                bad += int((a != r).sum()); tot += a.size
            for a, r in zip(got[2:], ref[2:]):
                du = np.abs(a.view(np.int16).astype(np.int64) - r.view(np.int16).astype(np.int64))
                assert du.max(initial=0) <= 1
    assert bad <= max(4, 1e-4 * tot), (bad, tot)


def _decode_vs_oracle(pool, st, q, pt, Rk, Rv, GS, Hkv, lens_dev, scale):
    """Decode with the device-updated lengths; oracle on the GPU's stored codes."""
    B = q.shape[0]
    sl, hl, rl, rs = lens_dev
    mh = int(st["hist_len"].max())
    ws_bytes = native.kv_decode_workspace_bytes(pool.handle, B, mh)
    ws = torch.empty(max(ws_bytes, 16) // 4 + 4, dtype=torch.float32, device="cuda")
    out = torch.full((B, q.shape[1], 128), float("nan"), dtype=torch.float32, device="cuda")
    native.kv_decode_attention(pool.handle, 0, B, gu.bf16_dev(q), sl, hl, rl, rs, gu.i32_dev(pt),
                               pt.shape[1], mh, scale, out, ws, ws_bytes)
    torch.cuda.synchronize()
    assert pool.error() == 0
    pages = pool.hist_view(0).cpu().numpy()
    hist = lambda b, g: kq.read_history(pages, pt[b], int(st["hist_len"][b]), g, pool.cfg.page_size, GS)
    ref = att.decode_three_tier(q, Rk, Rv, st["sink_k"], st["sink_v"], st["sink_len"], hist,
                                st["hist_len"], st["rec_k"], st["rec_v"], st["rec_len"],
                                st["rec_start"], Hkv, GS, scale)
    ma, rl2 = gu.metrics(out.cpu().numpy(), ref)
    assert ma <= MAX_ABS and rl2 <= REL_L2, (ma, rl2)


@pytest.mark.parametrize("P,GS", [(16, 128), (32, 64)])
def test_stream_from_empty(P, GS):
    rng = np.random.default_rng(40 + P + GS)
    B, Hkv, Hq, S, W, n_hist = 2, 2, 8, 4, 8, 45
    N = S + W + n_hist
    pages_per = (n_hist + P - 1) // P
    num_pages = B * pages_per + 3
    pt = rng.permutation(num_pages).astype(np.int32)[:B * pages_per].reshape(B, pages_per)
    make, Rk, Rv, ck, cv = _setup(rng, B, Hkv, Hq, P, GS, S, W, num_pages)
    tk, tv = _tokens(rng, N, B, Hkv), _tokens(rng, N, B, Hkv)

    pool = make()
    kd, vd = gu.bf16_dev(tk), gu.bf16_dev(tv)
    lens = [gu.i32_dev(np.zeros(B)) for _ in range(4)]
    ptd = gu.i32_dev(pt)
    for i in range(N):
        native.kv_append_step(pool.handle, 0, B, kd[i], vd[i], *lens, ptd, pages_per)
    torch.cuda.synchronize()
    assert pool.error() == 0

    st = _empty_state(B, Hkv, S, W, num_pages, P, GS)
    for i in range(N):
        assert tiers.append_step(st, tk[i], tv[i], pt, Rk, Rv, ck, cv, P, GS) == []
    for name, d in zip(("sink_len", "hist_len", "rec_len", "rec_start"), lens):
        assert np.array_equal(d.cpu().numpy(), st[name]), name
    for got, key in zip(_gpu_tiers(pool, B), ("sink_k", "sink_v", "rec_k", "rec_v")):
        assert np.array_equal(got, st[key]), key
    gpu_pages = pool.hist_view(0).cpu().numpy()
    _history_close(gpu_pages, st["pages"], pt, st["hist_len"], Hkv, P, GS)

    # the same tokens through the bulk append: identical pages, bit for bit
    bulk = make()
    hk = np.concatenate([tk[S:S + n_hist, b] for b in range(B)])
    hv = np.concatenate([tv[S:S + n_hist, b] for b in range(B)])
    native.kv_append_quantize(bulk.handle, 0, B, gu.bf16_dev(hk), gu.bf16_dev(hv),
                              gu.i32_dev([0, n_hist, 2 * n_hist]), gu.i32_dev(np.zeros(B)), ptd,
                              pages_per, n_hist)
    torch.cuda.synchronize()
    assert np.array_equal(bulk.hist_view(0).cpu().numpy(), gpu_pages)
    bulk.close()

    q = synth.f32_to_bf16_bits(rng.standard_normal((B, Hq, 128)).astype(np.float32))
    _decode_vs_oracle(pool, st, q, pt, Rk, Rv, GS, Hkv, lens, 1.0 / np.sqrt(128.0))
    pool.close()


def test_mixed_phases_tile_crossing_and_missing_page():
    """Four sequences in different phases: sink filling, ring filling, ring
    full and crossing a tile and a page, ring full with the next history page
    missing (its steps are refused and reported; the others go on)."""
    rng = np.random.default_rng(77)
    B, Hkv, Hq, P, GS, S, W = 4, 2, 4, 16, 128, 4, 8
    num_pages = 8
    pt = np.array([[0, 1], [2, 3], [4, 5], [6, -1]], np.int32)
    make, Rk, Rv, ck, cv = _setup(rng, B, Hkv, Hq, P, GS, S, W, num_pages)
    st = _empty_state(B, Hkv, S, W, num_pages, P, GS)
    st["sink_len"][:] = [2, S, S, S]
    st["rec_len"][:] = [0, 3, W, W]
    st["rec_start"][:] = [0, 6, 5, 2]
    st["hist_len"][:] = [0, 0, 14, 16]
    for key in ("sink_k", "sink_v", "rec_k", "rec_v"):
        st[key][:] = _tokens(rng, 1, B * Hkv * st[key].shape[2], 1)[0].reshape(st[key].shape)
    # existing history of sequences 2 and 3 (quantized by the oracle)
    for b in (2, 3):
        n = int(st["hist_len"][b])
        hk, hv = _tokens(rng, n, 1, Hkv)[:, 0], _tokens(rng, n, 1, Hkv)[:, 0]
        kq.pack_history_full(hk, hv, Rk, Rv, ck, cv, pt[b], num_pages, Hkv, P, GS, st["pages"])

    pool = make()
    sk, sv, rk, rv = pool.tier_views(0)
    for view, key in zip((sk, sv, rk, rv), ("sink_k", "sink_v", "rec_k", "rec_v")):
        view[:B].copy_(gu.bf16_dev(st[key]))
    gu.upload_pages(pool, st["pages"])
    lens = [gu.i32_dev(st[k]) for k in ("sink_len", "hist_len", "rec_len", "rec_start")]
    ptd = gu.i32_dev(pt)
    steps = 3
    tk, tv = _tokens(rng, steps, B, Hkv), _tokens(rng, steps, B, Hkv)
    kd, vd = gu.bf16_dev(tk), gu.bf16_dev(tv)
    for i in range(steps):
        native.kv_append_step(pool.handle, 0, B, kd[i], vd[i], *lens, ptd, pt.shape[1])
    torch.cuda.synchronize()
    assert pool.error() == 1                          # KV_DEVERR_PAGE_ID (sequence 3)
    assert pool.error() == 0                          # cleared by the read

    for i in range(steps):
        assert tiers.append_step(st, tk[i], tv[i], pt, Rk, Rv, ck, cv, P, GS) == [3]
    for name, d in zip(("sink_len", "hist_len", "rec_len", "rec_start"), lens):
        assert np.array_equal(d.cpu().numpy(), st[name]), name
    assert list(st["hist_len"]) == [0, 0, 17, 16] and list(st["sink_len"]) == [S, S, S, S]
    for got, key in zip(_gpu_tiers(pool, B), ("sink_k", "sink_v", "rec_k", "rec_v")):
        assert np.array_equal(got, st[key]), key
    _history_close(pool.hist_view(0).cpu().numpy(), st["pages"], pt, st["hist_len"], Hkv, P, GS)
    q = synth.f32_to_bf16_bits(rng.standard_normal((B, Hq, 128)).astype(np.float32))
    _decode_vs_oracle(pool, st, q, pt, Rk, Rv, GS, Hkv, lens, 0.09)
    pool.close()


def test_pages_sized_tiers_evict_after_sink_and_recent_fill():
    """The pages' capacities (64 sink, 256 recent): 330 steps from empty leave
    64 sink tokens, 256 recent and 10 history tokens."""
    rng = np.random.default_rng(91)
    B, Hkv, Hq, P, GS = 1, 2, 8, 16, 128
    make, Rk, Rv, ck, cv = _setup(rng, B, Hkv, Hq, P, GS, 64, 256, 2)
    pool = make()
    N = 330
    tk, tv = _tokens(rng, N, B, Hkv), _tokens(rng, N, B, Hkv)
    kd, vd = gu.bf16_dev(tk), gu.bf16_dev(tv)
    lens = [gu.i32_dev(np.zeros(B)) for _ in range(4)]
    pt = np.array([[1]], np.int32)
    ptd = gu.i32_dev(pt)
    for i in range(N):
        native.kv_append_step(pool.handle, 0, B, kd[i], vd[i], *lens, ptd, 1)
    torch.cuda.synchronize()
    assert pool.error() == 0
    assert [int(x.item()) for x in lens] == [64, 10, 256, 10]
    st = _empty_state(B, Hkv, 64, 256, 2, P, GS)
    for i in range(N):
        tiers.append_step(st, tk[i], tv[i], pt, Rk, Rv, ck, cv, P, GS)
    for got, key in zip(_gpu_tiers(pool, B), ("sink_k", "sink_v", "rec_k", "rec_v")):
        assert np.array_equal(got, st[key]), key
    _history_close(pool.hist_view(0).cpu().numpy(), st["pages"], pt, st["hist_len"], Hkv, P, GS)
    pool.close()
