"""Multi-layer pools with distinct rotations (GPU).

The gist.science OSCAR explainer (section 2.2 A) fixes one pair of rotations
and clip thresholds per layer, offline; the zingnex.cn forum summary
("离线优化的优势") notes that layers may also share them.  A pool holds every
layer's history pages, tiers, R_k, R_v and clips side by side: appending to
and decoding one layer must use that layer's rotations and must not disturb
any other layer."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from bit_kv_cache_12_gb300 import native, synth
from oracle import kvquant as kq
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 1e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    native.lib()


def _layer_workload(seed, shared_rotation=None):
    """A one-layer workload whose V rotation differs from its K rotation (the
    V clip is disabled so that it stays consistent with the new R_v)."""
    wl = synth.make_decode_workload(f"layer{seed}", seed, B=2, Hq=8, Hkv=2, ctx=[900, 1500],
                                    page_size=16, outliers_per_head=4)
    rng = np.random.default_rng(seed + 1000)
    wl.Rv = np.stack([synth.haar_orthogonal(rng) for _ in range(wl.Hkv)]).astype(wl.Rk.dtype)
    wl.clip_v = np.full_like(wl.clip_v, np.inf)
    if shared_rotation is not None:
        wl.Rk, wl.Rv = shared_rotation
    return wl


def test_two_layers_distinct_rotations_append_and_decode():
    wls = [_layer_workload(71), _layer_workload(72)]
    assert not np.allclose(wls[0].Rk, wls[1].Rk) and not np.allclose(wls[0].Rk, wls[0].Rv)
    w0 = wls[0]
    num_pages = max(w.num_pages for w in wls)
    pool = native.KVPool(native.KV_POOL_INT2_3TIER, 2, w0.Hq, w0.Hkv, w0.page_size, num_pages, w0.B,
                         group_size=w0.group_size)
    keep = []
    for layer, wl in enumerate(wls):
        t = (gu.f32_dev(wl.Rk), gu.f32_dev(wl.Rv), gu.f32_dev(wl.clip_k), gu.f32_dev(wl.clip_v))
        keep.append(t)
        native.kv_pool_set_rotation(pool.handle, layer, *t)
        sk, sv, rk, rv = pool.tier_views(layer)
        sk[:wl.B].copy_(gu.bf16_dev(wl.sink_k)); sv[:wl.B].copy_(gu.bf16_dev(wl.sink_v))
        rk[:wl.B].copy_(gu.bf16_dev(wl.rec_k)); rv[:wl.B].copy_(gu.bf16_dev(wl.rec_v))
    # append layer 1 first, then layer 0: neither may touch the other
    for layer in (1, 0):
        wl = wls[layer]
        k = np.concatenate(wl.hist_k); v = np.concatenate(wl.hist_v)
        cu = np.zeros(wl.B + 1, np.int32); cu[1:] = np.cumsum(wl.hist_len)
        native.kv_append_quantize(pool.handle, layer, wl.B, gu.bf16_dev(k), gu.bf16_dev(v),
                                  gu.i32_dev(cu), gu.i32_dev(np.zeros(wl.B)), gu.i32_dev(wl.page_table),
                                  wl.page_table.shape[1], int(wl.hist_len.max()))
        torch.cuda.synchronize()
        if layer == 1:
            snap1 = pool.hist_view(1).cpu().numpy().copy()
    assert pool.error() == 0
    assert np.array_equal(pool.hist_view(1).cpu().numpy(), snap1)     # layer 0's append left layer 1 alone

    for layer, wl in enumerate(wls):
        mh = int(wl.hist_len.max())
        ws_bytes = native.kv_decode_workspace_bytes(pool.handle, wl.B, mh)
        ws = torch.empty(max(ws_bytes, 16) // 4 + 4, dtype=torch.float32, device="cuda")
        out = torch.full((wl.B, wl.Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
        native.kv_decode_attention(pool.handle, layer, wl.B, gu.bf16_dev(wl.q), gu.i32_dev(wl.sink_len),
                                   gu.i32_dev(wl.hist_len), gu.i32_dev(wl.rec_len), gu.i32_dev(wl.rec_start),
                                   gu.i32_dev(wl.page_table), wl.page_table.shape[1], mh, wl.scale, out,
                                   ws, ws_bytes)
        torch.cuda.synchronize()
        assert pool.error() == 0
        pages = pool.hist_view(layer).cpu().numpy()
        ref = gu.oracle_decode(wl, pages)
        ma, rl = gu.metrics(out.cpu().numpy(), ref)
        assert ma <= MAX_ABS and rl <= REL_L2, (layer, ma, rl)
        # the codes the library stored are the oracle's quantization of this layer's
        # tokens with this layer's rotation (up to rounding-boundary flips)
        bad = tot = 0
        own = gu.oracle_pages(wl, num_pages=num_pages)
        for b in range(wl.B):
            for g in range(wl.Hkv):
                got = kq.read_history(pages, wl.page_table[b], int(wl.hist_len[b]), g, wl.page_size, wl.group_size)
                exp = kq.read_history(own, wl.page_table[b], int(wl.hist_len[b]), g, wl.page_size, wl.group_size)
                bad += int((got[0] != exp[0]).sum() + (got[1] != exp[1]).sum()); tot += got[0].size * 2
        assert bad <= max(4, 1e-4 * tot), (layer, bad, tot)
    pool.close()


def test_layers_sharing_one_rotation():
    """Cross-layer shared rotation: the same R in two layers gives each layer's
    decode the result of a one-layer pool with that R."""
    base = _layer_workload(73)
    wls = [base, _layer_workload(74, shared_rotation=(base.Rk, base.Rv))]
    outs = []
    for two_layer in (True, False):
        res = []
        for layer, wl in enumerate(wls):
            pool = gu.make_int2_pool(wl) if not two_layer else None
            if two_layer:
                if layer == 0:
                    shared = native.KVPool(native.KV_POOL_INT2_3TIER, 2, wl.Hq, wl.Hkv, wl.page_size,
                                           max(w.num_pages for w in wls), wl.B, group_size=wl.group_size)
                    shared._keep = []
                pool = shared
                t = (gu.f32_dev(wl.Rk), gu.f32_dev(wl.Rv), gu.f32_dev(wl.clip_k), gu.f32_dev(wl.clip_v))
                shared._keep.append(t)
                native.kv_pool_set_rotation(pool.handle, layer, *t)
                sk, sv, rk, rv = pool.tier_views(layer)
                sk[:wl.B].copy_(gu.bf16_dev(wl.sink_k)); sv[:wl.B].copy_(gu.bf16_dev(wl.sink_v))
                rk[:wl.B].copy_(gu.bf16_dev(wl.rec_k)); rv[:wl.B].copy_(gu.bf16_dev(wl.rec_v))
            lay = layer if two_layer else 0
            pool.hist_view(lay).copy_(torch.from_numpy(gu.oracle_pages(wl, num_pages=pool.cfg.num_pages)))
            mh = int(wl.hist_len.max())
            ws_bytes = native.kv_decode_workspace_bytes(pool.handle, wl.B, mh)
            ws = torch.empty(max(ws_bytes, 16) // 4 + 4, dtype=torch.float32, device="cuda")
            out = torch.empty((wl.B, wl.Hq, 128), dtype=torch.float32, device="cuda")
            native.kv_decode_attention(pool.handle, lay, wl.B, gu.bf16_dev(wl.q), gu.i32_dev(wl.sink_len),
                                       gu.i32_dev(wl.hist_len), gu.i32_dev(wl.rec_len),
                                       gu.i32_dev(wl.rec_start), gu.i32_dev(wl.page_table),
                                       wl.page_table.shape[1], mh, wl.scale, out, ws, ws_bytes)
            torch.cuda.synchronize()
            res.append(out.cpu().numpy())
            if not two_layer:
                pool.close()
        if two_layer:
            shared.close()
        outs.append(res)
    for layer in range(2):
        assert np.array_equal(outs[0][layer], outs[1][layer])
