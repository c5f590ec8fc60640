"""GPU parity of several queries per sequence over the INT2 cache
(``kv_decode_attention_multi``): a chunk continuing on a cached prefix, or
draft tokens being verified, each attending over the whole cache, with the
log-sum-exp a caller needs to merge in attention over the chunk's own tokens
(zingnex.cn forum summary of OSCAR, "与其他优化的协同").  Compared with the
oracle on identical stored codes and with single-query decodes."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from bit_kv_cache_12_gb300 import native, synth
from oracle import attention as att
from oracle import kvquant as kq
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 1e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    native.lib()


def _multi(pool, wl, qm, lens=None, with_lse=True):
    B, T = qm.shape[0], qm.shape[1]
    sl, hl, rl, rs = lens if lens is not None else (wl.sink_len, wl.hist_len, wl.rec_len, wl.rec_start)
    mh = int(max(np.max(hl), 0))
    ws_bytes = native.kv_decode_multi_workspace_bytes(pool.handle, B, T, mh)
    ws = torch.empty(max(ws_bytes, 16) // 4 + 4, dtype=torch.float32, device="cuda")
    out = torch.full((B, T, wl.Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((B, T, wl.Hq), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
    native.kv_decode_attention_multi(pool.handle, 0, B, T, gu.bf16_dev(qm), gu.i32_dev(sl), gu.i32_dev(hl),
                                     gu.i32_dev(rl), gu.i32_dev(rs), gu.i32_dev(wl.page_table),
                                     wl.page_table.shape[1], mh, wl.scale, out, lse, ws, ws_bytes)
    torch.cuda.synchronize()
    return out.cpu().numpy(), (lse.cpu().numpy() if with_lse else None)


@pytest.mark.parametrize("G,T,gs", [(4, 2, 128), (2, 4, 64), (1, 8, 128), (2, 2, 128)])
def test_multi_query_matches_oracle(G, T, gs):
    wl = synth.make_decode_workload(f"mq{G}{T}", 50 + G * T, B=3, Hq=2 * G, Hkv=2,
                                    ctx=[1500, 333, 900], page_size=16, group_size=gs,
                                    outliers_per_head=4)
    rng = np.random.default_rng(7 * G + T)
    qm = synth.f32_to_bf16_bits(rng.standard_normal((wl.B, T, wl.Hq, 128)).astype(np.float32))
    pages = gu.oracle_pages(wl)
    pool = gu.make_int2_pool(wl)
    gu.upload_pages(pool, pages)
    out, lse = _multi(pool, wl, qm)
    assert pool.error() == 0
    hist = lambda b, g: kq.read_history(pages, wl.page_table[b], int(wl.hist_len[b]), g, wl.page_size,
                                        wl.group_size)
    ref, ref_lse = att.decode_three_tier_multi(qm, wl.Rk, wl.Rv, wl.sink_k, wl.sink_v, wl.sink_len, hist,
                                               wl.hist_len, wl.rec_k, wl.rec_v, wl.rec_len, wl.rec_start,
                                               wl.Hkv, wl.group_size, wl.scale)
    ma, rl = gu.metrics(out, ref)
    assert ma <= MAX_ABS and rl <= REL_L2, (ma, rl)
    assert np.abs(lse - ref_lse).max() <= 1e-4 * max(1.0, np.abs(ref_lse).max())
    # every query position equals the single-query decode of that query, up to
    # the rounding of the BF16 tier rows: their softmax weights enter the tensor
    # cores as bf16 hi + lo pairs (relative error <= 2^-16 each), and the
    # multi-query kernel spreads the rows over a different number of warps
    for t in range(T):
        one = gu.gpu_decode(pool, wl, q=np.ascontiguousarray(qm[:, t]))
        assert gu.metrics(out[:, t], one)[1] <= 1e-5
    out2, _ = _multi(pool, wl, qm, with_lse=False)       # lse is optional
    assert np.array_equal(out2, out)
    pool.close()


def test_unsupported_query_count_and_empty_cache():
    wl = synth.make_decode_workload("mqe", 61, B=2, Hq=8, Hkv=2, ctx=[500, 700], page_size=16)
    pool = gu.make_int2_pool(wl)
    q3 = np.zeros((wl.B, 3, wl.Hq, 128), np.uint16)
    with pytest.raises(native.KVError):                   # 3 * 4 columns per KV head
        _multi(pool, wl, q3)
    z = np.zeros(wl.B, np.int32)
    rng = np.random.default_rng(3)
    qm = synth.f32_to_bf16_bits(rng.standard_normal((wl.B, 2, wl.Hq, 128)).astype(np.float32))
    out, lse = _multi(pool, wl, qm, lens=(z, z, z, z))
    assert pool.error() == 0
    assert np.all(out == 0.0) and np.all(np.isneginf(lse))
    pool.close()
