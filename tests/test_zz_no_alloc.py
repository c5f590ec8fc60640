"""kv_decode_attention_noalloc: the decode entry point for callers that cannot
allocate device memory (an engine whose memory manager owns every
allocation, or a latency-critical path where cudaMalloc may synchronise).

It must give the same results as kv_decode_attention with a caller workspace,
bit for bit (same kernel, same split plan, same merge order), also on a
second, smaller call right after the first (the fixed buffer then still holds
partials of the larger plan beyond what the second call writes), and must
refuse calls whose partials would not fit its 16 MiB buffer.  This file is
collected last on purpose."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from bit_kv_cache_12_gb300 import native, synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    native.lib()


def _call(pool, wl, q, B, noalloc):
    """Sequences 0..B-1 of wl with queries q, through either entry point."""
    mh = int(wl.hist_len[:B].max())
    out = torch.full((B, wl.Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    args = [gu.i32_dev(wl.sink_len[:B]), gu.i32_dev(wl.hist_len[:B]), gu.i32_dev(wl.rec_len[:B]),
            gu.i32_dev(wl.rec_start[:B])]
    pt = gu.i32_dev(wl.page_table[:B])
    if noalloc:
        native.kv_decode_attention_noalloc(pool.handle, 0, B, gu.bf16_dev(q[:B]), *args, pt,
                                           wl.page_table.shape[1], mh, wl.scale, out)
    else:
        ws_bytes = native.kv_decode_workspace_bytes(pool.handle, B, mh)
        ws = torch.empty(ws_bytes // 4 + 4, dtype=torch.float32, device="cuda")
        native.kv_decode_attention(pool.handle, 0, B, gu.bf16_dev(q[:B]), *args, pt,
                                   wl.page_table.shape[1], mh, wl.scale, out, ws, ws_bytes)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("G,P,gs", [(4, 16, 128), (8, 32, 64)])
def test_noalloc_matches_workspace_entry_on_two_calls(G, P, gs):
    wl = synth.make_decode_workload(f"na{G}{P}", 70 + G, B=3, Hq=2 * G, Hkv=2,
                                    ctx=[2500, 700, 1300], page_size=P, group_size=gs,
                                    outliers_per_head=4)
    pool = gu.make_int2_pool(wl)
    gu.upload_pages(pool, gu.oracle_pages(wl))
    q2 = synth.f32_to_bf16_bits(np.random.default_rng(5).standard_normal(wl.q.shape)
                                .astype(np.float32))
    # the whole batch, then a smaller batch with a shorter maximum history and
    # other queries: fewer partials than the first call left in the buffer
    for q, B in ((wl.q, 3), (q2, 2)):
        ref = _call(pool, wl, q, B, noalloc=False)
        got = _call(pool, wl, q, B, noalloc=True)
        assert np.all(np.isfinite(got))
        assert np.array_equal(got, ref)
    assert pool.error() == 0
    pool.close()


def test_noalloc_rejects_oversize_calls():
    """64 sequences x 8 KV heads x GQA 8 with 400k-token histories need far more
    than the fixed buffer: refused on the host, nothing launched."""
    B, Hq, Hkv, P = 64, 64, 8, 16
    pool = native.KVPool(native.KV_POOL_INT2_3TIER, 1, Hq, Hkv, P, 16, B)
    max_pages = 25600
    need = native.kv_decode_workspace_bytes(pool.handle, B, max_pages * P)
    assert need > native.KV_NOALLOC_SCRATCH_BYTES
    pt = torch.full((B, max_pages), -1, dtype=torch.int32, device="cuda")
    zeros = torch.zeros(B, dtype=torch.int32, device="cuda")
    q = torch.zeros((B, Hq, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((B, Hq, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(native.KVError) as ei:
        native.kv_decode_attention_noalloc(pool.handle, 0, B, q, zeros, zeros, zeros, zeros, pt,
                                           max_pages, max_pages * P, 0.088, out)
    assert ei.value.status == native.KV_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert pool.error() == 0
    pool.close()
