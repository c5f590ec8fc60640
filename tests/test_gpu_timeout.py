"""The decode's bounded waits, made to run out on purpose without a fault.

Every wait of the history loop on a bulk copy is bounded; when one runs out
the kernel records KV_DEVERR_TIMEOUT, waits (bounded) for the copies it did
issue, skips its split and returns, so the context stays usable.  The test
hook ``kv_debug_stall_first_copy`` arms the first ring stage of the first
history split for a copy that is never issued (nothing is in flight on it, so
nothing can land late) and shortens the poll limit; the call must return with
the error word set and finite outputs, and a normal call on the same pool
afterwards must match the oracle again.  The same hook makes the bulk
append's first CTA never start the x load of its first chunk: the waits of
its warps run out, the call returns with the error word set, and a normal
append afterwards stores exactly what a pool that never saw the hook stores."""

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


@pytest.mark.parametrize("G,P", [(4, 16), (8, 32)])
def test_stalled_copy_times_out_and_context_survives(G, P):
    wl = synth.make_decode_workload(f"stall{G}", 80 + G, B=2, Hq=2 * G, Hkv=2, ctx=[2000, 5000],
                                    page_size=P)
    pages = gu.oracle_pages(wl)
    pool = gu.make_int2_pool(wl)
    gu.upload_pages(pool, pages)
    ref = gu.oracle_decode(wl, pages)
    for _ in range(2):                                   # the hook twice in a row
        native.kv_debug_stall_first_copy(pool.handle, 1, 4096)
        out = gu.gpu_decode(pool, wl)                    # returns: the wait is bounded
        assert pool.error() == 4                         # KV_DEVERR_TIMEOUT
        assert np.all(np.isfinite(out))
        assert gu.metrics(out, ref)[1] > 1e-3            # a split really was skipped
    native.kv_debug_stall_first_copy(pool.handle, 0, 0)
    out = gu.gpu_decode(pool, wl)
    assert pool.error() == 0
    ma, rl = gu.metrics(out, ref)
    assert ma <= 1e-2 and rl <= 1e-3, (ma, rl)
    pool.close()


def _append_pool(aw, stall):
    pool = native.KVPool(native.KV_POOL_INT2_3TIER, 1, 2 * aw.Hkv, aw.Hkv, aw.page_size, aw.num_pages,
                         aw.n_seqs, group_size=aw.group_size)
    native.kv_pool_set_rotation(pool.handle, 0, gu.f32_dev(aw.Rk), gu.f32_dev(aw.Rv),
                                gu.f32_dev(aw.clip_k), gu.f32_dev(aw.clip_v))
    args = (pool.handle, 0, aw.n_seqs, gu.bf16_dev(aw.k), gu.bf16_dev(aw.v), gu.i32_dev(aw.cu_tokens),
            gu.i32_dev(aw.hist_start), gu.i32_dev(aw.page_table), aw.page_table.shape[1],
            int(np.max(aw.tokens_per_seq)))
    if stall:
        for _ in range(2):                               # the hook twice in a row
            native.kv_debug_stall_first_copy(pool.handle, 1, 4096)
            native.kv_append_quantize(*args)             # returns: the waits are bounded
            torch.cuda.synchronize()
            assert pool.error() == 4                     # KV_DEVERR_TIMEOUT
        native.kv_debug_stall_first_copy(pool.handle, 0, 0)
    native.kv_append_quantize(*args)
    torch.cuda.synchronize()
    assert pool.error() == 0
    pages = pool.hist_view(0).cpu().numpy().copy()
    pool.close()
    return pages


@pytest.mark.parametrize("gs", [64, 128])
def test_append_stalled_load_times_out_and_context_survives(gs):
    aw = synth.make_append_workload(f"stallapp{gs}", 95 + gs, n_seqs=3, Hkv=2,
                                    tokens_per_seq=[700, 300, 517], hist_start=[0, 16, 5],
                                    page_size=16, group_size=gs)
    ref = _append_pool(aw, stall=False)
    got = _append_pool(aw, stall=True)
    assert np.array_equal(got, ref)
