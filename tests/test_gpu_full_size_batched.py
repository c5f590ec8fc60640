"""Parity at the full size of the batched workloads, in the launch
configuration the benchmark times, and on grids of several waves.

Workloads (``bit_kv_cache_12_gb300.workloads``, the benchmark's own seeded
device generators): Qwen3-8B shape, batch 64, 32 q / 8 KV heads, context
U[8192, 32768], page 16; Qwen3-32B shape, batch 16, 64 q / 8 KV heads
(GQA 8, the 12-warp kernel), context 131,072, page 32.  The pool is filled by
the library's append and one decode call covers the whole batch.  The oracle
recomputes sampled KV heads (every query head of each) from the codes the
pool stores, including the last (sequence, KV head) pair, whose history splits
run in the grid's last wave; every output is finite.

Smaller cases force what the batched shapes reach only at size: the longest
split (128 tiles per warp at GQA 4 with 16 warps = 2,048 page ids, the staging
limit being 2,056; 96 per warp at GQA 8 with 12 warps = 1,152) and a second,
shorter split per pair, on grids of several waves with ragged lengths.  The gist.science OSCAR
explainer, section 4 (system results), reports the method at large batch."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from bit_kv_cache_12_gb300 import native, workloads
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 1e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    native.lib()


def _check(c, pairs):
    pool = gu.fill_pool_from_case(c)
    assert pool.error() == 0
    out = gu.decode_case(pool, c)
    assert pool.error() == 0
    assert np.all(np.isfinite(out))
    G = c.Hq // c.Hkv
    worst = (0.0, 0.0)
    for b, g in pairs:
        ref = gu.oracle_kv_head(pool, c, b, g)
        ma, rl = gu.metrics(out[b, g * G:(g + 1) * G], ref)
        worst = (max(worst[0], ma), max(worst[1], rl))
        assert ma <= MAX_ABS and rl <= REL_L2, (b, g, ma, rl)
    print(f"{c.name}: worst sampled max_abs {worst[0]:.3e} rel_l2 {worst[1]:.3e}")
    pool.close()


def test_batch64_full_size():
    c = workloads.batch64(torch, torch.device("cuda"))
    longest, shortest = int(np.argmax(c.hist_len)), int(np.argmin(c.hist_len))
    _check(c, [(0, 0), (longest, 3), (shortest, 5), (c.B - 1, c.Hkv - 1)])


def test_long16_full_size():
    c = workloads.long16(torch, torch.device("cuda"))
    _check(c, [(0, 0), (7, 3), (c.B - 1, c.Hkv - 1)])


@pytest.mark.parametrize("G,P,B,lo,hi", [(8, 16, 64, 18800, 19400), (4, 16, 40, 33000, 33900),
                                         (8, 32, 64, 18800, 19400)])
def test_split_bound_multi_wave(G, P, B, lo, hi):
    Hkv = 2
    c = workloads.generate(torch, torch.device("cuda"), f"wave_g{G}_p{P}", 90 + G + P, B, G * Hkv,
                           Hkv, P, ctx_range=(lo, hi), outlier_channels=4)
    ws = native.kv_decode_workspace_bytes
    pool = native.KVPool(native.KV_POOL_INT2_3TIER, 1, c.Hq, Hkv, P, 4, B)
    per_part = ws(pool.handle, B, int(c.hist_len.max()))
    pool.close()
    # 2 history splits per (sequence, KV head), the first with the longest split
    # (128 tiles per warp of 16 at 4 query columns, 96 of 12 at 8): their
    # partials (132 floats per query head), then the q' fragments
    qwords = 32 * (16 * (1 if G <= 4 else 2) + 4)
    assert per_part == B * Hkv * (2 * G * 132 * 4 + qwords * 4)
    _check(c, [(0, 0), (B // 2, 1), (B - 1, 0), (B - 1, 1), (int(np.argmax(c.hist_len)), 1)])
