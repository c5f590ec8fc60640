"""Decode with the per-step buffers in page-locked host memory.

A host caller may hand kv_decode_attention and kv_decode_attention_multi its
query, the four length arrays and the output (and log-sum-exp) in pinned host
memory: under unified addressing the kernel reads and writes them across the
CPU-GPU link in the same launch, with no staging copies.  The result must be
bit-identical to the same call with device buffers (same kernel, same plan),
and within the parity tolerance of the oracle."""

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


def _pinned(a, dtype):
    a = np.ascontiguousarray(a)
    if dtype == torch.bfloat16:                  # bf16 bit patterns held as uint16
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()
    return torch.from_numpy(a).pin_memory()


def _lens(wl):
    return [np.asarray(x, np.int32) for x in (wl.sink_len, wl.hist_len, wl.rec_len, wl.rec_start)]


def test_decode_host_buffers_bit_identical():
    wl = synth.make_decode_workload("hostmap", 61, B=3, Hq=8, Hkv=2, ctx=[2100, 333, 900],
                                    page_size=16, group_size=128, outliers_per_head=4)
    pages = gu.oracle_pages(wl)
    pool = gu.make_int2_pool(wl)
    gu.upload_pages(pool, pages)
    mh = int(wl.hist_len.max())
    ref_dev = gu.gpu_decode(pool, wl)

    ws_bytes = native.kv_decode_workspace_bytes(pool.handle, wl.B, mh)
    ws = torch.empty(ws_bytes // 4 + 4, dtype=torch.float32, device="cuda")
    q_h = _pinned(wl.q, torch.bfloat16)
    lens_h = [_pinned(x, torch.int32) for x in _lens(wl)]
    out_h = torch.full((wl.B, wl.Hq, 128), float("nan"), dtype=torch.float32).pin_memory()
    native.kv_decode_attention(pool.handle, 0, wl.B, q_h, *lens_h, gu.i32_dev(wl.page_table),
                               wl.page_table.shape[1], mh, wl.scale, out_h, ws, ws_bytes)
    torch.cuda.synchronize()
    err = pool.error()
    pool.close()
    assert err == 0
    out = out_h.numpy()
    assert np.array_equal(out, ref_dev)
    ma, rl = gu.metrics(out, gu.oracle_decode(wl, pages))
    assert ma <= MAX_ABS and rl <= REL_L2


def test_multi_query_host_buffers_bit_identical():
    T = 2
    wl = synth.make_decode_workload("hostmapm", 62, B=2, Hq=8, Hkv=2, ctx=[1700, 640],
                                    page_size=16, group_size=64, outliers_per_head=4)
    rng = np.random.default_rng(62)
    qm = synth.f32_to_bf16_bits(rng.standard_normal((wl.B, T, wl.Hq, 128)).astype(np.float32))
    pages = gu.oracle_pages(wl)
    pool = gu.make_int2_pool(wl)
    gu.upload_pages(pool, pages)
    mh = int(wl.hist_len.max())
    ws_bytes = native.kv_decode_multi_workspace_bytes(pool.handle, wl.B, T, mh)
    ws = torch.empty(ws_bytes // 4 + 4, dtype=torch.float32, device="cuda")
    pt = gu.i32_dev(wl.page_table)

    def run(host):
        if host:
            q = _pinned(qm, torch.bfloat16)
            lens = [_pinned(x, torch.int32) for x in _lens(wl)]
            out = torch.full((wl.B, T, wl.Hq, 128), float("nan"), dtype=torch.float32).pin_memory()
            lse = torch.full((wl.B, T, wl.Hq), float("nan"), dtype=torch.float32).pin_memory()
        else:
            q = gu.bf16_dev(qm)
            lens = [gu.i32_dev(x) for x in _lens(wl)]
            out = torch.full((wl.B, T, wl.Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
            lse = torch.full((wl.B, T, wl.Hq), float("nan"), dtype=torch.float32, device="cuda")
        native.kv_decode_attention_multi(pool.handle, 0, wl.B, T, q, *lens, pt, wl.page_table.shape[1],
                                         mh, wl.scale, out, lse, ws, ws_bytes)
        torch.cuda.synchronize()
        return out.cpu().numpy(), lse.cpu().numpy()

    out_d, lse_d = run(False)
    out_h, lse_h = run(True)
    err = pool.error()
    pool.close()
    assert err == 0
    assert np.array_equal(out_h, out_d) and np.array_equal(lse_h, lse_d)
    hist = lambda b, g: kq.read_history(pages, wl.page_table[b], int(wl.hist_len[b]), g, wl.page_size,
                                        wl.group_size)
    ref, _ = att.decode_three_tier_multi(qm, wl.Rk, wl.Rv, wl.sink_k, wl.sink_v, wl.sink_len, hist,
                                         wl.hist_len, wl.rec_k, wl.rec_v, wl.rec_len, wl.rec_start,
                                         wl.Hkv, wl.group_size, wl.scale)
    ma, rl = gu.metrics(out_h, ref)
    assert ma <= MAX_ABS and rl <= REL_L2
