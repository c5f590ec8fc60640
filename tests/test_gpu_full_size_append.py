"""Parity of the bulk append at the full size of the append workload, in the
launch configuration the benchmark times.

Workload (``bit_kv_cache_12_gb300.workloads.append_workload``, the
benchmark's own seeded device generator): 64 sequences x 8 KV heads x 4096
tokens of Student-t(4) K and V rows, per-head Haar R_k and R_v, clips at 0.9 x
the rotated per-channel absmax, group 64, page 16, a shuffled page table; one
``kv_append_quantize`` call over the whole batch (per tensor one CTA per SM,
each walking about a hundred chunks of 128 tokens in two teams).  The oracle
rotates sampled 128-token chunks in fp64, clips and quantizes them with the
scalar IEEE quantizer, and the stored codes, scales and zeros must agree: s and
z within one fp16 ulp, codes equal except where the exact quotient lies within
1e-4 of a rounding boundary (the kernel's rotation is an fp32 accumulation of
bf16 hi / lo terms of R).  The samples include the batch's first and last
chunk and chunks spread over the batch.  The yunpan.plus OSCAR write-up, section
"2. 在线量化与反量化", describes the step (rotate, clip, quantize, pack)."""

import types

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from bit_kv_cache_12_gb300 import native, workloads
from tests.test_gpu_parity import _compare_codes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def appended():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda")
    w = workloads.append_workload(torch, dev)
    n_seqs, Hkv, T, P, GS = w["n_seqs"], w["Hkv"], w["T"], w["page_size"], w["group_size"]
    pool = native.KVPool(native.KV_POOL_INT2_3TIER, 1, Hkv, Hkv, P, w["num_pages"], n_seqs, group_size=GS)
    native.kv_pool_set_rotation(pool.handle, 0, torch.as_tensor(w["Rk"]).to(dev),
                                torch.as_tensor(w["Rv"]).to(dev), torch.as_tensor(w["clip_k"]).to(dev),
                                torch.as_tensor(w["clip_v"]).to(dev))
    cu = torch.as_tensor(np.arange(n_seqs + 1, dtype=np.int32) * T, device=dev)
    hs = torch.zeros(n_seqs, dtype=torch.int32, device=dev)
    pt = torch.as_tensor(w["page_table"], device=dev)
    native.kv_append_quantize(pool.handle, 0, n_seqs, w["k"], w["v"], cu, hs, pt, w["pages_per_seq"], T)
    torch.cuda.synchronize()
    err = pool.error()
    pages = pool.hist_view(0).cpu().numpy().copy()
    pool.close()
    return w, err, pages


def test_full_size_append_no_device_error(appended):
    _, err, _ = appended
    assert err == 0


@pytest.mark.parametrize("b,c0", [(0, 0), (0, 31), (17, 1), (17, 16), (40, 22), (63, 30), (63, 31)])
def test_full_size_append_sampled_chunks_match_oracle(appended, b, c0):
    w, _, pages = appended
    T = w["T"]
    aw = types.SimpleNamespace(group_size=w["group_size"], Hkv=w["Hkv"], page_table=w["page_table"],
                               page_size=w["page_size"], Rk=w["Rk"], Rv=w["Rv"], clip_k=w["clip_k"],
                               clip_v=w["clip_v"])
    p0 = 128 * c0
    rows = slice(b * T + p0, b * T + p0 + 128)
    k_bits = w["k"][rows].cpu().view(torch.int16).numpy().view(np.uint16)
    v_bits = w["v"][rows].cpu().view(torch.int16).numpy().view(np.uint16)
    bad, tot = _compare_codes(pages, k_bits, v_bits, aw, b, p0, 128)
    assert tot == 2 * w["Hkv"] * 128 * 128
    assert bad <= max(4, 1e-4 * tot), (bad, tot)
