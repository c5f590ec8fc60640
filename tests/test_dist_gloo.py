"""Multi-rank path on CPU: two gloo ranks on 127.0.0.1.

The decode shards by sequence with no collective on the data path: each rank
decodes its own contiguous slice of the batch, and the slices together equal
the whole-batch result.  The host-side collectives of the benchmark (barrier,
maximum of per-rank times) are exercised on the same process group.  The
per-rank decode here is the oracle (the CPU stand-in for a GPU replica)."""

import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp

from bit_kv_cache_12_gb300 import dist as kvdist


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _workload():
    from bit_kv_cache_12_gb300 import synth
    return synth.make_decode_workload("dist", 21, B=5, Hq=8, Hkv=2, ctx=[300, 700, 65, 400, 1000],
                                      page_size=16)


def _decode_slice(wl, pages, b0, b1):
    """Oracle decode of sequences [b0, b1) only."""
    from oracle import attention as att
    from oracle import kvquant as kq
    sl = slice(b0, b1)
    hist = lambda b, g: kq.read_history(pages, wl.page_table[b0 + b], int(wl.hist_len[b0 + b]), g,
                                        wl.page_size, wl.group_size)
    return att.decode_three_tier(wl.q[sl], wl.Rk, wl.Rv, wl.sink_k[sl], wl.sink_v[sl],
                                 wl.sink_len[sl], hist, wl.hist_len[sl], wl.rec_k[sl], wl.rec_v[sl],
                                 wl.rec_len[sl], wl.rec_start[sl], wl.Hkv, wl.group_size, wl.scale)


def _pages(wl):
    from oracle import kvquant as kq
    tb = kq.tile_bytes(wl.group_size) * (wl.page_size // 16)
    pages = np.zeros((wl.num_pages, wl.Hkv, tb), np.uint8)
    for b in range(wl.B):
        if wl.hist_len[b]:
            kq.pack_history_full(wl.hist_k[b], wl.hist_v[b], wl.Rk, wl.Rv, wl.clip_k, wl.clip_v,
                                 wl.page_table[b], wl.num_pages, wl.Hkv, wl.page_size,
                                 wl.group_size, pages)
    return pages


def _worker(rank, world, port, outdir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    r, w, local = kvdist.init("gloo")
    assert (r, w, local) == (rank, world, rank)
    mx = kvdist.max_over_ranks([rank + 0.5, 10.0 - rank])
    kvdist.barrier()
    wl = _workload()
    b0, b1 = kvdist.shard(wl.B, r, w)
    out = _decode_slice(wl, _pages(wl), b0, b1)
    kvdist.barrier()
    kvdist.shutdown()
    np.savez(os.path.join(outdir, f"rank{rank}.npz"), mx=np.array(mx), b=np.array([b0, b1]), out=out)


def test_shard_partitions_the_batch():
    for n in range(0, 40):
        for world in range(1, 9):
            spans = [kvdist.shard(n, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(spans[i][1] == spans[i + 1][0] for i in range(world - 1))
            sizes = [e - s for s, e in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        kvdist.shard(4, 2, 2)


def test_single_process_helpers_without_group():
    assert kvdist.max_over_ranks([1.0, 2.5]) == [1.0, 2.5]
    kvdist.barrier()   # no group: a no-op


def test_two_gloo_ranks_shard_the_decode(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [np.load(os.path.join(tmp_path, f"rank{r}.npz")) for r in range(world)]
    for r in range(world):
        assert list(res[r]["mx"]) == [1.5, 10.0]          # element-wise max over ranks
    assert [tuple(res[r]["b"]) for r in range(world)] == [(0, 3), (3, 5)]
    wl = _workload()
    whole = _decode_slice(wl, _pages(wl), 0, wl.B)
    sharded = np.concatenate([res[r]["out"] for r in range(world)])
    assert np.array_equal(sharded, whole)
