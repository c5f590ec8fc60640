"""GPU parity: the CUDA library through its C ABI against the CPU oracle.

Tolerances: packed codes and fp16 scale/zero are bit-exact when both sides get
the same fp32 rotated input; attention outputs must be within max-abs 1e-2
and rel-L2 1e-3 of the fp64 oracle on identical stored codes."""

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


# ---------------------------------------------------------------------------
# quantizer parity entry: bit-exact
# ---------------------------------------------------------------------------

def _quant_inputs(rng, n, hkv):
    x = rng.standard_normal((n, hkv, 128)).astype(np.float32)
    x[:, :, 5] *= 30.0                                 # outlier channel
    x[0] = 1.25                                        # constant rows: s = 0
    x[1] = -0.0
    x[2, :, :64] = 0.0; x[2, :, 64:] = 1e-8            # fp16 underflow of s
    x[3] = np.linspace(-1e6, 1e6, 128, dtype=np.float32)   # saturation
    # exact ties: y = z + (k + 0.5) s with fp16-exact z, s
    k = rng.integers(0, 3, (hkv, 128)); k[:, 0] = 0; k[:, 1] = 3
    y = (-2.0 + k * 0.5).astype(np.float32); y[:, 2:64:7] += 0.25; y[:, 66:128:7] += 0.25
    x[4] = y
    return x


@pytest.mark.parametrize("gs", [64, 128])
def test_quantize_pack_bit_exact(gs):
    rng = np.random.default_rng(100 + gs)
    hkv, n = 4, 3001
    x = _quant_inputs(rng, n, hkv)
    clip = np.abs(rng.standard_normal((2, hkv, 128))).astype(np.float32) * 2 + 0.5
    clip[:, :, :16] = np.inf
    pool = native.KVPool(native.KV_POOL_INT2_3TIER, 1, hkv, hkv, 16, 4, 1, group_size=gs)
    eye = gu.f32_dev(np.stack([np.eye(128)] * hkv))
    native.kv_pool_set_rotation(pool.handle, 0, eye, eye, gu.f32_dev(clip[0]), gu.f32_dev(clip[1]))
    xd = gu.f32_dev(x)
    for tensor in (0, 1):
        codes = torch.zeros((n, hkv, 32), dtype=torch.uint8, device="cuda")
        sz = torch.zeros((n, hkv, 128 // gs, 2), dtype=torch.float16, device="cuda")
        native.kv_quantize_pack_f32(pool.handle, 0, tensor, n, xd, codes, sz)
        torch.cuda.synchronize()
        c_ref, s_ref, z_ref = kq.quantize_rows(x, clip[tensor][None], gs)
        assert np.array_equal(codes.cpu().numpy(), kq.pack_canonical(c_ref))
        sz_h = sz.cpu().numpy()
        assert np.array_equal(sz_h[..., 0].view(np.uint16), s_ref.view(np.uint16))
        assert np.array_equal(sz_h[..., 1].view(np.uint16), z_ref.view(np.uint16))
    assert pool.error() == 0
    pool.close()


# ---------------------------------------------------------------------------
# fused append: GPU pages vs oracle pages
# ---------------------------------------------------------------------------

def _compare_codes(gpu_pages, wl_k, wl_v, aw, b, hist_start, n):
    """Compare one sequence's appended tokens; returns (mismatch, total)."""
    gs = aw.group_size
    bad = tot = 0
    for g in range(aw.Hkv):
        kc, vc, sk, zk, sv, zv = kq.read_history(gpu_pages, aw.page_table[b], hist_start + n, g,
                                                 aw.page_size, gs)
        sl = slice(hist_start, hist_start + n)
        for x_bits, R, clip, codes, s, z in ((wl_k[:, g], aw.Rk[g], aw.clip_k[g], kc[sl], sk[sl], zk[sl]),
                                             (wl_v[:, g], aw.Rv[g], aw.clip_v[g], vc[sl], sv[sl], zv[sl])):
            x64 = kq.rotate(kq.bf16_bits_to_f64(x_bits), R)
            c_ref, s_ref, z_ref = kq.quantize_rows(x64.astype(np.float32), clip, gs)
            # scale / zero within one fp16 ulp
            ds = np.abs(s.view(np.uint16).astype(np.int32) - s_ref.view(np.uint16).astype(np.int32))
            dz = np.abs(z.view(np.uint16).astype(np.int32) - z_ref.view(np.uint16).astype(np.int32))
            assert ds.max() <= 1 and (dz.max() <= 1 or np.all(np.abs(z - z_ref) <= 1e-6))
            same_group = (ds == 0) & (dz == 0)
            # code flips only next to a rounding boundary of the exact quotient
            y = kq.clip(x64, clip.astype(np.float64))
            ng = 128 // gs
            sf = s_ref.astype(np.float64); zf = z_ref.astype(np.float64)
            with np.errstate(divide="ignore", invalid="ignore"):
                qv = (y.reshape(-1, ng, gs) - zf[..., None]) / sf[..., None]
            # the kernel's rotated value carries fp32 rounding (relative ~1e-6 of the
            # group's range), so a flip needs the exact quotient within 1e-4 of a boundary
            near = np.abs(np.abs(qv - np.floor(qv)) - 0.5) < 1e-4
            diff = (codes != c_ref).reshape(-1, ng, gs)
            explained = near | ~same_group[..., None]
            assert not np.any(diff & ~explained), "code flip away from a rounding boundary"
            bad += int(diff.sum()); tot += diff.size
    return bad, tot


@pytest.mark.parametrize("gs,P", [(64, 16), (128, 32), (64, 32)])
def test_append_matches_oracle(gs, P):
    aw = synth.make_append_workload(f"app{gs}{P}", 30 + gs + P, n_seqs=3, Hkv=2,
                                    tokens_per_seq=[37, 64, 5], hist_start=[0, 16, 29],
                                    page_size=P, group_size=gs)
    pool = native.KVPool(native.KV_POOL_INT2_3TIER, 1, 8, 2, P, aw.num_pages, 3, group_size=gs)
    native.kv_pool_set_rotation(pool.handle, 0, gu.f32_dev(aw.Rk), gu.f32_dev(aw.Rv),
                                gu.f32_dev(aw.clip_k), gu.f32_dev(aw.clip_v))
    native.kv_append_quantize(pool.handle, 0, 3, gu.bf16_dev(aw.k), gu.bf16_dev(aw.v),
                              gu.i32_dev(aw.cu_tokens), gu.i32_dev(aw.hist_start),
                              gu.i32_dev(aw.page_table), aw.page_table.shape[1], 64)
    torch.cuda.synchronize()
    assert pool.error() == 0
    pages = pool.hist_view(0).cpu().numpy()
    bad = tot = 0
    for b in range(3):
        sl = slice(aw.cu_tokens[b], aw.cu_tokens[b + 1])
        x, y = _compare_codes(pages, aw.k[sl], aw.v[sl], aw, b, int(aw.hist_start[b]),
                              int(aw.tokens_per_seq[b]))
        bad += x; tot += y
    assert bad <= max(4, 1e-4 * tot), (bad, tot)
    pool.close()


def _append(aw, page_table, max_tokens):
    pool = native.KVPool(native.KV_POOL_INT2_3TIER, 1, 2 * aw.Hkv, aw.Hkv, aw.page_size, aw.num_pages,
                         aw.n_seqs, group_size=aw.group_size)
    native.kv_pool_set_rotation(pool.handle, 0, gu.f32_dev(aw.Rk), gu.f32_dev(aw.Rv),
                                gu.f32_dev(aw.clip_k), gu.f32_dev(aw.clip_v))
    native.kv_append_quantize(pool.handle, 0, aw.n_seqs, gu.bf16_dev(aw.k), gu.bf16_dev(aw.v),
                              gu.i32_dev(aw.cu_tokens), gu.i32_dev(aw.hist_start), gu.i32_dev(page_table),
                              page_table.shape[1], max_tokens)
    torch.cuda.synchronize()
    err = pool.error()
    pages = pool.hist_view(0).cpu().numpy()
    pool.close()
    return err, pages


def _seq_ok(aw, pages, b, n=None):
    sl = slice(aw.cu_tokens[b], aw.cu_tokens[b + 1])
    n = int(aw.tokens_per_seq[b]) if n is None else n
    bad, tot = _compare_codes(pages, aw.k[sl][:n], aw.v[sl][:n], aw, b, int(aw.hist_start[b]), n)
    assert bad <= max(4, 1e-4 * tot), (b, bad, tot)


def test_append_missing_page_and_empty_sequence():
    """A sequence whose last page id is missing: KV_DEVERR_PAGE_ID, its other
    pages and every other sequence still hold the oracle's codes; an empty
    sequence between them is no error."""
    aw = synth.make_append_workload("apppid", 91, n_seqs=4, Hkv=2, tokens_per_seq=[120, 0, 90, 100],
                                    hist_start=[0, 0, 0, 5], page_size=16, group_size=128)
    pt = aw.page_table.copy()
    pt[2, (90 - 1) // 16] = -1                      # positions 80..89 have no page
    err, pages = _append(aw, pt, 128)
    assert err == 1                                 # KV_DEVERR_PAGE_ID
    _seq_ok(aw, pages, 0)
    _seq_ok(aw, pages, 3)
    _seq_ok(aw, pages, 2, n=80)


def test_append_over_length_keeps_later_sequences_exact():
    """A sequence far above max_tokens_per_seq: KV_DEVERR_LENGTH.  The input
    rows of the valid sequence after it lie beyond n_seqs * max_tokens_per_seq
    rows, where the tensor-map loads stop; its chunks take the per-thread copies
    and its codes stay the oracle's."""
    aw = synth.make_append_workload("applen", 92, n_seqs=4, Hkv=2, tokens_per_seq=[120, 600, 100, 128],
                                    page_size=16, group_size=64)
    # sequences 2 and 3: every 128-row chunk lies below T but past the map's 4 * 128 rows
    assert aw.cu_tokens[2] >= 4 * 128 and aw.cu_tokens[2] + 128 <= aw.cu_tokens[4]
    err, pages = _append(aw, aw.page_table, 128)
    assert err == 2                                 # KV_DEVERR_LENGTH
    _seq_ok(aw, pages, 0)
    _seq_ok(aw, pages, 2)
    _seq_ok(aw, pages, 3)
    _seq_ok(aw, pages, 1, n=256)                    # the chunks the grid covers


def test_append_continues_partial_tiles():
    """Two appends into the same pages (unaligned split) equal one append."""
    aw = synth.make_append_workload("cont", 77, n_seqs=1, Hkv=2, tokens_per_seq=45, page_size=32,
                                    group_size=128, kv_kind="normal")
    outs = []
    for parts in ([45], [13, 20, 12]):
        pool = native.KVPool(native.KV_POOL_INT2_3TIER, 1, 2, 2, 32, aw.num_pages, 1, group_size=128)
        native.kv_pool_set_rotation(pool.handle, 0, gu.f32_dev(aw.Rk), gu.f32_dev(aw.Rv),
                                    gu.f32_dev(aw.clip_k), gu.f32_dev(aw.clip_v))
        start = 0
        for n in parts:
            native.kv_append_quantize(pool.handle, 0, 1, gu.bf16_dev(aw.k[start:start + n]),
                                      gu.bf16_dev(aw.v[start:start + n]), gu.i32_dev([0, n]),
                                      gu.i32_dev([start]), gu.i32_dev(aw.page_table),
                                      aw.page_table.shape[1], n)
            start += n
        torch.cuda.synchronize()
        outs.append(pool.hist_view(0).cpu().numpy())
        pool.close()
    assert np.array_equal(outs[0], outs[1])


# ---------------------------------------------------------------------------
# decode: identical stored codes (packed by the oracle) -> attention parity
# ---------------------------------------------------------------------------

def _decode_case(wl, **kw):
    pages = gu.oracle_pages(wl)
    pool = gu.make_int2_pool(wl)
    gu.upload_pages(pool, pages)
    out = gu.gpu_decode(pool, wl, **kw)
    ref = gu.oracle_decode(wl, pages, **{k: v for k, v in kw.items() if k != "max_hist"})
    err = pool.error()
    pool.close()
    return out, ref, err


def test_decode_tiny_workload():
    wl = synth.tiny_decode()
    out, ref, err = _decode_case(wl)
    assert err == 0
    ma, rl = gu.metrics(out, ref)
    print(f"tiny: max_abs {ma:.3e} rel_l2 {rl:.3e}")
    assert ma <= MAX_ABS and rl <= REL_L2


@pytest.mark.parametrize("G,P,gs", [(4, 16, 128), (8, 32, 128), (4, 32, 64), (2, 16, 64),
                                    (1, 16, 128), (8, 16, 64)])
def test_decode_shapes(G, P, gs):
    wl = synth.make_decode_workload(f"d{G}{P}{gs}", 40 + G + P + gs, B=3, Hq=2 * G, Hkv=2,
                                    ctx=[1500, 333, 700], page_size=P, group_size=gs,
                                    outliers_per_head=4)
    out, ref, err = _decode_case(wl)
    assert err == 0
    ma, rl = gu.metrics(out, ref)
    print(f"G{G} P{P} gs{gs}: max_abs {ma:.3e} rel_l2 {rl:.3e}")
    assert ma <= MAX_ABS and rl <= REL_L2


def test_decode_edge_lengths():
    """Partial tiles, history 0 and 1, short sink and recent tiers."""
    wl = synth.make_decode_workload("edges", 9, B=6, Hq=8, Hkv=2,
                                    ctx=[1, 64, 65, 321, 337, 350], page_size=16)
    assert list(wl.hist_len) == [0, 0, 0, 1, 17, 30]
    out, ref, err = _decode_case(wl)
    assert err == 0
    ma, rl = gu.metrics(out, ref)
    assert ma <= MAX_ABS and rl <= REL_L2


def test_decode_split_count_invariance():
    wl = synth.make_decode_workload("split", 10, B=1, Hq=8, Hkv=2, ctx=20000, page_size=16)
    pages = gu.oracle_pages(wl)
    pool = gu.make_int2_pool(wl)
    gu.upload_pages(pool, pages)
    a = gu.gpu_decode(pool, wl)
    b = gu.gpu_decode(pool, wl)                                   # same plan: deterministic
    pt2 = np.concatenate([wl.page_table, np.full((1, 300), -1, np.int32)], axis=1)
    c = gu.gpu_decode(pool, wl, page_table=pt2, max_hist=pt2.shape[1] * 16)   # other split count
    pool.close()
    assert np.array_equal(a, b)
    # another split count regroups the fp32 sums and re-rounds the fp16 hi + lo
    # softmax weights (relative to another running maximum); both results lie
    # within about 2e-5 of the oracle, so they must agree far inside the
    # parity tolerance
    assert gu.metrics(c, a)[1] <= 1e-4


def test_decode_page_permutation_is_bit_identical():
    wl = synth.make_decode_workload("perm", 11, B=2, Hq=8, Hkv=2, ctx=[900, 1300], page_size=16)
    outs = []
    rng = np.random.default_rng(3)
    for trial in range(2):
        perm = np.arange(wl.num_pages) if trial == 0 else rng.permutation(wl.num_pages)
        pt = np.where(wl.page_table >= 0, perm[np.maximum(wl.page_table, 0)], -1).astype(np.int32)
        pages = gu.oracle_pages(wl, page_table=pt)
        pool = gu.make_int2_pool(wl)
        gu.upload_pages(pool, pages)
        outs.append(gu.gpu_decode(pool, wl, page_table=pt))
        pool.close()
    assert np.array_equal(outs[0], outs[1])


def test_decode_hist0_equals_bf16_path():
    """With no history the INT2 decode is plain attention over BF16 tokens, as is
    the BF16 decode.  The BF16 decode applies each softmax weight as a bf16
    hi + lo pair on the tensor cores (relative error <= 2^-16 per weight), so
    the two agree to 1e-5 rel-L2, not to fp32 rounding."""
    wl = synth.make_decode_workload("h0", 12, B=3, Hq=8, Hkv=2, ctx=[70, 320, 200], page_size=16)
    assert int(wl.hist_len.max()) == 0
    pool = gu.make_int2_pool(wl)
    out = gu.gpu_decode(pool, wl)
    pool.close()
    bpool, pt, lens = gu.make_bf16_pool(wl)
    ref = gu.gpu_decode_bf16(bpool, wl, pt, lens)
    bpool.close()
    ma, rl = gu.metrics(out, ref)
    print(f"hist0 vs bf16: max_abs {ma:.3e} rel_l2 {rl:.3e}")
    assert rl <= 1e-5


def test_decode_grid_exact_equals_bf16_path():
    """R = I, no clip, history on the quantization grid: INT2 is lossless, so the
    INT2 decode equals the BF16 decode of the same tokens."""
    wl = synth.make_decode_workload("grid", 13, B=2, Hq=8, Hkv=2, ctx=[700, 1000], page_size=16,
                                    rotation="identity", clip_ratio=None)
    rng = np.random.default_rng(5)
    for b in range(wl.B):
        for arr in (wl.hist_k, wl.hist_v):
            k = rng.integers(0, 4, arr[b].shape); k[..., 0] = 0; k[..., 1] = 3
            arr[b] = synth.f32_to_bf16_bits((-1.5 + 0.5 * k).astype(np.float32))
    out, ref, err = _decode_case(wl)
    assert gu.metrics(out, ref)[1] <= 1e-5
    bpool, pt, lens = gu.make_bf16_pool(wl)
    bf = gu.gpu_decode_bf16(bpool, wl, pt, lens)
    bpool.close()
    assert gu.metrics(out, bf)[1] <= 1e-5


def test_decode_bad_page_id_sets_error_and_stays_finite():
    wl = synth.make_decode_workload("badpage", 14, B=1, Hq=8, Hkv=2, ctx=600, page_size=16)
    pages = gu.oracle_pages(wl)
    pool = gu.make_int2_pool(wl)
    gu.upload_pages(pool, pages)
    pt = wl.page_table.copy()
    pt[0, 3] = wl.num_pages + 100
    out = gu.gpu_decode(pool, wl, page_table=pt)
    assert pool.error() == 1          # KV_DEVERR_PAGE_ID
    assert np.all(np.isfinite(out))
    assert pool.error() == 0          # cleared by the read
    pool.close()


# ---------------------------------------------------------------------------
# BF16 baseline decode
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("G,P", [(4, 16), (8, 32), (1, 16)])
def test_decode_bf16_matches_oracle(G, P):
    wl = synth.make_decode_workload(f"bf{G}{P}", 60 + G + P, B=3, Hq=2 * G, Hkv=2,
                                    ctx=[1400, 257, 3000], page_size=P)
    bpool, pt, lens = gu.make_bf16_pool(wl)
    out = gu.gpu_decode_bf16(bpool, wl, pt, lens)
    assert bpool.error() == 0
    kp, vp = bpool.bf16_views(0)
    kb = kp.view(torch.int16).cpu().numpy().view(np.uint16)
    vb = vp.view(torch.int16).cpu().numpy().view(np.uint16)
    bpool.close()
    ref = att.decode_bf16_paged(wl.q, kb, vb, pt, lens, wl.Hkv, P, wl.scale)
    ma, rl = gu.metrics(out, ref)
    print(f"bf16 G={G} P={P}: max_abs {ma:.3e} rel_l2 {rl:.3e}")
    assert ma <= 1e-4 and rl <= 1e-5


# ---------------------------------------------------------------------------
# end to end: GPU append then GPU decode vs the oracle's own pipeline
# ---------------------------------------------------------------------------

def test_end_to_end_append_then_decode():
    """GPU append + GPU decode against the oracle's own rotate/quantize/attend
    pipeline.  The stored codes may differ in a handful of rounding-boundary
    flips (bounded in the append tests); one flipped V code of a token with
    weight ~1/N moves an output channel by ~s/N, which at N ~ 1e3 is of the
    order of 1e-3 of the output norm, so this end-to-end check uses the
    max-abs bound and a 1e-2 rel-L2 bound; the 1e-3 rel-L2 bound applies to
    identical stored codes (tests above)."""
    wl = synth.make_decode_workload("e2e", 15, B=2, Hq=8, Hkv=2, ctx=[2100, 900], page_size=16,
                                    outliers_per_head=4)
    pool = gu.make_int2_pool(wl)
    gu.gpu_append_history(pool, wl)
    out = gu.gpu_decode(pool, wl)
    assert pool.error() == 0
    pool.close()
    ref = gu.oracle_decode(wl, gu.oracle_pages(wl))
    ma, rl = gu.metrics(out, ref)
    print(f"e2e: max_abs {ma:.3e} rel_l2 {rl:.3e}")
    assert ma <= MAX_ABS and rl <= 1e-2


# ---------------------------------------------------------------------------
# lengths beyond what the call covers
# ---------------------------------------------------------------------------

def test_decode_history_beyond_max_hist_len_is_flagged():
    """hist_len[b] above max_hist_len: KV_DEVERR_LENGTH, and the sequence's
    first max_hist_len history tokens (the ones the grid covers) are attended;
    the other sequence is unaffected."""
    wl = synth.make_decode_workload("overlen", 16, B=2, Hq=8, Hkv=2, ctx=[1100, 700], page_size=16)
    assert list(wl.hist_len) == [780, 380]
    pages = gu.oracle_pages(wl)
    pool = gu.make_int2_pool(wl)
    gu.upload_pages(pool, pages)
    out = gu.gpu_decode(pool, wl, max_hist=500)
    assert pool.error() == 2                                   # KV_DEVERR_LENGTH
    assert np.all(np.isfinite(out))
    ref = gu.oracle_decode(wl, pages, hist_len=np.array([500, 380]))
    ma, rl = gu.metrics(out, ref)
    assert ma <= MAX_ABS and rl <= REL_L2, (ma, rl)
    pool.close()


def test_decode_bf16_length_beyond_max_seq_len_is_flagged():
    wl = synth.make_decode_workload("overlen_bf", 17, B=2, Hq=8, Hkv=2, ctx=[900, 400], page_size=16)
    bpool, pt, lens = gu.make_bf16_pool(wl)
    ws_bytes = native.kv_decode_workspace_bytes(bpool.handle, wl.B, 600)
    ws = torch.empty(ws_bytes // 4 + 4, dtype=torch.float32, device="cuda")
    out = torch.full((wl.B, wl.Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    native.kv_decode_attention_bf16(bpool.handle, 0, wl.B, gu.bf16_dev(wl.q), gu.i32_dev(lens),
                                    gu.i32_dev(pt), pt.shape[1], 600, wl.scale, out, ws, ws_bytes)
    torch.cuda.synchronize()
    assert bpool.error() == 2                                  # KV_DEVERR_LENGTH
    kp, vp = bpool.bf16_views(0)
    kb = kp.view(torch.int16).cpu().numpy().view(np.uint16)
    vb = vp.view(torch.int16).cpu().numpy().view(np.uint16)
    bpool.close()
    ref = att.decode_bf16_paged(wl.q, kb, vb, pt, np.minimum(lens, 600), wl.Hkv, 16, wl.scale)
    ma, rl = gu.metrics(out.cpu().numpy(), ref)
    assert ma <= 1e-4 and rl <= 1e-5, (ma, rl)
