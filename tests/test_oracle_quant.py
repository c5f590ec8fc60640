"""Pins for the oracle's quantizer, packer and tile layout (CPU only).

Each test checks the oracle against something that does not come from the
oracle: hand-worked fixtures (tests/golden), closed forms, or exhaustive
enumeration."""

import numpy as np
import pytest

from oracle import kvquant as kq
from bit_kv_cache_12_gb300 import synth
from tests.conftest import read_golden


# --------------------------------------------------------------------------
# quantizer
# --------------------------------------------------------------------------

def test_quantizer_golden_cases():
    for y_s, sz, codes_s, note in read_golden("quantizer_cases.txt"):
        y = np.array([float(v) for v in y_s.split()], np.float32)
        s_hex, z_hex = sz.split()
        exp_codes = np.array([int(c) for c in codes_s.split()])
        codes, s, z = kq.quantize_groups(y[None, :], 4)
        assert codes[0].tolist() == exp_codes.tolist(), note
        assert int(s.view(np.uint16)[0, 0]) == int(s_hex, 16), note
        assert int(z.view(np.uint16)[0, 0]) == int(z_hex, 16), note


def test_f16_saturation_and_rounding():
    # 65519.99 rounds to 65504 (RNE), 65520 would overflow -> saturate
    v = np.array([65519.0, 65520.0, 1e9, -1e9, 1.0 / 3.0], np.float32)
    h = kq.to_f16_sat(v).view(np.uint16)
    assert h.tolist() == [0x7BFF, 0x7BFF, 0x7BFF, 0xFBFF, 0x3555]


def test_quantizer_error_bound_and_extremes():
    """|y - deq| <= s/2 + |z - mn| + 3|s - s32| + 4 ulp for unclipped values;
    codes in 0..3; min -> 0 and max -> 3 when fp16 rounding is small vs s."""
    rng = np.random.default_rng(11)
    for gs in (64, 128):
        y = rng.standard_normal((500, 128)).astype(np.float32)
        y[:, 7] *= 10.0
        codes, s_h, z_h = kq.quantize_groups(y, gs)
        assert codes.max() <= 3
        deq = kq.dequant(codes, s_h, z_h, gs)
        ng = 128 // gs
        yg = y.reshape(500, ng, gs).astype(np.float64)
        mn, mx = yg.min(-1), yg.max(-1)
        s32 = ((y.reshape(500, ng, gs).max(-1) - y.reshape(500, ng, gs).min(-1))
               / np.float32(3)).astype(np.float64)
        s = s_h.astype(np.float64); z = z_h.astype(np.float64)
        ulp = np.spacing(np.maximum(np.abs(mn), np.abs(mx)).astype(np.float32)).astype(np.float64)
        bound = s / 2 + np.abs(z - mn) + 3 * np.abs(s - s32) + 4 * ulp
        err = np.abs(yg - deq.reshape(500, ng, gs)).max(-1)
        assert np.all(err <= bound + 1e-12)
        cg = codes.reshape(500, ng, gs)
        ok = (np.abs(z - mn) < s / 4) & (3 * np.abs(s - s32) < s / 4)
        argmn = yg.argmin(-1); argmx = yg.argmax(-1)
        cmin = np.take_along_axis(cg, argmn[..., None], -1)[..., 0]
        cmax = np.take_along_axis(cg, argmx[..., None], -1)[..., 0]
        assert np.all(cmin[ok] == 0) and np.all(cmax[ok] == 3)
        assert ok.mean() > 0.99


def test_grid_exact_values_roundtrip():
    """Values on the quantization grid z + k s (fp16-exact z, s; bf16-exact y)
    come back exactly through quantize + dequant."""
    rng = np.random.default_rng(5)
    z = np.float32(-1.5); s = np.float32(0.5)
    for _ in range(20):
        k = rng.integers(0, 4, size=(8, 128))
        k[:, 0] = 0; k[:, 1] = 3            # pin min and max of each group
        y = (z + k * s).astype(np.float32)
        codes, s_h, z_h = kq.quantize_groups(y, 128)
        assert np.array_equal(codes, k)
        assert np.all(s_h == np.float16(0.5)) and np.all(z_h == np.float16(-1.5))
        assert np.array_equal(kq.dequant(codes, s_h, z_h, 128), y.astype(np.float64))


def test_clip_hand_cases():
    y = np.array([[-5.0, -1.0, 0.5, 7.0]], np.float32)
    c = np.array([2.0, 2.0, np.inf, 3.0], np.float32)
    assert kq.clip(y, c).tolist() == [[-2.0, -1.0, 0.5, 3.0]]


# --------------------------------------------------------------------------
# packing
# --------------------------------------------------------------------------

def test_pack_golden_cases():
    for codes_s, byte_hex in read_golden("pack_cases.txt"):
        c = np.array([[int(v) for v in codes_s.split()]], np.uint8)
        assert int(kq.pack_canonical(c)[0, 0]) == int(byte_hex, 16)


def test_pack_unpack_all_bytes_bijective():
    allb = np.arange(256, dtype=np.uint8)[None, :]
    codes = kq.unpack_canonical(allb)
    assert codes.shape == (1, 1024)
    assert np.array_equal(kq.pack_canonical(codes), allb)
    # every 4-code combination appears exactly once
    quads = codes.reshape(256, 4)
    assert len({tuple(q) for q in quads}) == 256
    rng = np.random.default_rng(2)
    c = rng.integers(0, 4, size=(33, 128)).astype(np.uint8)
    assert np.array_equal(kq.unpack_canonical(kq.pack_canonical(c)), c)


# --------------------------------------------------------------------------
# tile layout
# --------------------------------------------------------------------------

def test_tile_layout_golden_positions():
    for spec, pos in read_golden("tile_layout_cases.txt"):
        tensor, t, c = spec.split(); t = int(t); c = int(c)
        byte, shift = (int(v) for v in pos.split())
        if tensor == "K":
            b, s = kq.tile_code_bit(t, c % 16, c // 16)
        else:
            b, s = kq.tile_code_bit(c % 16, t, c // 16)
        assert (int(b), int(s)) == (byte, shift), spec


@pytest.mark.parametrize("tensor", ["K", "V"])
def test_tile_layout_is_a_bijection(tensor):
    seen = set()
    for t in range(16):
        for c in range(128):
            b, s = (kq.tile_code_bit(t, c % 16, c // 16) if tensor == "K"
                    else kq.tile_code_bit(c % 16, t, c // 16))
            b = int(b); s = int(s)
            assert 0 <= b < 512 and s in (0, 2, 4, 6)
            seen.add((b, s))
    assert len(seen) == 2048


@pytest.mark.parametrize("gs", [64, 128])
def test_tile_record_positions(gs):
    """Byte positions of the s/z records, worked by hand from the documented
    layout: after the 1024 code bytes, 16 K slots of 4 * (128 / gs) bytes, then
    16 V slots; slot 2 (t % 8) + t / 8 holds token t as (s, z) fp16 per group."""
    ng = 128 // gs
    sk = np.zeros((16, ng), np.float16); zk = np.zeros((16, ng), np.float16)
    sv = np.zeros((16, ng), np.float16); zv = np.zeros((16, ng), np.float16)
    sk[0, 0], zk[0, 0] = 1.5, -2.0       # token 0: slot 0
    sk[8, 0], zk[8, 0] = 3.0, 0.25       # token 8: slot 1
    sk[1, ng - 1] = 6.0                  # token 1: slot 2, last group
    sv[0, 0], zv[0, 0] = 0.5, -1.0       # V block, token 0
    sv[15, ng - 1] = 7.0                 # V block, token 15: slot 15, last group
    z = np.zeros((16, 128), np.uint8)
    tile = kq.pack_tile(z, z, sk, zk, sv, zv, gs)
    f16 = lambda off: float(tile[off:off + 2].view(np.float16)[0])
    kb, vb = 1024, 1024 + 16 * 4 * ng
    assert (f16(kb), f16(kb + 2)) == (1.5, -2.0)
    assert (f16(kb + 4 * ng), f16(kb + 4 * ng + 2)) == (3.0, 0.25)
    assert f16(kb + 2 * 4 * ng + 4 * (ng - 1)) == 6.0
    assert (f16(vb), f16(vb + 2)) == (0.5, -1.0)
    assert f16(vb + 15 * 4 * ng + 4 * (ng - 1)) == 7.0
    assert len(tile) == 1024 + 2 * 16 * 4 * ng
    back = kq.unpack_tile(tile, gs)
    for got, want in zip(back[2:], (sk, zk, sv, zv)):
        assert np.array_equal(got, want)


@pytest.mark.parametrize("gs", [64, 128])
def test_tile_pack_roundtrip_and_partial_merge(gs):
    rng = np.random.default_rng(9)
    ng = 128 // gs
    kc = rng.integers(0, 4, (16, 128)).astype(np.uint8); vc = rng.integers(0, 4, (16, 128)).astype(np.uint8)
    sk, zk, sv, zv = (rng.standard_normal((16, ng)).astype(np.float16) for _ in range(4))
    buf = kq.pack_tile(kc, vc, sk, zk, sv, zv, gs)
    assert buf.size == kq.tile_bytes(gs)
    out = kq.unpack_tile(buf, gs)
    for a, b in zip(out, (kc, vc, sk, zk, sv, zv)):
        assert np.array_equal(a, b)
    # partial write keeps other tokens
    kc2 = rng.integers(0, 4, (16, 128)).astype(np.uint8)
    valid = np.zeros(16, bool); valid[3:11] = True
    buf2 = kq.pack_tile(kc2, vc, sk, zk, sv, zv, gs, base=buf, valid=valid)
    k_back = kq.unpack_tile(buf2, gs)[0]
    assert np.array_equal(k_back[valid], kc2[valid]) and np.array_equal(k_back[~valid], kc[~valid])


def test_history_pages_roundtrip_across_appends():
    """Two appends at unaligned history positions, then a read back."""
    aw = synth.make_append_workload("t", 3, n_seqs=1, Hkv=2, tokens_per_seq=37, page_size=32,
                                    group_size=64, kv_kind="normal")
    ps, gs = 32, 64
    pages = np.zeros((aw.num_pages, 2, (ps // 16) * kq.tile_bytes(gs)), np.uint8)
    q_all = {}
    for g in range(2):
        q = kq.quantize_tokens(aw.k[:, g], aw.v[:, g], aw.Rk[g], aw.Rv[g], aw.clip_k[g],
                               aw.clip_v[g], gs)
        q_all[g] = q
        first = {kk: v[:20] for kk, v in q.items()}
        second = {kk: v[20:] for kk, v in q.items()}
        kq.pack_history(pages, aw.page_table[0], 0, first, g, 2, ps, gs)
        kq.pack_history(pages, aw.page_table[0], 20, second, g, 2, ps, gs)
    for g in range(2):
        kc, vc, sk, zk, sv, zv = kq.read_history(pages, aw.page_table[0], 37, g, ps, gs)
        q = q_all[g]
        assert np.array_equal(kc, q["kc"]) and np.array_equal(vc, q["vc"])
        assert np.array_equal(sk, q["sk"]) and np.array_equal(zv, q["zv"])


@pytest.mark.parametrize("gs", [64, 128])
def test_vectorised_tile_packer_matches_per_code_packer(gs):
    rng = np.random.default_rng(17)
    ng = 128 // gs
    n = 3
    kc = rng.integers(0, 4, (n, 16, 128)).astype(np.uint8); vc = rng.integers(0, 4, (n, 16, 128)).astype(np.uint8)
    sk, zk, sv, zv = (rng.standard_normal((n, 16, ng)).astype(np.float16) for _ in range(4))
    fast = kq.pack_tiles_full(kc, vc, sk, zk, sv, zv, gs)
    for i in range(n):
        slow = kq.pack_tile(kc[i], vc[i], sk[i], zk[i], sv[i], zv[i], gs)
        assert np.array_equal(fast[i], slow)


def test_pack_history_full_matches_incremental():
    aw = synth.make_append_workload("t", 4, n_seqs=1, Hkv=2, tokens_per_seq=45, page_size=16,
                                    group_size=128, kv_kind="normal")
    a = kq.pack_history_full(aw.k, aw.v, aw.Rk, aw.Rv, aw.clip_k, aw.clip_v, aw.page_table[0],
                             aw.num_pages, 2, 16, 128)
    b = np.zeros_like(a)
    for g in range(2):
        q = kq.quantize_tokens(aw.k[:, g], aw.v[:, g], aw.Rk[g], aw.Rv[g], aw.clip_k[g],
                               aw.clip_v[g], 128)
        kq.pack_history(b, aw.page_table[0], 0, q, g, 2, 16, 128)
    assert np.array_equal(a, b)
