"""Bit-exact parity of the quantizer that stores the history.

The yunpan.plus OSCAR write-up ("2. 在线量化与反量化") quantizes every token
leaving the recent window: rotate, clip, asymmetric INT2 with fp16 scale and
zero per group, pack.  The codes the pool keeps come from the tensor-core
append kernels (``kv_append_quantize`` in bulk, ``kv_append_step`` per decode
step), whose epilogue forms fl(fl(y - z) * fl(1/s)), rounds it with the
1.5 * 2^23 trick and falls back to the IEEE division when a quotient of the
warp lies within 2^-18 of a half-integer.  With R = I the tensor-core product
of bf16 rows with [I | 0] is exact, so both paths see exactly the fp32 input
the oracle quantizes, and codes, scales and zeros must agree bit for bit (no
flip budget).

The rows are built to reach every branch: exact half-integer ties (fp16-exact
z and s; whole warps of them, a single one among random rows, and none), a
reciprocal 1/s that is not exact, quotients 2^-20 below and above a tie,
constant groups (s = 0), -0 rows, s below the fp16 range, a subnormal fp16 s,
saturation at +-65504, clipped and unclipped channels, group 64 and 128, K
and V."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from bit_kv_cache_12_gb300 import native, synth
from oracle import kvquant as kq
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    native.lib()


# ---------------------------------------------------------------------------
# crafted groups (float32 values that are exact in bf16)
# ---------------------------------------------------------------------------

def _fill(rng, n, values, ends):
    """n values drawn from `values`, with the group's min and max `ends` present."""
    g = rng.choice(np.asarray(values, np.float32), n)
    pos = rng.choice(n, 2, replace=False)
    g[pos[0]], g[pos[1]] = ends
    return g


def _tie_group(rng, n):
    # z = -2, s = 0.5: the quotients of -1.75, -1.25, -0.75 are exactly 0.5, 1.5, 2.5
    if rng.random() < 0.5:
        return _fill(rng, n, [-2.0, -1.75, -1.5, -1.25, -1.0, -0.75, -0.5], (-2.0, -0.5))
    # z = -1, s = 0.75 (1/s not exact in fp32): ties at -0.625, 0.125, 0.875
    return _fill(rng, n, [-1.0, -0.625, -0.25, 0.125, 0.5, 0.875, 1.25], (-1.0, 1.25))


def _near_tie_group(rng, n):
    """Quotients 2^-20 (or 2^-21) off a half-integer: inside the fix-up band, not ties."""
    e = np.float32(2.0 ** -20)
    kind = rng.integers(0, 3)
    if kind == 0:     # z = 2^-20, s = 1: 0.5, 1.5, 2.5 give quotients just below .5
        return _fill(rng, n, [e, 0.5, 1.0, 1.5, 2.0, 2.5, 3.0], (e, 3.0))
    if kind == 1:     # z = -2^-20, s = 1: just above .5
        return _fill(rng, n, [-e, 0.0, 0.5, 1.0, 1.5, 2.5, 3.0], (-e, 3.0))
    e2 = np.float32(2.0 ** -22)   # z = 2^-22, s = 0.5
    return _fill(rng, n, [e2, 0.25, 0.5, 0.75, 1.0, 1.25, 1.5], (e2, 1.5))


def _special_group(rng, n, which):
    if which == 0:                                   # constant: s = 0
        return np.full(n, 1.25, np.float32)
    if which == 1:                                   # -0: s = 0, z = +0
        return np.full(n, -0.0, np.float32)
    if which == 2:                                   # range 1e-8: s underflows fp16
        return (rng.random(n) * 1e-8).astype(np.float32)
    if which == 3:                                   # s = 2^-20 (fp16 subnormal), ties
        u = np.float32(2.0 ** -20)
        return _fill(rng, n, u * np.array([0, 0.5, 1, 1.5, 2, 2.5, 3], np.float32), (0.0, 3 * u))
    if which == 4:                                   # saturation: s and z at +-65504
        return (rng.uniform(-1.0, 1.0, n) * 1e6).astype(np.float32)
    # wide range, mostly clamped codes after saturation of z
    g = (rng.uniform(0.0, 1.0, n) * 3e5).astype(np.float32)
    g[rng.integers(0, n)] = -2e5
    return g


def _random_group(rng, n):
    g = rng.standard_normal(n).astype(np.float32)
    g[rng.integers(0, n)] *= 12.0
    return g


def _row(rng, kind, gs):
    """One 128-channel row of one head, built from groups of gs channels."""
    parts = []
    for _ in range(128 // gs):
        if kind == "tie":
            parts.append(_tie_group(rng, gs))
        elif kind == "near":
            parts.append(_near_tie_group(rng, gs))
        elif kind == "mixed":
            parts.append(_tie_group(rng, gs) if rng.random() < 0.5 else _random_group(rng, gs))
        elif isinstance(kind, tuple):
            parts.append(_special_group(rng, gs, kind[1]))
        else:
            parts.append(_random_group(rng, gs))
    return np.concatenate(parts)


def _row_kind(i):
    """Row i of a 128-row chunk: warp quarters (32 rows each) take different
    paths of the epilogue's fix-up (taken by the whole warp when any lane
    needs it)."""
    m = i % 128
    q = m // 32
    if q == 0:
        return "tie" if m % 3 else "near"            # every lane near a tie
    if q == 1:
        return "tie" if m == 40 else "random"        # one lane in the warp
    if q == 2:
        return "random"                              # the fast path only
    return ("special", (m // 2) % 6) if m % 2 else "mixed"


def crafted_rows(rng, n, hkv, gs):
    """bf16 bits [n, hkv, 128]; the tie, near-tie and special groups are exact
    in bf16 by construction, random groups are rounded to bf16."""
    x = np.zeros((n, hkv, 128), np.float32)
    for i in range(n):
        for g in range(hkv):
            x[i, g] = _row(rng, _row_kind(i + 7 * g), gs)
    return synth.f32_to_bf16_bits(x)


def clip_thresholds(hkv):
    """K: +inf on channels 0..95, 2.5 on 96..127; V: 1.7 on 0..15, +inf elsewhere."""
    ck = np.full((hkv, 128), np.inf, np.float32); ck[:, 96:] = 2.5
    cv = np.full((hkv, 128), np.inf, np.float32); cv[:, :16] = 1.7
    return ck, cv


def expected(bits, clip, gs):
    """Codes, s, z of the oracle on the exact fp32 input (R = I)."""
    return kq.quantize_rows(synth.bf16_bits_to_f32(bits), clip[None], gs)


def _assert_same(got, ref, where):
    codes, s, z = got
    c_ref, s_ref, z_ref = ref
    assert np.array_equal(codes, c_ref), f"{where}: {int((codes != c_ref).sum())} codes differ"
    assert np.array_equal(s.view(np.uint16), s_ref.view(np.uint16)), f"{where}: scales differ"
    assert np.array_equal(z.view(np.uint16), z_ref.view(np.uint16)), f"{where}: zeros differ"


def _identity_pool(hkv, P, gs, num_pages, max_seqs, ck, cv, sink=64, recent=256):
    pool = native.KVPool(native.KV_POOL_INT2_3TIER, 1, 2 * hkv, hkv, P, num_pages, max_seqs,
                         group_size=gs, sink_tokens=sink, recent_tokens=recent)
    eye = gu.f32_dev(np.stack([np.eye(128, dtype=np.float32)] * hkv))
    keep = (eye, gu.f32_dev(ck), gu.f32_dev(cv))
    native.kv_pool_set_rotation(pool.handle, 0, eye, eye, keep[1], keep[2])
    pool._keep = keep
    return pool


# ---------------------------------------------------------------------------
# bulk append (kv_append_quantize)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("gs,P", [(64, 16), (128, 16), (128, 32), (64, 32)])
def test_bulk_append_codes_bit_exact(gs, P):
    rng = np.random.default_rng(500 + gs + P)
    hkv = 2
    tokens = np.array([300, 128, 45])                # several chunks, an exact chunk, a ragged one
    starts = np.array([0, 16, 7])                    # aligned, tile-aligned, unaligned starts
    n = int(tokens.sum())
    kb = crafted_rows(rng, n, hkv, gs)
    vb = crafted_rows(rng, n, hkv, gs)
    ck, cv = clip_thresholds(hkv)
    pages_per = (starts + tokens + P - 1) // P
    num_pages = int(pages_per.sum()) + 2
    perm = rng.permutation(num_pages).astype(np.int32)
    pt = np.full((3, int(pages_per.max())), -1, np.int32)
    o = 0
    for b in range(3):
        pt[b, :pages_per[b]] = perm[o:o + pages_per[b]]; o += pages_per[b]
    cu = np.concatenate([[0], np.cumsum(tokens)]).astype(np.int32)
    pool = _identity_pool(hkv, P, gs, num_pages, 3, ck, cv)
    native.kv_append_quantize(pool.handle, 0, 3, gu.bf16_dev(kb), gu.bf16_dev(vb), gu.i32_dev(cu),
                              gu.i32_dev(starts), gu.i32_dev(pt), pt.shape[1], int(tokens.max()))
    torch.cuda.synchronize()
    assert pool.error() == 0
    pages = pool.hist_view(0).cpu().numpy()
    pool.close()
    for b in range(3):
        sl = slice(cu[b], cu[b + 1])
        for g in range(hkv):
            kc, vc, sk, zk, sv, zv = kq.read_history(pages, pt[b], int(starts[b] + tokens[b]), g, P, gs)
            h = slice(int(starts[b]), None)
            _assert_same((kc[h], sk[h], zk[h]), expected(kb[sl, g], ck[g], gs), f"K seq {b} head {g}")
            _assert_same((vc[h], sv[h], zv[h]), expected(vb[sl, g], cv[g], gs), f"V seq {b} head {g}")


def test_crafted_rows_reach_every_branch():
    """The crafted inputs really contain exact ties, near ties inside the
    2^-18 band, s = 0 groups, a subnormal s and saturated s and z (checked on
    the oracle's own quantities, so the bit-exact tests above cover them)."""
    rng = np.random.default_rng(9)
    for gs in (64, 128):
        bits = crafted_rows(rng, 128, 2, gs)
        y = synth.bf16_bits_to_f32(bits).reshape(128, 2, 128 // gs, gs)
        c, s, z = kq.quantize_groups(y.reshape(128, 2, 128), gs)
        sf = s.astype(np.float64)[..., None]; zf = z.astype(np.float64)[..., None]
        with np.errstate(divide="ignore", invalid="ignore"):
            qv = (y.astype(np.float64) - zf) / sf
            frac = np.abs(qv - np.floor(qv) - 0.5)   # nan where s = 0: not live below
        live = np.isfinite(qv) & (qv >= 0) & (qv <= 3)
        assert np.any(live & (frac == 0)), "exact ties"
        assert np.any(live & (frac > 0) & (frac < 2.0 ** -18)), "near ties"
        assert np.any(s == 0), "s = 0 groups"
        assert np.any((s > 0) & (np.abs(s.astype(np.float32)) < 2.0 ** -14)), "subnormal s"
        assert np.any(s.astype(np.float32) == 65504.0) and np.any(z.astype(np.float32) == -65504.0)


# ---------------------------------------------------------------------------
# per-step eviction (kv_append_step)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("gs,P", [(128, 16), (64, 32)])
def test_step_eviction_codes_bit_exact(gs, P):
    """128 sequences whose rings hold crafted rows: every step evicts the oldest
    ring row into history, so after n steps history positions 0..n-1 hold the
    crafted stream c_0, c_1, ..; sequence b is row b of the eviction chunk,
    so warp quarters again see all-tie, one-tie, tie-free and special rows."""
    rng = np.random.default_rng(700 + gs + P)
    hkv, B, S, W, n_steps = 2, 128, 4, 8, 40
    ck, cv = clip_thresholds(hkv)
    stream_k = np.zeros((B, W + n_steps, hkv, 128), np.uint16)
    stream_v = np.zeros_like(stream_k)
    for b in range(B):
        for i in range(W + n_steps):
            for g in range(hkv):
                kind = _row_kind(b) if i % 5 else "random"
                stream_k[b, i, g] = synth.f32_to_bf16_bits(_row(rng, kind, gs))
                stream_v[b, i, g] = synth.f32_to_bf16_bits(_row(rng, kind, gs))
    pages_per = (n_steps + P - 1) // P
    num_pages = B * pages_per + 1
    pt = rng.permutation(num_pages).astype(np.int32)[:B * pages_per].reshape(B, pages_per)
    pool = _identity_pool(hkv, P, gs, num_pages, B, ck, cv, sink=S, recent=W)
    sk, sv, rk, rv = pool.tier_views(0)
    rk[:B].copy_(gu.bf16_dev(stream_k[:, :W].transpose(0, 2, 1, 3)))   # ring [B][Hkv][W][128]
    rv[:B].copy_(gu.bf16_dev(stream_v[:, :W].transpose(0, 2, 1, 3)))
    lens = [gu.i32_dev(np.full(B, S)), gu.i32_dev(np.zeros(B)), gu.i32_dev(np.full(B, W)),
            gu.i32_dev(np.zeros(B))]
    ptd = gu.i32_dev(pt)
    new_k = gu.bf16_dev(stream_k[:, W:])                                # [B][n][Hkv][128]
    new_v = gu.bf16_dev(stream_v[:, W:])
    for i in range(n_steps):
        native.kv_append_step(pool.handle, 0, B, new_k[:, i].contiguous(), new_v[:, i].contiguous(),
                              *lens, ptd, pt.shape[1])
    torch.cuda.synchronize()
    assert pool.error() == 0
    assert np.all(lens[1].cpu().numpy() == n_steps)
    pages = pool.hist_view(0).cpu().numpy()
    pool.close()
    for b in range(B):
        for g in range(hkv):
            kc, vc, skk, zk, svv, zv = kq.read_history(pages, pt[b], n_steps, g, P, gs)
            _assert_same((kc, skk, zk), expected(stream_k[b, :n_steps, g], ck[g], gs), f"K seq {b} head {g}")
            _assert_same((vc, svv, zv), expected(stream_v[b, :n_steps, g], cv[g], gs), f"V seq {b} head {g}")
