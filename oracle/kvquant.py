"""Oracle: rotate -> clip -> asymmetric INT2 quantize -> pack (CPU, numpy).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

What the method does to a token leaving the BF16 recent window
(yunpan.plus OSCAR write-up, "2. 在线量化与反量化": rotate, clip, quantize,
pack, four 2-bit values per byte; gist.science OSCAR explainer, section 2.2 B:
history is kept in INT2 after the fixed rotation and the clip):

1. rotate   x' = x . R           row-vector convention, R orthogonal d x d,
                                  fixed offline (section 2.2 A, R = U H P_br)
2. clip     y_j = min(max(x'_j, -c_j), c_j)   per rotated channel
3. quantize per token and per group of Gs contiguous rotated channels:
              mn, mx = min, max of the group (fp32)
              s32 = (mx - mn) / 3            fp32, round-to-nearest-even
              s = fp16(s32), z = fp16(mn + 0)  saturated to +-65504
              code = 0 if s == 0 else clamp(rint((y - z) / s), 0, 3)
   (asymmetric INT2, fp16 scale and zero per token per group; the pages give
   no formula, so this is the plain reading: zero = the group minimum, codes
   computed with the rounded fp16 scale/zero so quantizer and dequantizer
   agree, IEEE fp32 subtraction and division, ties to even.)
4. dequant  deq = code * s + z
5. pack     byte b of a row holds channels 4b..4b+3, channel 4b+j in bits
            [2j, 2j+2)  ("每4个2bit数值打包进1个Byte")

Paged storage: the library keeps each 16-token tile of a (page, KV head) in
the order its decode kernel consumes (``tile_code_bit``).  The oracle states
that order as an explicit index map and packs / unpacks through it.
"""

import numpy as np

F16_MAX = np.float32(65504.0)
TILE = 16          # tokens per history tile
HEAD_DIM = 128


# --------------------------------------------------------------------------
# bf16 helpers (inputs are bf16 bit patterns stored as uint16)
# --------------------------------------------------------------------------

def bf16_bits_to_f32(u16):
    """Exact widening of bf16 bit patterns to float32."""
    u16 = np.asarray(u16, dtype=np.uint16)
    return (u16.astype(np.uint32) << 16).view(np.float32)


def bf16_bits_to_f64(u16):
    return bf16_bits_to_f32(u16).astype(np.float64)


# --------------------------------------------------------------------------
# 1. rotation, 2. clip
# --------------------------------------------------------------------------

def rotate(x, R):
    """x' = x . R in fp64.  x: [..., d] (float), R: [d, d] (float).

    Row-vector convention: column j of R is the j-th basis vector of the
    rotated space (R = U_Q H P_br, the eigenbasis in the columns)."""
    x = np.asarray(x, dtype=np.float64)
    R = np.asarray(R, dtype=np.float64)
    return x @ R


def clip(y, c):
    """Symmetric per-channel clip to [-c_j, c_j]; c_j = +inf disables it.
    Works in the dtype of ``y`` (fp32 for the quantizer path)."""
    c = np.asarray(c, dtype=y.dtype)
    return np.minimum(np.maximum(y, -c), c)


# --------------------------------------------------------------------------
# 3. quantize (fp32 arithmetic, bit-exact definition)
# --------------------------------------------------------------------------

def to_f16_sat(x32):
    """fp32 -> fp16 with round-to-nearest-even, overflow saturated to +-65504."""
    x32 = np.asarray(x32, dtype=np.float32)
    with np.errstate(over="ignore"):
        h = x32.astype(np.float16)
    h = np.where(np.isinf(h) & np.isfinite(x32),
                 np.copysign(np.float16(65504.0), x32).astype(np.float16), h)
    return h.astype(np.float16)


def quantize_groups(y, group_size):
    """Quantize clipped rotated rows.

    y: float32 [..., d].  Returns (codes uint8 [..., d] in 0..3,
    s fp16 [..., d/Gs], z fp16 [..., d/Gs])."""
    y = np.asarray(y, dtype=np.float32)
    d = y.shape[-1]
    assert d % group_size == 0
    ng = d // group_size
    yg = y.reshape(y.shape[:-1] + (ng, group_size))
    mn = yg.min(axis=-1)
    mx = yg.max(axis=-1)
    s32 = (mx - mn) / np.float32(3.0)                       # fp32 sub, fp32 div
    s_h = to_f16_sat(s32)
    z_h = to_f16_sat(mn + np.float32(0.0))                  # +0 canonicalises -0
    s = s_h.astype(np.float32)[..., None]
    z = z_h.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        q = (yg - z) / s                                    # fp32 sub, fp32 div
        code = np.clip(np.rint(q), 0.0, 3.0)
    code = np.where(s == 0, 0.0, code)
    return code.astype(np.uint8).reshape(y.shape), s_h, z_h


def dequant(codes, s_h, z_h, group_size):
    """deq = code * s + z in fp64.  codes [..., d], s/z [..., d/Gs]."""
    codes = np.asarray(codes, dtype=np.float64)
    d = codes.shape[-1]
    ng = d // group_size
    cg = codes.reshape(codes.shape[:-1] + (ng, group_size))
    s = np.asarray(s_h, dtype=np.float64)[..., None]
    z = np.asarray(z_h, dtype=np.float64)[..., None]
    return (cg * s + z).reshape(codes.shape)


def quantize_rows(x_rot32, clip_c, group_size):
    """Clip then quantize fp32 rotated rows (the library's parity entry)."""
    y = clip(np.asarray(x_rot32, dtype=np.float32), np.asarray(clip_c, dtype=np.float32))
    return quantize_groups(y, group_size)


# --------------------------------------------------------------------------
# 5. canonical packing (four codes per byte, little-endian within the byte)
# --------------------------------------------------------------------------

def pack_canonical(codes):
    """codes uint8 [..., d] (0..3) -> bytes uint8 [..., d/4]."""
    c = np.asarray(codes, dtype=np.uint8)
    c4 = c.reshape(c.shape[:-1] + (c.shape[-1] // 4, 4)).astype(np.uint32)
    b = c4[..., 0] | (c4[..., 1] << 2) | (c4[..., 2] << 4) | (c4[..., 3] << 6)
    return b.astype(np.uint8)


def unpack_canonical(packed):
    p = np.asarray(packed, dtype=np.uint8).astype(np.uint32)
    out = np.stack([(p >> (2 * j)) & 3 for j in range(4)], axis=-1)
    return out.reshape(p.shape[:-1] + (p.shape[-1] * 4,)).astype(np.uint8)


# --------------------------------------------------------------------------
# Paged tile layout of the INT2 history (the library's storage order)
# --------------------------------------------------------------------------
#
# A page of P tokens (P = 16 or 32) of one KV head is P/16 tiles.  Each tile:
#   [ K codes 512 B ][ V codes 512 B ][ K records 16 * rec B ][ V records 16 * rec B ]
# rec = 2 halves per group, (s, z) for each group of the tensor; Gs=128 -> 4 B
# per token and tensor, Gs=64 -> 8 B.  Records are stored by token pairs:
# slot 2r holds token r, slot 2r + 1 token r + 8 (r = 0..7).
#
# Code bits.  A code is addressed by (m, k, step): m in [0,16) and k in [0,16)
# index a 16 x 16 block, step in [0,8) selects one of the eight blocks that
# tile the 16 x 128 slab.  Its bit lies in the 16-byte group of "lane"
# L = 4*(m % 8) + (k % 8) // 2, in 32-bit little-endian word w = step // 2,
# at bit 16*(k % 2) + 2*pi with pi = 2*(step % 2) + (m // 8) + 4*(k // 8).
#   K tile: m = token, k = channel % 16, step = channel // 16
#   V tile: m = channel % 16, k = token, step = channel // 16

def tile_code_bit(m, k, step):
    """Return (byte offset within the 512-B code block, bit shift in byte)."""
    m = np.asarray(m); k = np.asarray(k); step = np.asarray(step)
    lane = 4 * (m % 8) + (k % 8) // 2
    word = step // 2
    pi = 2 * (step % 2) + (m // 8) + 4 * (k // 8)
    bit = 16 * (k % 2) + 2 * pi
    byte = 16 * lane + 4 * word + bit // 8
    return byte, bit % 8


def _tile_maps():
    t = np.arange(TILE)[:, None]
    c = np.arange(HEAD_DIM)[None, :]
    kb, ks = tile_code_bit(t, c % 16, c // 16)
    vb, vs = tile_code_bit(c % 16, t, c // 16)
    return (np.broadcast_to(kb, (TILE, HEAD_DIM)), np.broadcast_to(ks, (TILE, HEAD_DIM)),
            np.broadcast_to(vb, (TILE, HEAD_DIM)), np.broadcast_to(vs, (TILE, HEAD_DIM)))


_KB, _KS, _VB, _VS = _tile_maps()


def _inverse_map(bmap, smap):
    """For each (byte, 2-bit slot) of a code block, the (token, channel) stored there."""
    inv_t = np.empty((512, 4), np.int64)
    inv_c = np.empty((512, 4), np.int64)
    for t in range(TILE):
        for c in range(HEAD_DIM):
            inv_t[bmap[t, c], smap[t, c] // 2] = t
            inv_c[bmap[t, c], smap[t, c] // 2] = c
    return inv_t, inv_c


_KINV = _inverse_map(_KB, _KS)
_VINV = _inverse_map(_VB, _VS)
_SLOT_SHIFT = np.array([0, 2, 4, 6], np.uint16)


def tile_bytes(group_size):
    ng = HEAD_DIM // group_size
    return 1024 + TILE * 8 * ng


def pack_tile(kc, vc, sk, zk, sv, zv, group_size, base=None, valid=None):
    """Pack one 16-token tile.

    kc, vc: uint8 [16, 128] codes; sk, zk, sv, zv: fp16 [16, ng].
    base: existing tile bytes (tokens outside ``valid`` keep their bits).
    valid: bool [16] tokens to write (default all)."""
    ng = HEAD_DIM // group_size
    out = np.zeros(tile_bytes(group_size), np.uint8) if base is None else base.copy()
    if valid is None:
        valid = np.ones(TILE, bool)
    for t in range(TILE):
        if not valid[t]:
            continue
        for c in range(HEAD_DIM):
            for (blk, bmap, smap, code) in ((0, _KB, _KS, kc), (512, _VB, _VS, vc)):
                byte = blk + int(bmap[t, c]); sh = int(smap[t, c])
                out[byte] = (out[byte] & ~np.uint8(3 << sh)) | np.uint8((int(code[t, c]) & 3) << sh)
        slot = 2 * (t % 8) + t // 8
        for blk, s_, z_ in ((1024, sk, zk), (1024 + TILE * 4 * ng, sv, zv)):
            rec = np.empty(2 * ng, np.float16)
            rec[0::2] = s_[t]; rec[1::2] = z_[t]
            off = blk + slot * 4 * ng
            out[off:off + 4 * ng] = rec.view(np.uint8)
    return out


def pack_tiles_full(kc, vc, sk, zk, sv, zv, group_size):
    """Vectorised ``pack_tile`` for n complete tiles.

    kc, vc uint8 [n, 16, 128]; s/z fp16 [n, 16, ng] -> uint8 [n, tile_bytes].
    Each stored byte gathers its four codes through the inverse index map."""
    n = kc.shape[0]
    ng = HEAD_DIM // group_size
    out = np.zeros((n, tile_bytes(group_size)), np.uint8)
    for blk, codes, (it, ic) in ((0, kc, _KINV), (512, vc, _VINV)):
        g = codes[:, it, ic].astype(np.uint16) << _SLOT_SHIFT
        out[:, blk:blk + 512] = g.sum(axis=-1).astype(np.uint8)
    order = np.array([t for r in range(8) for t in (r, r + 8)])   # record slot -> token
    for blk, s_, z_ in ((1024, sk, zk), (1024 + TILE * 4 * ng, sv, zv)):
        rec = np.empty((n, TILE, 2 * ng), np.float16)
        rec[:, :, 0::2] = s_; rec[:, :, 1::2] = z_
        out[:, blk:blk + TILE * 4 * ng] = rec[:, order].reshape(n, -1).view(np.uint8)
    return out


def pack_history_full(k_bf16, v_bf16, Rk, Rv, clip_k, clip_v, page_table_row, num_pages,
                      num_heads, page_size, group_size, pages_buf=None):
    """Quantize and pack a whole history (positions 0..T-1) of one sequence,
    all heads, vectorised.  k/v_bf16 [T, Hkv, 128] bf16 bits.  Tokens past T in
    the last tile are zero codes with zero scale/zero."""
    T = k_bf16.shape[0]
    tb = tile_bytes(group_size)
    tpp = page_size // TILE
    if pages_buf is None:
        pages_buf = np.zeros((num_pages, num_heads, tpp * tb), np.uint8)
    ntiles = (T + TILE - 1) // TILE
    pad = ntiles * TILE - T
    ng = HEAD_DIM // group_size
    for g in range(num_heads):
        q = quantize_tokens(k_bf16[:, g], v_bf16[:, g], Rk[g], Rv[g], clip_k[g], clip_v[g],
                            group_size)
        def tiles(a, dtype):
            a = np.concatenate([a, np.zeros((pad,) + a.shape[1:], dtype)]) if pad else a
            return a.reshape((ntiles, TILE) + a.shape[1:])
        blocks = pack_tiles_full(tiles(q["kc"], np.uint8), tiles(q["vc"], np.uint8),
                                 tiles(q["sk"], np.float16), tiles(q["zk"], np.float16),
                                 tiles(q["sv"], np.float16), tiles(q["zv"], np.float16), group_size)
        ti = np.arange(ntiles)
        pages = np.asarray(page_table_row)[(ti * TILE) // page_size]
        within = (ti * TILE % page_size) // TILE
        for w in range(tpp):
            sel = within == w
            pages_buf[pages[sel], g, w * tb:(w + 1) * tb] = blocks[sel]
    return pages_buf


def unpack_tile(buf, group_size):
    """Inverse of ``pack_tile``: returns kc, vc [16,128] and sk, zk, sv, zv [16, ng]."""
    ng = HEAD_DIM // group_size
    buf = np.asarray(buf, dtype=np.uint8)
    kc = (buf[_KB] >> _KS) & 3
    vc = (buf[512 + _VB] >> _VS) & 3
    rk = np.empty((TILE, 2 * ng), np.float16)
    rv = np.empty((TILE, 2 * ng), np.float16)
    for t in range(TILE):
        slot = 2 * (t % 8) + t // 8
        rk[t] = buf[1024 + slot * 4 * ng:1024 + (slot + 1) * 4 * ng].view(np.float16)
        off = 1024 + TILE * 4 * ng + slot * 4 * ng
        rv[t] = buf[off:off + 4 * ng].view(np.float16)
    sk = rk[:, 0::2]; zk = rk[:, 1::2]
    sv = rv[:, 0::2]; zv = rv[:, 1::2]
    return kc.astype(np.uint8), vc.astype(np.uint8), sk, zk, sv, zv


def quantize_tokens(k_bf16, v_bf16, Rk, Rv, clip_k, clip_v, group_size, rot_dtype=np.float64):
    """Full append pipeline for one KV head, token rows of bf16 bits.

    Returns fp32 rotated K/V (the quantizer input), codes and fp16 s/z.
    Rotation is fp64 (``rot_dtype``) and rounded once to fp32."""
    xk = rotate(bf16_bits_to_f64(k_bf16), Rk).astype(np.float32)
    xv = rotate(bf16_bits_to_f64(v_bf16), Rv).astype(np.float32)
    kc, sk, zk = quantize_rows(xk, clip_k, group_size)
    vc, sv, zv = quantize_rows(xv, clip_v, group_size)
    return dict(xk=xk, xv=xv, kc=kc, sk=sk, zk=zk, vc=vc, sv=sv, zv=zv)


def pack_history(pages_buf, page_table_row, hist_start, q, head, num_heads, page_size,
                 group_size):
    """Write quantized tokens into a flat history buffer (one layer).

    pages_buf: uint8 [num_pages, num_heads, page_size/16 * tile_bytes].
    q: dict from ``quantize_tokens`` for T tokens at history positions
    hist_start .. hist_start+T-1.  Partial tiles keep the bits of other tokens."""
    T = q["kc"].shape[0]
    tb = tile_bytes(group_size)
    pos = hist_start + np.arange(T)
    tiles = {}
    for i, p in enumerate(pos):
        tiles.setdefault(p // TILE, []).append((p % TILE, i))
    ng = HEAD_DIM // group_size
    for tile_idx, items in tiles.items():
        page = int(page_table_row[(tile_idx * TILE) // page_size])
        within = (tile_idx * TILE % page_size) // TILE
        blk = pages_buf[page, head, within * tb:(within + 1) * tb]
        kc = np.zeros((TILE, HEAD_DIM), np.uint8); vc = np.zeros_like(kc)
        sk = np.zeros((TILE, ng), np.float16); zk = sk.copy(); sv = sk.copy(); zv = sk.copy()
        valid = np.zeros(TILE, bool)
        for (slot, i) in items:
            kc[slot] = q["kc"][i]; vc[slot] = q["vc"][i]
            sk[slot] = q["sk"][i]; zk[slot] = q["zk"][i]
            sv[slot] = q["sv"][i]; zv[slot] = q["zv"][i]
            valid[slot] = True
        pages_buf[page, head, within * tb:(within + 1) * tb] = pack_tile(
            kc, vc, sk, zk, sv, zv, group_size, base=blk, valid=valid)
    return pages_buf


def unpack_tiles(blocks, group_size):
    """Vectorised ``unpack_tile`` for blocks uint8 [n, tile_bytes]."""
    ng = HEAD_DIM // group_size
    blocks = np.asarray(blocks, dtype=np.uint8)
    kc = (blocks[:, _KB] >> _KS) & 3
    vc = (blocks[:, 512 + _VB] >> _VS) & 3
    order = np.array([2 * (t % 8) + t // 8 for t in range(TILE)])   # token -> record slot
    rk = np.ascontiguousarray(blocks[:, 1024:1024 + TILE * 4 * ng]).view(np.float16).reshape(-1, TILE, 2 * ng)[:, order]
    rv = np.ascontiguousarray(blocks[:, 1024 + TILE * 4 * ng:]).view(np.float16).reshape(-1, TILE, 2 * ng)[:, order]
    return (kc.astype(np.uint8), vc.astype(np.uint8), rk[:, :, 0::2], rk[:, :, 1::2], rv[:, :, 0::2], rv[:, :, 1::2])


def read_history(pages_buf, page_table_row, hist_len, head, page_size, group_size):
    """Decode history tokens 0..hist_len-1 of one head back to codes and s/z."""
    tb = tile_bytes(group_size)
    ng = HEAD_DIM // group_size
    ntiles = (hist_len + TILE - 1) // TILE
    if ntiles == 0:
        z = np.zeros((0, HEAD_DIM), np.uint8); zs = np.zeros((0, ng), np.float16)
        return z, z.copy(), zs, zs.copy(), zs.copy(), zs.copy()
    ti = np.arange(ntiles)
    pages = np.asarray(page_table_row)[(ti * TILE) // page_size]
    within = (ti * TILE % page_size) // TILE
    blocks = np.stack([pages_buf[p, head, w * tb:(w + 1) * tb] for p, w in zip(pages, within)])
    out = unpack_tiles(blocks, group_size)
    return tuple(a.reshape((ntiles * TILE,) + a.shape[2:])[:hist_len] for a in out)
