"""Oracle: where a newly generated token goes in the three-tier pool (CPU, numpy).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The yunpan.plus OSCAR write-up ("1. 三段式 Token 池", "2. 在线量化与反量化")
describes the pool and its online update:
- the sink tier holds the sequence's first 64 tokens in BF16;
- the recent tier holds the latest 256 tokens in BF16;
- the history tier holds everything in between as INT2;
- a new token is written to the recent tier first; when the recent tier is
  full, its oldest token goes through rotate -> clip -> quantize -> pack and
  moves down into the INT2 history.

Readings where the pages are silent:
- a token whose position is below the sink capacity is one of "the first 64
  tokens", so it is written to the sink (the sink fills before the recent tier);
- the recent tier is a ring of capacity W with a start index (its oldest slot);
  the evicted token leaves from the start slot, the new token takes that slot,
  and the start index advances;
- the evicted token is appended at history position hist_len of its sequence,
  in the page the caller's page table names for that position; if that page id
  is missing or out of range the sequence's step is not applied and reported.
"""

import numpy as np

from . import kvquant as kq


def append_step(state, k_new, v_new, page_table, Rk, Rv, clip_k, clip_v, page_size,
                group_size):
    """Place one new token per sequence (all KV heads), in place.

    state: dict of numpy arrays
        sink_k, sink_v  uint16 [B, Hkv, S_cap, 128]  bf16 bits
        rec_k, rec_v    uint16 [B, Hkv, W_cap, 128]  bf16 bits (ring)
        sink_len, hist_len, rec_len, rec_start  int [B]
        pages           uint8 [num_pages, Hkv, page_size/16 * tile_bytes]
    k_new, v_new: uint16 [B, Hkv, 128] bf16 bits.
    Returns the list of sequences whose step was refused (missing page)."""
    sink_k, sink_v = state["sink_k"], state["sink_v"]
    rec_k, rec_v = state["rec_k"], state["rec_v"]
    pages = state["pages"]
    B, Hkv, S_cap = sink_k.shape[:3]
    W_cap = rec_k.shape[2]
    num_pages = pages.shape[0]
    refused = []
    for b in range(B):
        if state["sink_len"][b] < S_cap:                       # one of the first S_cap tokens
            s = state["sink_len"][b]
            sink_k[b, :, s] = k_new[b]
            sink_v[b, :, s] = v_new[b]
            state["sink_len"][b] = s + 1
            continue
        if state["rec_len"][b] < W_cap:                        # the recent tier has room
            slot = (state["rec_start"][b] + state["rec_len"][b]) % W_cap
            rec_k[b, :, slot] = k_new[b]
            rec_v[b, :, slot] = v_new[b]
            state["rec_len"][b] += 1
            continue
        pos = int(state["hist_len"][b])                       # evict the oldest recent token
        pidx = pos // page_size
        if pidx >= page_table.shape[1] or not (0 <= int(page_table[b, pidx]) < num_pages):
            refused.append(b)
            continue
        start = int(state["rec_start"][b])
        for g in range(Hkv):
            q = kq.quantize_tokens(rec_k[b, g, start][None], rec_v[b, g, start][None], Rk[g], Rv[g],
                                   clip_k[g], clip_v[g], group_size)
            kq.pack_history(pages, page_table[b], pos, q, g, Hkv, page_size, group_size)
        rec_k[b, :, start] = k_new[b]
        rec_v[b, :, start] = v_new[b]
        state["rec_start"][b] = (start + 1) % W_cap
        state["hist_len"][b] = pos + 1
    return refused
