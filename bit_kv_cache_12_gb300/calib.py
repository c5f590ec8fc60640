"""Offline calibration: rotations and clip thresholds from calibration activations.

Host-side (numpy, fp64), run once per layer before serving; its outputs are
the R_k, R_v and clip arguments of ``kv_pool_set_rotation``.

The method (gist.science OSCAR explainer, sections 2.1 and 2.2 A):
- the key rotation follows the query covariance, because the error a key
  quantization causes in the attention logits is weighted by the queries:
      C_Q = (1/N) sum_n q_n^T q_n
- the value rotation follows the covariance of the attention outputs, because
  value errors reach the output through the attention weights S:
      C_S = (1/N) V^T S^T S V
- each covariance is eigendecomposed; its eigenbasis U (columns by decreasing
  eigenvalue) is followed by a normalised Hadamard transform H, which spreads
  every important direction's energy over all channels, and a bit-reversal
  permutation P_br, which interleaves high- and low-variance channels so that
  every contiguous quantization group sees a balanced dynamic range:
      R_K = U_Q H P_br,   R_V = U_S H P_br
- clip thresholds are estimated from the rotated calibration activations.

Readings where the explainer is silent:
- N counts query rows; for a KV head the queries of every query head that
  reads it (its GQA group) are pooled;
- S is the causal softmax attention of the calibration sequence, with the
  softmax scale used at inference;
- eigenvalue ties are broken by the order numpy's eigh returns;
- a clip threshold is per rotated channel: ratio x the largest absolute value
  of that channel over the calibration tokens (ratio 0.95 unless given).
"""

import numpy as np


def hadamard(d):
    """Normalised Sylvester Hadamard matrix, d a power of two: H H^T = I."""
    if d <= 0 or d & (d - 1):
        raise ValueError("d must be a power of two")
    h = np.array([[1.0]])
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h / np.sqrt(d)


def bit_reversal(d):
    """Permutation matrix P with (x P)_j = x_{bitrev(j)} (d a power of two)."""
    if d <= 0 or d & (d - 1):
        raise ValueError("d must be a power of two")
    nb = d.bit_length() - 1
    idx = np.array([int(format(i, f"0{nb}b")[::-1], 2) if nb else 0 for i in range(d)])
    p = np.zeros((d, d))
    p[idx, np.arange(d)] = 1.0
    return p


def query_covariance(q):
    """C_Q = (1/N) sum_n q_n^T q_n over query rows q [N, d] (any leading shape)."""
    q = np.asarray(q, np.float64).reshape(-1, np.shape(q)[-1])
    return q.T @ q / q.shape[0]


def causal_attention(q, k, scale):
    """Softmax attention weights S [N, N] of rows q [N, d] over keys k [N, d],
    query n seeing keys 0..n."""
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
    logits = scale * (q @ k.T)
    n = logits.shape[0]
    logits[np.triu(np.ones((n, n), bool), 1)] = -np.inf
    logits -= logits.max(axis=1, keepdims=True)
    w = np.exp(logits)
    return w / w.sum(axis=1, keepdims=True)


def score_covariance(S, v):
    """C_S = (1/N) V^T S^T S V for attention weights S [N, M] and values v [M, d]."""
    sv = np.asarray(S, np.float64) @ np.asarray(v, np.float64)
    return sv.T @ sv / sv.shape[0]


def eigenbasis(C):
    """Eigenvectors of the symmetric C as columns, by decreasing eigenvalue."""
    w, u = np.linalg.eigh(np.asarray(C, np.float64))
    order = np.argsort(w, kind="stable")[::-1]
    return u[:, order], w[order]


def rotation(C):
    """R = U H P_br for the covariance C."""
    d = C.shape[0]
    u, _ = eigenbasis(C)
    return u @ hadamard(d) @ bit_reversal(d)


def clip_thresholds(x, R, ratio=0.95):
    """ratio x per-channel max |x R| over the rows of x [N, d]."""
    y = np.asarray(x, np.float64) @ R
    return ratio * np.abs(y).max(axis=0)


def calibrate_layer(q, k, v, scale, clip_ratio_k=0.95, clip_ratio_v=0.95):
    """Rotations and clips of one layer from a calibration sequence.

    q [N, Hq, d], k and v [N, Hkv, d] (float); query head h reads KV head
    h // (Hq / Hkv).  Returns R_k, R_v [Hkv, d, d] and clip_k, clip_v
    [Hkv, d] as float32, ready for ``kv_pool_set_rotation``."""
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    N, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    Rk = np.zeros((Hkv, d, d)); Rv = np.zeros((Hkv, d, d))
    ck = np.zeros((Hkv, d)); cv = np.zeros((Hkv, d))
    for g in range(Hkv):
        qg = q[:, g * G:(g + 1) * G]                             # [N, G, d]
        Rk[g] = rotation(query_covariance(qg))
        outs = [causal_attention(qg[:, j], k[:, g], scale) @ v[:, g] for j in range(G)]
        sv = np.concatenate(outs)                                 # rows of S V for every query
        Rv[g] = rotation(sv.T @ sv / sv.shape[0])
        ck[g] = clip_thresholds(k[:, g], Rk[g], clip_ratio_k)
        cv[g] = clip_thresholds(v[:, g], Rv[g], clip_ratio_v)
    return (Rk.astype(np.float32), Rv.astype(np.float32), ck.astype(np.float32), cv.astype(np.float32))
