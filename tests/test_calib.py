"""Pins for the offline calibration (``bit_kv_cache_12_gb300.calib``), CPU.

gist.science OSCAR explainer, sections 2.1 and 2.2 A: C_Q = (1/N) sum q^T q,
C_S = (1/N) V^T S^T S V, eigenbases by decreasing eigenvalue, R = U H P_br,
per-channel clips from the rotated calibration activations."""

import numpy as np
import pytest

from bit_kv_cache_12_gb300 import calib


def test_hadamard_definition():
    for d in (1, 2, 8, 128):
        h = calib.hadamard(d)
        assert np.allclose(h @ h.T, np.eye(d), atol=1e-14)
        assert np.allclose(np.abs(h), 1.0 / np.sqrt(d))
    h4 = calib.hadamard(4) * 2
    assert np.array_equal(h4, [[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]])
    with pytest.raises(ValueError):
        calib.hadamard(12)


def test_bit_reversal_definition():
    p = calib.bit_reversal(8)
    x = np.arange(8.0)
    assert list(x @ p) == [0, 4, 2, 6, 1, 5, 3, 7]
    p128 = calib.bit_reversal(128)
    assert np.array_equal(p128 @ p128, np.eye(128))            # an involution
    assert np.array_equal(p128.sum(0), np.ones(128)) and np.array_equal(p128.sum(1), np.ones(128))


def test_query_covariance_closed_form():
    d = 8
    rows = [3.0 * np.eye(d)[0]] * 5 + [-2.0 * np.eye(d)[2]] * 3   # N = 8
    c = calib.query_covariance(np.array(rows))
    exp = np.zeros((d, d)); exp[0, 0] = 9 * 5 / 8; exp[2, 2] = 4 * 3 / 8
    assert np.allclose(c, exp, atol=1e-15)
    # leading axes are pooled: [N, G, d] counts N*G rows
    assert np.allclose(calib.query_covariance(np.array(rows).reshape(4, 2, d)), exp)


def test_causal_attention_worked_case():
    q = np.array([[1.0, 0.0], [0.0, 1.0]])
    k = np.array([[0.0, 0.0], [0.0, np.log(3.0)]])
    S = calib.causal_attention(q, k, scale=1.0)
    # row 0 sees only key 0; row 1 sees logits 0 and ln 3 -> weights 1/4, 3/4
    assert np.allclose(S, [[1.0, 0.0], [0.25, 0.75]], atol=1e-15)


def test_score_covariance_closed_forms():
    rng = np.random.default_rng(1)
    v = rng.standard_normal((6, 4))
    assert np.allclose(calib.score_covariance(np.eye(6), v), v.T @ v / 6)
    S = np.array([[1.0, 0.0], [0.25, 0.75]])
    v2 = rng.standard_normal((2, 3))
    o = np.stack([v2[0], 0.25 * v2[0] + 0.75 * v2[1]])
    assert np.allclose(calib.score_covariance(S, v2), (np.outer(o[0], o[0]) + np.outer(o[1], o[1])) / 2)


def test_eigenbasis_and_rotation():
    rng = np.random.default_rng(2)
    a = rng.standard_normal((300, 16)) * np.linspace(5, 0.1, 16)
    C = a.T @ a / 300
    u, w = calib.eigenbasis(C)
    assert np.all(np.diff(w) <= 0)
    assert np.allclose(u.T @ C @ u, np.diag(w), atol=1e-10 * w[0])
    R = calib.rotation(C)
    assert np.abs(R @ R.T - np.eye(16)).max() <= 1e-12
    assert np.allclose(R, u @ calib.hadamard(16) @ calib.bit_reversal(16))
    # the most important direction ends up spread evenly over every channel
    assert np.allclose(np.abs(u[:, 0] @ R), 1.0 / 4.0, atol=1e-12)


def test_clip_thresholds_are_scaled_channel_absmax():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((50, 8))
    R = calib.rotation(np.cov(x.T))
    c = calib.clip_thresholds(x, R, ratio=0.9)
    assert np.allclose(c, 0.9 * np.abs(x @ R).max(axis=0))


def test_calibrate_layer_shapes_and_definitions():
    rng = np.random.default_rng(4)
    N, Hq, Hkv, d = 40, 4, 2, 128
    q = rng.standard_normal((N, Hq, d)); k = rng.standard_normal((N, Hkv, d)); v = rng.standard_normal((N, Hkv, d))
    q[..., 3] *= 8.0                                   # a dominant query direction
    Rk, Rv, ck, cv = calib.calibrate_layer(q, k, v, scale=1 / np.sqrt(d))
    assert Rk.shape == (Hkv, d, d) and ck.shape == (Hkv, d) and Rk.dtype == np.float32
    for g in range(Hkv):
        for R in (Rk[g], Rv[g]):
            assert np.abs(R.astype(np.float64) @ R.T - np.eye(d)).max() <= 2e-6
        exp = calib.rotation(calib.query_covariance(q[:, 2 * g:2 * g + 2]))
        assert np.allclose(Rk[g], exp, atol=1e-6)
        outs = np.concatenate([calib.causal_attention(q[:, h], k[:, g], 1 / np.sqrt(d)) @ v[:, g]
                               for h in (2 * g, 2 * g + 1)])
        assert np.allclose(Rv[g], calib.rotation(outs.T @ outs / outs.shape[0]), atol=1e-6)
        assert np.allclose(ck[g], 0.95 * np.abs(k[:, g] @ Rk[g].astype(np.float64)).max(0), rtol=1e-5)
