"""Pins the decoder layer composed from oracle functions (tests/decoder_oracle.py),
the reference the GPU layer and training-step tests compare against: its
forward against a float64 NumPy statement of the layer's mathematics, and its
backward (every weight gradient and the input gradient) against central
differences of that float64 forward.

"Verde与RepOps" §4.3 (Llama-style training as the workload).  A wrong index, a
transposed operand, a missing rotation or a wrong derivative in the oracle's
composition moves a gradient by far more than the tolerance.
"""
import math

import numpy as np
import pytest

from verifiable_repops_gemm_gb300.decoder import DecoderConfig
from decoder_oracle import oracle_layer_with_grads

try:
    from scipy.special import erf as _erf
except ImportError:                                 # pragma: no cover
    _erf = np.vectorize(math.erf)

TINY = {
    "swiglu": DecoderConfig(d=32, heads=4, kv_heads=2, ffn=24, seq_len=8),
    "gelu": DecoderConfig(d=32, heads=4, kv_heads=2, ffn=24, seq_len=8, mlp="gelu", rope_base=0.0),
}


def weights(cfg, seed):
    from verifiable_repops_gemm_gb300.decoder import weight_shapes
    rng = np.random.default_rng(seed)
    w = {}
    for name, shape in weight_shapes(cfg).items():
        v = rng.standard_normal(shape)
        w[name] = (v * 0.1 + 1.0 if name in ("g1", "g2") else v * 0.3).astype(np.float32)
    return w


def ref_forward(x, w, cfg):
    """The layer in float64: RMSNorm, rotary on q and k, causal grouped-query
    attention, residual, RMSNorm, the MLP, residual."""
    S, dh, group = cfg.seq_len, cfg.d_head, cfg.heads // cfg.kv_heads

    def rms(v, g):
        return v / np.sqrt((v * v).mean(1, keepdims=True) + cfg.eps) * g

    h1 = rms(x, w["g1"])
    qkv = h1 @ w["w_qkv"]
    if cfg.rope_base:
        width = (cfg.heads + cfg.kv_heads) * dh
        pos = np.arange(x.shape[0]) % S
        freq = cfg.rope_base ** (-2.0 * np.arange(dh // 2) / dh)
        ang = pos[:, None] * freq[None, :]
        c, s = np.cos(ang), np.sin(ang)
        v = qkv[:, :width].reshape(x.shape[0], -1, dh // 2, 2)
        x0, x1 = v[..., 0], v[..., 1]
        rot = np.stack([x0 * c[:, None] - x1 * s[:, None], x0 * s[:, None] + x1 * c[:, None]], -1)
        qkv = np.concatenate([rot.reshape(x.shape[0], width), qkv[:, width:]], 1)
    attn = np.zeros_like(x)
    k0, v0 = cfg.d, cfg.d + cfg.kv_heads * dh
    mask = np.tril(np.ones((S, S), bool))
    for sq in range(x.shape[0] // S):
        rows = slice(sq * S, (sq + 1) * S)
        for q in range(cfg.heads):
            k = q // group
            Q = qkv[rows, q * dh:(q + 1) * dh]
            K = qkv[rows, k0 + k * dh:k0 + (k + 1) * dh]
            V = qkv[rows, v0 + k * dh:v0 + (k + 1) * dh]
            sc = np.where(mask, Q @ K.T / math.sqrt(dh), -np.inf)
            P = np.exp(sc - sc.max(1, keepdims=True))
            P /= P.sum(1, keepdims=True)
            attn[rows, q * dh:(q + 1) * dh] = P @ V
    x1 = x + attn @ w["w_o"]
    h2 = rms(x1, w["g2"])
    if cfg.mlp == "swiglu":
        gu = h2 @ w["w_gu"]
        gg, uu = gu[:, :cfg.ffn], gu[:, cfg.ffn:]
        a = gg / (1 + np.exp(-gg)) * uu
        return x1 + a @ w["w_down"]
    pre = h2 @ w["w_up"] + w["b_up"]
    a = 0.5 * pre * (1 + _erf(pre / math.sqrt(2)))
    return x1 + a @ w["w_down"] + w["b_down"]


@pytest.mark.parametrize("mlp", sorted(TINY))
def test_oracle_decoder_against_float64(orc, mlp):
    cfg = TINY[mlp]
    rng = np.random.default_rng(1)
    T = 2 * cfg.seq_len
    x = rng.standard_normal((T, cfg.d)).astype(np.float32)
    r = rng.standard_normal((T, cfg.d)).astype(np.float32)          # dL/dy of L = sum(y * r)
    w = weights(cfg, 2)
    y, dx, grads = oracle_layer_with_grads(orc, x, w, cfg, r)
    w64 = {k: v.astype(np.float64) for k, v in w.items()}
    y64 = ref_forward(x.astype(np.float64), w64, cfg)
    assert np.max(np.abs(y - y64)) < 2e-4 * max(1.0, np.max(np.abs(y64)))
    assert set(grads) == set(w)

    def loss(xv, wv):
        return float((ref_forward(xv, wv, cfg) * r).sum())

    h = 1e-5
    pick = np.random.default_rng(3)
    for name in sorted(w):
        for _ in range(6):
            idx = tuple(int(pick.integers(0, n)) for n in w[name].shape)
            wp = dict(w64)
            wp[name] = w64[name].copy()
            wp[name][idx] += h
            lp = loss(x.astype(np.float64), wp)
            wp[name][idx] -= 2 * h
            lm = loss(x.astype(np.float64), wp)
            fd = (lp - lm) / (2 * h)
            got = float(grads[name][idx])
            assert abs(got - fd) <= 2e-3 * max(1.0, abs(fd)), (name, idx, got, fd)
    x64 = x.astype(np.float64)
    for _ in range(10):
        idx = (int(pick.integers(0, T)), int(pick.integers(0, cfg.d)))
        xp = x64.copy()
        xp[idx] += h
        lp = loss(xp, w64)
        xp[idx] -= 2 * h
        fd = (lp - loss(xp, w64)) / (2 * h)
        assert abs(float(dx[idx]) - fd) <= 2e-3 * max(1.0, abs(fd)), (idx, float(dx[idx]), fd)
