"""The decoder layer (forward, and forward with backward) composed from oracle
functions in the library's order of operations: test infrastructure for the
GPU parity tests of the layer and of the training step.

The attention products run over the full score matrices here; the library
runs them over the causal band only.  The skipped terms multiply probabilities
(or their gradients) that are +0 by finite values, so both give the same bits
(pinned on the oracle in test_oracle_llama.py)."""
import math

import numpy as np

F32 = np.float32
C = np.ascontiguousarray


def rope_tables(orc, cfg):
    if not cfg.rope_base:
        return None
    freq = orc.rope_frequencies(cfg.d_head // 2, float(F32(math.log(cfg.rope_base))))
    return orc.rope_table(cfg.seq_len, freq)


def rotate(orc, qkv, cfg, tables, inverse):
    """The rotary embedding (or its transpose) of the query and key heads."""
    if tables is None:
        return qkv
    width = (cfg.heads + cfg.kv_heads) * cfg.d_head
    out = qkv.copy()
    out[:, :width] = orc.rope(qkv[:, :width], cfg.heads + cfg.kv_heads, tables[0], tables[1], 0, cfg.seq_len,
                              inverse)
    return out


def _heads(qkv, cfg, rows, q):
    dh, group = cfg.d_head, cfg.heads // cfg.kv_heads
    k0, v0 = cfg.d, cfg.d + cfg.kv_heads * dh
    k = q // group
    return (C(qkv[rows, q * dh:(q + 1) * dh]), C(qkv[rows, k0 + k * dh:k0 + (k + 1) * dh]),
            C(qkv[rows, v0 + k * dh:v0 + (k + 1) * dh]))


def _forward(orc, x, w, cfg):
    """Forward keeping every activation the backward needs."""
    S, dh, f = cfg.seq_len, cfg.d_head, cfg.ffn
    scale = F32(1.0 / dh ** 0.5)                          # 1/8: exact scaling
    act = {"x0": x}
    act["h1"] = orc.rmsnorm_rows(x, w["g1"], cfg.eps)
    act["qkv"] = rotate(orc, orc.gemm(act["h1"], w["w_qkv"]), cfg, rope_tables(orc, cfg), False)
    attn = np.empty_like(x)
    probs = {}
    for s in range(x.shape[0] // S):
        rows = slice(s * S, (s + 1) * S)
        for q in range(cfg.heads):
            Q, K, V = _heads(act["qkv"], cfg, rows, q)
            P = orc.softmax_rows_causal((orc.gemm(Q, C(K.T)) * scale).astype(F32), 0)
            probs[s, q] = P
            attn[rows, q * dh:(q + 1) * dh] = orc.gemm(P, V)
    act["attn"], act["probs"] = attn, probs
    act["x1"] = (x + orc.gemm(attn, w["w_o"])).astype(F32)
    act["h2"] = orc.rmsnorm_rows(act["x1"], w["g2"], cfg.eps)
    if cfg.mlp == "swiglu":
        act["gu"] = orc.gemm(act["h2"], w["w_gu"])
        act["a"] = orc.swiglu(act["gu"][:, :f], act["gu"][:, f:])
        y = (orc.gemm(act["a"], w["w_down"]) + act["x1"]).astype(F32)
    else:
        act["pre"] = (orc.gemm(act["h2"], w["w_up"]) + w["b_up"]).astype(F32)
        act["a"] = orc.gelu(act["pre"])
        y = ((orc.gemm(act["a"], w["w_down"]) + w["b_down"]).astype(F32) + act["x1"]).astype(F32)
    return y, act


def oracle_layer(orc, x, w, cfg):
    return _forward(orc, x, w, cfg)[0]


def oracle_layer_with_grads(orc, x, w, cfg, dy):
    """The layer forward and its backward, composed from oracle functions in
    the library's order: (y, dx, grads)."""
    S, dh, group, f = cfg.seq_len, cfg.d_head, cfg.heads // cfg.kv_heads, cfg.ffn
    k0, v0 = cfg.d, cfg.d + cfg.kv_heads * dh
    scale = F32(1.0 / dh ** 0.5)
    T = x.shape[0]
    y, act = _forward(orc, x, w, cfg)
    g = {}
    g["w_down"] = orc.gemm(C(act["a"].T), dy)
    da = orc.gemm(dy, C(w["w_down"].T))
    if cfg.mlp == "swiglu":
        dg, du = orc.swiglu_backward(act["gu"][:, :f], act["gu"][:, f:], da)
        dgu = np.concatenate([dg, du], axis=1)
        g["w_gu"] = orc.gemm(C(act["h2"].T), dgu)
        dh2 = orc.gemm(dgu, C(w["w_gu"].T))
    else:
        g["b_down"] = orc.colsum(dy)
        dpre = orc.gelu_backward(act["pre"], da)
        g["w_up"] = orc.gemm(C(act["h2"].T), dpre)
        g["b_up"] = orc.colsum(dpre)
        dh2 = orc.gemm(dpre, C(w["w_up"].T))
    dx1, p2 = orc.rmsnorm_backward(act["x1"], w["g2"], cfg.eps, dh2, dy)
    g["g2"] = orc.colsum(p2)
    g["w_o"] = orc.gemm(C(act["attn"].T), dx1)
    dattn = orc.gemm(dx1, C(w["w_o"].T))
    qkv = act["qkv"]
    dqkv = np.empty_like(qkv)
    for s in range(T // S):
        rows = slice(s * S, (s + 1) * S)
        for k in range(cfg.kv_heads):
            dV = dK = None
            for h in range(group):
                q = k * group + h
                Q, K, V = _heads(qkv, cfg, rows, q)
                P = act["probs"][s, q]
                dO = C(dattn[rows, q * dh:(q + 1) * dh])
                pv = orc.gemm(C(P.T), dO)
                dV = pv if dV is None else (pv + dV).astype(F32)
                dS = orc.softmax_backward_causal(P, orc.gemm(dO, C(V.T)), 0)
                dqkv[rows, q * dh:(q + 1) * dh] = (orc.gemm(dS, K) * scale).astype(F32)
                kq = (orc.gemm(C(dS.T), Q) * scale).astype(F32)
                dK = kq if dK is None else (kq + dK).astype(F32)
            dqkv[rows, k0 + k * dh:k0 + (k + 1) * dh] = dK
            dqkv[rows, v0 + k * dh:v0 + (k + 1) * dh] = dV
    dqkv = rotate(orc, dqkv, cfg, rope_tables(orc, cfg), True)
    g["w_qkv"] = orc.gemm(C(act["h1"].T), dqkv)
    dh1 = orc.gemm(dqkv, C(w["w_qkv"].T))
    dx0, p1 = orc.rmsnorm_backward(x, w["g1"], cfg.eps, dh1, dx1)
    g["g1"] = orc.colsum(p1)
    return y, dx0, g
