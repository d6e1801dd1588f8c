"""The decoder layer (forward, and forward with backward) composed from oracle
functions in the library's order of operations: test infrastructure for the
GPU parity tests of the layer and of the training step."""
import numpy as np


def oracle_layer(orc, x, w, cfg):
    f32 = np.float32
    S, dh, group = cfg.seq_len, cfg.d_head, cfg.heads // cfg.kv_heads
    h = orc.rmsnorm_rows(x, w["g1"], cfg.eps)
    qkv = orc.gemm(h, w["w_qkv"])
    attn = np.empty_like(x)
    scale = f32(1.0 / dh ** 0.5)                          # 1/8: exact scaling
    for s in range(x.shape[0] // S):
        rows = slice(s * S, (s + 1) * S)
        for q in range(cfg.heads):
            k = q // group
            Q = np.ascontiguousarray(qkv[rows, q * dh:(q + 1) * dh])
            K = np.ascontiguousarray(qkv[rows, cfg.d + k * dh:cfg.d + (k + 1) * dh])
            V = np.ascontiguousarray(qkv[rows, cfg.d + (cfg.kv_heads + k) * dh:cfg.d + (cfg.kv_heads + k + 1) * dh])
            scores = (orc.gemm(Q, np.ascontiguousarray(K.T)) * scale).astype(f32)
            P = orc.softmax_rows_causal(scores, 0)
            attn[rows, q * dh:(q + 1) * dh] = orc.gemm(P, V)
    x1 = (x + orc.gemm(attn, w["w_o"])).astype(f32)
    h2 = orc.rmsnorm_rows(x1, w["g2"], cfg.eps)
    u = orc.gelu((orc.gemm(h2, w["w_up"]) + w["b_up"]).astype(f32))
    return ((orc.gemm(u, w["w_down"]) + w["b_down"]).astype(f32) + x1).astype(f32)


def oracle_layer_with_grads(orc, x, w, cfg, dy):
    """The layer forward and its backward, composed from oracle functions in
    the library's order: (y, dx, grads)."""
    f32 = np.float32
    S, dh, group = cfg.seq_len, cfg.d_head, cfg.heads // cfg.kv_heads
    k0, v0 = cfg.d, cfg.d + cfg.kv_heads * dh
    scale = f32(1.0 / dh ** 0.5)
    T = x.shape[0]
    C = np.ascontiguousarray
    h1 = orc.rmsnorm_rows(x, w["g1"], cfg.eps)
    qkv = orc.gemm(h1, w["w_qkv"])
    attn = np.empty_like(x)
    probs = {}
    for s in range(T // S):
        rows = slice(s * S, (s + 1) * S)
        for q in range(cfg.heads):
            k = q // group
            Q = C(qkv[rows, q * dh:(q + 1) * dh])
            K = C(qkv[rows, k0 + k * dh:k0 + (k + 1) * dh])
            V = C(qkv[rows, v0 + k * dh:v0 + (k + 1) * dh])
            P = orc.softmax_rows_causal((orc.gemm(Q, C(K.T)) * scale).astype(f32), 0)
            probs[s, q] = P
            attn[rows, q * dh:(q + 1) * dh] = orc.gemm(P, V)
    x1 = (x + orc.gemm(attn, w["w_o"])).astype(f32)
    h2 = orc.rmsnorm_rows(x1, w["g2"], cfg.eps)
    a = (orc.gemm(h2, w["w_up"]) + w["b_up"]).astype(f32)
    u = orc.gelu(a)
    y = ((orc.gemm(u, w["w_down"]) + w["b_down"]).astype(f32) + x1).astype(f32)
    g = {}
    g["w_down"] = orc.gemm(C(u.T), dy)
    g["b_down"] = orc.colsum(dy)
    da = orc.gelu_backward(a, orc.gemm(dy, C(w["w_down"].T)))
    g["w_up"] = orc.gemm(C(h2.T), da)
    g["b_up"] = orc.colsum(da)
    dh2 = orc.gemm(da, C(w["w_up"].T))
    dx1, p2 = orc.rmsnorm_backward(x1, w["g2"], cfg.eps, dh2, dy)
    g["g2"] = orc.colsum(p2)
    g["w_o"] = orc.gemm(C(attn.T), dx1)
    dattn = orc.gemm(dx1, C(w["w_o"].T))
    dqkv = np.empty_like(qkv)
    for s in range(T // S):
        rows = slice(s * S, (s + 1) * S)
        for k in range(cfg.kv_heads):
            K = C(qkv[rows, k0 + k * dh:k0 + (k + 1) * dh])
            V = C(qkv[rows, v0 + k * dh:v0 + (k + 1) * dh])
            dV = dK = None
            for h in range(group):
                q = k * group + h
                P = probs[s, q]
                dO = C(dattn[rows, q * dh:(q + 1) * dh])
                Q = C(qkv[rows, q * dh:(q + 1) * dh])
                pv = orc.gemm(C(P.T), dO)
                dV = pv if dV is None else (pv + dV).astype(f32)
                dS = orc.softmax_backward(P, orc.gemm(dO, C(V.T)))
                dqkv[rows, q * dh:(q + 1) * dh] = (orc.gemm(dS, K) * scale).astype(f32)
                kq = (orc.gemm(C(dS.T), Q) * scale).astype(f32)
                dK = kq if dK is None else (kq + dK).astype(f32)
            dqkv[rows, k0 + k * dh:k0 + (k + 1) * dh] = dK
            dqkv[rows, v0 + k * dh:v0 + (k + 1) * dh] = dV
    g["w_qkv"] = orc.gemm(C(h1.T), dqkv)
    dh1 = orc.gemm(dqkv, C(w["w_qkv"].T))
    dx0, p1 = orc.rmsnorm_backward(x, w["g1"], cfg.eps, dh1, dx1)
    g["g1"] = orc.colsum(p1)
    return y, dx0, g
