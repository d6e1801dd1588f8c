"""One transformer decoder layer, forward and backward, built only from the
library's order-fixed operators: the workload of a verifiable training step on
a Llama-style model ("Verde与RepOps" §4.3, the Llama-1B training measurement),
driven with synthetic weights.

Layer (pre-norm, causal, grouped-query attention):

    h    = RMSNorm(x; g1)
    qkv  = h W_qkv                                  one GEMM
    q, k = rotary(q, k)                             in place, the heads' pairs
                                                    rotated to each token's position
    for every sequence (each GEMM call covers every query head; the
    `group` query heads of a key/value head share its K and V):
        S = (Q K^T) / sqrt(d_head)                  batched GEMM, alpha epilogue,
                                                    tiles above the diagonal skipped
        P = causal softmax of every head's rows     one row-operator call
        O = P V                                     batched GEMM over k <= i only,
                                                    written as the heads' column blocks
    x    = x + O W_o                                GEMM, residual epilogue (in place)
    h    = RMSNorm(x; g2)
    SwiGLU MLP (mlp="swiglu", Llama):
        [g | u] = h W_gu                            one GEMM, gate and up side by side
        a    = SiLU(g) * u                          element-wise kernel
        x    = x + a W_down                         GEMM, residual epilogue
    GeLU MLP (mlp="gelu"):
        a    = GeLU(h W_up + b_up)                  GEMM, bias epilogue; GeLU kernel
        x    = x + a W_down + b_down                GEMM, bias + residual epilogue

The causal attention GEMMs run over the band where the probabilities are not
+0 (P V over k <= i; the gradients P^T dO and dS^T Q over k >= i, dS K over
k <= i): the skipped terms would add fl(+0 * v) = +-0 to each chain, so the
bits equal those of the full chains while the work halves.

`backward` runs the layer's backward pass from saved activations: weight,
bias and gain gradients and the input gradient, every step again a library
call (transposed GEMMs, the backward row operators, column sums, the inverse
rotation); the key and value gradients of a key/value head accumulate its
query heads in head order through the GEMM's residual epilogue.

Every step is a library call (this module only slices tensors); the bits of
the result depend on nothing but the inputs.  In the GeLU layer, GeLU runs as
its own kernel by default: inside the GEMM's epilogue it measured 2.5x its
stand-alone cost (the GEMM is bound by the FP32 pipe, and its epilogue runs on
few warps), more than the memory pass it saves; `gelu_epilogue=True` fuses it
anyway.  `fused=False` runs every epilogue as a separate step (GEMM, then
element-wise adds in PyTorch): the same bits, more memory traffic; it exists
to measure what the fusion saves.
"""
import math
from dataclasses import dataclass

import torch

from . import (gemm, gemm_batched, gelu, rmsnorm_rows, softmax_rows, ACT_GELU, colsum, gelu_backward,
               rmsnorm_backward, softmax_backward, swiglu, swiglu_backward, rope_frequencies, rope_table, rope)


@dataclass(frozen=True)
class DecoderConfig:
    d: int = 2048              # model width
    heads: int = 32            # query heads
    kv_heads: int = 8          # key/value heads (grouped-query attention)
    ffn: int = 8192            # MLP width
    seq_len: int = 2048        # tokens per sequence
    eps: float = 1e-5
    mlp: str = "swiglu"        # "swiglu" (Llama: gate and up, no biases) or "gelu" (up + bias)
    rope_base: float = 500000.0  # rotary base; 0 turns the rotary embedding off

    @property
    def d_head(self) -> int:
        return self.d // self.heads

    @property
    def qkv_width(self) -> int:
        return self.d + 2 * self.kv_heads * self.d_head

    def flops(self, tokens: int) -> float:
        """Multiply-adds x 2 of the layer's GEMMs, attention counted over the
        causal band only (S (S + 1) / 2 scores per head): the work the layer
        needs, not the full score matrix."""
        d, f, w = self.d, self.ffn, self.qkv_width
        seqs = tokens // self.seq_len
        S = self.seq_len
        attn = 2 * 2.0 * seqs * self.heads * (S * (S + 1) / 2) * self.d_head
        mlp = 3 * d * f if self.mlp == "swiglu" else 2 * d * f
        return 2.0 * tokens * (d * w + d * d + mlp) + attn


def weight_shapes(cfg: DecoderConfig) -> dict:
    """Every weight of a layer and its shape, in a fixed order."""
    d, w, f = cfg.d, cfg.qkv_width, cfg.ffn
    if cfg.mlp == "swiglu":
        return {"g1": (d,), "w_qkv": (d, w), "w_o": (d, d), "g2": (d,), "w_gu": (d, 2 * f), "w_down": (f, d)}
    if cfg.mlp == "gelu":
        return {"g1": (d,), "w_qkv": (d, w), "w_o": (d, d), "g2": (d,), "w_up": (d, f), "b_up": (f,),
                "w_down": (f, d), "b_down": (d,)}
    raise ValueError("mlp must be 'swiglu' or 'gelu'")


def init_weights(cfg: DecoderConfig, seed: int, device) -> dict:
    """Synthetic weights: N(0, 0.02) matrices and biases, norm gains
    N(1, 0.1); seeded, generated on `device`."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = {}
    for name, shape in weight_shapes(cfg).items():
        t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        out[name] = t * 0.1 + 1.0 if name in ("g1", "g2") else t * 0.02
    return out


def rope_tables(cfg: DecoderConfig, device):
    """(cos, sin), seq_len x d_head/2, of the layer's rotary embedding, or
    None when it is off: frequencies base^(-2i/d_head) from the binary32
    value of ln(base), angles p * f_i for positions p < seq_len."""
    if not cfg.rope_base:
        return None
    freq = rope_frequencies(cfg.d_head // 2, math.log(cfg.rope_base), device)
    return rope_table(cfg.seq_len, freq)


def _rotate(qkv, cfg: DecoderConfig, tables, inverse: bool):
    """The rotary embedding (or its transpose) of the query and key heads:
    columns [0, (heads + kv_heads) * d_head) of every row, position = the row's
    index within its sequence."""
    if tables is not None:
        rope(qkv, cfg.heads + cfg.kv_heads, tables[0], tables[1], first=0, period=cfg.seq_len, inverse=inverse)


def _after(stream, *others):
    """Work queued on `stream` from now on waits for everything queued so far
    on `others`."""
    for o in others:
        e = torch.cuda.Event()
        e.record(o)
        stream.wait_event(e)


def side_streams(cfg: DecoderConfig, tokens: int, device):
    """The side streams one layer's attention runs its independent work on:
    three per sequence (the scores, softmax and products of a sequence, or in
    the backward its dP / dQ; the dV chain; the dK chain)."""
    return [torch.cuda.Stream(device) for _ in range(tokens // cfg.seq_len * 3)]


def _per_kv(t, rows, col0, kv, group, h, dh):
    """(kv, S, dh) view of query head h of every key/value group: the column
    block (k*group + h)*dh of rows, k = 0 .. kv-1 (a batch stride of
    group*dh)."""
    return t[rows, col0:col0 + kv * group * dh].unflatten(1, (kv, group, dh))[:, :, h, :].transpose(0, 1)


def _kv(t, rows, col0, kv, dh):
    """(kv, S, dh) view of the key or value heads: column block col0 + k*dh."""
    return t[rows, col0:col0 + kv * dh].unflatten(1, (kv, dh)).transpose(0, 1)


def _heads(t, rows, col0, n, dh):
    """(n, S, dh) view of n consecutive heads: column block col0 + h*dh."""
    return t[rows, col0:col0 + n * dh].unflatten(1, (n, dh)).transpose(0, 1)


def attention(qkv, cfg: DecoderConfig, out, scores, probs=None, streams=None, fused: bool = False):
    """Causal grouped-query attention of every sequence into `out` (T x d).
    scores: (sequences * kv_heads, group, S, S) scratch (or (kv_heads, group,
    S, S), shared by the sequences in turn); probs: optional buffer shaped
    like the first that keeps every head's softmax output for the backward
    pass.

    fused: one launch of the fused kernel (repops_attention_causal_f32:
    scores, causal softmax and the banded product per block of 16 query rows in
    shared memory) where its limits allow; it computes the same bits as the
    operators below and needs no S x S scratch (`scores` is not touched), but
    it is slower at decoder sizes, so the unfused operators are the default.
    Unfused: one GEMM call covers every query head of a sequence: a key/value
    head's K or V is shared by the `group` consecutive query heads of its
    group.  streams (from
    `side_streams`): the sequences run concurrently -- their outputs are
    disjoint, so the bits do not change -- and the caller's stream waits for
    all of them."""
    S, dh, kv, H = cfg.seq_len, cfg.d_head, cfg.kv_heads, cfg.heads
    k0, v0 = cfg.d, cfg.d + kv * dh
    scale = 1.0 / float(dh) ** 0.5
    seqs = qkv.shape[0] // S
    if fused:
        from . import attention_causal
        from ._capi import RepopsError, ERR_UNSUPPORTED
        try:
            attention_causal(qkv[:, :H * dh], qkv[:, k0:k0 + kv * dh], qkv[:, v0:v0 + kv * dh], out,
                             seq_len=S, heads=H, kv_heads=kv, scale=scale,
                             probs=probs.view(seqs * H, S, S) if probs is not None else None)
            return
        except RepopsError as e:
            if e.code != ERR_UNSUPPORTED:
                raise
    buf = probs if probs is not None else scores
    shared = buf.shape[0] < seqs * kv
    main = torch.cuda.current_stream()
    prev, joined = None, []
    if streams is not None:
        fork = torch.cuda.Event()
        fork.record(main)
    for s in range(seqs):
        rows = slice(s * S, (s + 1) * S)
        sc = (buf if shared else buf[s * kv:(s + 1) * kv]).view(H, S, S)       # head q = k*group + h
        st = main if streams is None else streams[3 * s]
        if streams is not None:
            st.wait_event(fork)
            if shared and prev is not None:    # a shared scratch is reused after the previous sequence
                _after(st, prev)
        with torch.cuda.stream(st):
            # tiles wholly above the diagonal are skipped: the causal softmax
            # never reads them
            gemm_batched(_heads(qkv, rows, 0, H, dh), _kv(qkv, rows, k0, kv, dh).transpose(1, 2), out=sc,
                         alpha=scale, causal_first=0)
            P = sc.view(H * S, S)
            softmax_rows(P, out=P, causal_first=0, causal_period=S)
            # P is +0 past the diagonal: row i's chain stops at k = i
            gemm_batched(sc, _kv(qkv, rows, v0, kv, dh), out=_heads(out, rows, 0, H, dh), k_hi=0)
        prev = st
        joined.append(st)
    if streams is not None:
        _after(main, *joined)


def forward(x, w: dict, cfg: DecoderConfig, *, fused: bool = True, gelu_epilogue: bool = False,
            work: dict = None, save: dict = None, fused_attention: bool = False):
    """Runs the layer on x (T x d, T a multiple of seq_len) in place and
    returns it.  `work`: reusable buffers from `workspace` (allocated when
    absent).  `save`: a dict (from `activations`) that receives what
    `backward` needs; a GeLU layer then keeps its GeLU input and runs GeLU as
    its own kernel."""
    T = x.shape[0]
    if T % cfg.seq_len:
        raise ValueError("tokens must be a whole number of sequences")
    ws = work if work is not None else workspace(cfg, T, x.device)
    f = cfg.ffn
    if save is not None:
        save["x0"].copy_(x)
        h, qkv, attn, a = save["h1"], save["qkv"], save["attn"], save["a"]
    else:
        h, qkv, attn, a = ws["h"], ws["qkv"], ws["attn"], ws["a"]
    rmsnorm_rows(x, w["g1"], cfg.eps, out=h)
    gemm(h, w["w_qkv"], out=qkv)
    _rotate(qkv, cfg, ws["rope"], inverse=False)
    attention(qkv, cfg, attn, ws["scores"], save["probs"] if save is not None else None, ws.get("streams"),
              fused=fused_attention)
    if fused:
        gemm_batched(attn, w["w_o"], out=x, residual=x)
    else:
        x += gemm(attn, w["w_o"], out=ws["tmp_d"])
    if save is not None:
        save["x1"].copy_(x)
        h = save["h2"]
    rmsnorm_rows(x, w["g2"], cfg.eps, out=h)
    if cfg.mlp == "swiglu":
        gu = save["gu"] if save is not None else ws["gu"]
        gemm(h, w["w_gu"], out=gu)
        swiglu(gu[:, :f], gu[:, f:], out=a)
        if fused:
            gemm_batched(a, w["w_down"], out=x, residual=x)
        else:
            x += gemm(a, w["w_down"], out=ws["tmp_d"])
        return x
    if save is not None:
        gemm_batched(h, w["w_up"], out=save["pre"], bias=w["b_up"])
        gelu(save["pre"], out=a)
        gemm_batched(a, w["w_down"], out=x, bias=w["b_down"], residual=x)
    elif fused:
        if gelu_epilogue:
            gemm_batched(h, w["w_up"], out=a, bias=w["b_up"], act=ACT_GELU)
        else:
            gemm_batched(h, w["w_up"], out=a, bias=w["b_up"])
            gelu(a, out=a)
        gemm_batched(a, w["w_down"], out=x, bias=w["b_down"], residual=x)
    else:
        gemm(h, w["w_up"], out=a)
        a += w["b_up"]
        gelu(a, out=a)
        y = gemm(a, w["w_down"], out=ws["tmp_d"])
        y += w["b_down"]
        x += y
    return x


def activations(cfg: DecoderConfig, tokens: int, device) -> dict:
    """Buffers for the activations `forward(save=...)` keeps for `backward`
    (every head's attention probabilities included: seqs * heads * S^2)."""
    e = dict(dtype=torch.float32, device=device)
    group, S = cfg.heads // cfg.kv_heads, cfg.seq_len
    out = {"x0": torch.empty(tokens, cfg.d, **e), "h1": torch.empty(tokens, cfg.d, **e),
           "qkv": torch.empty(tokens, cfg.qkv_width, **e), "attn": torch.empty(tokens, cfg.d, **e),
           "probs": torch.empty(tokens // S * cfg.kv_heads, group, S, S, **e),
           "x1": torch.empty(tokens, cfg.d, **e), "h2": torch.empty(tokens, cfg.d, **e),
           "a": torch.empty(tokens, cfg.ffn, **e)}
    if cfg.mlp == "swiglu":
        out["gu"] = torch.empty(tokens, 2 * cfg.ffn, **e)
    else:
        out["pre"] = torch.empty(tokens, cfg.ffn, **e)
    return out


def backward(dy, w: dict, cfg: DecoderConfig, saved: dict, *, work: dict = None, grads: dict = None):
    """Gradients of the layer given dy = dL/d(output): returns (dx, grads) with
    grads holding one tensor per weight of `init_weights` (written into the
    tensors of `grads` when given, e.g. views of one flat gradient buffer).
    dy is consumed (used as scratch) and dx is returned in its storage; a
    SwiGLU layer's saved["gu"] is overwritten with its gradient.  Every step
    is a library call:

        SwiGLU MLP:
          dW_down = a^T dy, da = dy W_down^T
          [dg | du] = SwiGLU'(g, u; da), dW_gu = h2^T [dg | du], dh2 = [dg | du] W_gu^T
        GeLU MLP:
          dW_down = a^T dy, db_down = colsum(dy), da = dy W_down^T
          dpre = GeLU'(pre) da, dW_up = h2^T dpre, db_up = colsum(dpre), dh2 = dpre W_up^T
        dx1 = RMSNorm'(x1; dh2) + dy, dg2 = colsum(dh2 * xhat2)
        dW_o = attn^T dx1, dattn = dx1 W_o^T
        attention, per sequence and key/value head k (its query heads h):
            dP_h = dO_h V_k^T (on and below the diagonal);
            dV_k = sum_h P_h^T dO_h (head order, k >= i)
            dS_h = causal softmax'(P_h; dP_h)
            dQ_h = s dS_h K_k (k <= i);  dK_k = sum_h s dS_h^T Q_h (head order,
            k >= i), s = 1/sqrt(d_head)
        dq, dk rotated back (the rotary embedding's transpose)
        dW_qkv = h1^T dqkv, dh1 = dqkv W_qkv^T
        dx0 = RMSNorm'(x0; dh1) + dx1, dg1 = colsum(dh1 * xhat1)
    """
    T, f = dy.shape[0], cfg.ffn
    ws = work if work is not None else backward_workspace(cfg, T, dy.device)
    g = {}
    o = grads if grads is not None else {}
    g["w_down"] = gemm(saved["a"].t(), dy, out=o.get("w_down"))
    da = gemm(dy, w["w_down"].t(), out=ws["t_ffn"])
    if cfg.mlp == "swiglu":
        gu = saved["gu"]
        swiglu_backward(gu[:, :f], gu[:, f:], da, dg=gu[:, :f], du=gu[:, f:])     # gu <- [dg | du]
        g["w_gu"] = gemm(saved["h2"].t(), gu, out=o.get("w_gu"))
        dh2 = gemm(gu, w["w_gu"].t(), out=ws["t_d"])
    else:
        g["b_down"] = colsum(dy, out=o.get("b_down"))
        dpre = gelu_backward(saved["pre"], da, out=da)
        g["w_up"] = gemm(saved["h2"].t(), dpre, out=o.get("w_up"))
        g["b_up"] = colsum(dpre, out=o.get("b_up"))
        dh2 = gemm(dpre, w["w_up"].t(), out=ws["t_d"])
    dx1, p2 = rmsnorm_backward(saved["x1"], w["g2"], cfg.eps, dh2, dx=dy, dyxh=ws["t_d2"], res=dy)
    g["g2"] = colsum(p2, out=o.get("g2"))
    g["w_o"] = gemm(saved["attn"].t(), dx1, out=o.get("w_o"))
    dattn = gemm(dx1, w["w_o"].t(), out=ws["t_d"])
    _attention_backward(dattn, ws["dqkv"], saved, cfg, ws["dp"], ws.get("streams"))
    dqkv = ws["dqkv"]
    _rotate(dqkv, cfg, ws["rope"], inverse=True)
    g["w_qkv"] = gemm(saved["h1"].t(), dqkv, out=o.get("w_qkv"))
    dh1 = gemm(dqkv, w["w_qkv"].t(), out=ws["t_d"])
    dx0, p1 = rmsnorm_backward(saved["x0"], w["g1"], cfg.eps, dh1, dx=dx1, dyxh=ws["t_d2"], res=dx1)
    g["g1"] = colsum(p1, out=o.get("g1"))
    return dx0, g


def _attention_backward(dattn, dqkv, saved, cfg: DecoderConfig, dp, streams):
    """The attention's part of dqkv (before the inverse rotation), per
    sequence, every query head q = k*group + h of key/value head k:
        dP_q = dO_q V_k^T (on and below the diagonal); dV_k = sum_h P_q^T dO_q
        dS_q = causal softmax'(P_q; dP_q)
        dQ_q = s dS_q K_k;  dK_k = sum_h s dS_q^T Q_q
    with dP and dQ one GEMM call per sequence, the dV and dK sums in head
    order through the residual epilogue.  dp: (sequences * kv_heads, group,
    S, S) scratch, or (kv_heads, group, S, S) shared by the sequences in turn.
    With `streams` the sequences run concurrently, and within one the dV
    chain and the dK chain beside dP / dQ; the bits do not change."""
    S, dh, kv, H = cfg.seq_len, cfg.d_head, cfg.kv_heads, cfg.heads
    group = H // kv
    scale = 1.0 / float(dh) ** 0.5
    k0, v0 = cfg.d, cfg.d + kv * dh
    qkv = saved["qkv"]
    seqs = qkv.shape[0] // S
    shared = dp.shape[0] < seqs * kv
    main = torch.cuda.current_stream()
    used, joined = [], []
    if streams is not None:
        fork = torch.cuda.Event()
        fork.record(main)
    for s in range(seqs):
        rows = slice(s * S, (s + 1) * S)
        P = saved["probs"][s * kv:(s + 1) * kv]                               # (kv, group, S, S)
        dP = dp if shared else dp[s * kv:(s + 1) * kv]
        V, K = _kv(qkv, rows, v0, kv, dh), _kv(qkv, rows, k0, kv, dh)
        dV, dK = _kv(dqkv, rows, v0, kv, dh), _kv(dqkv, rows, k0, kv, dh)
        if streams is None:
            sp = sv = sk = main
        else:
            sp, sv, sk = streams[3 * s:3 * s + 3]
            for st in (sp, sv):
                st.wait_event(fork)
            if shared:
                _after(sp, *used)
        with torch.cuda.stream(sp):
            # dP = dO V^T on and below the diagonal (the causal backward reads no more)
            gemm_batched(_heads(dattn, rows, 0, H, dh), V.transpose(1, 2), out=dP.view(H, S, S), causal_first=0)
        with torch.cuda.stream(sv):
            for h in range(group):
                # dV = sum over the group's heads, in head order, of P_h^T dO_h;
                # row i of P^T is +0 before k = i
                gemm_batched(P[:, h].transpose(1, 2), _per_kv(dattn, rows, 0, kv, group, h, dh), out=dV,
                             residual=dV if h else None, k_lo=0)
        with torch.cuda.stream(sp):
            dS = dP.view(H * S, S)
            softmax_backward(P.view(H * S, S), dS, out=dS, causal_first=0, causal_period=S)
            gemm_batched(dP.view(H, S, S), K, out=_heads(dqkv, rows, 0, H, dh), alpha=scale, k_hi=0)
        if streams is not None:
            _after(sk, sp)
        with torch.cuda.stream(sk):
            for h in range(group):
                # dK = sum over the group's heads, in head order, of s dS_h^T Q_h
                gemm_batched(dP[:, h].transpose(1, 2), _per_kv(qkv, rows, 0, kv, group, h, dh), out=dK,
                             alpha=scale, residual=dK if h else None, k_lo=0)
        if streams is not None:
            used = [sp, sv, sk]
            joined += used
    if streams is not None:
        _after(main, *joined)


def backward_workspace(cfg: DecoderConfig, tokens: int, device) -> dict:
    e = dict(dtype=torch.float32, device=device)
    group, S = cfg.heads // cfg.kv_heads, cfg.seq_len
    seqs = tokens // S
    return {"t_ffn": torch.empty(tokens, cfg.ffn, **e), "t_d": torch.empty(tokens, cfg.d, **e),
            "t_d2": torch.empty(tokens, cfg.d, **e), "dqkv": torch.empty(tokens, cfg.qkv_width, **e),
            "dp": torch.empty(seqs * cfg.kv_heads, group, S, S, **e), "rope": rope_tables(cfg, device),
            "streams": side_streams(cfg, tokens, device)}


def workspace(cfg: DecoderConfig, tokens: int, device) -> dict:
    e = dict(dtype=torch.float32, device=device)
    group = cfg.heads // cfg.kv_heads
    seqs = tokens // cfg.seq_len
    out = {"h": torch.empty(tokens, cfg.d, **e), "qkv": torch.empty(tokens, cfg.qkv_width, **e),
           "attn": torch.empty(tokens, cfg.d, **e), "a": torch.empty(tokens, cfg.ffn, **e),
           "scores": torch.empty(seqs * cfg.kv_heads, group, cfg.seq_len, cfg.seq_len, **e),
           "tmp_d": torch.empty(tokens, cfg.d, **e), "rope": rope_tables(cfg, device),
           "streams": side_streams(cfg, tokens, device)}
    if cfg.mlp == "swiglu":
        out["gu"] = torch.empty(tokens, 2 * cfg.ffn, **e)
    return out
