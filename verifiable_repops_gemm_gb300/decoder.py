"""One transformer decoder layer, forward, built only from the library's
order-fixed operators: the workload of a verifiable training step on a
Llama-style model ("Verde与RepOps" §4.3, the Llama-1B training measurement),
driven with synthetic weights.

Layer (pre-norm, causal, grouped-query attention):

    h    = RMSNorm(x; g1)
    qkv  = h W_qkv                                  one GEMM
    for every sequence s and key/value head k (its H/KV query heads batched):
        S = (Q K^T) / sqrt(d_head)                  batched GEMM, alpha epilogue,
                                                    tiles above the diagonal skipped
        P = causal softmax of the heads' rows       one row-operator call
        O = P V                                     batched GEMM, written as the
                                                    heads' column blocks
    x    = x + O W_o                                GEMM, residual epilogue (in place)
    h    = RMSNorm(x; g2)
    u    = GeLU(h W_up + b_up)                      GEMM, bias epilogue; GeLU kernel
    x    = x + u W_down + b_down                    GEMM, bias + residual epilogue

Every step is a library call (this module only slices tensors); the bits of
the result depend on nothing but the inputs.  GeLU runs as its own kernel by
default: inside the GEMM's epilogue it measured 2.5x its stand-alone cost (the
GEMM is bound by the FP32 pipe, and its epilogue runs on few warps), more than
the memory pass it saves; `gelu_epilogue=True` fuses it anyway.  `fused=False`
runs every epilogue as a separate step (GEMM, then element-wise adds in
PyTorch, then the library's GeLU): the same bits, more memory traffic; it
exists to measure what the fusion saves.
"""
from dataclasses import dataclass

import torch

from . import gemm, gemm_batched, gelu, rmsnorm_rows, softmax_rows, ACT_GELU


@dataclass(frozen=True)
class DecoderConfig:
    d: int = 2048            # model width
    heads: int = 32          # query heads
    kv_heads: int = 8        # key/value heads (grouped-query attention)
    ffn: int = 8192          # MLP width
    seq_len: int = 2048      # tokens per sequence
    eps: float = 1e-5

    @property
    def d_head(self) -> int:
        return self.d // self.heads

    @property
    def qkv_width(self) -> int:
        return self.d + 2 * self.kv_heads * self.d_head

    def flops(self, tokens: int) -> float:
        """Multiply-adds x 2 of the layer's GEMMs (attention computed over the
        full score matrix, masked entries included)."""
        d, f, w = self.d, self.ffn, self.qkv_width
        seqs = tokens // self.seq_len
        attn = 2 * 2.0 * seqs * self.heads * self.seq_len * self.seq_len * self.d_head
        return 2.0 * tokens * (d * w + d * d + 2 * d * f) + attn


def init_weights(cfg: DecoderConfig, seed: int, device) -> dict:
    """Synthetic weights: N(0, 0.02) matrices, N(0, 0.02) biases, norm gains
    N(1, 0.1); seeded, generated on `device`."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)

    def n(shape, std, mean=0.0):
        return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std + mean

    return {
        "g1": n((cfg.d,), 0.1, 1.0), "g2": n((cfg.d,), 0.1, 1.0),
        "w_qkv": n((cfg.d, cfg.qkv_width), 0.02),
        "w_o": n((cfg.d, cfg.d), 0.02),
        "w_up": n((cfg.d, cfg.ffn), 0.02), "b_up": n((cfg.ffn,), 0.02),
        "w_down": n((cfg.ffn, cfg.d), 0.02), "b_down": n((cfg.d,), 0.02),
    }


def attention(qkv, cfg: DecoderConfig, out, scores):
    """Causal grouped-query attention of every sequence into `out` (T x d)."""
    S, dh, group = cfg.seq_len, cfg.d_head, cfg.heads // cfg.kv_heads
    k0, v0 = cfg.d, cfg.d + cfg.kv_heads * dh
    scale = 1.0 / float(dh) ** 0.5
    for s in range(qkv.shape[0] // S):
        rows = slice(s * S, (s + 1) * S)
        for k in range(cfg.kv_heads):
            q_cols = slice(k * group * dh, (k + 1) * group * dh)
            Q = qkv[rows, q_cols].unflatten(1, (group, dh)).transpose(0, 1)     # (group, S, dh)
            Kt = qkv[rows, k0 + k * dh:k0 + (k + 1) * dh].t()                   # (dh, S), shared
            V = qkv[rows, v0 + k * dh:v0 + (k + 1) * dh]                        # (S, dh), shared
            # tiles wholly above the diagonal are skipped: the causal softmax
            # never reads them
            gemm_batched(Q, Kt, out=scores, alpha=scale, causal_first=0)
            P = scores.view(group * S, S)
            softmax_rows(P, out=P, causal_first=0, causal_period=S)
            O = out[rows, q_cols].unflatten(1, (group, dh)).transpose(0, 1)     # heads' column blocks
            gemm_batched(scores, V, out=O)


def forward(x, w: dict, cfg: DecoderConfig, *, fused: bool = True, gelu_epilogue: bool = False,
            work: dict = None):
    """Runs the layer on x (T x d, T a multiple of seq_len) in place and
    returns it.  `work`: reusable buffers from `workspace` (allocated when
    absent)."""
    T = x.shape[0]
    if T % cfg.seq_len:
        raise ValueError("tokens must be a whole number of sequences")
    ws = work if work is not None else workspace(cfg, T, x.device)
    h, qkv, attn, u = ws["h"], ws["qkv"], ws["attn"], ws["u"]
    rmsnorm_rows(x, w["g1"], cfg.eps, out=h)
    gemm(h, w["w_qkv"], out=qkv)
    attention(qkv, cfg, attn, ws["scores"])
    if fused:
        gemm_batched(attn, w["w_o"], out=x, residual=x)
    else:
        x += gemm(attn, w["w_o"], out=ws["tmp_d"])
    rmsnorm_rows(x, w["g2"], cfg.eps, out=h)
    if fused:
        if gelu_epilogue:
            gemm_batched(h, w["w_up"], out=u, bias=w["b_up"], act=ACT_GELU)
        else:
            gemm_batched(h, w["w_up"], out=u, bias=w["b_up"])
            gelu(u, out=u)
        gemm_batched(u, w["w_down"], out=x, bias=w["b_down"], residual=x)
    else:
        gemm(h, w["w_up"], out=u)
        u += w["b_up"]
        gelu(u, out=u)
        y = gemm(u, w["w_down"], out=ws["tmp_d"])
        y += w["b_down"]
        x += y
    return x


def workspace(cfg: DecoderConfig, tokens: int, device) -> dict:
    e = dict(dtype=torch.float32, device=device)
    group = cfg.heads // cfg.kv_heads
    return {"h": torch.empty(tokens, cfg.d, **e), "qkv": torch.empty(tokens, cfg.qkv_width, **e),
            "attn": torch.empty(tokens, cfg.d, **e), "u": torch.empty(tokens, cfg.ffn, **e),
            "scores": torch.empty(group, cfg.seq_len, cfg.seq_len, **e),
            "tmp_d": torch.empty(tokens, cfg.d, **e)}
