"""GPU parity of one decoder layer forward (every step a library call) against
the same layer composed from oracle functions.

"Verde与RepOps" §4.3 (Llama-1B training as the workload).  Bar: bit-exact, for
the fused layer (epilogues inside the GEMMs) and the unfused one (epilogues as
separate steps), whose bits must also equal each other.
"""
import numpy as np
import pytest
import torch

from verifiable_repops_gemm_gb300 import decoder

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
SMALL = decoder.DecoderConfig(d=256, heads=4, kv_heads=2, ffn=512, seq_len=64)


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


@pytest.mark.parametrize("fused,ge", [(True, False), (True, True), (False, False)])
def test_decoder_layer_matches_oracle(rp, orc, fused, ge):
    w = decoder.init_weights(SMALL, 7, DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(8)
    x = torch.randn(2 * SMALL.seq_len, SMALL.d, generator=g, device=DEV)
    want = oracle_layer(orc, x.cpu().numpy(), {k: v.cpu().numpy() for k, v in w.items()}, SMALL)
    y = decoder.forward(x.clone(), w, SMALL, fused=fused, gelu_epilogue=ge)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), want.view(np.uint32))


def test_decoder_layer_is_deterministic_across_calls(rp):
    w = decoder.init_weights(SMALL, 9, DEV)
    x = torch.randn(3 * SMALL.seq_len, SMALL.d, device=DEV)
    a = decoder.forward(x.clone(), w, SMALL)
    b = decoder.forward(x.clone(), w, SMALL, fused=False)
    assert torch.equal(a, b)
