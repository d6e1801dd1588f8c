"""GPU parity of the fused causal attention kernel (repops_attention_causal_f32).

The definition is the composition of the library's operators: scores as the
batched GEMM's k-chain times the scale, the causal softmax of every row's
prefix, and the banded product with V ("Verde与RepOps" §3.2: fixed order in
the order-critical reductions; §4.3: Llama-style training).  The oracle side
composes the same steps from oracle functions; the bar is bit-exact outputs
and probabilities, grouped heads, ragged sequence lengths and several
sequences per call.
"""
import numpy as np
import pytest
import torch

from verifiable_repops_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
F32 = np.float32
DH = 64


def C(a):
    return np.ascontiguousarray(a, dtype=F32)


def u32(a):
    return np.ascontiguousarray(a, dtype=F32).view(np.uint32)


def make_qkv(T, heads, kv, seed, pad=8):
    """A (T, width + pad) matrix holding [Q | K | V] column blocks, like the
    decoder's qkv projection output, and its three views."""
    width = (heads + 2 * kv) * DH
    X = inputs.normal((T, width + pad), 1.0, seed, DEV)
    q = X[:, :heads * DH]
    k = X[:, heads * DH:(heads + kv) * DH]
    v = X[:, (heads + kv) * DH:width]
    return X, q, k, v


def oracle_attention(orc, q, k, v, S, heads, kv, scale, head_list=None):
    """(out, probs) of the composition, per sequence and head, on host copies."""
    Q, K, V = (C(t.cpu().numpy()) for t in (q, k, v))
    T = Q.shape[0]
    group = heads // kv
    out = np.zeros((T, heads * DH), F32)
    probs = {}
    for b in range(T // S):
        rows = slice(b * S, (b + 1) * S)
        for h in (head_list if head_list is not None else range(heads)):
            g = h // group
            qh, kh, vh = C(Q[rows, h * DH:(h + 1) * DH]), C(K[rows, g * DH:(g + 1) * DH]), C(V[rows, g * DH:(g + 1) * DH])
            sc = np.zeros(S * S, F32)
            orc.gemm_batched(0, 1, 1, S, S, DH, qh.reshape(-1), DH, 0, kh.reshape(-1), DH, 0, sc, S, 0,
                             alpha=scale)
            P = C(orc.softmax_rows_causal(sc.reshape(S, S), 0))
            o = np.zeros(S * DH, F32)
            orc.gemm_batched(0, 0, 1, S, DH, S, P.reshape(-1), S, 0, vh.reshape(-1), DH, 0, o, DH, 0, k_hi=0)
            out[rows, h * DH:(h + 1) * DH] = o.reshape(S, DH)
            probs[b, h] = P
    return out, probs


@pytest.mark.parametrize("seqs,S,heads,kv,scale", [(1, 1, 2, 1, 0.125), (2, 16, 4, 2, 0.125),
                                                   (2, 17, 4, 4, 1.0), (1, 100, 6, 2, 0.125),
                                                   (3, 129, 6, 3, 0.1), (1, 300, 4, 1, 0.125),
                                                   (2, 260, 8, 2, 0.3)])
def test_fused_attention_matches_oracle(rp, orc, seqs, S, heads, kv, scale):
    T = seqs * S
    X, q, k, v = make_qkv(T, heads, kv, 500 + S)
    out = torch.full((T, heads * DH + 4), float("nan"), device=DEV)[:, :heads * DH]
    probs = torch.full((seqs * heads, S, S), float("nan"), device=DEV) if S % 4 == 0 else None
    rp.attention_causal(q, k, v, out, seq_len=S, heads=heads, kv_heads=kv, scale=scale, probs=probs)
    torch.cuda.synchronize()
    want, wprobs = oracle_attention(orc, q, k, v, S, heads, kv, F32(scale))
    assert np.array_equal(u32(out.cpu().numpy()), u32(want))
    if probs is not None:
        P = probs.cpu().numpy()
        for (b, h), Pw in wprobs.items():
            assert np.array_equal(u32(P[b * heads + h]), u32(Pw)), (b, h)


def test_fused_attention_equals_unfused_operators(rp):
    # the same bits as the three library operators it fuses (the decoder's
    # unfused path), outputs and every probability, at a ragged length
    from verifiable_repops_gemm_gb300 import decoder
    cfg = decoder.DecoderConfig(d=512, heads=8, kv_heads=2, ffn=1024, seq_len=300)
    T = 2 * cfg.seq_len
    X, q, k, v = make_qkv(T, cfg.heads, cfg.kv_heads, 77, pad=0)
    qkv = X
    out_u = torch.empty((T, cfg.d), device=DEV)
    probs_u = torch.empty((2 * cfg.kv_heads, cfg.heads // cfg.kv_heads, cfg.seq_len, cfg.seq_len), device=DEV)
    decoder.attention(qkv, cfg, out_u, probs_u, probs=probs_u, fused=False)
    out_f = torch.empty_like(out_u)
    probs_f = torch.empty_like(probs_u)
    decoder.attention(qkv, cfg, out_f, probs_f, probs=probs_f, fused=True)
    torch.cuda.synchronize()
    assert torch.equal(out_u.view(torch.int32), out_f.view(torch.int32))
    assert torch.equal(probs_u.view(torch.int32), probs_f.view(torch.int32))


def test_fused_attention_special_values(rp, orc):
    # a key/value row with infinities and NaN past some rows' prefixes: rows
    # before it are untouched (their terms past the prefix are skipped, not
    # multiplied by +0), rows after it follow the definition; huge query
    # values push exp to its overflow and underflow branches
    S, heads, kv = 64, 2, 1
    X, q, k, v = make_qkv(S, heads, kv, 91)
    v[40, 3] = float("inf")
    v[41, 5] = float("nan")
    k[50, :] = 0.0
    q[10, :] = 50.0                                   # scores of +-thousands: exp overflow / underflow
    q[20, 0] = -3.0e38
    out = torch.empty((S, heads * DH), device=DEV)
    probs = torch.empty((heads, S, S), device=DEV)
    rp.attention_causal(q, k, v, out, seq_len=S, heads=heads, kv_heads=kv, scale=0.125, probs=probs)
    torch.cuda.synchronize()
    want, wprobs = oracle_attention(orc, q, k, v, S, heads, kv, F32(0.125))
    got = out.cpu().numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(u32(got[~nan]), u32(want[~nan]))
    # rows that see neither the inf/NaN values nor row 20's overflowing query
    finite_rows = [i for i in range(40) if i != 20]
    assert np.isfinite(got[finite_rows]).all()
    P = probs.cpu().numpy()
    for (b, h), Pw in wprobs.items():
        pn = np.isnan(Pw)
        assert np.array_equal(np.isnan(P[h]), pn)
        assert np.array_equal(u32(P[h][~pn]), u32(Pw[~pn]))


def test_fused_attention_limits_and_errors(rp):
    S, heads, kv = 32, 2, 1
    X, q, k, v = make_qkv(S, heads, kv, 3)
    out = torch.empty((S, heads * DH), device=DEV)
    L = rp.load()
    s = torch.cuda.current_stream().cuda_stream
    # head dimension other than 64, sequences past 2048, unaligned rows
    assert L.repops_attention_causal_f32(1, S, heads * 2, kv * 2, 32, q.data_ptr(), q.stride(0), k.data_ptr(),
                                         k.stride(0), v.data_ptr(), v.stride(0), 0.125, out.data_ptr(),
                                         out.stride(0), None, s) == -7
    big = torch.empty((2049, 3 * DH), device=DEV)
    ob = torch.empty((2049, DH), device=DEV)
    assert L.repops_attention_causal_f32(1, 2049, 1, 1, DH, big.data_ptr(), big.stride(0),
                                         big[:, DH:].data_ptr(), big.stride(0), big[:, 2 * DH:].data_ptr(),
                                         big.stride(0), 0.125, ob.data_ptr(), ob.stride(0), None, s) == -7
    assert L.repops_attention_causal_f32(1, S, heads, kv, DH, q.data_ptr() + 4, q.stride(0), k.data_ptr(),
                                         k.stride(0), v.data_ptr(), v.stride(0), 0.125, out.data_ptr(),
                                         out.stride(0), None, s) == -7
    # heads not a multiple of kv heads; the output over the input
    assert L.repops_attention_causal_f32(1, S, 3, 2, DH, q.data_ptr(), q.stride(0), k.data_ptr(), k.stride(0),
                                         v.data_ptr(), v.stride(0), 0.125, out.data_ptr(), out.stride(0),
                                         None, s) == -1
    assert L.repops_attention_causal_f32(1, S, heads, kv, DH, q.data_ptr(), q.stride(0), k.data_ptr(),
                                         k.stride(0), v.data_ptr(), v.stride(0), 0.125, X.data_ptr(),
                                         X.stride(0), None, s) == -2
    # nothing to do
    assert L.repops_attention_causal_f32(0, S, heads, kv, DH, None, 0, None, 0, None, 0, 0.125, None, 0,
                                         None, s) == 0


@pytest.mark.slow
def test_fused_attention_llama_sized(rp, orc):
    # 2 sequences x 2048 tokens, 32 query heads over 8 key/value heads: the
    # decoder layer's attention.  Every output and probability equals the
    # unfused operators'; heads of both sequences, first and last of a group,
    # against the oracle composition
    from verifiable_repops_gemm_gb300 import decoder
    cfg = decoder.DecoderConfig()
    S, H, kv = cfg.seq_len, cfg.heads, cfg.kv_heads
    T = 2 * S
    X, q, k, v = make_qkv(T, H, kv, 123, pad=0)
    out_u = torch.empty((T, cfg.d), device=DEV)
    probs_u = torch.empty((2 * kv, H // kv, S, S), device=DEV)
    decoder.attention(X, cfg, out_u, probs_u, probs=probs_u, fused=False)
    out_f = torch.empty_like(out_u)
    probs_f = torch.empty_like(probs_u)
    decoder.attention(X, cfg, out_f, probs_f, probs=probs_f, fused=True)
    torch.cuda.synchronize()
    assert torch.equal(out_u.view(torch.int32), out_f.view(torch.int32))
    assert torch.equal(probs_u.view(torch.int32), probs_f.view(torch.int32))
    del probs_u
    heads = [0, 3, 4, 31]
    want, wprobs = oracle_attention(orc, q, k, v, S, H, kv, F32(1.0 / 8.0), head_list=heads)
    got = out_f.cpu().numpy()
    P = probs_f.view(2 * H, S, S)
    for b in range(2):
        rows = slice(b * S, (b + 1) * S)
        for h in heads:
            cols = slice(h * DH, (h + 1) * DH)
            assert np.array_equal(u32(got[rows, cols]), u32(want[rows, cols])), (b, h)
            assert np.array_equal(u32(P[b * H + h].cpu().numpy()), u32(wprobs[b, h])), (b, h)
