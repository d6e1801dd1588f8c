"""Seeded random parity cases for the remaining "next" entry points: the fused
causal attention ("Verde与RepOps" §4.3), the GEMM on half-precision storage
(§3.3, §5.3), Merkle inclusion proofs and membership checks (§2.4), and the
block replay ("Zoo Per-LLM Chain Soundness" §7 "Reproducibility test plan").

Attention: 1 to 3 sequences of 1 to 300 tokens, 1 to 8 query heads over 1 to
4 key/value groups, random scales and padded (16-byte) row pitches, outputs
and probabilities against the oracle composition.  Typed GEMM: every pair of
binary32 / binary16 / bfloat16 operands and output type, both storage orders.
Proofs: 1 to 5,000 leaves of 64 or 4096 bytes, a random leaf, the proof
against the oracle's, membership true and false after a flipped bit.
Replay: 1 to 4 blocks of 1 to 8 contributors.
"""
import numpy as np
import pytest
import torch

from verifiable_repops_gemm_gb300 import inputs

from test_gpu_attention import oracle_attention

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
DH = 64
F32, F16, BF16 = 0, 1, 2
TORCH = {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}


def u32(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


@pytest.mark.parametrize("case", range(24))
def test_random_fused_attention(rp, orc, case):
    rng = np.random.default_rng(19_000 + case)
    seqs = int(rng.integers(1, 4))
    S = int(np.exp(rng.uniform(0.0, np.log(300.0))))
    kv = int(rng.integers(1, 5))
    heads = kv * int(rng.integers(1, 3))
    scale = float(np.float32(rng.choice([0.125, 1.0, 0.3])))
    T = seqs * S
    width = (heads + 2 * kv) * DH
    pad = 4 * int(rng.integers(0, 4))
    X = inputs.normal((T, width + pad), 1.0, 19_100 + case, DEV)
    q, k, v = X[:, :heads * DH], X[:, heads * DH:(heads + kv) * DH], X[:, (heads + kv) * DH:width]
    opad = 2 * int(rng.integers(0, 3))
    obuf = torch.full((T, heads * DH + opad), float("nan"), device=DEV)
    out = obuf[:, :heads * DH]
    probs = torch.full((seqs * heads, S, S), float("nan"), device=DEV) if S % 4 == 0 else None
    rp.attention_causal(q, k, v, out, seq_len=S, heads=heads, kv_heads=kv, scale=scale, probs=probs)
    torch.cuda.synchronize()
    want, wprobs = oracle_attention(orc, q, k, v, S, heads, kv, np.float32(scale))
    what = dict(seqs=seqs, S=S, heads=heads, kv=kv, scale=scale, pad=pad, opad=opad)
    assert np.array_equal(u32(out.cpu().numpy()), u32(want)), what
    if opad:
        assert torch.isnan(obuf[:, heads * DH:]).all(), what
    if probs is not None:
        P = probs.cpu().numpy()
        for (b, h), Pw in wprobs.items():
            assert np.array_equal(u32(P[b * heads + h]), u32(Pw)), (what, b, h)


def storage(t):
    """The oracle's view: float32 values or the uint16 bits of a half tensor."""
    t = t.contiguous().cpu()
    return t.numpy() if t.dtype == torch.float32 else t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("case", range(60))
def test_random_typed_gemm(rp, orc, case):
    rng = np.random.default_rng(20_000 + case)
    M, N, K = (int(np.exp(rng.uniform(0.0, np.log(400.0)))) for _ in range(3))
    ta, tb, tc = (int(rng.integers(3)) for _ in range(3))
    A = inputs.normal((M, K), 1.0, 20_100 + case, DEV).to(TORCH[ta])
    B = inputs.normal((K, N), 1.0, 20_200 + case, DEV).to(TORCH[tb])
    want = orc.gemm_typed(storage(A), ta, storage(B), tb, tc)
    Aop = A.t().contiguous().t() if rng.integers(2) else A
    Bop = B.t().contiguous().t() if rng.integers(2) else B
    C = rp.gemm_typed(Aop, Bop, out_dtype=TORCH[tc])
    torch.cuda.synchronize()
    got = storage(C)
    what = dict(M=M, N=N, K=K, types=(ta, tb, tc))
    if tc == F32:
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(got), nan), what
        assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32)), what
    else:
        assert np.array_equal(got, want), what


@pytest.mark.parametrize("case", range(40))
def test_random_proofs_and_membership(rp, orc, case):
    rng = np.random.default_rng(21_000 + case)
    leaf = int(rng.choice([64, 4096]))
    nleaves = int(np.exp(rng.uniform(0.0, np.log(5000.0))))
    nbytes = (nleaves - 1) * leaf + int(rng.integers(1, leaf + 1))
    g = torch.Generator(device=DEV).manual_seed(21_100 + case)
    data = torch.randint(0, 256, (nbytes,), generator=g, dtype=torch.uint8, device=DEV)
    tree, root = rp.merkle_tree(data, leaf)
    index = int(rng.integers(0, nleaves))
    proof = rp.merkle_proof(tree, nleaves, index)
    torch.cuda.synchronize()
    th = tree.cpu().numpy()
    what = dict(leaf=leaf, nleaves=nleaves, index=index)
    assert np.array_equal(proof.cpu().numpy(), orc.merkle_proof(th, nleaves, index)), what
    lb = data[index * leaf:min((index + 1) * leaf, nbytes)]
    assert int(rp.merkle_verify(lb, nleaves, index, proof, root).item()) == 1, what
    assert orc.merkle_verify(lb.cpu().numpy(), nleaves, index, proof.cpu().numpy(), bytes(root.cpu().numpy()))
    bad = lb.clone()
    bad[int(rng.integers(0, bad.numel()))] ^= 1 << int(rng.integers(0, 8))
    assert int(rp.merkle_verify(bad, nleaves, index, proof, root).item()) == 0, what
    if proof.shape[0]:
        bp = proof.clone()
        bp[int(rng.integers(0, bp.shape[0])), int(rng.integers(0, 32))] ^= 1
        assert int(rp.merkle_verify(lb, nleaves, index, bp, root).item()) == 0, what


@pytest.mark.parametrize("case", range(20))
def test_random_replay(rp, orc, case):
    rng = np.random.default_rng(22_000 + case)
    steps = int(rng.integers(1, 5))
    nC = int(rng.integers(1, 9))
    n = int(np.exp(rng.uniform(0.0, np.log(100_000.0))))
    leaf = int(rng.choice([64, 4096]))
    grads = [[inputs.normal((n,), 1e-2, 22_100 + 97 * case + 11 * t + r, DEV) for r in range(nC)]
             for t in range(steps)]
    orders = [[int(x) for x in rng.permutation(nC)] for _ in range(steps)]
    etas = [float(np.float32(10.0 ** rng.uniform(-4, -1))) for _ in range(steps)]
    theta = inputs.normal((n,), 0.02, 22_000 + case, DEV)
    want_theta, want_roots = orc.replay([[g.cpu().numpy() for g in gs] for gs in grads], orders, etas,
                                        theta.cpu().numpy(), leaf)
    roots = rp.replay(grads, orders, etas, theta, leaf)
    torch.cuda.synchronize()
    what = dict(steps=steps, nC=nC, n=n, leaf=leaf)
    assert np.array_equal(u32(theta.cpu().numpy()), u32(want_theta)), what
    assert [bytes(r) for r in roots.cpu().numpy()] == want_roots, what
