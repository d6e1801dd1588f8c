"""GPU parity of the batched GEMM with the fused epilogue against the oracle,
through the C ABI.

"Verde与RepOps" §3.2 (the k-chain), §4.3 (GeLU).  Bar: bit-exact for every tile
configuration, loader, storage layout and batch-stride pattern (stacked,
interleaved attention heads, shared operands), every epilogue part, in place
and at decoder sizes (sampled rows).
"""
import itertools

import numpy as np
import pytest
import torch

from verifiable_repops_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def u32(a):
    return np.ascontiguousarray(a).view(np.uint32)


def flat(n, seed, scale=1.0):
    return inputs.normal((n,), scale, seed, DEV)


def view(buf, batch, rows, cols, ld, stride, trans):
    """(batch, rows, cols) view of a flat buffer: row-major with pitch ld, or
    stored transposed (element (r, c) at c*ld + r)."""
    st = (stride, 1, ld) if trans else (stride, ld, 1)
    return torch.as_strided(buf, (batch, rows, cols), st)


def extent(batch, rows, cols, ld, stride, trans):
    r, c = (cols, rows) if trans else (rows, cols)
    return (batch - 1) * stride + (r - 1) * ld + c


def run_both(rp, orc, *, tA, tB, batch, M, N, K, lda, sA, ldb, sB, ldc, sC, alpha=1.0, bias=False,
             act=0, res="none", config=-1, loader=0, seed=0):
    """Runs the library and the oracle on the same flat buffers; returns both C
    buffers (numpy) for comparison, padding included."""
    A = flat(extent(batch, M, K, lda, sA, tA) + 3, seed + 1)
    B = flat(extent(batch, K, N, ldb, sB, tB) + 3, seed + 2)
    C = flat(extent(batch, M, N, ldc, sC, 0) + 3, seed + 3)
    bvec = flat(N, seed + 4) if bias else None
    R = flat(C.numel(), seed + 5) if res == "separate" else None
    Ah, Bh, Ch = A.cpu().numpy(), B.cpu().numpy(), C.cpu().numpy().copy()
    Cv = view(C, batch, M, N, ldc, sC, 0)
    Rv = Cv if res == "inplace" else (view(R, batch, M, N, ldc, sC, 0) if R is not None else None)
    rp.gemm_batched(view(A, batch, M, K, lda, sA, tA), view(B, batch, K, N, ldb, sB, tB), out=Cv,
                    alpha=alpha, bias=bvec, act=act, residual=Rv, config=config, loader=loader)
    Rh = Ch if res == "inplace" else (R.cpu().numpy() if R is not None else None)
    orc.gemm_batched(tA, tB, batch, M, N, K, Ah, lda, sA, Bh, ldb, sB, Ch, ldc, sC, alpha,
                     bvec.cpu().numpy() if bias else None, act, Rh, ldc, sC)
    return C.cpu().numpy(), Ch


LAYOUTS = list(itertools.product([0, 1], [0, 1]))


@pytest.mark.parametrize("config", range(5))
@pytest.mark.parametrize("loader", [0, 1, 2])
@pytest.mark.parametrize("tA,tB", LAYOUTS)
def test_every_config_loader_and_layout(rp, orc, config, loader, tA, tB):
    batch, M, N, K = 3, 70, 68, 45          # ragged against every tile, K tail of 13
    lda = (M if tA else K) + 3              # pitches that keep TMA eligible (multiples of 4)
    lda += (-lda) % 4
    ldb = (K if tB else N) + 4
    ldb += (-ldb) % 4
    ldc = N + 4
    rows_a = K if tA else M
    rows_b = N if tB else K
    sA = rows_a * lda + 8
    sB = rows_b * ldb + 4
    sC = M * ldc + 4
    got, want = run_both(rp, orc, tA=tA, tB=tB, batch=batch, M=M, N=N, K=K, lda=lda, sA=sA, ldb=ldb,
                         sB=sB, ldc=ldc, sC=sC, alpha=-0.75, bias=True, act=1, res="separate",
                         config=config, loader=loader, seed=10 * config + loader)
    assert np.array_equal(u32(got), u32(want))


@pytest.mark.parametrize("alpha,bias,act,res", [(1.0, False, 0, "none"), (2.0, True, 0, "none"),
                                                (1.0, False, 1, "none"), (0.5, True, 1, "inplace"),
                                                (1.0, False, 0, "inplace"), (-3.0, True, 0, "separate")])
def test_epilogue_parts(rp, orc, alpha, bias, act, res):
    got, want = run_both(rp, orc, tA=0, tB=0, batch=2, M=129, N=200, K=97, lda=100, sA=129 * 100,
                         ldb=200, sB=97 * 200, ldc=204, sC=129 * 204, alpha=alpha, bias=bias, act=act,
                         res=res, seed=40)
    assert np.array_equal(u32(got), u32(want))


def test_attention_heads_interleaved(rp, orc):
    # QKV [T, 3*H*d] row-major; head h of Q at column h*d: S_h = alpha Q_h K_h^T,
    # then O_h = S_h V_h written back as column block h of O [T, H*d]
    T, H, d = 200, 4, 64
    qkv = flat(T * 3 * H * d, 50)
    Q = qkv.view(T, 3, H, d)[:, 0].transpose(0, 1)         # (H, T, d), stride d, ld 3Hd
    Kt = qkv.view(T, 3, H, d)[:, 1].permute(1, 2, 0)       # (H, d, T): K_h^T as a transposed view
    V = qkv.view(T, 3, H, d)[:, 2].transpose(0, 1)         # (H, T, d)
    S = rp.gemm_batched(Q, Kt, alpha=0.125)                # (H, T, T) stacked
    O = torch.empty(T, H * d, device=DEV)
    rp.gemm_batched(S, V, out=O.view(T, H, d).transpose(0, 1))
    qh = qkv.cpu().numpy()
    Sh = np.empty(H * T * T, np.float32)
    orc.gemm_batched(0, 1, H, T, T, d, qh, 3 * H * d, d, qh[H * d:].copy(), 3 * H * d, d,
                     Sh, T, T * T, 0.125)
    assert np.array_equal(u32(S.cpu().numpy().reshape(-1)), u32(Sh))
    Oh = np.empty(T * H * d, np.float32)
    orc.gemm_batched(0, 0, H, T, d, T, Sh, T, T * T, qh[2 * H * d:].copy(), 3 * H * d, d,
                     Oh, H * d, d)
    assert np.array_equal(u32(O.cpu().numpy().reshape(-1)), u32(Oh))


def test_shared_weights_and_unaligned_strides(rp, orc):
    # B shared by all batches (stride 0); odd strides and pitches force the
    # 4-byte loader, same bits
    got, want = run_both(rp, orc, tA=0, tB=0, batch=5, M=33, N=47, K=61, lda=63, sA=33 * 63 + 1,
                         ldb=49, sB=0, ldc=47, sC=33 * 47 + 3, bias=True, act=1, seed=60)
    assert np.array_equal(u32(got), u32(want))
    got, want = run_both(rp, orc, tA=1, tB=1, batch=4, M=64, N=64, K=64, lda=64, sA=0,
                         ldb=64, sB=64 * 64, ldc=64, sC=64 * 64, res="inplace", seed=61)
    assert np.array_equal(u32(got), u32(want))


def test_empty_k_is_the_epilogue_of_zero(rp, orc):
    got, want = run_both(rp, orc, tA=0, tB=0, batch=2, M=9, N=12, K=0, lda=1, sA=0, ldb=12, sB=0,
                         ldc=12, sC=9 * 12, alpha=-1.0, bias=True, act=1, res="separate", seed=70)
    assert np.array_equal(u32(got), u32(want))


def test_fused_equals_unfused_sequence(rp):
    # the epilogue runs after the whole k-chain: the bits equal GEMM, then the
    # element-wise steps as separate library calls
    X = inputs.normal((300, 256), 1.0, 80, DEV)
    W = inputs.normal((256, 520), 0.05, 81, DEV)
    b = inputs.normal((520,), 0.1, 82, DEV)
    res = inputs.normal((300, 520), 1.0, 83, DEV)
    fused = rp.gemm_batched(X, W, bias=b, act=rp.ACT_GELU, residual=res)
    y = rp.gemm(X, W)
    y = y + b                                   # one float32 rounding per element
    y = rp.gelu(y)
    y = y + res
    assert torch.equal(fused, y)
    assert torch.equal(rp.gemm_batched(X, W), rp.gemm(X, W))


@pytest.mark.slow
def test_decoder_sized_fused_gemms_sampled(rp, orc):
    T, D = inputs.DECODER_TOKENS, inputs.DECODER_DIM
    X = inputs.normal((T, D), 1.0, 90, DEV)
    Wu = inputs.normal((D, 4 * D), 0.02, 91, DEV)
    bu = inputs.normal((4 * D,), 0.02, 92, DEV)
    Hid = rp.gemm_batched(X, Wu, bias=bu, act=rp.ACT_GELU)          # up-projection + GeLU
    Wd = inputs.normal((4 * D, D), 0.02, 93, DEV)
    Y = X.clone()
    rp.gemm_batched(Hid, Wd, out=Y, residual=Y)                     # down-projection + residual, in place
    rows = [0, 1, 2047, T - 1]
    Xh, Wuh, buh, Wdh = X[rows].cpu().numpy(), Wu.cpu().numpy(), bu.cpu().numpy(), Wd.cpu().numpy()
    Hh = np.empty(len(rows) * 4 * D, np.float32)
    orc.gemm_batched(0, 0, 1, len(rows), 4 * D, D, np.ascontiguousarray(Xh).reshape(-1), D, 0,
                     Wuh.reshape(-1), 4 * D, 0, Hh, 4 * D, 0, 1.0, buh, 1)
    assert np.array_equal(u32(Hid[rows].cpu().numpy().reshape(-1)), u32(Hh))
    Yh = np.ascontiguousarray(Xh).reshape(-1).copy()
    orc.gemm_batched(0, 0, 1, len(rows), D, 4 * D, Hh, 4 * D, 0, Wdh.reshape(-1), D, 0, Yh, D, 0,
                     1.0, None, 0, Yh, D, 0)
    assert np.array_equal(u32(Y[rows].cpu().numpy().reshape(-1)), u32(Yh))


@pytest.mark.parametrize("config", [-1, 0, 3])
@pytest.mark.parametrize("first", [0, 70])
def test_causal_tile_skip_keeps_the_lower_part_exact(rp, orc, config, first):
    # scores of 3 heads, 300 queries x 300 keys: every element on or below
    # j = first + i equals the oracle's; tiles wholly above are not written
    H, T, d = 3, 300, 64
    Q = inputs.normal((H, T, d), 1.0, 400 + first, DEV)
    K = inputs.normal((H, T, d), 1.0, 401 + first, DEV)
    S = torch.full((H, T, T), 12345.0, device=DEV)
    rp.gemm_batched(Q, K.transpose(1, 2), out=S, alpha=0.125, causal_first=first, config=config)
    Sh = np.empty(H * T * T, np.float32)
    orc.gemm_batched(0, 1, H, T, T, d, Q.cpu().numpy().reshape(-1), d, T * d, K.cpu().numpy().reshape(-1), d,
                     T * d, Sh, T, T * T, 0.125)
    lower = np.tril(np.ones((T, T), bool), k=first)
    got = S.cpu().numpy()
    want = Sh.reshape(H, T, T)
    for h in range(H):
        assert np.array_equal(u32(got[h][lower]), u32(want[h][lower]))
    assert (got == 12345.0).any()                     # some tiles were skipped
    P = rp.softmax_rows(S.view(H * T, T), causal_first=first, causal_period=T)
    Ph = orc.softmax_rows_causal(want.reshape(H * T, T), first, T)
    assert np.array_equal(u32(P.cpu().numpy()), u32(Ph))


@pytest.mark.parametrize("act", [0, 1])
def test_epilogue_special_values(rp, orc, act):
    # infinities and NaN in the operands, a product that overflows, a bias at
    # +inf, a residual at -inf: the epilogue (alpha, bias, GeLU, residual) gives
    # the same bits as the oracle wherever its value is not NaN
    batch, M, N, K = 2, 37, 40, 24
    g = np.random.default_rng(20000 + act)
    A = (g.standard_normal((batch, M, K)) * 2).astype(np.float32)
    B = (g.standard_normal((batch, K, N)) * 2).astype(np.float32)
    A[0, 3, 5] = np.inf
    A[1, 4, :] = 0.0
    A[1, 4, 2] = np.nan
    A[0, 9, 0] = 3.0e38
    B[0, 0, :] = 3.0e38
    bias = (g.standard_normal(N)).astype(np.float32)
    bias[7] = np.inf
    R = (g.standard_normal((batch, M, N))).astype(np.float32)
    R[1, 30, :] = -np.inf
    C = np.zeros((batch, M, N), dtype=np.float32)
    Ad, Bd, bd, Rd = (torch.from_numpy(x.copy()).to(DEV) for x in (A, B, bias, R))
    got = rp.gemm_batched(Ad, Bd, alpha=0.5, bias=bd, act=act, residual=Rd).cpu().numpy()
    orc.gemm_batched(0, 0, batch, M, N, K, A.reshape(-1), K, M * K, B.reshape(-1), N, K * N,
                     C.reshape(-1), N, M * N, 0.5, bias, act, R.reshape(-1), N, M * N)
    nan = np.isnan(C)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(u32(got[~nan]), u32(C[~nan]))


# ------------------------------------------------- attention-sized ----
# Batched, causal and banded products with many tiles (attention's shapes,
# shrunk): the automatic choice against explicit configurations and the
# oracle -- causal scores of grouped heads, both bands, an epilogue with bias
# and residual over 24 batches, and B shared by groups of batches.

def _oracle_batched(orc, A, B, alpha=1.0, k_lo=-1, k_hi=-1, b_group=1, bias=None, R=None):
    """Oracle of out[b] = A[b] @ B[b // b_group] on contiguous host copies."""
    A = np.ascontiguousarray(A.cpu().numpy(), dtype=np.float32)
    B = np.ascontiguousarray(B.cpu().numpy(), dtype=np.float32)
    batch, M, K = A.shape
    N = B.shape[2]
    C = np.zeros(batch * M * N, np.float32)
    Rh = np.ascontiguousarray(R.cpu().numpy(), dtype=np.float32).reshape(-1) if R is not None else None
    orc.gemm_batched(0, 0, batch, M, N, K, A.reshape(-1), K, M * K, B.reshape(-1), N, K * N, C, N, M * N, alpha,
                     bias.cpu().numpy() if bias is not None else None, 0, Rh, N, M * N, k_lo=k_lo, k_hi=k_hi,
                     b_group=b_group)
    return C.reshape(batch, M, N)


@pytest.mark.parametrize("case", ["scores", "band_hi", "band_lo", "epilogue", "grouped"])
def test_attention_sized_batched_products(rp, orc, case):
    g = 1000 + ["scores", "band_hi", "band_lo", "epilogue", "grouped"].index(case)
    if case == "scores":          # Q K^T of 12 heads over 3 key/value heads, causal tiles skipped
        Q = inputs.normal((12, 700, 64), 1.0, g, DEV)
        Kt = inputs.normal((3, 700, 64), 1.0, g + 1, DEV).transpose(1, 2)
        kw = dict(alpha=0.125, causal_first=0)
        got = rp.gemm_batched(Q, Kt, **kw)
        ref = rp.gemm_batched(Q, Kt, config=1, loader=rp.LOADER_TMA, **kw)
        # only tiles on or below the diagonal are specified: compare the lower triangle
        mask = torch.tril(torch.ones(700, 700, dtype=torch.bool, device=DEV)).expand(12, -1, -1)
        assert torch.equal(got[mask].view(torch.int32), ref[mask].view(torch.int32))
        Qh, Kh = Q.cpu().numpy(), Kt.cpu().numpy()
        for h in (0, 5, 11):
            want = orc.gemm(np.ascontiguousarray(Qh[h]), np.ascontiguousarray(Kh[h // 4])) * np.float32(0.125)
            tri = np.tril(np.ones((700, 700), bool))
            assert np.array_equal(u32(got[h].cpu().numpy()[tri]), u32(want.astype(np.float32)[tri])), h
        return
    if case in ("band_hi", "band_lo"):   # P V over k <= i, and P^T dO over k >= i
        S = 900
        P = torch.tril(inputs.uniform_pm1((10, S, S), g, DEV))
        V = inputs.normal((10, S, 64), 1.0, g + 1, DEV)
        if case == "band_hi":
            A, kw = P, dict(k_hi=0)
        else:
            A, kw = P.transpose(1, 2).contiguous(), dict(k_lo=0)
        got = rp.gemm_batched(A, V, **kw)
        for cfg in (3, 4):
            ref = rp.gemm_batched(A, V, config=cfg, loader=rp.LOADER_TMA, **kw)
            assert torch.equal(got.view(torch.int32), ref.view(torch.int32)), cfg
        want = _oracle_batched(orc, A, V, **kw)
        assert np.array_equal(u32(got.cpu().numpy()), u32(want))
        return
    if case == "epilogue":        # bias and a residual, 24 batches
        A = inputs.normal((24, 300, 200), 1.0, g, DEV)
        B = inputs.normal((24, 200, 260), 1.0, g + 1, DEV)
        bias = inputs.normal((260,), 1.0, g + 2, DEV)
        R = inputs.normal((24, 300, 260), 1.0, g + 3, DEV)
        got = rp.gemm_batched(A, B, alpha=0.5, bias=bias, residual=R)
        ref = rp.gemm_batched(A, B, alpha=0.5, bias=bias, residual=R, config=3, loader=rp.LOADER_TMA)
        assert torch.equal(got.view(torch.int32), ref.view(torch.int32))
        want = _oracle_batched(orc, A, B, alpha=0.5, bias=bias, R=R)
        assert np.array_equal(u32(got.cpu().numpy()), u32(want))
        return
    # grouped: 16 batches over 4 shared B matrices (a stride-0 expansion per group)
    A = inputs.normal((16, 400, 96), 1.0, g, DEV)
    B = inputs.normal((4, 96, 320), 1.0, g + 1, DEV)
    Bx = B.repeat_interleave(4, dim=0)        # the oracle's view: batch b reads B[b // 4]
    got = rp.gemm_batched(A, B)
    ref = rp.gemm_batched(A, B, config=1, loader=rp.LOADER_TMA)
    assert torch.equal(got.view(torch.int32), ref.view(torch.int32))
    want = _oracle_batched(orc, A, Bx)
    assert np.array_equal(u32(got.cpu().numpy()), u32(want))
