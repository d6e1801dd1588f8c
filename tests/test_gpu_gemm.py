"""GPU parity of the order-fixed GEMM against the oracle, through the C ABI.

Bar: bit-exact (0 ULP, identical bytes) for every tile configuration, loader
path, operand layout and alignment ("Verde与RepOps" §3.1: operation order,
core count and strides must not change the result; §3.2: k in a fixed order).
"""
import numpy as np
import pytest
import torch

from verifiable_repops_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def bits(t):
    return t.contiguous().view(torch.int32).cpu()


def np_bits(a):
    return torch.from_numpy(np.ascontiguousarray(a)).view(torch.int32)


def all_configs(rp):
    return list(range(rp.gemm_config_count()))


def run(rp, A, B, config=-1, loader=0, out=None):
    C = rp.gemm(A, B, out=out, config=config, loader=loader)
    torch.cuda.synchronize()
    assert rp.device_status() == 0
    return C


def oracle_full(orc, A, B):
    return orc.gemm(A.cpu().numpy(), B.cpu().numpy())


def test_gemm_256_uniform_bit_exact(rp, orc):
    # 256^3, U[-1,1), seeds 0 (A) and 1 (B)
    A = inputs.uniform_pm1((256, 256), 0, DEV)
    B = inputs.uniform_pm1((256, 256), 1, DEV)
    want = np_bits(oracle_full(orc, A, B))
    for cfg in all_configs(rp):
        for loader in (rp.LOADER_TMA, rp.LOADER_CPASYNC):
            C = run(rp, A, B, cfg, loader)
            assert torch.equal(bits(C), want), (cfg, loader)
    assert torch.equal(bits(run(rp, A, B, -1, rp.LOADER_DIRECT)), want)
    # the automatic choice runs this size on the small-output kernel
    assert rp.gemm_small_output(256, 256, 256)
    assert torch.equal(bits(run(rp, A, B)), want)


LAYOUTS = [(False, False), (True, False), (False, True), (True, True)]


def make_operand(X, transposed):
    """Same logical matrix, stored row-major or as a transposed view."""
    return X.t().contiguous().t() if transposed else X.contiguous()


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (7, 5, 3), (129, 257, 33), (300, 200, 100),
                                   (64, 64, 32), (65, 129, 97), (256, 130, 1000), (17, 19, 20011)])
def test_gemm_ragged_all_configs_layouts_loaders(rp, orc, M, N, K):
    A = inputs.normal((M, K), 1.0, 10 + M, DEV)
    B = inputs.normal((K, N), 1.0, 20 + N, DEV)
    want = np_bits(oracle_full(orc, A, B))
    for ta, tb in LAYOUTS:
        Aop, Bop = make_operand(A, ta), make_operand(B, tb)
        for cfg in all_configs(rp):
            loaders = [rp.LOADER_CPASYNC]
            # TMA needs 16-byte aligned bases and leading dims that are multiples of 4
            lda = Aop.stride(1) if ta else Aop.stride(0)
            ldb = Bop.stride(1) if tb else Bop.stride(0)
            if lda % 4 == 0 and ldb % 4 == 0:
                loaders.append(rp.LOADER_TMA)
            for loader in loaders:
                C = run(rp, Aop, Bop, cfg, loader)
                assert torch.equal(bits(C), want), (ta, tb, cfg, loader)
        C = run(rp, Aop, Bop, -1, rp.LOADER_DIRECT)
        assert torch.equal(bits(C), want), (ta, tb, "direct")


def test_gemm_crafted_detectors_all_configs(rp, golden):
    od, fd = golden["gemm_order_detector"], golden["gemm_fma_detector"]
    M, N, K = 70, 68, 40      # ldb = 68 keeps the TMA loader eligible; both edges ragged
    A = inputs.integer_matrix((M, K), -3, 3, 5, DEV)
    B = torch.ones((K, N), device=DEV)
    a_od = torch.tensor(od["a_row"], dtype=torch.float32, device=DEV)
    a_fd = torch.tensor([int(x, 16) for x in fd["a_row_bits"]], dtype=torch.int64).to(torch.int32).view(torch.float32).to(DEV)
    b_fd = torch.tensor([int(x, 16) for x in fd["b_col_bits"]], dtype=torch.int64).to(torch.int32).view(torch.float32).to(DEV)
    # order detector in row 33, columns of B all ones over k = 10..13, zeros elsewhere
    A[33].zero_(); A[33, 10:14] = a_od
    # FMA detector in row 69 (a ragged tile edge) against column 67
    A[69].zero_(); A[69, 38:40] = a_fd
    B[:, 67].zero_(); B[38:40, 67] = b_fd
    cases = [(c, l) for c in all_configs(rp) for l in (rp.LOADER_TMA, rp.LOADER_CPASYNC)]
    for cfg, loader in cases + [(-1, rp.LOADER_DIRECT)]:
        C = run(rp, A, B, cfg, loader).cpu()
        assert int(C[33, 0].view(torch.int32)) == int(od["expected_bits"], 16)
        assert int(C[69, 67].view(torch.int32)) == int(fd["expected_bits"], 16), (cfg, loader)


def test_gemm_integer_exact_large(rp):
    # entries in [-8, 8], K = 4096: every partial sum < 2^24, so C is the exact
    # integer product
    M, N, K = 512, 384, 4096
    A = inputs.integer_matrix((M, K), -8, 8, 1, DEV)
    B = inputs.integer_matrix((K, N), -8, 8, 2, DEV)
    want = (A.cpu().to(torch.int64) @ B.cpu().to(torch.int64)).to(torch.float32)
    for cfg in all_configs(rp):
        assert torch.equal(run(rp, A, B, cfg).cpu(), want), cfg
    assert torch.equal(run(rp, A, B, -1, rp.LOADER_DIRECT).cpu(), want)


def test_gemm_unaligned_and_padded_operands(rp, orc):
    M, N, K = 131, 97, 75
    base_a = inputs.normal((M * 80 + 1,), 1.0, 3, DEV)
    base_b = inputs.normal((K * 101 + 3,), 1.0, 4, DEV)
    A = base_a[1:1 + M * 80].view(M, 80)[:, :K]          # 4-byte aligned only, lda = 80
    B = base_b[3:3 + K * 101].view(K, 101)[:, :N]        # ldb = 101
    want = np_bits(oracle_full(orc, A, B))
    Cbuf = torch.full((M, 104), float("nan"), device=DEV)
    C = Cbuf[:, 1:1 + N]                                  # ldc = 104, unaligned
    for cfg, loader in [(c, 0) for c in all_configs(rp)] + [(-1, rp.LOADER_DIRECT)]:
        C.fill_(float("nan"))
        run(rp, A, B, cfg, loader, out=C)
        assert torch.equal(bits(C), want), (cfg, loader)
    # padding columns untouched
    assert torch.isnan(Cbuf[:, 0]).all() and torch.isnan(Cbuf[:, 1 + N:]).all()
    with pytest.raises(rp.RepopsError):
        rp.gemm(A, B, config=0, loader=rp.LOADER_TMA)


def test_gemm_zero_k_and_empty(rp):
    A = torch.empty((5, 0), device=DEV)
    B = torch.empty((0, 7), device=DEV)
    C = torch.full((5, 7), float("nan"), device=DEV)
    run(rp, A, B, out=C)
    assert torch.equal(bits(C), torch.zeros((5, 7), dtype=torch.int32))
    E = torch.full((0, 7), 1.0, device=DEV)
    rp.gemm(torch.empty((0, 3), device=DEV), torch.empty((3, 7), device=DEV), out=E)


def test_gemm_output_guard_band(rp):
    # canaries around C stay untouched
    M, N, K = 67, 45, 33
    A = inputs.normal((M, K), 1.0, 8, DEV)
    B = inputs.normal((K, N), 1.0, 9, DEV)
    buf = torch.full((M * N + 2048,), 12345.0, device=DEV)
    C = buf[1024:1024 + M * N].view(M, N)
    for cfg, loader in [(c, 0) for c in all_configs(rp)] + [(-1, rp.LOADER_DIRECT)]:
        run(rp, A, B, cfg, loader, out=C)
        assert (buf[:1024] == 12345.0).all() and (buf[1024 + M * N:] == 12345.0).all()


def sampled_check(orc, A, B, C, rows, cols):
    """Oracle on the selected rows x cols only (any order over i, j)."""
    Ar = A[rows].cpu().numpy()
    Bc = B[:, cols].cpu().numpy()
    want = orc.gemm(Ar, Bc)
    got = C[rows][:, cols].cpu().numpy()
    assert np.array_equal(np_bits(got), np_bits(want))


@pytest.mark.slow
@pytest.mark.parametrize("n", inputs.SQUARE_SWEEP)
def test_gemm_square_sweep_sampled_and_layout_invariant(rp, orc, n):
    idx = inputs.SQUARE_SWEEP.index(n)
    A = inputs.normal((n, n), 1.0, 10 + idx, DEV)
    B = inputs.normal((n, n), 1.0, 20 + idx, DEV)
    C = run(rp, A, B)
    g = torch.Generator().manual_seed(n)
    rows = torch.cat([torch.tensor([0, n - 1]), torch.randint(0, n, (6,), generator=g)])
    cols = torch.cat([torch.tensor([0, n - 1]), torch.randint(0, n, (30,), generator=g)])
    sampled_check(orc, A, B, C, rows, cols)
    # B column-major (same logical B, transposed storage): identical bytes
    Bcm = B.t().contiguous().t()
    C2 = run(rp, A, Bcm)
    assert torch.equal(C.view(torch.int32), C2.view(torch.int32))
    # another tile configuration: identical bytes
    C3 = run(rp, A, B, config=3 if n <= 2048 else 1)
    assert torch.equal(C.view(torch.int32), C3.view(torch.int32))
    # Merkle root of the output matches the oracle's root of the same bytes
    root = rp.merkle_sha256(C).cpu().numpy().tobytes()
    assert root == orc.merkle_root(C.cpu().numpy(), 4096)


@pytest.mark.slow
def test_gemm_ragged_4097_1023_3001(rp, orc):
    M, N, K = inputs.RAGGED
    A = inputs.normal((M, K), 1.0, 30, DEV)
    B = inputs.normal((K, N), 1.0, 31, DEV)
    C = run(rp, A, B)
    rows = torch.tensor([0, 1, 2047, 4095, 4096])
    cols = torch.tensor(list(range(0, N, 61)) + [N - 2, N - 1])
    sampled_check(orc, A, B, C, rows, cols)
    C2 = run(rp, A.t().contiguous().t(), B.t().contiguous().t())
    assert torch.equal(C.view(torch.int32), C2.view(torch.int32))
    root = rp.merkle_sha256(C).cpu().numpy().tobytes()
    assert root == orc.merkle_root(C.cpu().numpy(), 4096)


@pytest.mark.slow
def test_gemm_decoder_layer_set(rp, orc):
    T, D = inputs.DECODER_TOKENS, inputs.DECODER_DIM
    X = inputs.normal((T, D), 1.0, 100, DEV)
    g = torch.Generator().manual_seed(7)
    for li, (name, kin, nout) in enumerate(inputs.DECODER_LAYERS):
        Xin = X if kin == D else inputs.normal((T, kin), 1.0, 150 + li, DEV)
        W = inputs.normal((kin, nout), 0.02, 110 + li, DEV)
        dY = inputs.normal((T, nout), 1e-3, 120 + li, DEV)
        Y = run(rp, Xin, W)                       # forward
        dX = run(rp, dY, W.t())                   # dX = dY W^T (B as a transposed view)
        dW = run(rp, Xin.t(), dY)                 # dW = X^T dY (A as a transposed view)
        for out, a, b in ((Y, Xin, W), (dX, dY, W.t()), (dW, Xin.t(), dY)):
            m, n = out.shape
            rows = torch.cat([torch.tensor([m - 1]), torch.randint(0, m, (3,), generator=g)])
            cols = torch.cat([torch.tensor([n - 1]), torch.randint(0, n, (16,), generator=g)])
            sampled_check(orc, a, b, out, rows, cols)
        # transposed views give the bytes of materialised transposes
        assert torch.equal(dX.view(torch.int32), run(rp, dY, W.t().contiguous()).view(torch.int32))
        assert torch.equal(dW.view(torch.int32), run(rp, Xin.t().contiguous(), dY).view(torch.int32))


def test_gemm_repacked_operands_match_every_loader(rp, orc):
    # 2*1601^3 = 8.2 GFLOP with lda = ldb = 1601: the automatic path copies both
    # operands to a 16-byte pitch and runs the TMA kernels
    n = 1601
    A = inputs.normal((n, n), 1.0, 41, DEV)
    B = inputs.normal((n, n), 1.0, 42, DEV)
    C_auto = run(rp, A, B)
    C_cp = run(rp, A, B, config=rp.gemm_auto_config(n, n, n), loader=rp.LOADER_CPASYNC)
    assert torch.equal(C_auto.view(torch.int32), C_cp.view(torch.int32))
    rows = torch.tensor([0, 777, n - 1])
    cols = torch.tensor([0, 5, 1000, n - 2, n - 1])
    sampled_check(orc, A, B, C_auto, rows, cols)
    # transposed storage of both operands (ld = 1601 again)
    C_t = run(rp, A.t().contiguous().t(), B.t().contiguous().t())
    assert torch.equal(C_auto.view(torch.int32), C_t.view(torch.int32))


@pytest.mark.parametrize("M,N,K,pinned", [(300, 260, 70, True), (1000, 129, 33, False), (4097, 1023, 3001, True),
                                          (64, 64, 0, True)])
def test_host_buffer_gemm_same_bits(rp, M, N, K, pinned):
    # row blocks of C are independent k-chains: the pipelined host-buffer call
    # gives the device GEMM's bits, for pinned and pageable host memory
    A = torch.randn(M, K + 1)[:, :K] if K else torch.randn(M, 0)
    B = torch.randn(K, N)
    if pinned:
        A, B = A.pin_memory(), B.pin_memory()
    s = torch.cuda.Stream()
    C = rp.gemm_host(A, B, stream=s)
    s.synchronize()
    want = rp.gemm(A.cuda(), B.cuda()).cpu()
    assert torch.equal(C.view(torch.int32), want.view(torch.int32))


def test_transposed_b_large_problem_same_bits(rp):
    # >= 4 GFLOP with B stored transposed: B is transposed into padded scratch
    # and the row-major kernels run; the bits equal row-major B's and the
    # forced 4-byte loader's (which reads the transposed storage directly)
    M, N, K = 1024, 1001, 2048
    A = inputs.normal((M, K), 1.0, 700, DEV)
    B = inputs.normal((K, N), 1.0, 701, DEV)
    Bcm = B.t().contiguous().t()
    C_rm = run(rp, A, B)
    C_cm = run(rp, A, Bcm)
    C_forced = run(rp, A, Bcm, config=1, loader=2)
    assert torch.equal(C_rm.view(torch.int32), C_cm.view(torch.int32))
    assert torch.equal(C_rm.view(torch.int32), C_forced.view(torch.int32))


def test_row_major_a_large_problem_same_bits(rp, orc):
    # >= 4 GFLOP with A row-major: A^T is copied into padded scratch and the
    # M-inner kernels run; the bits equal the K-inner kernels' (explicit TMA
    # loader, no copy) and the oracle's on sampled rows; M and K not multiples
    # of the tile or of 4
    M, N, K = 1029, 1024, 2051
    A = inputs.normal((M, K), 1.0, 710, DEV)
    B = inputs.normal((K, N), 1.0, 711, DEV)
    C_auto = run(rp, A, B)
    C_kin = run(rp, A, B, config=1, loader=2)
    assert torch.equal(C_auto.view(torch.int32), C_kin.view(torch.int32))
    rows = [0, 1, 517, M - 1]
    want = orc.gemm(A[rows].cpu().numpy(), B.cpu().numpy())
    assert np.array_equal(C_auto[rows].cpu().numpy().view(np.uint32), want.view(np.uint32))
    # both transposes: B column-major as well
    Bcm = B.t().contiguous().t()
    assert torch.equal(run(rp, A, Bcm).view(torch.int32), C_auto.view(torch.int32))


def test_gemm_direct_loader_typed_and_batched(rp, orc):
    # the typed call widens its operands and runs the plain GEMM: the small-output
    # kernel gives the same bytes as the tiled one; the batched call refuses it
    M, N, K = 45, 70, 129
    A = inputs.normal((M, K), 1.0, 41, DEV).half()
    B = inputs.normal((K, N), 1.0, 42, DEV).half()
    want = np_bits(orc.gemm(A.float().cpu().numpy(), B.float().cpu().numpy()))
    for loader in (rp.LOADER_AUTO, rp.LOADER_DIRECT):
        C = rp.gemm_typed(A, B, loader=loader)
        torch.cuda.synchronize()
        assert torch.equal(bits(C), want), loader
    with pytest.raises(rp.RepopsError):
        rp.gemm_batched(A.float().unsqueeze(0), B.float().unsqueeze(0), loader=rp.LOADER_DIRECT)


def test_gemm_special_values_every_kernel(rp, orc):
    # infinities, NaN, values whose products or sums overflow, subnormals and
    # signed zeros, on ragged edges: the same bits as the oracle (NaN where the
    # oracle has NaN; payloads are not pinned) on every tile configuration,
    # loader and the small-output kernel
    M, N, K = 70, 68, 44                 # leading dimensions TMA can describe
    g = np.random.default_rng(17000)
    A = (g.standard_normal((M, K)) * 2).astype(np.float32)
    B = (g.standard_normal((K, N)) * 2).astype(np.float32)
    A[3, 7] = np.inf
    A[5, :] = 0.0
    A[5, 43] = -np.inf
    B[43, 9] = 0.0                       # -inf * 0 = NaN in column 9 of row 5
    A[11, 2] = np.nan
    A[20, 0] = 3.0e38
    B[0, :] = 3.0e38                     # row 20 overflows to +inf
    A[30, 1] = -3.0e38
    B[1, 30] = 3.0e38                    # row 30, column 30: -inf
    A[40, :] = -0.0
    A[50, 3] = 1e-40                     # subnormal products
    B[3, 50] = 1e-3
    A[69, :] = -1e-45
    B[:, 67] = 1e-45                     # products round to -0 / +0
    want = orc.gemm(A, B)
    nan = np.isnan(want)
    Ad, Bd = torch.from_numpy(A).to(DEV), torch.from_numpy(B).to(DEV)
    cases = [(c, l) for c in all_configs(rp) for l in (rp.LOADER_TMA, rp.LOADER_CPASYNC)]
    for cfg, loader in cases + [(-1, rp.LOADER_DIRECT)]:
        got = run(rp, Ad, Bd, cfg, loader).cpu().numpy()
        assert np.array_equal(np.isnan(got), nan), (cfg, loader)
        assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32)), (cfg, loader)
