"""GPU parity of the order-fixed GEMM against the oracle, through the C ABI.

Bar: bit-exact (0 ULP, identical bytes) for every tile configuration, loader
path, operand layout and alignment ("Verde与RepOps" §3.1: operation order,
core count and strides must not change the result; §3.2: k in a fixed order).
"""
import numpy as np
import pytest
import torch

from verifiable_repops_gemm_gb300 import inputs

import oracle_par

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
    rows = [int(r) for r in rows]
    cols = [int(c) for c in cols]
    want = oracle_par.gemm(orc, A, B, rows=rows, cols=cols)
    got = C[rows][:, cols].cpu().numpy()
    assert np.array_equal(np_bits(got), np_bits(want))


def plant_detectors(A, B, golden, seed):
    """Plants the hand-derived order and FMA detectors into the logical
    operands A (M x K) and B (K x N), in place, whatever their storage.

    Each detector gets a row of A of its own (zero apart from the detector's
    entries) and a column of B of its own (its entries set over the
    detector's k positions, random elsewhere).  The zero products before and
    after the detector add ±0 to an accumulator that starts at +0, so the
    element's value is the detector's hand-derived one.  k positions: the
    chain's start, a 32-wide k-slice boundary crossed, the chain's end, and a
    random offset; rows include the last (a ragged tile edge) and columns the
    last.  Returns [(i, j, expected bits)]."""
    od, fd = golden["gemm_order_detector"], golden["gemm_fma_detector"]
    M, K = A.shape
    N = B.shape[1]
    dev = A.device
    g = np.random.default_rng(seed)
    n_det = 8
    rows = [M - 1, 0] + [int(x) for x in g.choice(np.arange(1, M - 1), n_det - 2, replace=False)]
    cols = [N - 1, 0] + [int(x) for x in g.choice(np.arange(1, N - 1), n_det - 2, replace=False)]
    a_od = torch.tensor(od["a_row"], dtype=torch.float32, device=dev)
    b_od = torch.tensor(od["b_col"], dtype=torch.float32, device=dev)

    def from_bits(lst):
        return torch.tensor([int(x, 16) for x in lst], dtype=torch.int64).to(torch.int32).view(torch.float32).to(dev)

    a_fd, b_fd = from_bits(fd["a_row_bits"]), from_bits(fd["b_col_bits"])
    k_order = [0, 30, K - 4, int(g.integers(0, K - 4))]
    k_fma = [31, K - 2, 0, int(g.integers(0, K - 2))]
    planted = []
    for d in range(n_det):
        i, j = rows[d], cols[d]
        A[i].zero_()
        if d % 2 == 0:
            k0 = k_order[d // 2]
            A[i, k0:k0 + 4] = a_od
            B[k0:k0 + 4, j] = b_od
            planted.append((i, j, int(od["expected_bits"], 16)))
        else:
            k0 = k_fma[d // 2]
            A[i, k0:k0 + 2] = a_fd
            B[k0:k0 + 2, j] = b_fd
            planted.append((i, j, int(fd["expected_bits"], 16)))
    return planted


def check_planted(C, planted, what):
    Cb = C.view(torch.int32) if isinstance(C, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(C)).view(torch.int32)
    for i, j, bits_ in planted:
        assert int(Cb[i, j]) & 0xFFFFFFFF == bits_, (what, i, j)


def assert_same_bits(got, want_bits, what):
    """got: device tensor; want_bits: int32 CPU tensor of the oracle's bytes."""
    g = got.contiguous().view(torch.int32).cpu()
    if not torch.equal(g, want_bits):
        bad = (g != want_bits).nonzero()
        raise AssertionError("%s: %d elements differ from the oracle, first at %s"
                             % (what, bad.shape[0], tuple(bad[0].tolist())))


def full_parity(rp, orc, A, B, want_bits, configs, what, loaders=None):
    """Every configuration (and loader) gives the oracle's bytes on the whole
    output."""
    for cfg in configs:
        for loader in (loaders or [rp.LOADER_TMA]):
            assert_same_bits(run(rp, A, B, cfg, loader), want_bits, (what, cfg, loader))


@pytest.mark.slow
@pytest.mark.parametrize("n", inputs.SQUARE_SWEEP)
def test_gemm_square_sweep_full_output(rp, orc, golden, n):
    # N(0,1) operands with the order and FMA detectors planted; the whole
    # output against the oracle for the automatic choice with B row-major and
    # column-major, A transposed, and every tile configuration with both
    # loaders (each configuration has its own CTA shape and thread count)
    idx = inputs.SQUARE_SWEEP.index(n)
    A = inputs.normal((n, n), 1.0, 10 + idx, DEV)
    B = inputs.normal((n, n), 1.0, 20 + idx, DEV)
    planted = plant_detectors(A, B, golden, 900 + idx)
    want = oracle_par.gemm(orc, A, B)
    check_planted(want, planted, "oracle")
    want_bits = np_bits(want)
    C = run(rp, A, B)
    assert_same_bits(C, want_bits, "auto")
    check_planted(C.cpu(), planted, "auto")
    Bcm = B.t().contiguous().t()
    assert_same_bits(run(rp, A, Bcm), want_bits, "B column-major")
    Atr = A.t().contiguous().t()
    assert_same_bits(run(rp, Atr, B), want_bits, "A transposed")
    del Atr
    full_parity(rp, orc, A, B, want_bits, all_configs(rp), n)
    full_parity(rp, orc, A, Bcm, want_bits, all_configs(rp), (n, "B column-major"))
    for cfg in (0, 2, 3):
        assert_same_bits(run(rp, A, B, cfg, rp.LOADER_CPASYNC), want_bits, (n, cfg, "cp.async"))
    # Merkle root of the output equals the oracle's root of the oracle's bytes
    root = rp.merkle_sha256(C).cpu().numpy().tobytes()
    assert root == orc.merkle_root(want, 4096)


@pytest.mark.slow
def test_gemm_ragged_4097_1023_3001_full_output(rp, orc, golden):
    M, N, K = inputs.RAGGED
    A = inputs.normal((M, K), 1.0, 30, DEV)
    B = inputs.normal((K, N), 1.0, 31, DEV)
    planted = plant_detectors(A, B, golden, 930)
    want = oracle_par.gemm(orc, A, B)
    check_planted(want, planted, "oracle")
    want_bits = np_bits(want)
    C = run(rp, A, B)                       # operands repacked to 16-byte pitches, TMA
    assert_same_bits(C, want_bits, "auto")
    # lda = 3001, ldb = 1023: only the 4-byte loader reads the caller's storage
    full_parity(rp, orc, A, B, want_bits, all_configs(rp), "ragged", [rp.LOADER_CPASYNC])
    At, Bt = A.t().contiguous().t(), B.t().contiguous().t()
    assert_same_bits(run(rp, At, Bt), want_bits, "both transposed")
    assert_same_bits(run(rp, At, B, 1, rp.LOADER_CPASYNC), want_bits, "A transposed, cp.async")
    root = rp.merkle_sha256(C).cpu().numpy().tobytes()
    assert root == orc.merkle_root(want, 4096)


def decoder_gemms():
    return [(li, name, kind) for li, (name, _, _) in enumerate(inputs.DECODER_LAYERS)
            for kind in ("forward", "dX", "dW")]


@pytest.mark.slow
@pytest.mark.parametrize("li,name,kind", decoder_gemms())
def test_gemm_decoder_layer_set_full_output(rp, orc, golden, li, name, kind):
    # the 15 GEMMs of the 1B-class layer set, each on its whole output with
    # the detectors planted: forward Y = X W, dX = dY W^T (B a transposed
    # view), dW = X^T dY (A a transposed view)
    T, D = inputs.DECODER_TOKENS, inputs.DECODER_DIM
    _, kin, nout = inputs.DECODER_LAYERS[li]
    X = inputs.normal((T, D), 1.0, 100, DEV) if kin == D else inputs.normal((T, kin), 1.0, 150 + li, DEV)
    W = inputs.normal((kin, nout), 0.02, 110 + li, DEV)
    dY = inputs.normal((T, nout), 1e-3, 120 + li, DEV)
    a, b = {"forward": (X, W), "dX": (dY, W.t()), "dW": (X.t(), dY)}[kind]
    planted = plant_detectors(a, b, golden, 940 + 3 * li + ("forward", "dX", "dW").index(kind))
    want = oracle_par.gemm(orc, a, b)
    check_planted(want, planted, "oracle")
    want_bits = np_bits(want)
    C = run(rp, a, b)
    assert_same_bits(C, want_bits, (name, kind))
    # a materialised copy of a transposed operand gives the same bytes
    assert_same_bits(run(rp, a.contiguous(), b.contiguous()), want_bits, (name, kind, "row-major copies"))
    assert_same_bits(run(rp, a, b, 3), want_bits, (name, kind, "64x64 tiles"))


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


# ---------------------------------------------------------------- chained ----
# The chained k-split schedule: persistent workers, the last tiles' k-slices
# shared out so that a tile's chain may be begun by one worker and continued
# by the next.  Every worker count must give the oracle's bytes ("Verde与RepOps"
# §3.2: only who computes which part of the serial chain changes).

@pytest.mark.parametrize("M,N,K", [(300, 260, 1000), (129, 257, 33), (64, 64, 32), (257, 130, 4099)])
def test_chained_split_every_worker_count_bit_exact(rp, orc, golden, M, N, K):
    A = inputs.normal((M, K), 1.0, 60 + M, DEV)
    B = inputs.normal((K, N), 1.0, 61 + N, DEV)
    planted = plant_detectors(A, B, golden, 62 + K) if K >= 40 and M >= 8 and N >= 8 else []
    want = orc.gemm(A.cpu().numpy(), B.cpu().numpy())
    check_planted(want, planted, "oracle")
    want_bits = np_bits(want)
    for cfg in all_configs(rp):
        info = rp.gemm_config_info(cfg)
        tiles = -(-M // info["bm"]) * -(-N // info["bn"])
        slots = rp.gemm_config_occupancy(cfg) * torch.cuda.get_device_properties(0).multi_processor_count
        counts = sorted({w for w in (1, 2, 3, 5, 7, tiles - 1, tiles, 0) if 0 <= w <= min(tiles, slots)})
        for w in counts:
            for ta, tb in LAYOUTS:
                Aop, Bop = make_operand(A, ta), make_operand(B, tb)
                lda = Aop.stride(1) if ta else Aop.stride(0)
                ldb = Bop.stride(1) if tb else Bop.stride(0)
                if lda % 4 or ldb % 4:
                    continue
                C = rp.gemm_chained(Aop, Bop, config=cfg, workers=w)
                torch.cuda.synchronize()
                assert rp.device_status() == 0
                assert_same_bits(C, want_bits, ("chained", cfg, w, ta, tb))


def test_chained_split_rejects_what_it_cannot_run(rp):
    A = inputs.normal((100, 64), 1.0, 1, DEV)
    B = inputs.normal((64, 96), 1.0, 2, DEV)
    with pytest.raises(rp.RepopsError):
        rp.gemm_chained(A, B, config=3, workers=1000)          # more workers than tiles
    Au = inputs.normal((100 * 65 + 1,), 1.0, 3, DEV)[1:].view(100, 65)[:, :64]
    with pytest.raises(rp.RepopsError):
        rp.gemm_chained(Au, B, config=3, workers=2)            # not TMA-readable
    with pytest.raises(rp.RepopsError):
        rp.gemm_chained(A, B, config=3, workers=-1)


@pytest.mark.slow
@pytest.mark.parametrize("M,N,K", [(2048, 2048, 2048), (4096, 3072, 2048), (4097, 1023, 3001)])
def test_chained_split_auto_and_worker_counts_same_bytes(rp, orc, M, N, K):
    # shapes the automatic choice runs on the chained split; every worker count
    # and the one-tile-per-CTA kernel of every configuration give the same bytes,
    # and rows spread over the tiles match the oracle
    A = inputs.normal((M, K), 1.0, 70, DEV)
    B = inputs.normal((K, N), 1.0, 71, DEV)
    C = run(rp, A, B)
    ref = run(rp, A, B, config=1, loader=rp.LOADER_CPASYNC)
    assert torch.equal(C.view(torch.int32), ref.view(torch.int32))
    rows = sorted({0, 63, 64, M // 2, M - 1})
    want = oracle_par.gemm(orc, A, B, rows=rows)
    assert np.array_equal(C[rows].cpu().numpy().view(np.uint32), want.view(np.uint32))
    if M % 4 == 0 and N % 4 == 0 and K % 4 == 0:
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        for cfg in all_configs(rp):
            info = rp.gemm_config_info(cfg)
            tiles = -(-M // info["bm"]) * -(-N // info["bn"])
            most = min(tiles, rp.gemm_config_occupancy(cfg) * sms)
            for w in sorted({0, 151, most - 1, most}):
                Cw = rp.gemm_chained(A, B, config=cfg, workers=w)
                assert torch.equal(Cw.view(torch.int32), ref.view(torch.int32)), (cfg, w)
            Cw = rp.gemm_chained(A.t().contiguous().t(), B, config=cfg, workers=0)
            assert torch.equal(Cw.view(torch.int32), ref.view(torch.int32)), (cfg, "A transposed")
    torch.cuda.synchronize()
    assert rp.device_status() == 0


def test_chained_split_is_the_automatic_choice_where_waves_are_uneven(rp):
    # 2048^3 with 64 x 128 tiles is 512 tiles on 304 resident CTAs: the last
    # wave would be two-thirds empty; 8192^3 (8192 tiles) is not split
    assert rp.gemm_auto_chained(2048, 2048, 2048)
    assert not rp.gemm_auto_chained(8192, 8192, 8192)
    assert not rp.gemm_auto_chained(256, 256, 256)


@pytest.mark.slow
@pytest.mark.parametrize("M,N,K", [(2048, 2048, 2048), (4097, 1024, 3000), (3000, 3000, 1000)])
def test_chained_split_repeated_runs_identical(rp, M, N, K):
    # the heads' stores and the tails' flag-acquired loads race only if the
    # release/acquire protocol is wrong: 200 runs across worker counts (every
    # resident slot, one per SM, odd counts) must all give the one-CTA-per-tile
    # bytes, with no bounded wait giving up
    A = inputs.normal((M, K), 1.0, 31, DEV)
    B = inputs.normal((K, N), 1.0, 32, DEV)
    ref = rp.gemm(A, B, config=0, loader=rp.LOADER_TMA).view(torch.int32).clone()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    mismatches = 0
    for w in (0, sms, sms - 1, 97, 64):
        for _ in range(40):
            C = rp.gemm_chained(A, B, config=0, workers=w)
            mismatches += int(not torch.equal(C.view(torch.int32), ref))
    torch.cuda.synchronize()
    assert mismatches == 0
    assert rp.device_status() == 0
