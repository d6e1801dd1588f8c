"""Host-only checks of the C ABI: the library loads without a GPU, exports
every entry point include/repops.h declares, and rejects bad arguments before
launching anything (those paths touch no CUDA call, so fake pointers are safe:
they are never dereferenced)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "repops.h")


@pytest.fixture(scope="module")
def L():
    from verifiable_repops_gemm_gb300 import build, _capi
    build.build()
    return _capi.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(repops_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for need in ("repops_gemm_f32", "repops_fixed_order_mean_sgd", "repops_merkle_sha256"):
        assert need in names


def test_every_declared_symbol_is_exported(L):
    from verifiable_repops_gemm_gb300 import _capi
    for name in declared_functions():
        assert hasattr(L, name), name
        assert name in _capi.SIGNATURES, "binding lacks " + name


def test_manifest_names_arithmetic_flags(L):
    v = L.repops_version().decode()
    for s in ("sm_103a", "-fmad=false", "-ftz=false", "-prec-div=true", "no tensor cores"):
        assert s in v, s
    # the release build; the checked build's manifest adds -DREPOPS_DEBUG_BOUNDS
    if not os.environ.get("REPOPS_LIBRARY"):
        assert "REPOPS_DEBUG_BOUNDS" not in v


def test_status_strings(L):
    for code in range(-8, 1):
        assert L.repops_status_string(code).decode() != "unknown status"


FAKE_A, FAKE_B, FAKE_C = 0x10000000, 0x20000000, 0x30000000


def test_gemm_rejects_bad_arguments(L):
    g = L.repops_gemm_f32_ex
    assert g(0, 0, -1, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4, None) == -1
    assert g(0, 0, 4, 4, 4, FAKE_A, 3, FAKE_B, 4, FAKE_C, 4, None) == -1     # lda < K
    assert g(0, 0, 4, 4, 4, FAKE_A, 4, FAKE_B, 3, FAKE_C, 4, None) == -1     # ldb < N
    assert g(0, 0, 4, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 3, None) == -1     # ldc < N
    assert g(1, 0, 8, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4, None) == -1     # transA: lda < M
    assert g(0, 1, 4, 8, 4, FAKE_A, 4, FAKE_B, 3, FAKE_C, 8, None) == -1     # transB: ldb < K
    assert g(0, 0, 4, 4, 4, None, 4, FAKE_B, 4, FAKE_C, 4, None) == -1       # null A
    assert g(0, 0, 4, 4, 4, FAKE_A, 4, FAKE_B, 4, None, 4, None) == -1       # null C
    # C overlapping A or B
    assert g(0, 0, 4, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_A + 32, 4, None) == -2
    assert g(0, 0, 4, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_B + 60, 4, None) == -2
    # empty output: nothing to do, no launch
    assert g(0, 0, 0, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4, None) == 0
    assert g(0, 0, 4, 0, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4, None) == 0
    # overflowing spans
    assert g(0, 0, 1 << 62, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4, None) == -1
    # bad config / loader ids
    assert L.repops_gemm_f32_config(99, 0, 0, 0, 4, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4, None) == -1
    assert L.repops_gemm_f32_config(0, 7, 0, 0, 4, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4, None) == -1


def test_gemm_config_table(L):
    n = L.repops_gemm_config_count()
    assert n >= 3
    seen = set()
    for c in range(n):
        v = [ctypes.c_int() for _ in range(5)]
        assert L.repops_gemm_config_info(c, *[ctypes.byref(x) for x in v]) == 0
        bm, bn, th, tm, tn = (x.value for x in v)
        assert bm % 8 == 0 and bn % 8 == 0 and th % 32 == 0
        assert (bm // (4 * tm)) * (bn // (8 * tn)) * 32 == th
        seen.add((bm, bn, th))
    assert len(seen) == n
    assert L.repops_gemm_config_info(n, None, None, None, None, None) == -1


def _mean(L, nC, ln, ptrs, order, theta):
    P = (ctypes.c_void_p * max(nC, 1))(*ptrs)
    O = (ctypes.c_int * max(len(order), 1))(*order)
    return L.repops_fixed_order_mean_sgd(nC, ln, ctypes.cast(P, ctypes.c_void_p),
                                         ctypes.cast(O, ctypes.c_void_p), ctypes.c_float(1e-3),
                                         theta, None)


def test_mean_rejects_bad_arguments(L):
    p = [FAKE_A, FAKE_A + 4096, FAKE_A + 8192]
    assert _mean(L, 0, 16, [], [], FAKE_C) == -1
    assert _mean(L, 1025, 16, [FAKE_A] * 1025, list(range(1025)), FAKE_C) == -1
    assert _mean(L, 3, -1, p, [0, 1, 2], FAKE_C) == -1
    assert _mean(L, 3, 16, p, [0, 1, 1], FAKE_C) == -3      # duplicate
    assert _mean(L, 3, 16, p, [0, 1, 3], FAKE_C) == -3      # out of range
    assert _mean(L, 3, 16, p, [2, 0, 1], FAKE_A + 4096 + 8) == -2   # theta inside a gradient
    assert _mean(L, 3, 0, p, [2, 0, 1], FAKE_C) == 0        # empty: no launch
    assert _mean(L, 3, 16, p, [2, 0, 1], None) == -1


def test_merkle_rejects_bad_arguments(L):
    m = L.repops_merkle_sha256
    assert m(FAKE_A, 0, 4096, FAKE_C, None) == -1
    assert m(FAKE_A, 100, 100, FAKE_C, None) == -1          # leaf not a multiple of 64
    assert m(FAKE_A, 100, 0, FAKE_C, None) == -1
    assert m(None, 100, 4096, FAKE_C, None) == -1
    assert m(FAKE_A, 100, 4096, None, None) == -1
    assert m(FAKE_A, 100, 4096, FAKE_A + 50, None) == -2    # root inside the input
    ws = L.repops_merkle_workspace_bytes
    assert ws(1 << 32, 4096) == (8192 + 16) * 32            # 2^20 leaves, 128 per CTA
    assert ws(4096 * 128, 4096) == 0                        # one CTA writes the root
    assert ws(0, 4096) == 0
    mw = L.repops_merkle_sha256_ws
    n = 4096 * 1000
    need = ws(n, 4096)
    assert need > 0
    assert mw(FAKE_A, n, 4096, FAKE_C, FAKE_B, need - 1, None) == -1     # too small
    assert mw(FAKE_A, n, 4096, FAKE_C, FAKE_B + 4, need, None) == -1     # misaligned
    assert mw(FAKE_A, n, 4096, FAKE_C, FAKE_A + 16, need, None) == -2    # overlaps input


def test_sort_ids_matches_oracle(L, orc):
    import numpy as np
    import verifiable_repops_gemm_gb300 as rp
    rng = np.random.default_rng(11)
    for n in (1, 2, 16, 100):
        ids = [rng.bytes(int(rng.integers(1, 40))) for _ in range(n)]
        ids = list(dict.fromkeys(ids))
        assert rp.sort_ids(ids) == orc.sort_ids(ids)
    ids = [b"did:a", b"did:", b"did:ab", b"\x80", b"\x7f\xff"]
    assert rp.sort_ids(ids) == orc.sort_ids(ids)
    with pytest.raises(rp.RepopsError):
        rp.sort_ids([b"x", b"y", b"x"])


def test_sha256_constant_table_matches_derivation(orc):
    # the CUDA source's FIPS 180-4 table, read as text, against the oracle's
    # derivation from the primes
    src = open(os.path.join(ROOT, "verifiable_repops_gemm_gb300", "csrc", "merkle.cu")).read()
    k_block = src[src.index("c_K[64]"):src.index("};", src.index("c_K[64]"))]
    h_block = src[src.index("c_H0[8]"):src.index("};", src.index("c_H0[8]"))]
    K = [int(x, 16) for x in re.findall(r"0x([0-9a-f]{8})u", k_block)]
    H = [int(x, 16) for x in re.findall(r"0x([0-9a-f]{8})u", h_block)]
    K0, H0 = orc.sha256_constants()
    assert K == K0
    assert H == H0


def test_product_path_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "verifiable_repops_gemm_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "repops_oracle" not in text and "liboracle" not in text, f


def test_proof_shape_and_tree_size_match_oracle(L, orc):
    import numpy as np
    for nl in (1, 2, 3, 5, 8, 13, 128, 129, 1000):
        data = np.zeros(nl * 64, np.uint8)
        tree = orc.merkle_tree(data, 64)
        assert L.repops_merkle_tree_bytes(nl * 64, 64) == 32 * tree.shape[0]
        for i in sorted({0, nl // 2, nl - 1}):
            assert L.repops_merkle_proof_steps(nl, i) == orc.merkle_proof(tree, nl, i).shape[0]
    assert L.repops_merkle_proof_steps(5, 5) == -1
    assert L.repops_merkle_proof_steps(0, 0) == -1


def test_replay_validates_every_block_before_launching(L):
    steps, nC, n = 3, 2, 1024
    P = (ctypes.c_void_p * (steps * nC))(*[FAKE_A + 0x100000 * i for i in range(steps * nC)])
    E = (ctypes.c_float * steps)(1e-3, 1e-3, 1e-3)

    def call(orders, theta=FAKE_C, roots=FAKE_B):
        O = (ctypes.c_int * (steps * nC))(*orders)
        return L.repops_replay_mean_sgd_commit(steps, nC, n, ctypes.cast(P, ctypes.c_void_p),
                                               ctypes.cast(O, ctypes.c_void_p),
                                               ctypes.cast(E, ctypes.c_void_p), theta, 4096, roots, None)
    assert call([0, 1, 1, 0, 0, 0]) == -3            # the last block repeats a contributor
    assert call([0, 1, 1, 0, 0, 1], theta=FAKE_A + 0x100000 * 5 + 64) == -2
    assert call([0, 1, 1, 0, 0, 1], roots=FAKE_C + 16) == -2
    assert L.repops_replay_mean_sgd_commit(0, nC, n, P, None, E, FAKE_C, 4096, FAKE_B, None) == -1


def test_row_operators_reject_bad_arguments(L):
    sm = L.repops_softmax_rows_f32
    assert sm(-1, 4, FAKE_A, 4, FAKE_B, 4, None) == -1
    assert sm(4, 4, FAKE_A, 3, FAKE_B, 4, None) == -1            # ldx < cols
    assert sm(4, 4, FAKE_A, 4, FAKE_A + 8, 4, None) == -2        # partial overlap
    assert sm(0, 4, FAKE_A, 4, FAKE_B, 4, None) == 0
    assert sm(4, 400000, FAKE_A, 400000, FAKE_B, 400000, None) == -7
    ln = L.repops_layernorm_rows_f32
    assert ln(4, 4, FAKE_A, 4, None, FAKE_C, ctypes.c_float(1e-5), FAKE_B, 4, None) == -1
    assert ln(4, 4, FAKE_A, 4, FAKE_B + 16, FAKE_C, ctypes.c_float(1e-5), FAKE_B, 4, None) == -2
    rn = L.repops_rmsnorm_rows_f32
    assert rn(4, 4, FAKE_A, 4, FAKE_B, ctypes.c_float(1e-5), FAKE_B, 4, None) == -2
    assert L.repops_gelu_f32(-1, FAKE_A, FAKE_B, None) == -1
    assert L.repops_gelu_f32(8, FAKE_A, FAKE_A + 4, None) == -2
    assert L.repops_gelu_f32(0, None, None, None) == 0


def _bat(L, batch=2, M=4, N=4, K=4, A=FAKE_A, lda=4, sA=16, B=FAKE_B, ldb=4, sB=16, C=FAKE_C, ldc=4,
         sC=16, alpha=1.0, bias=None, act=0, R=None, ldr=4, sR=16, config=-1, loader=0, tA=0, tB=0,
         causal=-1, k_lo=-1, k_hi=-1, b_group=1):
    return L.repops_gemm_f32_batched(config, loader, tA, tB, batch, M, N, K, A, lda, sA, B, ldb, sB,
                                     C, ldc, sC, ctypes.c_float(alpha), bias, act, R, ldr, sR, causal, k_lo, k_hi,
                                     b_group, None)


def test_batched_gemm_rejects_bad_arguments(L):
    assert _bat(L, batch=-1) == -1
    assert _bat(L, sA=-4) == -1                                    # negative stride
    assert _bat(L, act=2) == -1                                    # unknown activation
    assert _bat(L, causal=-2) == -1
    assert _bat(L, k_lo=-2) == -1 and _bat(L, k_hi=-5) == -1                 # k window bounds
    assert _bat(L, b_group=0) == -1
    assert _bat(L, ldc=3) == -1
    assert _bat(L, R=FAKE_B + 4096, ldr=3) == -1                   # residual ld < N
    assert _bat(L, config=99) == -1
    assert _bat(L, loader=7) == -1
    assert _bat(L, A=None) == -1
    assert _bat(L, batch=0) == 0                                   # empty: no launch
    assert _bat(L, M=0) == 0
    assert _bat(L, batch=70000) == -7                              # one grid row per batch
    # outputs of two batches overlap: neither stacked nor interleaved
    assert _bat(L, sC=8) == -2
    assert _bat(L, sC=2, ldc=6) == -2                              # interleaved, but 2 < N
    assert _bat(L, C=FAKE_A + 32, sA=0) == -2                      # C over A
    assert _bat(L, bias=FAKE_C + 8) == -2                          # bias inside C
    assert _bat(L, R=FAKE_C + 4) == -2                             # residual overlapping C, not in place
    assert _bat(L, R=FAKE_C, sR=20, sC=16) == -2                   # same base, other stride


def test_causal_softmax_rejects_bad_arguments(L):
    c = L.repops_softmax_rows_causal_f32
    assert c(4, 4, FAKE_A, 4, FAKE_B, 4, -1, 4, None) == -1                # first < 0
    assert c(4, 4, FAKE_A, 4, FAKE_B, 4, 0, 0, None) == -1                 # period < 1
    assert c(4, 4, FAKE_A, 4, FAKE_A + 8, 4, 0, 4, None) == -2
    assert c(0, 4, FAKE_A, 4, FAKE_B, 4, 0, 4, None) == 0


def test_half_storage_and_rolling_hash_reject_bad_arguments(L):
    cv = L.repops_convert
    assert cv(-1, FAKE_A, 0, FAKE_B, 1, None) == -1
    assert cv(8, FAKE_A, 3, FAKE_B, 1, None) == -1                     # unknown type
    assert cv(8, FAKE_A, 0, FAKE_A + 8, 1, None) == -2                 # overlap, not in place
    assert cv(8, FAKE_A, 0, FAKE_A, 1, None) == -2                     # in place needs equal sizes
    assert cv(0, None, 0, None, 1, None) == 0
    gt = L.repops_gemm_typed
    assert gt(-1, 0, 0, 0, 4, 4, 4, FAKE_A, 5, 4, FAKE_B, 1, 4, FAKE_C, 0, 4, None) == -1   # type 5
    assert gt(-1, 0, 0, 0, 4, 4, 4, FAKE_A, 1, 3, FAKE_B, 1, 4, FAKE_C, 0, 4, None) == -1   # lda < K
    assert gt(-1, 0, 0, 0, 4, 4, 4, FAKE_A, 1, 4, FAKE_B, 1, 4, FAKE_A + 8, 1, 4, None) == -2
    assert gt(-1, 0, 0, 0, 0, 4, 4, FAKE_A, 1, 4, FAKE_B, 1, 4, FAKE_C, 1, 4, None) == 0
    ms = L.repops_fixed_order_mean_sgd_typed
    p = (ctypes.c_void_p * 2)(FAKE_A, FAKE_A + 4096)
    o = (ctypes.c_int * 2)(1, 0)
    assert ms(2, 16, ctypes.cast(p, ctypes.c_void_p), 7, ctypes.cast(o, ctypes.c_void_p), ctypes.c_float(1e-3),
              FAKE_C, None) == -1                                                        # unknown type
    assert ms(2, 16, ctypes.cast(p, ctypes.c_void_p), 1, ctypes.cast(o, ctypes.c_void_p), ctypes.c_float(1e-3),
              FAKE_A + 16, None) == -2                                                   # theta over a gradient
    rh = L.repops_rolling_hash_u32
    assert rh(4, 10, FAKE_A, 10, 0, FAKE_B, 10, None) == -1          # window 0
    assert rh(4, 10, FAKE_A, 10, 11, FAKE_B, 10, None) == -1         # window above the row width
    assert rh(4, 10, FAKE_A, 9, 3, FAKE_B, 8, None) == -1            # ldw < width
    assert rh(4, 10, FAKE_A, 10, 3, FAKE_B, 7, None) == -1           # ldo < width - window + 1
    assert rh(4, 10, FAKE_A, 10, 3, FAKE_A + 40, 8, None) == -2
    assert rh(0, 10, FAKE_A, 10, 3, FAKE_B, 8, None) == 0


def test_backward_operators_reject_bad_arguments(L):
    assert L.repops_colsum_f32(-1, 4, FAKE_A, 4, FAKE_B, None) == -1
    assert L.repops_colsum_f32(4, 4, FAKE_A, 3, FAKE_B, None) == -1          # ldx < cols
    assert L.repops_colsum_f32(4, 4, FAKE_A, 4, FAKE_A + 8, None) == -2
    assert L.repops_colsum_f32(4, 0, FAKE_A, 4, FAKE_B, None) == 0
    assert L.repops_gelu_backward_f32(-1, FAKE_A, FAKE_B, FAKE_C, None) == -1
    assert L.repops_gelu_backward_f32(8, FAKE_A, FAKE_B, FAKE_A + 4, None) == -2
    assert L.repops_gelu_backward_f32(0, None, None, None, None) == 0
    rb = L.repops_rmsnorm_backward_f32
    eps = ctypes.c_float(1e-5)
    assert rb(4, 4, FAKE_A, 4, None, eps, FAKE_B, 4, None, 0, FAKE_C, 4, FAKE_C + 4096, 4, None) == -1   # null gamma
    assert rb(4, 4, FAKE_A, 4, FAKE_A + 4096, eps, FAKE_B, 4, None, 0, FAKE_A, 4, FAKE_C, 4, None) == -2  # dx over x
    assert rb(4, 4, FAKE_A, 4, FAKE_A + 4096, eps, FAKE_B, 4, None, 0, FAKE_C, 4, FAKE_C + 8, 4, None) == -2
    assert rb(4, 4, FAKE_A, 4, FAKE_A + 4096, eps, FAKE_B, 4, FAKE_C + 8, 4, FAKE_C, 4, FAKE_C + 4096, 4,
              None) == -2                                                                    # res partly over dx
    sb = L.repops_softmax_backward_f32
    assert sb(4, 4, FAKE_A, 3, FAKE_B, 4, FAKE_C, 4, None) == -1
    assert sb(4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_A + 8, 4, None) == -2
    assert sb(4, 400000, FAKE_A, 400000, FAKE_B, 400000, FAKE_C, 400000, None) == -7


def test_host_buffer_gemm_rejects_bad_arguments(L):
    g = L.repops_gemm_f32_host
    assert g(-1, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4, None) == -1
    assert g(4, 4, 4, FAKE_A, 3, FAKE_B, 4, FAKE_C, 4, None) == -1
    assert g(4, 4, 4, None, 4, FAKE_B, 4, FAKE_C, 4, None) == -1
    assert g(4, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_A + 16, 4, None) == -2
    assert g(0, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4, None) == 0


def test_llama_operators_reject_bad_arguments(L):
    f = ctypes.c_float
    sbc = L.repops_softmax_backward_causal_f32
    assert sbc(4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4, -1, 4, None) == -1        # first < 0
    assert sbc(4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4, 0, 0, None) == -1         # period < 1
    assert sbc(4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_A + 4, 4, 0, 4, None) == -2     # ds overlaps p
    sw = L.repops_swiglu_f32
    assert sw(-1, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4, None) == -1
    assert sw(4, 4, FAKE_A, 3, FAKE_B, 4, FAKE_C, 4, None) == -1                # ldg < cols
    assert sw(4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_A + 4, 4, None) == -2            # h overlaps g, not in place
    assert sw(4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_A, 8, None) == -2                # same start, other pitch
    assert sw(0, 4, None, 4, None, 4, None, 4, None) == 0
    sb = L.repops_swiglu_backward_f32
    assert sb(4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4, FAKE_A, 4, FAKE_A + 8, 4, None) == -2   # dg, du overlap
    assert sb(4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4, FAKE_B, 4, FAKE_C + 4096, 4, None) == -2  # dg on u
    assert sb(4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4, FAKE_C + 4096, 4, FAKE_A, 4, None) == -2  # du on g
    assert sb(4, 4, FAKE_A, 4, FAKE_B, 4, None, 4, FAKE_C, 4, FAKE_C + 4096, 4, None) == -1
    assert L.repops_rope_frequencies_f32(0, f(13.0), FAKE_A, None) == -1
    assert L.repops_rope_frequencies_f32(4, f(13.0), None, None) == -1
    rt = L.repops_rope_table_f32
    assert rt(0, 4, FAKE_A, FAKE_B, FAKE_C, None) == -1
    assert rt((1 << 24) + 1, 4, FAKE_A, FAKE_B, FAKE_C, None) == -1
    assert rt(16, 4, FAKE_A, FAKE_B, FAKE_B + 16, None) == -2                   # cos and sin overlap
    assert rt(16, 4, FAKE_A, FAKE_A + 4, FAKE_C, None) == -2                    # cos over freq
    rp = L.repops_rope_f32
    assert rp(4, 2, 0, FAKE_A, 8, FAKE_B, FAKE_C, 16, 0, 4, 0, None) == -1      # pairs < 1
    assert rp(4, 2, 2, FAKE_A, 7, FAKE_B, FAKE_C, 16, 0, 4, 0, None) == -1      # ldx < heads * 2 * pairs
    assert rp(4, 2, 2, FAKE_A, 8, FAKE_B, FAKE_C, 16, 13, 4, 0, None) == -1     # position 16 past the table
    assert rp(40, 2, 2, FAKE_B - 64, 8, FAKE_B, FAKE_C, 16, 12, 4, 0, None) == -2  # positions 12..15 fit; x runs into cos
    assert rp(4, 2, 2, FAKE_A, 8, FAKE_B, FAKE_C, 16, 0, 0, 0, None) == -1      # period < 1
    assert rp(4, 2, 2, FAKE_B + 8, 8, FAKE_B, FAKE_C, 16, 0, 4, 0, None) == -2  # x overlaps cos
    assert rp(0, 2, 2, None, 8, None, None, 16, 0, 4, 0, None) == 0


def test_selftest_rejects_bad_limits(L):
    assert L.repops_selftest_bounded_wait(0, None) == -1
    assert L.repops_selftest_bounded_wait(3_000_000_000, None) == -1
    assert L.repops_selftest_bounded_flag_wait(0, None) == -1
    assert L.repops_selftest_bounded_flag_wait(3_000_000_000, None) == -1


def test_added_entry_points_reject_bad_arguments(L):
    # the chained k-split: a negative worker count; the usual GEMM checks first
    assert L.repops_gemm_f32_chained(0, -1, 0, 0, 4, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4, None) == -1
    assert L.repops_gemm_f32_chained(0, 2, 0, 0, 4, 4, 4, FAKE_A, 3, FAKE_B, 4, FAKE_C, 4, None) == -1
    assert L.repops_gemm_f32_chained(0, 2, 0, 0, 4, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_A + 32, 4, None) == -2
    # fused attention: heads not a multiple of kv heads, short leading dims,
    # null pointers, nothing to do
    att = L.repops_attention_causal_f32
    assert att(1, 32, 3, 2, 64, FAKE_A, 256, FAKE_B, 256, FAKE_C, 256, 0.125, FAKE_C + (1 << 20), 256,
               None, None) == -1
    assert att(1, 32, 4, 2, 64, FAKE_A, 100, FAKE_B, 256, FAKE_C, 256, 0.125, FAKE_C + (1 << 20), 256,
               None, None) == -1
    assert att(1, 32, 4, 2, 64, None, 256, FAKE_B, 256, FAKE_C, 256, 0.125, FAKE_C + (1 << 20), 256,
               None, None) == -1
    assert att(0, 32, 4, 2, 64, None, 0, None, 0, None, 0, 0.125, None, 0, None, None) == 0
    assert att(1, 32, 4, -1, 64, FAKE_A, 256, FAKE_B, 256, FAKE_C, 256, 0.125, FAKE_C, 256, None, None) == -1
    # the per-thread status word must be 4-byte aligned; null restores the shared one
    assert L.repops_set_thread_status_word(FAKE_A + 2) == -1
    assert L.repops_set_thread_status_word(None) == 0
    # the scratch pool's size query needs somewhere to write
    assert L.repops_scratch_reserved_bytes(None) == -1
    # GEMM workspace: sizes of rejected arguments are 0; a misaligned or
    # null-but-sized workspace is refused before any launch
    assert L.repops_gemm_workspace_bytes(0, 0, -1, 8, 8, FAKE_A, 8, FAKE_B, 8) == 0
    assert L.repops_gemm_workspace_bytes(0, 0, 8, 8, 8, FAKE_A, 4, FAKE_B, 8) == 0
    assert L.repops_gemm_f32_ws(0, 0, 8, 8, 8, FAKE_A, 8, FAKE_B, 8, FAKE_C, 8, FAKE_C + (1 << 20) + 16, 4096,
                                None) == -1
    assert L.repops_gemm_f32_ws(0, 0, 8, 8, 8, FAKE_A, 8, FAKE_B, 8, FAKE_C, 8, None, 4096, None) == -1
    # host-buffer mean + SGD: counts, orders, aliasing host ranges
    import ctypes as C
    ptrs = (C.c_void_p * 2)(FAKE_A, FAKE_B)
    order_ok = (C.c_int * 2)(1, 0)
    order_dup = (C.c_int * 2)(0, 0)
    mh = L.repops_fixed_order_mean_sgd_host
    assert mh(0, 8, C.cast(ptrs, C.c_void_p), C.cast(order_ok, C.c_void_p), C.c_float(1e-3), FAKE_C, None) == -1
    assert mh(2, 8, C.cast(ptrs, C.c_void_p), C.cast(order_dup, C.c_void_p), C.c_float(1e-3), FAKE_C, None) == -3
    assert mh(2, 8, C.cast(ptrs, C.c_void_p), C.cast(order_ok, C.c_void_p), C.c_float(1e-3), FAKE_A + 4,
              None) == -2
    # host-buffer Merkle: empty input, bad leaf, the root over the input
    assert L.repops_merkle_sha256_host(FAKE_A, 0, 4096, FAKE_C, None) == -1
    assert L.repops_merkle_sha256_host(FAKE_A, 100, 100, FAKE_C, None) == -1
    assert L.repops_merkle_sha256_host(FAKE_A, 100, 4096, FAKE_A + 8, None) == -2


def test_host_allocator_arguments(L):
    import ctypes as C
    p = C.c_void_p(12345)
    # nothing to allocate: a null pointer and OK; nowhere to write: refused
    assert L.repops_host_alloc(0, C.byref(p)) == 0 and p.value is None
    assert L.repops_host_alloc(4096, None) == -1
    # freeing null is a no-op; a pointer the allocator did not return is refused
    assert L.repops_host_free(None) == 0
    assert L.repops_host_free(FAKE_A) == -1
    # a size no mapping can hold
    p = C.c_void_p(12345)
    assert L.repops_host_alloc((1 << 64) - 1, C.byref(p)) == -1 and p.value is None


def test_host_allocator_without_a_device_keeps_nothing(L):
    # with no usable GPU the registration fails: an error, a null pointer,
    # and the mapping is gone again (a free of whatever was returned is refused)
    import ctypes as C
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    p = C.c_void_p(12345)
    assert L.repops_host_alloc(1 << 20, C.byref(p)) == -4 and p.value is None


def declared_signatures():
    """name -> (return type text, [parameter texts]) for every declaration in
    include/repops.h (comments and preprocessor lines removed)."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = "\n".join(l for l in text.split("\n") if not l.lstrip().startswith("#"))
    out = {}
    for m in re.finditer(r"([A-Za-z_][\w\s\*]*?)\b(repops_\w+)\s*\(([^;{]*?)\)\s*;", text):
        ret, name, params = m.group(1).strip(), m.group(2), m.group(3).strip()
        ret = ret.split("\n")[-1].strip()
        plist = [] if params in ("", "void") else [p.strip() for p in params.split(",")]
        out[name] = (ret, plist)
    return out


def test_binding_signatures_match_the_header():
    import ctypes as C
    from verifiable_repops_gemm_gb300 import _capi
    decl = declared_signatures()
    assert set(decl) == set(_capi.SIGNATURES), set(decl) ^ set(_capi.SIGNATURES)
    ret_types = {"int": C.c_int, "uint64_t": C.c_uint64, "const char *": C.c_char_p}
    scalar = {"int": C.c_int, "int64_t": C.c_int64, "uint32_t": C.c_uint32, "uint64_t": C.c_uint64,
              "float": C.c_float}
    for name, (ret, params) in decl.items():
        restype, argtypes = _capi.SIGNATURES[name]
        assert ret in ret_types and restype is ret_types[ret], (name, ret, restype)
        assert len(argtypes) == len(params), (name, len(argtypes), len(params))
        for p, a in zip(params, argtypes):
            base = re.sub(r"\s+\w+$", "", p).replace("const ", "").strip()   # the type, without the name
            if "*" in p or base == "cudaStream_t":
                assert a is C.c_void_p, (name, p, a)       # pointers and the stream: passed as addresses
            else:
                assert base in scalar and a is scalar[base], (name, p, a)


def test_library_exports_exactly_the_declared_functions(L):
    # every extern "C" definition in the sources is declared in the header and
    # the other way round; and where binutils are at hand, the shared object's
    # exported repops_ symbols are exactly those
    import glob
    import shutil
    import subprocess
    decl = set(declared_signatures())
    csrc = os.path.join(ROOT, "verifiable_repops_gemm_gb300", "csrc")
    defs = set()
    for f in glob.glob(os.path.join(csrc, "*.cu")):
        defs |= set(re.findall(r'extern "C"[^;{(]*?\b(repops_\w+)\s*\(', open(f).read()))
    assert defs == decl, sorted(defs ^ decl)
    nm = shutil.which("nm")
    if nm:
        from verifiable_repops_gemm_gb300 import build
        r = subprocess.run([nm, "-D", "--defined-only", build.LIB], capture_output=True, text=True)
        if r.returncode == 0:
            exported = {line.split()[-1] for line in r.stdout.splitlines()
                        if line.split() and line.split()[-1].startswith("repops_")}
            assert exported == decl, sorted(exported ^ decl)
