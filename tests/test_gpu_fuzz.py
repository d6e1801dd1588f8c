"""Seeded random parity cases for the order-fixed GEMM ("Verde与RepOps" §3.1:
operation order, core count and memory layout must not change the bits;
§3.2: k in a fixed order from +0).

Each case draws its shape (1 to 900 a side: log-uniform in odd cases, so
most end inside one tile, uniform from 64 in even ones), the storage of A and B (row-major or transposed), padded
leading dimensions, base offsets that break 16-byte alignment, an output
buffer with padded rows and canaries, and the path: the automatic choice, an
explicit tile configuration with either loader, the chained k-split with a
random worker count, a batch of one through the batched entry point, or the
host-buffer call.  The whole output must equal the oracle's bit for bit and
nothing outside C may change.  Paths a case cannot take (the TMA loader on an
unaligned operand, more workers than tiles) must be refused with
REPOPS_ERR_UNSUPPORTED and launch nothing.
"""
import numpy as np
import pytest
import torch

from verifiable_repops_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
CASES = 320
CANARY = 7.25


def operand(rng, rows, cols, seed):
    """A (rows, cols) view with random storage order, leading-dimension
    padding and base offset, its values N(0,1) from `seed`."""
    trans = bool(rng.integers(2))
    pad = int(rng.integers(0, 9))
    off = int(rng.integers(0, 4))
    outer, inner = (cols, rows) if trans else (rows, cols)
    ld = inner + pad
    base = inputs.normal((off + outer * ld + 1,), 1.0, seed, DEV)
    M = base[off:off + outer * ld].view(outer, ld)[:, :inner]
    return (M.t() if trans else M), dict(trans=trans, pad=pad, off=off)


def tma_ready(X):
    # the TMA loader's rule: a 16-byte aligned base and a leading dimension
    # that is a multiple of 4 elements
    ld = X.stride(0) if X.stride(1) == 1 else X.stride(1)
    return X.data_ptr() % 16 == 0 and ld % 4 == 0


@pytest.mark.parametrize("case", range(CASES))
def test_random_gemm_case_matches_oracle(rp, orc, case):
    rng = np.random.default_rng(20261202 + case)
    if case % 2:
        M, N, K = (int(np.exp(rng.uniform(0.0, np.log(900.0)))) for _ in range(3))
    else:
        M, N, K = (int(rng.integers(64, 901)) for _ in range(3))
    A, da = operand(rng, M, K, 1000 + 3 * case)
    B, db = operand(rng, K, N, 1001 + 3 * case)
    want = orc.gemm(A.cpu().numpy(), B.cpu().numpy()).view(np.uint32)
    path = ["auto", "config", "chained", "batched", "host"][int(rng.integers(5))]
    ldc = N + int(rng.integers(0, 5))
    cbuf = torch.full((M + 2, ldc), CANARY, device=DEV)
    C = cbuf[1:1 + M, :N]
    what = dict(M=M, N=N, K=K, A=da, B=db, path=path, ldc=ldc)
    if path == "auto":
        rp.gemm(A, B, out=C)
    elif path == "config":
        cfg = int(rng.integers(rp.gemm_config_count()))
        loader = [rp.LOADER_TMA, rp.LOADER_CPASYNC, rp.LOADER_AUTO][int(rng.integers(3))]
        what.update(cfg=cfg, loader=loader)
        if loader == rp.LOADER_TMA and not (tma_ready(A) and tma_ready(B)):
            with pytest.raises(rp.RepopsError) as e:
                rp.gemm(A, B, out=C, config=cfg, loader=loader)
            assert e.value.code == -7, what
            assert (cbuf == CANARY).all(), what
            return
        rp.gemm(A, B, out=C, config=cfg, loader=loader)
    elif path == "chained":
        cfg = int(rng.integers(rp.gemm_config_count()))
        info = rp.gemm_config_info(cfg)
        tiles = -(-M // info["bm"]) * -(-N // info["bn"])
        workers = int(rng.integers(1, tiles + 2))
        slots = rp.gemm_config_occupancy(cfg) * torch.cuda.get_device_properties(0).multi_processor_count
        what.update(cfg=cfg, workers=workers, tiles=tiles)
        if not (tma_ready(A) and tma_ready(B)) or workers > tiles or workers > slots:
            with pytest.raises(rp.RepopsError) as e:
                rp.gemm_chained(A, B, out=C, config=cfg, workers=workers)
            assert e.value.code == -7, what
            assert (cbuf == CANARY).all(), what
            return
        rp.gemm_chained(A, B, out=C, config=cfg, workers=workers)
    elif path == "batched":
        rp.gemm_batched(A, B, out=C)
    else:
        Ah = A.cpu().contiguous()
        Bh = B.cpu().contiguous()
        Ch = torch.full((M, N), CANARY)
        s = torch.cuda.current_stream()
        rp.gemm_host(Ah, Bh, out=Ch, stream=s)
        s.synchronize()
        assert np.array_equal(Ch.numpy().view(np.uint32), want), what
        return
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy().view(np.uint32), want), what
    # rows above and below C, and the padding columns of its rows, untouched
    assert (cbuf[0] == CANARY).all() and (cbuf[M + 1] == CANARY).all(), what
    assert (cbuf[1:1 + M, N:] == CANARY).all(), what
