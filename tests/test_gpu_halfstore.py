"""GPU parity of half-precision storage (conversions, the typed GEMM, the mean
+ SGD over half gradients) and of the rolling hash, against the oracle,
through the C ABI.

"Verde与RepOps" §3.3, §5.3 (lower precision as future work); the ZKDV page's
rolling_window.  Bar: bit-exact (NaN compared as a class), every conversion
pair, every GEMM storage mix, transposition, config and loader; aligned and
unaligned gradients; every window length and row split.
"""
import numpy as np
import pytest
import torch

from verifiable_repops_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
F32, F16, BF16 = 0, 1, 2
TORCH = {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}


def bits(t):
    """Host uint bit patterns of a CUDA tensor of any 2- or 4-byte type."""
    if t.element_size() == 2:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.view(torch.int32).cpu().numpy().view(np.uint32)


def to_host_storage(t):
    """The oracle's view of a tensor: float32 values or uint16 half bits."""
    return t.cpu().numpy() if t.dtype == torch.float32 else bits(t)


def same(got_bits, want_bits, nan_mask):
    return np.array_equal(got_bits[~nan_mask], want_bits[~nan_mask])


def test_widen_every_half_pattern(rp, orc):
    h = torch.arange(1 << 16, dtype=torch.int32, device=DEV).to(torch.int16)
    for dt, t in ((torch.float16, F16), (torch.bfloat16, BF16)):
        x = h.view(dt)
        y = rp.convert(x, torch.float32)
        want = orc.convert(bits(x), t, F32)
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(y.cpu().numpy()), nan)
        assert same(bits(y), want.view(np.uint32), nan)


@pytest.mark.parametrize("dt,t", [(torch.float16, F16), (torch.bfloat16, BF16)])
def test_narrow_against_oracle(rp, orc, dt, t):
    rng = np.random.default_rng(t)
    x = (rng.standard_normal(1 << 20) * np.exp2(rng.integers(-140, 127, 1 << 20))).astype(np.float32)
    mids = np.arange(1 << 16, dtype=np.uint32) << 16 | 0x8000          # bfloat16 ties
    x = np.concatenate([x, mids.view(np.float32), np.array([65504, 65520, 65519.99, 2.0 ** -25, 2.0 ** -24,
                                                            -0.0, np.inf, -np.inf, 3.4e38], np.float32)])
    xd = torch.from_numpy(x).to(DEV)
    y = rp.convert(xd, dt)
    want = orc.convert(x, F32, t)
    nan = np.isnan(x)
    assert same(bits(y), want, nan)
    # unaligned source and destination, odd count
    y2 = torch.empty(x.size, dtype=dt, device=DEV)
    rp.convert(xd[1:], dt, out=y2[1:])
    assert same(bits(y2[1:]), want[1:], nan[1:])


def test_in_place_between_half_types(rp, orc):
    x = inputs.normal((100003,), 10.0, 5, DEV).to(torch.float16)
    want = orc.convert(bits(x), F16, BF16)
    y = x.view(torch.bfloat16)
    rp.convert(x, torch.bfloat16, out=y)
    assert np.array_equal(bits(y), want)


MIXES = [(F16, F16, F32), (BF16, BF16, F32), (BF16, BF16, BF16), (F16, BF16, F16), (F32, BF16, F32),
         (BF16, F32, F16)]


def stored(shape, t, seed, trans=False):
    x = inputs.normal(shape[::-1] if trans else shape, 1.0, seed, DEV)
    if t != F32:
        x = x.to(TORCH[t])
    return x.t() if trans else x


@pytest.mark.parametrize("ta,tb,tc", MIXES)
@pytest.mark.parametrize("transA,transB", [(0, 0), (1, 1)])
def test_typed_gemm_matches_oracle(rp, orc, ta, tb, tc, transA, transB):
    M, N, K = 67, 130, 75
    A = stored((M, K), ta, 10 + ta, transA)
    B = stored((K, N), tb, 20 + tb, transB)
    C = rp.gemm_typed(A, B, out_dtype=TORCH[tc])
    want = orc.gemm_typed(to_host_storage(A.contiguous()), ta, to_host_storage(B.contiguous()), tb, tc)
    assert np.array_equal(bits(C), want.view(np.uint32) if tc == F32 else want)


@pytest.mark.parametrize("config,loader", [(0, 1), (3, 2), (4, 0)])
def test_typed_gemm_every_path_same_bits(rp, orc, config, loader):
    A = stored((200, 96), BF16, 30)
    B = stored((96, 72), BF16, 31)
    C = rp.gemm_typed(A, B, config=config, loader=loader)
    want = orc.gemm_typed(to_host_storage(A), BF16, to_host_storage(B), BF16, F32)
    assert np.array_equal(bits(C), want.view(np.uint32))


@pytest.mark.parametrize("t,dt", [(F16, torch.float16), (BF16, torch.bfloat16)])
@pytest.mark.parametrize("nC", [1, 3, 16])
@pytest.mark.parametrize("offset", [0, 1])
def test_half_gradient_mean_matches_oracle(rp, orc, t, dt, nC, offset):
    n = 100003
    grads = [inputs.normal((n + offset,), 1e-2, 40 + r, DEV).to(dt)[offset:] for r in range(nC)]
    theta = inputs.normal((n,), 0.02, 60, DEV)
    order = list(np.random.default_rng(nC).permutation(nC))
    want = orc.mean_sgd_typed([bits(g) for g in grads], t, order, 1e-3, theta.cpu().numpy())
    rp.fixed_order_mean_sgd(grads, order, 1e-3, theta)
    assert np.array_equal(theta.cpu().numpy().view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("width,window", [(1, 1), (50, 1), (50, 2), (50, 50), (1000, 32), (1000, 7), (4096, 32),
                                          (2100, 1024), (2100, 1025), (3000, 1500)])
def test_rolling_hash_matches_oracle(rp, orc, width, window):
    g = torch.Generator(device=DEV)
    g.manual_seed(width + window)
    w = torch.randint(-(1 << 31), 1 << 31, (5, width + 3), generator=g, dtype=torch.int64, device=DEV)
    words = w.to(torch.int32)[:, :width]                  # pitch width + 3
    h = rp.rolling_hash(words, window)
    want = orc.rolling_hash(words.cpu().numpy().view(np.uint32), window)
    assert np.array_equal(h.cpu().numpy().view(np.uint64), want)


@pytest.mark.parametrize("width,window", [(5000, 1024), (6000, 700), (4200, 33), (4100, 1000)])
def test_rolling_hash_several_segments_per_row(rp, orc, width, window):
    # rows longer than one 2048-start segment with windows up to the staged
    # kernel's largest (1024 words): non-last segments stage their full
    # 2048 + W - 1 words, the largest per-warp stage, and more rows than warps
    # per block put warps of one block on different rows and segments
    rows = 9
    g = torch.Generator(device=DEV)
    g.manual_seed(width * 7 + window)
    w = torch.randint(-(1 << 31), 1 << 31, (rows, width + 5), generator=g, dtype=torch.int64, device=DEV)
    words = w.to(torch.int32)[:, :width]                  # pitch width + 5
    h = rp.rolling_hash(words, window)
    want = orc.rolling_hash(words.cpu().numpy().view(np.uint32), window)
    assert np.array_equal(h.cpu().numpy().view(np.uint64), want)


@pytest.mark.parametrize("width,window", [(1100, 32), (2100, 1025)])
def test_rolling_hash_extreme_words(rp, orc, width, window):
    # every word 0xFFFFFFFF gives the largest intermediate sums; runs of zeros
    # between them give windows whose hash is 0 or a single power of the base
    w = torch.full((3, width), -1, dtype=torch.int32, device=DEV)
    w[1, ::3] = 0
    w[2, width // 2:] = 0
    h = rp.rolling_hash(w, window)
    want = orc.rolling_hash(w.cpu().numpy().view(np.uint32), window)
    assert np.array_equal(h.cpu().numpy().view(np.uint64), want)


@pytest.mark.slow
def test_rolling_hash_large_batch_sampled(rp, orc):
    rows, width = 8192, 4096
    g = torch.Generator(device=DEV)
    g.manual_seed(7)
    words = torch.randint(-(1 << 31), 1 << 31, (rows, width), generator=g, dtype=torch.int64, device=DEV).to(torch.int32)
    h = rp.rolling_hash(words, 32)
    pick = [0, 1, 4095, rows - 1]
    want = orc.rolling_hash(words[pick].cpu().numpy().view(np.uint32), 32)
    assert np.array_equal(h[pick].cpu().numpy().view(np.uint64), want)
