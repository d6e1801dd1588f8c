"""GPU parity of the fixed-order contributor mean + SGD against the oracle.

"Zoo Per-LLM Chain Soundness" §2 Def. "Aggregation rule", §5 "Ordering
subroutine" / "Update step".  Bar: bit-exact theta.
"""
import numpy as np
import pytest
import torch

from verifiable_repops_gemm_gb300 import inputs

import oracle_par

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _hex(lst):
    return np.array([int(x, 16) for x in lst], dtype=np.uint32)


def run_both(rp, orc, grads, order, eta, theta):
    want = orc.mean_sgd([g.cpu().numpy() for g in grads], order, eta, theta.cpu().numpy())
    th = theta.clone()
    rp.fixed_order_mean_sgd(grads, order, eta, th)
    torch.cuda.synchronize()
    return th.cpu().numpy(), want


@pytest.mark.parametrize("nC,n", [(1, 1), (1, 1000), (2, 4099), (3, 1000003), (7, 513),
                                  (16, 1 << 20), (16, (1 << 20) + 3), (33, 10007), (100, 4096)])
def test_mean_sgd_bit_exact(rp, orc, nC, n):
    grads = [inputs.normal((n,), 1e-2, 1000 + r, DEV) for r in range(nC)]
    theta = inputs.normal((n,), 0.02, 999, DEV)
    ids = inputs.contributor_ids(nC, 7 + nC)
    order = rp.sort_ids(ids)
    got, want = run_both(rp, orc, grads, order, 1e-3, theta)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_mean_sgd_crafted_cases(rp, golden):
    c = golden["mean_order_detector"]
    gs = [torch.tensor(g, dtype=torch.float32, device=DEV) for g in c["grads"]]
    for case in c["cases"]:
        th = torch.tensor(c["theta"], dtype=torch.float32, device=DEV)
        rp.fixed_order_mean_sgd(gs, case["order"], c["eta"], th)
        assert np.array_equal(th.cpu().numpy().view(np.uint32), _hex(case["expected_bits"]))
    z = golden["mean_fold_starts_at_first_gradient"]
    gs = [torch.from_numpy(_hex(g).view(np.float32)).to(DEV) for g in z["grads_bits"]]
    th = torch.from_numpy(_hex(z["theta_bits"]).view(np.float32)).to(DEV)
    eta = float(_hex([z["eta_bits"]]).view(np.float32)[0])
    rp.fixed_order_mean_sgd(gs, z["order"], eta, th)
    assert np.array_equal(th.cpu().numpy().view(np.uint32), _hex(z["expected_bits"]))
    d = golden["mean_divides_by_count"]
    gs = [torch.tensor(g, dtype=torch.float32, device=DEV) for g in d["grads"]]
    th = torch.tensor(d["theta"], dtype=torch.float32, device=DEV)
    rp.fixed_order_mean_sgd(gs, d["order"], d["eta"], th)
    assert np.array_equal(th.cpu().numpy().view(np.uint32), _hex(d["expected_bits"]))


def test_mean_sgd_order_changes_bits(rp):
    n = 4096
    big = torch.full((n,), 1e8, device=DEV)
    one = torch.ones(n, device=DEV)
    gs = [big, one, -big, one]
    a = torch.zeros(n, device=DEV)
    b = torch.zeros(n, device=DEV)
    rp.fixed_order_mean_sgd(gs, [0, 1, 2, 3], 1.0, a)
    rp.fixed_order_mean_sgd(gs, [0, 2, 1, 3], 1.0, b)
    assert (a == -0.25).all() and (b == -0.5).all()


def test_mean_sgd_unaligned_and_guard_band(rp, orc):
    n, nC = 100003, 5
    bases = [inputs.normal((n + 8,), 1e-2, 50 + r, DEV) for r in range(nC)]
    grads = [b[r % 4 + 1:r % 4 + 1 + n] for r, b in enumerate(bases)]   # misaligned views
    tbuf = torch.full((n + 2048,), 777.0, device=DEV)
    theta = tbuf[1025:1025 + n]
    theta.copy_(inputs.normal((n,), 0.02, 49, DEV))
    order = [3, 1, 4, 0, 2]
    want = orc.mean_sgd([g.cpu().numpy() for g in grads], order, 1e-3, theta.cpu().numpy())
    rp.fixed_order_mean_sgd(grads, order, 1e-3, theta)
    assert np.array_equal(theta.cpu().numpy().view(np.uint32), want.view(np.uint32))
    assert (tbuf[:1025] == 777.0).all() and (tbuf[1025 + n:] == 777.0).all()


def test_mean_sgd_rejects_alias_and_order(rp):
    g = torch.zeros(1000, device=DEV)
    with pytest.raises(rp.RepopsError):
        rp.fixed_order_mean_sgd([g, g.clone()], [0, 0], 1e-3, torch.zeros(1000, device=DEV))
    with pytest.raises(rp.RepopsError):
        rp.fixed_order_mean_sgd([g, g.clone()], [0, 1], 1e-3, g)


@pytest.mark.slow
def test_mean_sgd_full_size_every_element(rp, orc):
    # 16 contributors x 2^28 fp32, N(0, 1e-2); theta 2^28, N(0, 0.02); eta = 1e-3.
    # Every element of theta after the update against the oracle on the same
    # buffers, in element ranges of 2^25 (the oracle split across the host cores)
    nC, n = inputs.MEAN_CONTRIBUTORS, inputs.MEAN_LEN
    grads = [inputs.normal((n,), 1e-2, 200 + r, DEV) for r in range(nC)]
    theta = inputs.normal((n,), 0.02, 199, DEV)
    order = rp.sort_ids(inputs.contributor_ids(nC, 200))
    before = theta.cpu().numpy()
    rp.fixed_order_mean_sgd(grads, order, 1e-3, theta)
    torch.cuda.synchronize()
    chunk = 1 << 25
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        gs = [g[lo:hi].cpu().numpy() for g in grads]
        want = oracle_par.mean_sgd(orc, gs, order, 1e-3, before[lo:hi], 0, hi - lo)
        got = theta[lo:hi].cpu().numpy()
        if not np.array_equal(got.view(np.uint32), want.view(np.uint32)):
            bad = np.nonzero(got.view(np.uint32) != want.view(np.uint32))[0]
            raise AssertionError("%d elements differ, first at %d" % (bad.size, lo + int(bad[0])))


@pytest.mark.parametrize("nC", [3, 16])
def test_mean_sgd_special_values(rp, orc, nC):
    # infinities of both signs (their sum NaN), NaN, sums that overflow, -0 and
    # subnormal gradients, θ at ±inf and ±0, on a ragged length (vector body and
    # scalar tail): the same bits as the oracle wherever it is not NaN
    n = 4099
    g = np.random.default_rng(19000 + nC)
    G = (g.standard_normal((nC, n)) * 1e-2).astype(np.float32)
    th = (g.standard_normal(n) * 0.02).astype(np.float32)
    G[0, 1] = np.inf
    G[1, 2] = np.inf
    G[2, 2] = -np.inf
    G[1, 3] = np.nan
    G[:, 4] = 3.0e38
    G[:, 5] = -0.0
    th[5] = -0.0
    G[:, 6] = 1e-45
    th[7] = np.inf
    th[8] = -np.inf
    G[:, 4098] = -3.0e38
    grads = [torch.from_numpy(G[r].copy()).to(DEV) for r in range(nC)]
    theta = torch.from_numpy(th.copy()).to(DEV)
    order = rp.sort_ids(inputs.contributor_ids(nC, 19100 + nC))
    got, want = run_both(rp, orc, grads, order, 1e-3, theta)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


@pytest.mark.parametrize("nC,n,pinned", [(16, (1 << 23) + 3, True), (3, 1000003, False), (1, 5, True)])
def test_host_buffer_mean_sgd_same_bits(rp, orc, nC, n, pinned):
    # chunks of the host call are independent element ranges: the bits equal
    # the device call's and the oracle's, pinned or pageable host memory
    grads = [inputs.normal((n,), 1e-2, 300 + r, "cpu") for r in range(nC)]
    theta = inputs.normal((n,), 0.02, 299, "cpu")
    if pinned:
        grads = [g.pin_memory() for g in grads]
        theta = theta.pin_memory()
    order = rp.sort_ids(inputs.contributor_ids(nC, 301))
    want = orc.mean_sgd([g.numpy() for g in grads], order, 1e-3, theta.numpy())
    dev = theta.to(DEV)
    rp.fixed_order_mean_sgd([g.to(DEV) for g in grads], order, 1e-3, dev)
    s = torch.cuda.Stream()
    rp.fixed_order_mean_sgd_host(grads, order, 1e-3, theta, stream=s)
    s.synchronize()
    assert np.array_equal(theta.numpy().view(np.uint32), want.view(np.uint32))
    assert np.array_equal(dev.cpu().numpy().view(np.uint32), want.view(np.uint32))
