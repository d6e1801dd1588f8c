"""GPU parity of the stored Merkle tree, inclusion proofs, membership checks
and the step-replay driver against the oracle.

"Verde与RepOps" §2.4 (membership proofs against the checkpoint hash);
"Zoo Per-LLM Chain Soundness" §7 (replay the blocks, then verify H(theta) = m).
Bar: byte-identical trees, proofs, roots and theta.
"""
import numpy as np
import pytest
import torch

from verifiable_repops_gemm_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def dev_bytes(n, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return torch.randint(0, 256, (n,), generator=g, device=DEV, dtype=torch.uint8)


@pytest.mark.parametrize("nleaves,leaf,tail", [(1, 64, 0), (2, 64, 7), (5, 4096, 100), (127, 64, 0),
                                               (128, 64, 1), (129, 64, 0), (1000, 4096, 17),
                                               (70001, 64, 0), (128 * 512 + 3, 64, 9)])
def test_tree_matches_oracle(rp, orc, nleaves, leaf, tail):
    n = nleaves * leaf - tail
    t = dev_bytes(n, nleaves)
    tree, root = rp.merkle_tree(t, leaf)
    torch.cuda.synchronize()
    want = orc.merkle_tree(t.cpu().numpy(), leaf)
    assert np.array_equal(tree.cpu().numpy(), want)
    assert root.cpu().numpy().tobytes() == want[-1].tobytes()
    assert root.cpu().numpy().tobytes() == rp.merkle_sha256(t, leaf).cpu().numpy().tobytes()


@pytest.mark.parametrize("nleaves", [1, 3, 129, 1000, 70001])
def test_proofs_match_oracle_and_verify(rp, orc, nleaves):
    leaf = 64
    n = nleaves * leaf - 5
    t = dev_bytes(n, 7 + nleaves)
    tree, root = rp.merkle_tree(t, leaf)
    host_tree = orc.merkle_tree(t.cpu().numpy(), leaf)
    idx = sorted({0, 1 % nleaves, nleaves // 2, nleaves - 2 if nleaves > 1 else 0, nleaves - 1})
    for i in idx:
        proof = rp.merkle_proof(tree, nleaves, i)
        want = orc.merkle_proof(host_tree, nleaves, i)
        assert np.array_equal(proof.cpu().numpy(), want), i
        lb = t[i * leaf:min((i + 1) * leaf, n)]
        assert int(rp.merkle_verify(lb, nleaves, i, proof, root).item()) == 1
        bad = lb.clone()
        bad[0] ^= 1
        assert int(rp.merkle_verify(bad, nleaves, i, proof, root).item()) == 0
        if proof.shape[0]:
            p2 = proof.clone()
            p2[-1, 3] ^= 0x40
            assert int(rp.merkle_verify(lb, nleaves, i, p2, root).item()) == 0


def test_replay_matches_oracle(rp, orc):
    steps, nC, n = 3, 5, 100003
    theta0 = inputs.normal((n,), 0.02, 400, DEV)
    G = [[inputs.normal((n,), 1e-2, 500 + 10 * t + r, DEV) for r in range(nC)] for t in range(steps)]
    orders = [rp.sort_ids(inputs.contributor_ids(nC, 600 + t)) for t in range(steps)]
    etas = [1e-3, 5e-4, 2.5e-4]
    theta = theta0.clone()
    roots = rp.replay(G, orders, etas, theta, 4096)
    torch.cuda.synchronize()
    th_want, roots_want = orc.replay([[g.cpu().numpy() for g in gs] for gs in G], orders, etas,
                                     theta0.cpu().numpy(), 4096)
    assert np.array_equal(theta.cpu().numpy().view(np.uint32), th_want.view(np.uint32))
    assert [r.tobytes() for r in roots.cpu().numpy()] == roots_want
    # replaying again from the same genesis state commits the same roots
    theta2 = theta0.clone()
    roots2 = rp.replay(G, orders, etas, theta2, 4096)
    assert torch.equal(roots, roots2)
    # a block aggregated in another order commits another state from there on
    theta3 = theta0.clone()
    swapped = [orders[0], orders[1][::-1], orders[2]]
    roots3 = rp.replay(G, swapped, etas, theta3, 4096)
    assert torch.equal(roots3[0], roots[0]) and not torch.equal(roots3[1], roots[1])


@pytest.mark.slow
def test_replay_full_size_block(rp, orc):
    # one block of the 16 x 2^28 workload: theta sampled against the oracle,
    # the committed root against the oracle's root of the same theta bytes
    nC, n = inputs.MEAN_CONTRIBUTORS, inputs.MEAN_LEN
    grads = [inputs.normal((n,), 1e-2, 200 + r, DEV) for r in range(nC)]
    theta = inputs.normal((n,), 0.02, 199, DEV)
    order = rp.sort_ids(inputs.contributor_ids(nC, 200))
    s0 = 12345 * 4096
    before = theta[s0:s0 + 4096].cpu().numpy()
    roots = rp.replay([grads], [order], [1e-3], theta, 4096)
    torch.cuda.synchronize()
    want = orc.mean_sgd([g[s0:s0 + 4096].cpu().numpy() for g in grads], order, 1e-3, before)
    assert np.array_equal(theta[s0:s0 + 4096].cpu().numpy().view(np.uint32), want.view(np.uint32))
    assert roots[0].cpu().numpy().tobytes() == orc.merkle_root(theta.cpu().numpy(), 4096)


def test_verify_on_a_side_stream(rp):
    # the result is written by the kernel on the caller's stream only
    t = dev_bytes(300 * 4096 + 11, 77)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        tree, root = rp.merkle_tree(t, 4096, stream=s)
        proof = rp.merkle_proof(tree, 301, 299, stream=s)
        ok = rp.merkle_verify(t[299 * 4096:300 * 4096], 301, 299, proof, root, stream=s)
    s.synchronize()
    assert int(ok.item()) == 1
