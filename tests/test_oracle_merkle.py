"""Pins the SHA-256 and Merkle oracle.

SHA-256 is checked against Python's hashlib, run as a black box.  The tree
rule (leaf = SHA256(0x00||bytes), node = SHA256(0x01||L||R), level by level,
unpaired last node promoted) is checked against a recursive restatement written
here on top of hashlib.  Sources: "Zoo Per-LLM Chain Soundness" §1 (batch hash
is a Merkle root), §6 (bytes32 roots); "Verde与RepOps" §2.3.2 (checkpoint hash
is a Merkle tree over node hashes).
"""
import hashlib
from decimal import Decimal, getcontext

import numpy as np
import pytest


def H(b: bytes) -> bytes:
    return hashlib.sha256(b).digest()


def ref_root(data: bytes, leaf: int) -> bytes:
    """Recursive statement: the node covering leaves [lo, hi) at the level where
    it sits; an unpaired node rises unchanged."""
    n = (len(data) + leaf - 1) // leaf
    leaves = [H(b"\x00" + data[i * leaf:(i + 1) * leaf]) for i in range(n)]

    def node(lo, span):
        # span = 2^level leaves; the node is hashed from its two halves if the
        # right half holds any leaf, else it is the left half carried up
        if span == 1:
            return leaves[lo]
        half = span // 2
        if lo + half >= n:
            return node(lo, half)
        return H(b"\x01" + node(lo, half) + node(lo + half, half))

    span = 1
    while span < n:
        span *= 2
    return node(0, span)


def test_sha256_matches_hashlib(orc):
    rng = np.random.default_rng(0)
    for n in list(range(0, 301)) + [4096, 4097, 4159, 4160, 10000]:
        msg = rng.bytes(n)
        assert orc.sha256(msg) == H(msg), n


def test_sha256_constants_from_primes(orc):
    # independent derivation in high-precision decimal arithmetic
    K, H0 = orc.sha256_constants()
    getcontext().prec = 60
    primes = [p for p in range(2, 400) if all(p % d for d in range(2, int(p ** 0.5) + 1))][:64]
    for t, p in enumerate(primes):
        r = Decimal(p) ** (Decimal(1) / Decimal(3))
        assert K[t] == int((r - int(r)) * (1 << 32)), t
    for i, p in enumerate(primes[:8]):
        r = Decimal(p).sqrt()
        assert H0[i] == int((r - int(r)) * (1 << 32)), i


@pytest.mark.parametrize("nleaves", [1, 2, 3, 4, 5, 6, 7, 8, 9, 16, 17, 33])
@pytest.mark.parametrize("leaf", [64, 4096])
def test_merkle_root_matches_recursive_definition(orc, nleaves, leaf):
    rng = np.random.default_rng(nleaves * 7 + leaf)
    for tail in (0, 1, leaf // 2 + 3):
        n = nleaves * leaf - (tail if nleaves > 0 and tail < leaf else 0)
        data = rng.bytes(n)
        assert orc.merkle_root(data, leaf) == ref_root(data, leaf), (n, tail)


def test_closed_forms(orc):
    rng = np.random.default_rng(1)
    d = rng.bytes(3 * 64)
    l0, l1, l2 = (H(b"\x00" + d[i * 64:(i + 1) * 64]) for i in range(3))
    assert orc.merkle_root(d[:64], 64) == l0
    assert orc.merkle_root(d[:128], 64) == H(b"\x01" + l0 + l1)
    assert orc.merkle_root(d, 64) == H(b"\x01" + H(b"\x01" + l0 + l1) + l2)
    # a short last leaf is hashed as it is
    assert orc.merkle_root(d[:100], 64) == H(b"\x01" + l0 + H(b"\x00" + d[64:100]))


def test_ragged_gemm_output_leaf_count(orc):
    # 4097 x 1023 fp32 = 16,764,924 bytes -> 4093 leaves, the last one 4092 bytes
    rng = np.random.default_rng(2)
    data = rng.bytes(4097 * 1023 * 4)
    leaves = orc.merkle_leaves(data, 4096)
    assert leaves.shape == (4093, 32)
    assert leaves[-1].tobytes() == H(b"\x00" + data[4092 * 4096:])
    assert orc.merkle_root(data, 4096) == ref_root(data, 4096)


def test_aligned_subtree_root_is_the_level_node(orc):
    # the node at level m, index j covers leaves [j*2^m, (j+1)*2^m); hashing
    # that slice alone gives the same digest
    rng = np.random.default_rng(3)
    data = rng.bytes(37 * 64 + 10)
    leaves = orc.merkle_leaves(data, 64)
    for m in (1, 2, 3, 4):
        span = 1 << m
        for j in range((len(leaves) + span - 1) // span):
            sub = data[j * span * 64:(j + 1) * span * 64]
            assert orc.merkle_root(sub, 64) == orc.merkle_reduce(leaves[j * span:(j + 1) * span])


def test_empty_input_rejected(orc):
    with pytest.raises(ValueError):
        orc.merkle_root(b"", 4096)


def ref_node(data: bytes, leaf: int, level: int, j: int) -> bytes:
    """Node j of `level`: it covers leaves [j*2^level, (j+1)*2^level); hashed
    from its two children when the right child covers any leaf, else the left
    child carried up."""
    n = (len(data) + leaf - 1) // leaf
    if level == 0:
        return H(b"\x00" + data[j * leaf:(j + 1) * leaf])
    left = ref_node(data, leaf, level - 1, 2 * j)
    if (2 * j + 1) << (level - 1) >= n:
        return left
    return H(b"\x01" + left + ref_node(data, leaf, level - 1, 2 * j + 1))


def ref_proof(data: bytes, leaf: int, i: int):
    n = (len(data) + leaf - 1) // leaf
    sibs, level, count = [], 0, n
    while count > 1:
        j = i >> level
        if j % 2 == 1:
            sibs.append(ref_node(data, leaf, level, j - 1))
        elif j + 1 < count:
            sibs.append(ref_node(data, leaf, level, j + 1))
        level += 1
        count = (count + 1) // 2
    return sibs


@pytest.mark.parametrize("nleaves", [1, 2, 3, 5, 6, 7, 8, 9, 13, 16, 17, 33])
def test_tree_levels_match_recursive_definition(orc, nleaves):
    rng = np.random.default_rng(100 + nleaves)
    data = rng.bytes(nleaves * 64 - 5)
    tree = orc.merkle_tree(data, 64)
    off, count, level = 0, nleaves, 0
    while True:
        for j in range(count):
            assert tree[off + j].tobytes() == ref_node(data, 64, level, j), (level, j)
        if count == 1:
            break
        off += count
        count = (count + 1) // 2
        level += 1
    assert off + 1 == tree.shape[0]
    assert tree[-1].tobytes() == orc.merkle_root(data, 64)


@pytest.mark.parametrize("nleaves", [1, 2, 3, 4, 5, 7, 11, 17, 33])
def test_proofs_match_independent_paths_and_verify(orc, nleaves):
    rng = np.random.default_rng(200 + nleaves)
    data = rng.bytes(nleaves * 64 - 3)
    tree = orc.merkle_tree(data, 64)
    root = tree[-1].tobytes()
    for i in range(nleaves):
        proof = orc.merkle_proof(tree, nleaves, i)
        assert [p.tobytes() for p in proof] == ref_proof(data, 64, i)
        leaf_bytes = data[i * 64:(i + 1) * 64]
        assert orc.merkle_verify(leaf_bytes, nleaves, i, proof, root)
        # tampering anywhere breaks membership
        if len(leaf_bytes):
            bad = bytearray(leaf_bytes)
            bad[0] ^= 1
            assert not orc.merkle_verify(bytes(bad), nleaves, i, proof, root)
        for s in range(proof.shape[0]):
            p2 = proof.copy()
            p2[s, 7] ^= 0x80
            assert not orc.merkle_verify(leaf_bytes, nleaves, i, p2, root)
        if nleaves > 1:
            other = (i + 1) % nleaves
            assert not orc.merkle_verify(leaf_bytes, nleaves, other, proof, root) or \
                data[other * 64:(other + 1) * 64] == leaf_bytes
        assert not orc.merkle_verify(leaf_bytes, nleaves, i, proof[:-1], root) or proof.shape[0] == 0


def test_three_leaf_proof_closed_form(orc):
    rng = np.random.default_rng(9)
    d = rng.bytes(3 * 64)
    l0, l1, l2 = (H(b"\x00" + d[i * 64:(i + 1) * 64]) for i in range(3))
    tree = orc.merkle_tree(d, 64)
    # leaf 2 is unpaired at level 0, then pairs with H(l0||l1) at level 1
    assert [p.tobytes() for p in orc.merkle_proof(tree, 3, 2)] == [H(b"\x01" + l0 + l1)]
    assert [p.tobytes() for p in orc.merkle_proof(tree, 3, 0)] == [l1, l2]


def test_replay_recomputes_the_committed_roots(orc):
    # "Zoo Per-LLM Chain Soundness" §7: replay the blocks in order from the
    # initial state, then H(theta) must equal the recorded model root
    rng = np.random.default_rng(5)
    n, steps, k = 3000, 3, 4
    theta0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    G = [[(rng.standard_normal(n) * 1e-2).astype(np.float32) for _ in range(k)] for _ in range(steps)]
    orders = [list(rng.permutation(k)) for _ in range(steps)]
    etas = [1e-3, 5e-4, 2.5e-4]
    th, roots = orc.replay(G, orders, etas, theta0, 1024)
    th_manual = theta0
    for t in range(steps):
        th_manual = orc.mean_sgd(G[t], orders[t], etas[t], th_manual)
        assert roots[t] == orc.merkle_root(th_manual, 1024)
    assert np.array_equal(th.view(np.uint32), th_manual.view(np.uint32))
    # a block replayed with another contributor order commits another state
    swapped = [orders[0], orders[1][::-1], orders[2]]
    _, roots2 = orc.replay(G, swapped, etas, theta0, 1024)
    assert roots2[0] == roots[0] and roots2[1] != roots[1] and roots2[2] != roots[2]
