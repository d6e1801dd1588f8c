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
