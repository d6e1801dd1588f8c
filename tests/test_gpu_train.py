"""GPU parity of the verifiable training step (contributors' gradients through a
decoder model, the fixed-order mean, SGD, the Merkle root of theta) against
the same step composed from oracle functions, and its order independence.

"Zoo Per-LLM Chain Soundness" §2 (Aggregation rule; Lemma "Order independence
within a batch"), §5 (Ordering subroutine, Update step), §1/§6 (the state
root); "Verde与RepOps" §4.3.  Bar: theta bit-exact and the root byte-exact;
the same root for every order in which the contributions arrive.
"""
import itertools

import numpy as np
import pytest
import torch

from verifiable_repops_gemm_gb300 import decoder, train

from decoder_oracle import oracle_layer, oracle_layer_with_grads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
SMALL = decoder.DecoderConfig(d=256, heads=4, kv_heads=2, ffn=512, seq_len=64)
DIDS = [b"did:zoo:charlie", b"did:zoo:alice", b"did:zoo:bob"]


def contributions(seed, tokens):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return [(did, torch.randn(tokens, SMALL.d, generator=g, device=DEV),
             torch.randn(tokens, SMALL.d, generator=g, device=DEV) * 1e-2) for did in DIDS]


def oracle_step(orc, model, contribs, eta):
    """Per contributor: the layers' forward, then their backward from dy, with
    the gradients laid out like theta; the mean + SGD in DID order; the root."""
    layers = model.layers
    w = [{k: v.cpu().numpy() for k, v in lw.items()} for lw in model.weights]
    grads = []
    for _, x, dy in contribs:
        xs = [x.cpu().numpy()]
        for layer in range(layers - 1):
            xs.append(oracle_layer(orc, xs[-1], w[layer], SMALL))
        flat = np.zeros(model.theta.numel(), np.float32)
        d = dy.cpu().numpy()
        for layer in reversed(range(layers)):
            _, d, g = oracle_layer_with_grads(orc, xs[layer], w[layer], SMALL, d)
            for lay, key, off, shape in model.slots:
                if lay == layer:
                    flat[off:off + g[key].size] = g[key].reshape(-1)
        grads.append(flat)
    order = orc.sort_ids([did for did, _, _ in contribs])
    theta = orc.mean_sgd(grads, order, eta, model.theta.cpu().numpy())
    return theta, orc.merkle_root(theta.tobytes())


def test_training_step_matches_oracle(rp, orc):
    model = train.Model(SMALL, 2, DEV, seed=20)
    T = 2 * SMALL.seq_len
    contribs = contributions(21, T)
    want_theta, want_root = oracle_step(orc, model, contribs, 1e-3)
    ws = train.Workspace(model, T, DEV)
    root, order = train.train_step(model, contribs, 1e-3, ws)
    assert order == [1, 2, 0]                                  # alice, bob, charlie
    assert np.array_equal(model.theta.cpu().numpy().view(np.uint32), want_theta.view(np.uint32))
    assert bytes(root.cpu().numpy()) == want_root


def test_training_step_is_order_independent(rp):
    T = 2 * SMALL.seq_len
    contribs = contributions(30, T)
    roots = set()
    for perm in itertools.permutations(range(len(contribs))):
        model = train.Model(SMALL, 2, DEV, seed=31)
        ws = train.Workspace(model, T, DEV)
        root, _ = train.train_step(model, [contribs[i] for i in perm], 1e-3, ws)
        roots.add(bytes(root.cpu().numpy()))
    assert len(roots) == 1


def test_two_steps_chain_roots(rp):
    # each step commits the state the next one starts from: replaying the same
    # blocks from the same start gives the same chain of roots
    T = 2 * SMALL.seq_len
    chains = []
    for _ in range(2):
        model = train.Model(SMALL, 1, DEV, seed=40)
        ws = train.Workspace(model, T, DEV)
        chain = [bytes(train.train_step(model, contributions(41 + step, T), 1e-3, ws)[0].cpu().numpy())
                 for step in range(2)]
        chains.append(chain)
    assert chains[0] == chains[1] and chains[0][0] != chains[0][1]
