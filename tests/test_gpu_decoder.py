"""GPU parity of one decoder layer forward (every step a library call) against
the same layer composed from oracle functions.

"Verde与RepOps" §4.3 (Llama-1B training as the workload).  Bar: bit-exact, for
the fused layer (epilogues inside the GEMMs) and the unfused one (epilogues as
separate steps), whose bits must also equal each other.
"""
import numpy as np
import pytest
import torch

from verifiable_repops_gemm_gb300 import decoder

from decoder_oracle import oracle_layer, oracle_layer_with_grads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
SMALL = decoder.DecoderConfig(d=256, heads=4, kv_heads=2, ffn=512, seq_len=64)


@pytest.mark.parametrize("fused,ge", [(True, False), (True, True), (False, False)])
def test_decoder_layer_matches_oracle(rp, orc, fused, ge):
    w = decoder.init_weights(SMALL, 7, DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(8)
    x = torch.randn(2 * SMALL.seq_len, SMALL.d, generator=g, device=DEV)
    want = oracle_layer(orc, x.cpu().numpy(), {k: v.cpu().numpy() for k, v in w.items()}, SMALL)
    y = decoder.forward(x.clone(), w, SMALL, fused=fused, gelu_epilogue=ge)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), want.view(np.uint32))


def test_decoder_layer_is_deterministic_across_calls(rp):
    w = decoder.init_weights(SMALL, 9, DEV)
    x = torch.randn(3 * SMALL.seq_len, SMALL.d, device=DEV)
    a = decoder.forward(x.clone(), w, SMALL)
    b = decoder.forward(x.clone(), w, SMALL, fused=False)
    assert torch.equal(a, b)


def test_decoder_layer_backward_matches_oracle(rp, orc):
    w = decoder.init_weights(SMALL, 11, DEV)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(12)
    T = 2 * SMALL.seq_len
    x = torch.randn(T, SMALL.d, generator=gen, device=DEV)
    dy = torch.randn(T, SMALL.d, generator=gen, device=DEV)
    wh = {k: v.cpu().numpy() for k, v in w.items()}
    y_want, dx_want, g_want = oracle_layer_with_grads(orc, x.cpu().numpy(), wh, SMALL, dy.cpu().numpy())
    saved = decoder.activations(SMALL, T, DEV)
    y = decoder.forward(x.clone(), w, SMALL, save=saved)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y_want.view(np.uint32))
    # the saving forward gives the same bits as the default one
    assert torch.equal(y, decoder.forward(x.clone(), w, SMALL))
    dx, grads = decoder.backward(dy.clone(), w, SMALL, saved)
    assert np.array_equal(dx.cpu().numpy().view(np.uint32), dx_want.view(np.uint32))
    assert set(grads) == set(w)
    for name, gv in grads.items():
        assert np.array_equal(gv.cpu().numpy().view(np.uint32), g_want[name].view(np.uint32)), name
