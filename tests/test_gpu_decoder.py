"""GPU parity of one decoder layer, forward and backward (every step a library
call), against the same layer composed from oracle functions: the Llama-style
layer (rotary embedding, SwiGLU MLP, banded attention GEMMs) and the GeLU
layer.

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
SMALL = decoder.DecoderConfig(d=256, heads=4, kv_heads=2, ffn=512, seq_len=64)              # SwiGLU, rotary
SMALL_GELU = decoder.DecoderConfig(d=256, heads=4, kv_heads=2, ffn=512, seq_len=64, mlp="gelu", rope_base=0.0)
CFGS = {"llama": SMALL, "gelu": SMALL_GELU}


@pytest.mark.parametrize("name,fused,ge", [("llama", True, False), ("llama", False, False), ("gelu", True, False),
                                           ("gelu", True, True), ("gelu", False, False)])
def test_decoder_layer_matches_oracle(rp, orc, name, fused, ge):
    cfg = CFGS[name]
    w = decoder.init_weights(cfg, 7, DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(8)
    x = torch.randn(2 * cfg.seq_len, cfg.d, generator=g, device=DEV)
    want = oracle_layer(orc, x.cpu().numpy(), {k: v.cpu().numpy() for k, v in w.items()}, cfg)
    y = decoder.forward(x.clone(), w, cfg, fused=fused, gelu_epilogue=ge)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("name", sorted(CFGS))
def test_decoder_layer_is_deterministic_across_calls(rp, name):
    cfg = CFGS[name]
    w = decoder.init_weights(cfg, 9, DEV)
    x = torch.randn(3 * cfg.seq_len, cfg.d, device=DEV)
    a = decoder.forward(x.clone(), w, cfg)
    b = decoder.forward(x.clone(), w, cfg, fused=False)
    assert torch.equal(a, b)


@pytest.mark.parametrize("name", sorted(CFGS))
def test_decoder_layer_backward_matches_oracle(rp, orc, name):
    cfg = CFGS[name]
    w = decoder.init_weights(cfg, 11, DEV)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(12)
    T = 2 * cfg.seq_len
    x = torch.randn(T, cfg.d, generator=gen, device=DEV)
    dy = torch.randn(T, cfg.d, generator=gen, device=DEV)
    wh = {k: v.cpu().numpy() for k, v in w.items()}
    y_want, dx_want, g_want = oracle_layer_with_grads(orc, x.cpu().numpy(), wh, cfg, dy.cpu().numpy())
    saved = decoder.activations(cfg, T, DEV)
    y = decoder.forward(x.clone(), w, cfg, save=saved)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y_want.view(np.uint32))
    # the saving forward gives the same bits as the default one
    assert torch.equal(y, decoder.forward(x.clone(), w, cfg))
    dx, grads = decoder.backward(dy.clone(), w, cfg, saved)
    assert np.array_equal(dx.cpu().numpy().view(np.uint32), dx_want.view(np.uint32))
    assert set(grads) == set(w)
    for key, gv in grads.items():
        assert np.array_equal(gv.cpu().numpy().view(np.uint32), g_want[key].view(np.uint32)), key


def test_side_streams_do_not_change_the_bits(rp):
    # the attention's sequences and heads on side streams, on the caller's
    # stream alone, and with one score scratch shared by the sequences
    cfg = SMALL
    T = 3 * cfg.seq_len
    w = decoder.init_weights(cfg, 13, DEV)
    x = torch.randn(T, cfg.d, device=DEV)
    dy = torch.randn(T, cfg.d, device=DEV)
    ws = decoder.workspace(cfg, T, DEV)
    serial = dict(ws, streams=None)
    shared = dict(ws, scores=ws["scores"][:cfg.kv_heads])
    ys = [decoder.forward(x.clone(), w, cfg, work=k) for k in (ws, serial, shared)]
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[0], ys[2])
    outs = []
    for streams in (True, False):
        saved = decoder.activations(cfg, T, DEV)
        bws = decoder.backward_workspace(cfg, T, DEV)
        if not streams:
            bws["streams"] = None
        decoder.forward(x.clone(), w, cfg, work=ws, save=saved)
        outs.append(decoder.backward(dy.clone(), w, cfg, saved, work=bws))
    (dx0, g0), (dx1, g1) = outs
    assert torch.equal(dx0, dx1) and all(torch.equal(g0[k], g1[k]) for k in g0)
