"""A verifiable data-parallel training step on one GPU, every step a library
call: contributors' gradients through a decoder model, the fixed-order
aggregation, the update and the commitment.

"Zoo Per-LLM Chain Soundness" §2 (Definition "Aggregation rule": the average of
the contributors' gradients; Lemma "Order independence within a batch"), §5
("Ordering subroutine": contributors sorted by DID bytes, the left fold;
"Update step": theta_t = theta_{t-1} - eta * gbar_t), §1 and §6 (the model
state committed as a Merkle root); "Verde与RepOps" §4.3 (Llama-style training
as the workload).

theta is one flat float32 vector holding every layer's weights, each at a
16-byte-aligned offset in a fixed order (the gaps stay +0); the Merkle root
commits exactly its bytes.  A contributor's gradient is a flat vector of the
same layout: forward through the layers keeping their activations, then the
backward pass from the contributor's upstream gradient.  A step sorts the
contributors' DIDs, folds their gradients in that order into the mean, applies
SGD to theta in place and returns the root of the new theta -- the same bits
whatever order the gradients were computed in.
"""
import torch

from . import decoder, fixed_order_mean_sgd, merkle_sha256, sort_ids

def layout(cfg: decoder.DecoderConfig, layers: int):
    """[(layer, key, offset, shape)] and the total length of theta: layer by
    layer, each layer's weights in `decoder.weight_shapes` order, every tensor
    starting at a multiple of 4 elements (16 bytes: TMA-describable)."""
    out, off = [], 0
    shapes = decoder.weight_shapes(cfg)
    for layer in range(layers):
        for key, shape in shapes.items():
            n = 1
            for s in shape:
                n *= s
            out.append((layer, key, off, shape))
            off += (n + 3) // 4 * 4
    return out, off


class Model:
    """`layers` decoder layers whose weights are views into one flat theta."""

    def __init__(self, cfg: decoder.DecoderConfig, layers: int, device, seed: int = 0):
        self.cfg, self.layers = cfg, layers
        self.slots, n = layout(cfg, layers)
        self.theta = torch.zeros(n, dtype=torch.float32, device=device)
        self.weights = self.views(self.theta)
        for layer in range(layers):
            init = decoder.init_weights(cfg, seed + layer, device)
            for key, v in init.items():
                self.weights[layer][key].copy_(v)

    def views(self, flat):
        """Per layer, {key: view} of a flat buffer with theta's layout."""
        vs = [{} for _ in range(self.layers)]
        for layer, key, off, shape in self.slots:
            n = 1
            for s in shape:
                n *= s
            vs[layer][key] = flat[off:off + n].view(shape)
        return vs

    def gradient_buffer(self):
        """A flat gradient vector (its alignment gaps stay +0)."""
        return torch.zeros_like(self.theta)


class Workspace:
    """Buffers one contributor's forward and backward reuse."""

    def __init__(self, model: Model, tokens: int, device):
        cfg = model.cfg
        self.saved = [decoder.activations(cfg, tokens, device) for _ in range(model.layers)]
        self.fwd = decoder.workspace(cfg, tokens, device)
        self.bwd = decoder.backward_workspace(cfg, tokens, device)
        self.h = torch.empty(tokens, cfg.d, dtype=torch.float32, device=device)
        self.d = torch.empty(tokens, cfg.d, dtype=torch.float32, device=device)


def contributor_gradient(model: Model, x, dy, grad_flat, ws: Workspace):
    """grad_flat <- the gradient of the model's parameters for input x and
    upstream gradient dy (both T x d); returns grad_flat."""
    cfg = model.cfg
    ws.h.copy_(x)
    for layer in range(model.layers):
        decoder.forward(ws.h, model.weights[layer], cfg, work=ws.fwd, save=ws.saved[layer])
    gviews = model.views(grad_flat)
    ws.d.copy_(dy)
    d = ws.d
    for layer in reversed(range(model.layers)):
        d, _ = decoder.backward(d, model.weights[layer], cfg, ws.saved[layer], work=ws.bwd, grads=gviews[layer])
    return grad_flat


def train_step(model: Model, contributions, eta: float, ws: Workspace, grads=None):
    """contributions: [(did bytes, x, dy)], in any order.  Computes every
    contributor's gradient, folds them in DID order into the mean, applies
    SGD to theta in place and returns (root of the new theta, the order)."""
    if grads is None:
        grads = [model.gradient_buffer() for _ in contributions]
    for (did, x, dy), g in zip(contributions, grads):
        contributor_gradient(model, x, dy, g, ws)
    order = sort_ids([did for did, _, _ in contributions])
    fixed_order_mean_sgd(grads, order, eta, model.theta)
    return merkle_sha256(model.theta), order
