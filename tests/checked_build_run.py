"""Test helper: one set of hot-path workloads through the library's binding,
run once on the release library and once -- in a child process -- on the
access-checking build (librepops_debug.so), whose kernels test every global
access against its buffer's span.  The two must give the same bytes, and the
checked run must report no skipped access (repops_device_status).

Usage as a child: python tests/checked_build_run.py <checked .so> <out .npz>
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEV = "cuda:0"


def workloads(rp):
    """Name -> host array of every result; raises if a kernel reported a
    skipped access or a timed-out wait."""
    import torch
    from verifiable_repops_gemm_gb300 import inputs
    out = {}

    def done(name, t):
        torch.cuda.synchronize()
        st = rp.device_status()
        if st != 0:
            raise RuntimeError("%s: device status %d" % (name, st))
        out[name] = t.detach().cpu().numpy().copy()

    # GEMM: the small-output kernel, every configuration with both loaders and
    # every storage layout on ragged shapes, the chained split, the repacked
    # large path, unaligned operands, a batched product with an epilogue
    A = inputs.normal((130, 301), 1.0, 1, DEV)
    B = inputs.normal((301, 67), 1.0, 2, DEV)
    done("small", rp.gemm(A, B))
    A = inputs.normal((300, 1000), 1.0, 3, DEV)
    B = inputs.normal((1000, 260), 1.0, 4, DEV)
    for cfg in range(rp.gemm_config_count()):
        for ta in (False, True):
            for tb in (False, True):
                Aop = A.t().contiguous().t() if ta else A
                Bop = B.t().contiguous().t() if tb else B
                for loader in (rp.LOADER_TMA, rp.LOADER_CPASYNC):
                    done("gemm_c%d_l%d_%d%d" % (cfg, loader, ta, tb), rp.gemm(Aop, Bop, config=cfg, loader=loader))
                done("chained_c%d_%d%d" % (cfg, ta, tb), rp.gemm_chained(Aop, Bop, config=cfg, workers=3))
    n = 1601
    A = inputs.normal((n, n), 1.0, 5, DEV)
    B = inputs.normal((n, n), 1.0, 6, DEV)
    done("repacked", rp.gemm(A, B))
    done("chained_auto", rp.gemm(inputs.normal((2048, 2048), 1.0, 7, DEV), inputs.normal((2048, 2048), 1.0, 8, DEV)))
    base = inputs.normal((131 * 80 + 1,), 1.0, 9, DEV)
    Au = base[1:1 + 131 * 80].view(131, 80)[:, :75]
    Bu = inputs.normal((75, 97), 1.0, 10, DEV)
    Cbuf = torch.zeros((131, 104), device=DEV)
    rp.gemm(Au, Bu, out=Cbuf[:, 1:98])
    done("unaligned", Cbuf)
    Ab = inputs.normal((3, 70, 90), 1.0, 11, DEV)
    Bb = inputs.normal((3, 90, 50), 1.0, 12, DEV)
    bias = inputs.normal((50,), 1.0, 13, DEV)
    R = inputs.normal((3, 70, 50), 1.0, 14, DEV)
    done("batched", rp.gemm_batched(Ab, Bb, bias=bias, residual=R, alpha=0.5))
    # mean + SGD: aligned, unaligned views, bfloat16 gradients
    for name, nC, n, off in (("mean", 16, 100003, 0), ("mean_unaligned", 5, 100003, 1)):
        gs = [inputs.normal((n + 4,), 1e-2, 20 + r, DEV)[off:off + n] for r in range(nC)]
        th = inputs.normal((n,), 0.02, 19, DEV)
        rp.fixed_order_mean_sgd(gs, list(range(nC))[::-1], 1e-3, th)
        done(name, th)
    gs = [inputs.normal((4099,), 1e-2, 30 + r, DEV).to(torch.bfloat16) for r in range(3)]
    th = inputs.normal((4099,), 0.02, 29, DEV)
    rp.fixed_order_mean_sgd(gs, [2, 0, 1], 1e-3, th)
    done("mean_bf16", th)
    # Merkle: several reduce passes, a ragged last leaf, the stored tree
    T = inputs.normal(((700 * 128 * 4096 + 333) // 4 + 1,), 0.02, 40, DEV)
    done("merkle", rp.merkle_sha256(T.view(torch.uint8)[:700 * 128 * 4096 + 333]))
    t = inputs.normal((1000 * 1024 + 5,), 0.02, 41, DEV)
    tree, root = rp.merkle_tree(t)
    done("merkle_tree", tree)
    done("merkle_tree_root", root)
    return out


if __name__ == "__main__":
    import verifiable_repops_gemm_gb300 as rp
    from verifiable_repops_gemm_gb300 import _capi
    _capi.load(sys.argv[1])
    # the manifest names the build that produced the bits
    assert "-DREPOPS_DEBUG_BOUNDS" in rp.version(), rp.version()
    res = workloads(rp)
    np.savez(sys.argv[2], **res)
    print("checked run ok:", len(res), "results")
