"""ctypes declarations for librepops (include/repops.h).

Argument marshalling only: every operation runs in the library's CUDA kernels.
The library must have been built (``verifiable_repops_gemm_gb300.build``);
loading fails loudly when it is missing -- there is no fallback path.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "librepops.so")

OK = 0
ERR_INVALID_ARG = -1
ERR_ALIAS = -2
ERR_ORDER = -3
ERR_CUDA = -4
ERR_TIMEOUT = -5
ERR_ALLOC = -6
ERR_UNSUPPORTED = -7

LOADER_AUTO = 0
LOADER_TMA = 1
LOADER_CPASYNC = 2
LOADER_DIRECT = 3

MEAN_MAX_CONTRIBUTORS = 1024

# name -> (restype, argtypes); the full exported surface of include/repops.h
_i32, _i64, _u32, _u64 = ctypes.c_int, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64
_vp, _f32, _cs = ctypes.c_void_p, ctypes.c_float, ctypes.c_char_p
SIGNATURES = {
    "repops_version": (_cs, []),
    "repops_status_string": (_cs, [_i32]),
    "repops_last_cuda_error": (_i32, []),
    "repops_device_status": (_i32, [_vp, _vp]),
    "repops_scratch_set_keep_bytes": (_i32, [ctypes.c_uint64]),
    "repops_scratch_release": (_i32, []),
    "repops_scratch_reserved_bytes": (_i32, [_vp]),
    "repops_host_alloc": (_i32, [_u64, _vp]),
    "repops_host_free": (_i32, [_vp]),
    "repops_set_thread_status_word": (_i32, [_vp]),
    "repops_gemm_f32": (_i32, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp]),
    "repops_gemm_f32_ex": (_i32, [_i32, _i32, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp]),
    "repops_gemm_workspace_bytes": (_u64, [_i32, _i32, _i64, _i64, _i64, _vp, _i64, _vp, _i64]),
    "repops_gemm_f32_ws": (_i32, [_i32, _i32, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _u64,
                                  _vp]),
    "repops_gemm_f32_config": (_i32, [_i32, _i32, _i32, _i32, _i64, _i64, _i64, _vp, _i64, _vp, _i64,
                                      _vp, _i64, _vp]),
    "repops_gemm_f32_chained": (_i32, [_i32, _i32, _i32, _i32, _i64, _i64, _i64, _vp, _i64, _vp, _i64,
                                       _vp, _i64, _vp]),
    "repops_attention_causal_f32": (_i32, [_i64, _i64, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _f32,
                                           _vp, _i64, _vp, _vp]),
    "repops_fixed_order_mean_sgd_host": (_i32, [_i32, _i64, _vp, _vp, _f32, _vp, _vp]),
    "repops_merkle_sha256_host": (_i32, [_vp, _u64, _u32, _vp, _vp]),
    "repops_gemm_config_count": (_i32, []),
    "repops_gemm_config_info": (_i32, [_i32, _vp, _vp, _vp, _vp, _vp]),
    "repops_gemm_auto_config": (_i32, [_i64, _i64, _i64]),
    "repops_gemm_small_output": (_i32, [_i64, _i64, _i64]),
    "repops_gemm_auto_chained": (_i32, [_i64, _i64, _i64]),
    "repops_sort_ids": (_i32, [_i32, _vp, _vp, _vp, _vp]),
    "repops_fixed_order_mean_sgd": (_i32, [_i32, _i64, _vp, _vp, _f32, _vp, _vp]),
    "repops_merkle_sha256": (_i32, [_vp, _u64, _u32, _vp, _vp]),
    "repops_merkle_workspace_bytes": (_u64, [_u64, _u32]),
    "repops_merkle_sha256_ws": (_i32, [_vp, _u64, _u32, _vp, _vp, _u64, _vp]),
    "repops_merkle_sha256_noalloc": (_i32, [_vp, _u64, _u32, _vp, _vp]),
    "repops_sha256_rate_probe": (_i32, [_u32, _u32, _vp, _vp]),
    "repops_merkle_tree_bytes": (_u64, [_u64, _u32]),
    "repops_merkle_tree_sha256": (_i32, [_vp, _u64, _u32, _vp, _u64, _vp, _vp]),
    "repops_merkle_proof_steps": (_i32, [_u64, _u64]),
    "repops_merkle_proof": (_i32, [_vp, _u64, _u64, _vp, _vp]),
    "repops_merkle_verify": (_i32, [_vp, _u64, _u64, _u64, _vp, _vp, _vp, _vp]),
    "repops_replay_mean_sgd_commit": (_i32, [_i32, _i32, _i64, _vp, _vp, _vp, _vp, _u32, _vp, _vp]),
    "repops_softmax_rows_f32": (_i32, [_i64, _i64, _vp, _i64, _vp, _i64, _vp]),
    "repops_layernorm_rows_f32": (_i32, [_i64, _i64, _vp, _i64, _vp, _vp, _f32, _vp, _i64, _vp]),
    "repops_rmsnorm_rows_f32": (_i32, [_i64, _i64, _vp, _i64, _vp, _f32, _vp, _i64, _vp]),
    "repops_gelu_f32": (_i32, [_i64, _vp, _vp, _vp]),
    "repops_fixed_order_mean_sgd_typed": (_i32, [_i32, _i64, _vp, _i32, _vp, ctypes.c_float, _vp, _vp]),
    "repops_convert": (_i32, [_i64, _vp, _i32, _vp, _i32, _vp]),
    "repops_gemm_typed": (_i32, [_i32, _i32, _i32, _i32, _i64, _i64, _i64, _vp, _i32, _i64, _vp, _i32, _i64,
                                 _vp, _i32, _i64, _vp]),
    "repops_rolling_hash_u32": (_i32, [_i64, _i64, _vp, _i64, _i64, _vp, _i64, _vp]),
    "repops_gemm_config_occupancy": (_i32, [_i32]),
    "repops_gemm_f32_host": (_i32, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp]),
    "repops_colsum_f32": (_i32, [_i64, _i64, _vp, _i64, _vp, _vp]),
    "repops_gelu_backward_f32": (_i32, [_i64, _vp, _vp, _vp, _vp]),
    "repops_rmsnorm_backward_f32": (_i32, [_i64, _i64, _vp, _i64, _vp, ctypes.c_float, _vp, _i64, _vp, _i64,
                                           _vp, _i64, _vp, _i64, _vp]),
    "repops_softmax_backward_f32": (_i32, [_i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp]),
    "repops_softmax_backward_causal_f32": (_i32, [_i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _i64, _i64,
                                                  _vp]),
    "repops_swiglu_f32": (_i32, [_i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp]),
    "repops_swiglu_backward_f32": (_i32, [_i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64,
                                          _vp]),
    "repops_rope_frequencies_f32": (_i32, [_i64, ctypes.c_float, _vp, _vp]),
    "repops_rope_table_f32": (_i32, [_i64, _i64, _vp, _vp, _vp, _vp]),
    "repops_rope_f32": (_i32, [_i64, _i64, _i64, _vp, _i64, _vp, _vp, _i64, _i64, _i64, _i32, _vp]),
    "repops_selftest_bounded_wait": (_i32, [_i64, _vp]),
    "repops_selftest_bounded_flag_wait": (_i32, [_i64, _vp]),
    "repops_softmax_rows_causal_f32": (_i32, [_i64, _i64, _vp, _i64, _vp, _i64, _i64, _i64, _vp]),
    "repops_gemm_f32_batched": (_i32, [_i32, _i32, _i32, _i32, _i64, _i64, _i64, _i64,
                                       _vp, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _i64,
                                       ctypes.c_float, _vp, _i32, _vp, _i64, _i64, _i64, _i64, _i64, _i64,
                                       _vp]),
}

ACT_NONE, ACT_GELU = 0, 1
TYPE_F32, TYPE_F16, TYPE_BF16 = 0, 1, 2

MERKLE_NOALLOC_SCRATCH_BYTES = 1 << 20

_lib = None


class RepopsError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        msg = "%s failed: %s (%d)" % (what, status_string(code), code)
        if code == ERR_CUDA and _lib is not None:
            msg += ", cudaError %d" % _lib.repops_last_cuda_error()
        super().__init__(msg)


def load(path: str = None) -> ctypes.CDLL:
    """Loads librepops.so (once).  Raises if it has not been built.

    Without `path`, the environment variable REPOPS_LIBRARY, when set, names
    the library file to load instead of the in-tree release build -- e.g. the
    access-checking build _build_checked/librepops_debug.so, to run a whole
    program or test suite with every hot-path global access checked."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or os.environ.get("REPOPS_LIBRARY") or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(
            "librepops.so is not built (%s); run `python -c \"import __graft_entry__ as g; g.build()\"` "
            "or verifiable_repops_gemm_gb300.build.build()" % path)
    L = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def status_string(code: int) -> str:
    if _lib is None:
        return "status %d" % code
    return _lib.repops_status_string(code).decode()


def check(code: int, what: str) -> None:
    if code != OK:
        raise RepopsError(code, what)
