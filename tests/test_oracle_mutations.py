"""The pins catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of oracle/repops_oracle.c, builds it
with the oracle's own flags, and runs the pin suite (tests/test_oracle_*.py)
against it in a subprocess (several at a time): the suite must fail.  The unmodified source must
pass.  Nothing here touches the CUDA library.
"""
import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "repops_oracle.c")
PINS = [os.path.join(ROOT, "tests", f) for f in
        ("test_oracle_gemm.py", "test_oracle_mean.py", "test_oracle_merkle.py", "test_oracle_rowops.py",
         "test_oracle_epilogue.py", "test_oracle_halfstore.py", "test_oracle_backward.py",
         "test_oracle_llama.py")]

MUTATIONS = {
    "gemm: fused multiply-add": (
        "float p = a * b;        /* product, rounded to binary32 */\n                sum = sum + p; ",
        "sum = __builtin_fmaf(a, b, sum); "),
    "gemm: k in decreasing order": (
        "for (int64_t k = 0; k < K; ++k) {", "for (int64_t k = K - 1; k >= 0; --k) {"),
    "gemm: sum starts at -0": ("float sum = 0.0f;", "float sum = -0.0f;"),
    "gemm: B indexed as if transposed": (
        "float b = transB ? B[j * ldb + k] : B[k * ldb + j];",
        "float b = transB ? B[k * ldb + j] : B[j * ldb + k];"),
    "gemm: product in double": ("float p = a * b; ", "float p = (float)((double)a * (double)b + 1e-30); "),
    "mean: fold starts at zero": (
        "float S = grads[order[0]][e];\n        for (int r = 1; r < nC; ++r) {",
        "float S = 0.0f;\n        for (int r = 0; r < nC; ++r) {"),
    "mean: multiply by the reciprocal": ("float gbar = S / count;", "float gbar = S * (1.0f / count);"),
    "mean: SGD adds the step": ("theta[e] = theta[e] - step;", "theta[e] = theta[e] + step;"),
    "mean: contributor order ignored": ("S = S + grads[order[r]][e];", "S = S + grads[r][e];"),
    "sort: signed byte comparison": ("if (a[i] != b[i]) return a[i] < b[i];",
                                     "if (a[i] != b[i]) return (signed char)a[i] < (signed char)b[i];"),
    "sort: longer prefix first": ("    return la < lb;\n}", "    return la > lb;\n}"),
    "sha256: rotate by 7 in Sigma1": ("uint32_t S1 = rotr32(e, 6)", "uint32_t S1 = rotr32(e, 7)"),
    "sha256: length in bytes, not bits": ("uint64_t bits = c->total * 8u;", "uint64_t bits = c->total;"),
    "merkle: node prefix 0x02": ("msg[0] = 0x01;", "msg[0] = 0x02;"),
    "merkle: no leaf prefix": ("osha_update(&c, &prefix, 1);\n    osha_update(&c, data + start, end - start);",
                               "osha_update(&c, data + start, end - start);"),
    "merkle: unpaired node hashed with itself": (
        "memmove(level + 32 * next, level + 32 * (count - 1), 32);",
        "merkle_node(level + 32 * (count - 1), level + 32 * (count - 1), level + 32 * next);"),
    "merkle: leaves one byte short": ("uint64_t end = start + leaf;", "uint64_t end = start + leaf - 1;"),
    "proof: sibling side swapped": ("merkle_node(proof + 32 * used++, h, t);", "merkle_node(h, proof + 32 * used++, t);"),
    "rows: runs of 16": ("#define ROW_RUN 32", "#define ROW_RUN 16"),
    "exp: degree-6 polynomial": ("float p = 1.98412701e-04f;          /* 1/5040 */\n    p = p * r + 1.38888892e-03f;",
                                 "float p = 1.38888892e-03f;"),
    "exp: one-part ln 2": ("    r = r - kf * ln2_lo;\n", ""),
    "erfc: final factor t dropped": ("return t * oracle_exp(arg);", "return oracle_exp(arg);"),
    "gelu: branches swapped": ("z >= 0.0f ? 2.0f - oracle_erfc_pos(z) : oracle_erfc_pos(-z)",
                               "z >= 0.0f ? oracle_erfc_pos(z) : 2.0f - oracle_erfc_pos(-z)"),
    "softmax: no max subtraction": ("e[j] = oracle_exp(xr[j] - m);", "e[j] = oracle_exp(xr[j]);"),
    "layernorm: variance over n - 1": ("float var = tree_reduce(v, cols, 0) / n;",
                                       "float var = tree_reduce(v, cols, 0) / (n - 1.0f);"),
    "rmsnorm: divide each element": ("y[i * ldy + j] = (xr[j] * inv) * gamma[j];",
                                     "y[i * ldy + j] = (xr[j] / sqrtf(ms + eps)) * gamma[j];"),
    "softmax: divide each element": ("y[i * ldy + j] = e[j] * inv;", "y[i * ldy + j] = e[j] / s;"),
    "epilogue: bias before alpha": ("float y = alpha * acc;\n                if (bias) y = y + bias[j];",
                                    "float y = acc;\n                if (bias) y = y + bias[j];\n"
                                    "                y = alpha * y;"),
    "batched: k in decreasing order": ("for (int64_t kk = k0; kk < k1; ++kk) {",
                                       "for (int64_t kk = k1 - 1; kk >= k0; --kk) {"),
    "batched: acc starts at -0": ("float acc = 0.0f;", "float acc = -0.0f;"),
    "batched: fused multiply-add": ("float p = a * bv;\n                    acc = acc + p;",
                                    "acc = __builtin_fmaf(a, bv, acc);"),
    "epilogue: residual before GeLU": ("if (act == 1) y = oracle_gelu(y);\n                if (Rb) y = y + Rb[i * ldr + j];",
                                       "if (Rb) y = y + Rb[i * ldr + j];\n                if (act == 1) y = oracle_gelu(y);"),
    "causal softmax: one key too many": ("int64_t L = first + i % period + 1;",
                                         "int64_t L = first + i % period + 2;"),
    "causal softmax: period ignored": ("int64_t L = first + i % period + 1;", "int64_t L = first + i + 1;"),
    "f16: ties rounded up": ("if (rem > half || (rem == half && (r & 1))) ++r;", "if (rem >= half) ++r;"),
    "f16: subnormals scaled by 2^-23": ("float v = (float)m * 5.9604644775390625e-08f;",
                                        "float v = (float)m * 1.1920928955078125e-07f;"),
    "bf16: truncation": ("uint32_t rounded = x + 0x7fffu + ((x >> 16) & 1u);", "uint32_t rounded = x;"),
    "rolling hash: wrong base": ("#define ROLL_B 4294967311ull", "#define ROLL_B 4294967291ull"),
    "typed gemm: q in decreasing order": ("for (int64_t q = 0; q < K; ++q) {", "for (int64_t q = K - 1; q >= 0; --q) {"),
    "typed mean: SGD adds the step": ("float updated = theta[e] - step;", "float updated = theta[e] + step;"),
    "typed mean: last gradient dropped": ("for (int r = 1; r < nC; ++r) S = S + load_as_f32(grads[order[r]], e, gtype);",
                                          "for (int r = 1; r < nC - 1; ++r) S = S + load_as_f32(grads[order[r]], e, gtype);"),
    "colsum: rows in reverse order": ("for (int64_t i = 0; i < rows; ++i) v[i] = x[i * ldx + j];",
                                      "for (int64_t i = 0; i < rows; ++i) v[i] = x[(rows - 1 - i) * ldx + j];"),
    "gelu grad: pdf without 1/sqrt(2 pi)": ("float pdf = oracle_exp(a) * 0.3989422917366028f;",
                                            "float pdf = oracle_exp(a);"),
    "gelu grad: cdf not halved": ("float cdf = 0.5f * phi2;", "float cdf = phi2;"),
    "rmsnorm backward: inv dropped": ("float d = inv * (gy - xh * c);", "float d = gy - xh * c;"),
    "rmsnorm backward: residual ignored": ("if (res) d = d + res[i * ldres + j];", ""),
    "rmsnorm backward: dgamma from gy": ("dyxh[i * ldp + j] = dr[j] * xh;", "dyxh[i * ldp + j] = gy * xh;"),
    "softmax backward: s not subtracted": ("ds[i * ldds + j] = p[i * ldp + j] * (dp[i * lddp + j] - s);",
                                           "ds[i * ldds + j] = p[i * ldp + j] * dp[i * lddp + j];"),
    "batched: A advanced by B's stride": ("const float *Ab = A + b * strideA;", "const float *Ab = A + b * strideB;"),
    "window: one k past the upper band": ("if (k_hi >= 0 && i + k_hi + 1 < k1) k1 = i + k_hi + 1;",
                                          "if (k_hi >= 0 && i + k_hi + 2 < k1) k1 = i + k_hi + 2;"),
    "batched: B group ignored": ("const float *Bb = B + (b / b_group) * strideB;",
                                 "const float *Bb = B + b * strideB;"),
    "window: lower band ignored": ("if (k_lo >= 0 && i - k_lo > k0) k0 = i - k_lo;", ""),
    "causal softmax backward: one entry too many": ("int64_t seen = first + (i % period) + 1;",
                                                    "int64_t seen = first + (i % period) + 2;"),
    "causal softmax backward: masked entries -0": ("ds[i * ldds + j] = 0.0f;", "ds[i * ldds + j] = -0.0f;"),
    "silu: sigma without the 1 +": ("float den = 1.0f + e;", "float den = e;"),
    "silu: exp of +x": ("float e = oracle_exp(-x);", "float e = oracle_exp(x);"),
    "swiglu backward: du from u": ("du[i] = dhi * a;", "du[i] = dhi * up;"),
    "swiglu backward: 1 - sigma as sigma": ("float one_minus = 1.0f - sg;", "float one_minus = sg;"),
    "rope frequencies: growing": ("freq[i] = oracle_exp(-x);", "freq[i] = oracle_exp(x);"),
    "rope table: quadrant 1 swapped": ("else if (q == 1) { sv = cr;  cv = -sr; }",
                                       "else if (q == 1) { sv = -cr; cv = sr; }"),
    "rope table: one-part pi/2": ("    r = r - k * RP_PIO2_2;\n    r = r - k * RP_PIO2_3;\n", ""),
    "rope table: cos series without z^2/4!": (
        "    qc = qc * z + 0x1.5555555555555p-5;                  /* 1/4! */\n", ""),
    "rope: sin term added": ("y0 = a - b;", "y0 = a + b;"),
    "rope: position ignores first": ("int64_t pos = first + r % period;", "int64_t pos = r % period;"),
    "rope inverse: forward formula": ("float e = x1 * c, f = x0 * sn;\n                    y1 = e - f;",
                                      "float e = x0 * sn, f = x1 * c;\n                    y1 = e + f;"),
}


def build_variant(tmp_path, name, source):
    sys.path.insert(0, ROOT)
    from oracle import build as ob
    src = tmp_path / (name + ".c")
    src.write_text(source)
    lib = tmp_path / (name + ".so")
    subprocess.run([os.environ.get("CC", "gcc")] + ob.CFLAGS + ["-o", str(lib), str(src)] + ob.LDLIBS,
                   check=True)
    return str(lib)


def run_pins(lib):
    env = dict(os.environ, REPOPS_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider"] + PINS,
                       capture_output=True, text=True, env=env, cwd=ROOT, timeout=600)
    return r.returncode, r.stdout[-2000:]


def _variant_result(tmp_path, name, source):
    return run_pins(build_variant(tmp_path, name, source))


@pytest.fixture(scope="session")
def results(tmp_path_factory):
    """Builds the unmodified source and every mutant and runs the pin suite on
    each, several subprocesses at a time; maps a case name (None: unmodified)
    to (return code, output tail)."""
    src = open(SRC).read()
    cases = {None: src}
    for name, (old, new) in MUTATIONS.items():
        if src.count(old) == 1:
            cases[name] = src.replace(old, new)
    workers = max(1, min(8, (os.cpu_count() or 2) - 1))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        futs = {name: ex.submit(_variant_result, tmp_path_factory.mktemp("mut"), "v", text)
                for name, text in cases.items()}
        return {name: f.result() for name, f in futs.items()}


def test_unmodified_source_passes_the_pins(results):
    rc, out = results[None]
    assert rc == 0, out


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_fails_a_pin(results, name):
    old, new = MUTATIONS[name]
    assert open(SRC).read().count(old) == 1, "mutation anchor not found exactly once: " + name
    rc, out = results[name]
    assert rc != 0, "the pins did not catch: " + name
