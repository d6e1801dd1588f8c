// llama.cu -- the element-wise operators of a Llama-style decoder layer: the
// SiLU-gated MLP activation (SwiGLU) with its backward, and rotary position
// embeddings (frequencies, the cos/sin table, the rotation and its inverse).
//
// "Verde与RepOps" §4.3 measures Llama-style training; the pages fix neither
// operator, so the library defines them with one IEEE rounding per step in a
// fixed order:
//   sigma(x) = 1 / (1 + exp(-x)) (the library's exp, one correctly rounded
//   reciprocal), SiLU(x) = x * sigma(x), h = SiLU(g) * u;
//   frequencies f_i = exp(-((i / pairs) * ln_base));
//   cos/sin of p * f_i in binary64 -- Cody and Waite's reduction by a
//   three-part pi/2, Taylor series of sin and cos on [-pi/4, pi/4] by Horner's
//   rule -- rounded once to binary32 (binary64 add and multiply are IEEE
//   operations with the same bits on any hardware);
//   adjacent pairs (x[2i], x[2i+1]) rotated by the position's angle.
// All kernels are memory-streaming: threads run along columns (coalesced,
// 16-byte accesses where the operands allow), the grid strides over rows.
#include <algorithm>

#include "fixed_math.cuh"
#include "internal.cuh"

namespace repops {
namespace {

// ----------------------------------------------------------------- SwiGLU ----

__device__ __forceinline__ float sigmoid_fixed(float x) {
    return __frcp_rn(__fadd_rn(1.0f, exp_fixed(-x)));   // correctly rounded 1/(1 + e)
}

// Two sigmoids: the same steps lane by lane, the exponentials and the 1 + e
// additions of the pair as packed adds (exp_fixed2): the same bits.
__device__ __forceinline__ float2 sigmoid_fixed2(float x0, float x1) {
    const float2 e = exp_fixed2(-x0, -x1);
    float d0, d1;
    unpack2(add2_rn(pack2(1.0f, 1.0f), pack2(e.x, e.y)), d0, d1);
    return make_float2(__frcp_rn(d0), __frcp_rn(d1));
}

__device__ __forceinline__ float swiglu1(float g, float u) {
    return __fmul_rn(__fmul_rn(g, sigmoid_fixed(g)), u);
}

__device__ __forceinline__ float swiglu_s(float g, float u, float sg) {
    return __fmul_rn(__fmul_rn(g, sg), u);
}

__device__ __forceinline__ void swiglu_grad_s(float g, float u, float dh, float sg, float &dg, float &du) {
    du = __fmul_rn(dh, __fmul_rn(g, sg));
    const float t = __fmul_rn(dh, u);
    const float d = __fmul_rn(sg, __fadd_rn(1.0f, __fmul_rn(g, __fsub_rn(1.0f, sg))));
    dg = __fmul_rn(t, d);
}

__device__ __forceinline__ void swiglu_grad1(float g, float u, float dh, float &dg, float &du) {
    swiglu_grad_s(g, u, dh, sigmoid_fixed(g), dg, du);
}

// Columns in units of 4 (vec) or 1; h may be g or u (each element is read
// before it is written, by the same thread).
__global__ void __launch_bounds__(256)
swiglu_kernel(int64_t rows, int64_t cols, const float *g, int64_t ldg, const float *u, int64_t ldu, float *h,
              int64_t ldh, int vec) {
    const int64_t units = vec ? cols / 4 : cols;
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
        const float *gr = g + r * ldg, *ur = u + r * ldu;
        float *hr = h + r * ldh;
        for (int64_t c = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; c < units;
             c += int64_t(gridDim.x) * blockDim.x) {
            if (vec) {
                const float4 a = reinterpret_cast<const float4 *>(gr)[c];
                const float4 b = reinterpret_cast<const float4 *>(ur)[c];
                const float2 s01 = sigmoid_fixed2(a.x, a.y), s23 = sigmoid_fixed2(a.z, a.w);
                reinterpret_cast<float4 *>(hr)[c] = make_float4(swiglu_s(a.x, b.x, s01.x), swiglu_s(a.y, b.y, s01.y),
                                                                swiglu_s(a.z, b.z, s23.x), swiglu_s(a.w, b.w, s23.y));
            } else {
                hr[c] = swiglu1(gr[c], ur[c]);
            }
        }
    }
}

__global__ void __launch_bounds__(256)
swiglu_backward_kernel(int64_t rows, int64_t cols, const float *g, int64_t ldg, const float *u, int64_t ldu,
                       const float *dh, int64_t lddh, float *dg, int64_t lddg, float *du, int64_t lddu, int vec) {
    const int64_t units = vec ? cols / 4 : cols;
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
        const float *gr = g + r * ldg, *ur = u + r * ldu, *dr = dh + r * lddh;
        float *dgr = dg + r * lddg, *dur = du + r * lddu;
        for (int64_t c = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; c < units;
             c += int64_t(gridDim.x) * blockDim.x) {
            if (vec) {
                const float4 a = reinterpret_cast<const float4 *>(gr)[c];
                const float4 b = reinterpret_cast<const float4 *>(ur)[c];
                const float4 d = reinterpret_cast<const float4 *>(dr)[c];
                float4 og, ou;
                const float2 s01 = sigmoid_fixed2(a.x, a.y), s23 = sigmoid_fixed2(a.z, a.w);
                swiglu_grad_s(a.x, b.x, d.x, s01.x, og.x, ou.x);
                swiglu_grad_s(a.y, b.y, d.y, s01.y, og.y, ou.y);
                swiglu_grad_s(a.z, b.z, d.z, s23.x, og.z, ou.z);
                swiglu_grad_s(a.w, b.w, d.w, s23.y, og.w, ou.w);
                reinterpret_cast<float4 *>(dgr)[c] = og;
                reinterpret_cast<float4 *>(dur)[c] = ou;
            } else {
                float og, ou;
                swiglu_grad1(gr[c], ur[c], dr[c], og, ou);
                dgr[c] = og;
                dur[c] = ou;
            }
        }
    }
}

// ----------------------------------------------------------------- rotary ----

__global__ void rope_frequencies_kernel(int64_t pairs, float ln_base, float *freq) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < pairs; i += int64_t(gridDim.x) * blockDim.x) {
        const float frac = __fdiv_rn(float(i), float(pairs));
        freq[i] = exp_fixed(-__fmul_rn(frac, ln_base));
    }
}

// pi/2 = P1 + P2 + P3: P1, P2 the leading 29-bit pieces (k * P exact for
// |k| < 2^24), P3 the rest rounded to binary64; and 2/pi rounded.
constexpr double kPio2_1 = 0x1.921fb54p+0;
constexpr double kPio2_2 = 0x1.10b4611p-30;
constexpr double kPio2_3 = 0x1.4c4c6628b80dcp-59;
constexpr double kTwoOverPi = 0x1.45f306dc9c883p-1;

__device__ __forceinline__ void rope_sincos(int64_t pos, float f, float &c_out, float &s_out) {
    const double a = __dmul_rn(double(pos), double(f));   // exact: 24 + 24 bits
    const double k = rint(__dmul_rn(a, kTwoOverPi));
    double r = __dsub_rn(a, __dmul_rn(k, kPio2_1));
    r = __dsub_rn(r, __dmul_rn(k, kPio2_2));
    r = __dsub_rn(r, __dmul_rn(k, kPio2_3));
    const double z = __dmul_rn(r, r);
    // Taylor coefficients (-1)^n / (2n+1)! and (-1)^n / (2n)!, rounded to binary64
    double qs = -0x1.ae7f3e733b81fp-41;                       // -1/15!
    qs = __dadd_rn(__dmul_rn(qs, z), 0x1.6124613a86d09p-33);  // 1/13!
    qs = __dadd_rn(__dmul_rn(qs, z), -0x1.ae64567f544e4p-26); // -1/11!
    qs = __dadd_rn(__dmul_rn(qs, z), 0x1.71de3a556c734p-19);  // 1/9!
    qs = __dadd_rn(__dmul_rn(qs, z), -0x1.a01a01a01a01ap-13); // -1/7!
    qs = __dadd_rn(__dmul_rn(qs, z), 0x1.1111111111111p-7);   // 1/5!
    qs = __dadd_rn(__dmul_rn(qs, z), -0x1.5555555555555p-3);  // -1/3!
    const double sr = __dadd_rn(r, __dmul_rn(__dmul_rn(r, z), qs));
    double qc = 0x1.ae7f3e733b81fp-45;                        // 1/16!
    qc = __dadd_rn(__dmul_rn(qc, z), -0x1.93974a8c07c9dp-37); // -1/14!
    qc = __dadd_rn(__dmul_rn(qc, z), 0x1.1eed8eff8d898p-29);  // 1/12!
    qc = __dadd_rn(__dmul_rn(qc, z), -0x1.27e4fb7789f5cp-22); // -1/10!
    qc = __dadd_rn(__dmul_rn(qc, z), 0x1.a01a01a01a01ap-16);  // 1/8!
    qc = __dadd_rn(__dmul_rn(qc, z), -0x1.6c16c16c16c17p-10); // -1/6!
    qc = __dadd_rn(__dmul_rn(qc, z), 0x1.5555555555555p-5);   // 1/4!
    qc = __dadd_rn(__dmul_rn(qc, z), -0.5);                   // -1/2!
    const double cr = __dadd_rn(1.0, __dmul_rn(z, qc));
    const long long q = static_cast<long long>(k) & 3;
    const double sv = q == 0 ? sr : q == 1 ? cr : q == 2 ? -sr : -cr;
    const double cv = q == 0 ? cr : q == 1 ? -sr : q == 2 ? -cr : sr;
    c_out = __double2float_rn(cv);
    s_out = __double2float_rn(sv);
}

__global__ void rope_table_kernel(int64_t positions, int64_t pairs, const float *__restrict__ freq,
                                  float *__restrict__ cosv, float *__restrict__ sinv) {
    const int64_t n = positions * pairs;
    for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < n; e += int64_t(gridDim.x) * blockDim.x) {
        const int64_t p = e / pairs, i = e - p * pairs;
        float c, s;
        rope_sincos(p, freq[i], c, s);
        cosv[e] = c;
        sinv[e] = s;
    }
}

// One thread per pair of a row (threads along the row, the grid's y along
// rows); 8-byte accesses when the rows allow them.
__global__ void __launch_bounds__(256)
rope_kernel(int64_t rows, int heads, int pairs, float *x, int64_t ldx, const float *__restrict__ cosv,
            const float *__restrict__ sinv, int64_t first, int64_t period, int inverse, int vec2) {
    const int per_row = heads * pairs;
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
        const int64_t pos = first + r % period;
        const float *ct = cosv + pos * pairs, *st = sinv + pos * pairs;
        float *xr = x + r * ldx;
        for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < per_row; e += gridDim.x * blockDim.x) {
            const int h = e / pairs, i = e - h * pairs;
            float *v = xr + int64_t(h) * 2 * pairs + 2 * i;
            float x0, x1;
            if (vec2) {
                const float2 w = *reinterpret_cast<const float2 *>(v);
                x0 = w.x; x1 = w.y;
            } else {
                x0 = v[0]; x1 = v[1];
            }
            const float c = __ldg(ct + i), s = __ldg(st + i);
            float y0, y1;
            if (!inverse) {
                y0 = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
                y1 = __fadd_rn(__fmul_rn(x0, s), __fmul_rn(x1, c));
            } else {
                y0 = __fadd_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
                y1 = __fsub_rn(__fmul_rn(x1, c), __fmul_rn(x0, s));
            }
            if (vec2) {
                *reinterpret_cast<float2 *>(v) = make_float2(y0, y1);
            } else {
                v[0] = y0; v[1] = y1;
            }
        }
    }
}

// ------------------------------------------------------------------- host ----

bool span2d(int64_t rows, int64_t cols, int64_t ld, uint64_t *bytes) {
    if (rows == 0 || cols == 0) { *bytes = 0; return true; }
    if (ld < cols || rows - 1 > (INT64_MAX / 4 - cols) / ld) return false;
    *bytes = uint64_t((rows - 1) * ld + cols) * 4u;
    return true;
}

bool aligned16(const void *p, int64_t ld) { return reinterpret_cast<uintptr_t>(p) % 16 == 0 && ld % 4 == 0; }

// 256-thread CTAs: x over column units, y over rows, about 16 CTAs per SM.
dim3 grid_2d(int64_t units, int64_t rows) {
    DeviceInfo di;
    const int64_t target = int64_t(current_device_info(&di) == REPOPS_OK ? di.sms : 152) * 16;
    const int64_t gx = std::max<int64_t>(1, std::min<int64_t>((units + 255) / 256, target));
    const int64_t gy = std::max<int64_t>(1, std::min<int64_t>({rows, std::max<int64_t>(1, target / gx), 65535}));
    return dim3(unsigned(gx), unsigned(gy));
}

// True when two rows x cols blocks of floats, at a (pitch lda) and b (pitch
// ldb), share an element.  With one pitch the test is exact, so column
// blocks of one matrix ([g | u] side by side) do not count as overlapping;
// with two pitches it falls back to the byte spans.
bool blocks_overlap(const float *a, int64_t lda, const float *b, int64_t ldb, int64_t rows, int64_t cols) {
    uint64_t ab = 0, bb = 0;
    span2d(rows, cols, lda, &ab);
    span2d(rows, cols, ldb, &bb);
    if (!ranges_overlap(a, ab, b, bb)) return false;
    const intptr_t db = reinterpret_cast<intptr_t>(b) - reinterpret_cast<intptr_t>(a);
    if (lda != ldb || db % 4 != 0) return true;
    // b = a + d elements: b's row r starts in a's row r + q at column rem
    const int64_t d = db / 4;
    int64_t q = d / lda, rem = d % lda;
    if (rem < 0) { rem += lda; --q; }
    auto rows_meet = [&](int64_t shift) { return shift > -rows && shift < rows; };
    if (rem < cols && rows_meet(q)) return true;               // columns [rem, rem + cols) of row r + q
    if (rem + cols > lda && rows_meet(q + 1)) return true;     // the part wrapping into row r + q + 1
    return false;
}

// `out` may be `in` itself with the same pitch; any other shared element is
// an alias.
bool bad_overlap(const float *out, int64_t ldo, const float *in, int64_t ldi, int64_t rows, int64_t cols) {
    if (out == in && ldo == ldi) return false;
    return blocks_overlap(out, ldo, in, ldi, rows, cols);
}

}  // namespace
}  // namespace repops

using namespace repops;

extern "C" int repops_swiglu_f32(int64_t rows, int64_t cols, const float *g, int64_t ldg, const float *u,
                                 int64_t ldu, float *h, int64_t ldh, cudaStream_t stream) {
    if (rows < 0 || cols < 0) return REPOPS_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return REPOPS_OK;
    if (!g || !u || !h) return REPOPS_ERR_INVALID_ARG;
    uint64_t gb, ub, hb;
    if (!span2d(rows, cols, ldg, &gb) || !span2d(rows, cols, ldu, &ub) || !span2d(rows, cols, ldh, &hb))
        return REPOPS_ERR_INVALID_ARG;
    if (bad_overlap(h, ldh, g, ldg, rows, cols) || bad_overlap(h, ldh, u, ldu, rows, cols)) return REPOPS_ERR_ALIAS;
    const int vec = cols % 4 == 0 && aligned16(g, ldg) && aligned16(u, ldu) && aligned16(h, ldh);
    swiglu_kernel<<<grid_2d(vec ? cols / 4 : cols, rows), 256, 0, stream>>>(rows, cols, g, ldg, u, ldu, h, ldh, vec);
    return check_launch();
}

extern "C" int repops_swiglu_backward_f32(int64_t rows, int64_t cols, const float *g, int64_t ldg, const float *u,
                                          int64_t ldu, const float *dh, int64_t lddh, float *dg, int64_t lddg,
                                          float *du, int64_t lddu, cudaStream_t stream) {
    if (rows < 0 || cols < 0) return REPOPS_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return REPOPS_OK;
    if (!g || !u || !dh || !dg || !du) return REPOPS_ERR_INVALID_ARG;
    uint64_t gb, ub, db, ogb, oub;
    if (!span2d(rows, cols, ldg, &gb) || !span2d(rows, cols, ldu, &ub) || !span2d(rows, cols, lddh, &db) ||
        !span2d(rows, cols, lddg, &ogb) || !span2d(rows, cols, lddu, &oub))
        return REPOPS_ERR_INVALID_ARG;
    if (blocks_overlap(dg, lddg, du, lddu, rows, cols)) return REPOPS_ERR_ALIAS;
    // dg may be g or dh, du may be u or dh (same pointer and pitch); no other overlap
    if (bad_overlap(dg, lddg, g, ldg, rows, cols) || blocks_overlap(dg, lddg, u, ldu, rows, cols) ||
        bad_overlap(dg, lddg, dh, lddh, rows, cols))
        return REPOPS_ERR_ALIAS;
    if (blocks_overlap(du, lddu, g, ldg, rows, cols) || bad_overlap(du, lddu, u, ldu, rows, cols) ||
        bad_overlap(du, lddu, dh, lddh, rows, cols))
        return REPOPS_ERR_ALIAS;
    const int vec = cols % 4 == 0 && aligned16(g, ldg) && aligned16(u, ldu) && aligned16(dh, lddh) &&
                    aligned16(dg, lddg) && aligned16(du, lddu);
    swiglu_backward_kernel<<<grid_2d(vec ? cols / 4 : cols, rows), 256, 0, stream>>>(
        rows, cols, g, ldg, u, ldu, dh, lddh, dg, lddg, du, lddu, vec);
    return check_launch();
}

extern "C" int repops_rope_frequencies_f32(int64_t pairs, float ln_base, float *freq, cudaStream_t stream) {
    if (pairs < 1 || pairs > (int64_t(1) << 24) || !freq) return REPOPS_ERR_INVALID_ARG;
    const int blocks = int(std::min<int64_t>((pairs + 255) / 256, 1024));
    rope_frequencies_kernel<<<blocks, 256, 0, stream>>>(pairs, ln_base, freq);
    return check_launch();
}

extern "C" int repops_rope_table_f32(int64_t positions, int64_t pairs, const float *freq, float *cos_out,
                                     float *sin_out, cudaStream_t stream) {
    if (positions < 1 || positions > (int64_t(1) << 24) || pairs < 1 || pairs > (int64_t(1) << 24))
        return REPOPS_ERR_INVALID_ARG;
    if (!freq || !cos_out || !sin_out) return REPOPS_ERR_INVALID_ARG;
    if (positions > INT64_MAX / 4 / pairs) return REPOPS_ERR_INVALID_ARG;
    const uint64_t tb = uint64_t(positions * pairs) * 4u, fb = uint64_t(pairs) * 4u;
    if (ranges_overlap(cos_out, tb, sin_out, tb) || ranges_overlap(cos_out, tb, freq, fb) ||
        ranges_overlap(sin_out, tb, freq, fb))
        return REPOPS_ERR_ALIAS;
    DeviceInfo di;
    const int64_t cap = int64_t(current_device_info(&di) == REPOPS_OK ? di.sms : 152) * 8;
    const int blocks = int(std::max<int64_t>(1, std::min<int64_t>((positions * pairs + 255) / 256, cap)));
    rope_table_kernel<<<blocks, 256, 0, stream>>>(positions, pairs, freq, cos_out, sin_out);
    return check_launch();
}

extern "C" int repops_rope_f32(int64_t rows, int64_t heads, int64_t pairs, float *x, int64_t ldx,
                               const float *cos_tab, const float *sin_tab, int64_t positions, int64_t first,
                               int64_t period, int inverse, cudaStream_t stream) {
    if (rows < 0 || heads < 0 || pairs < 1 || first < 0 || period < 1 || positions < 1)
        return REPOPS_ERR_INVALID_ARG;
    if (heads * pairs > (int64_t(1) << 30)) return REPOPS_ERR_INVALID_ARG;
    const int64_t width = heads * 2 * pairs;
    if (ldx < std::max<int64_t>(1, width)) return REPOPS_ERR_INVALID_ARG;
    if (rows == 0 || heads == 0) return REPOPS_OK;
    if (!x || !cos_tab || !sin_tab) return REPOPS_ERR_INVALID_ARG;
    // the largest position reached: first + min(rows, period) - 1
    if (first > positions - std::min(rows, period)) return REPOPS_ERR_INVALID_ARG;
    if (positions > INT64_MAX / 4 / pairs) return REPOPS_ERR_INVALID_ARG;
    uint64_t xb;
    if (!span2d(rows, width, ldx, &xb)) return REPOPS_ERR_INVALID_ARG;
    const uint64_t tb = uint64_t(positions * pairs) * 4u;
    if (ranges_overlap(x, xb, cos_tab, tb) || ranges_overlap(x, xb, sin_tab, tb)) return REPOPS_ERR_ALIAS;
    const int vec2 = reinterpret_cast<uintptr_t>(x) % 8 == 0 && ldx % 2 == 0;
    rope_kernel<<<grid_2d(heads * pairs, rows), 256, 0, stream>>>(rows, int(heads), int(pairs), x, ldx, cos_tab,
                                                                  sin_tab, first, period, inverse ? 1 : 0, vec2);
    return check_launch();
}
