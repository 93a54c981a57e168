// qkv_oracle.cpp -- plain, slow CPU oracle for the quantized paged KV-cache path.
//
// TEST INFRASTRUCTURE ONLY. Only the test suite, the package smoke check and the
// benchmark's CPU-baseline leg load this library. The product path (the CUDA
// library under quantized_paged_kv_append_gb300/) never calls it, and the two
// share no source: no header, helper, table or constant generator.
//
// Compile with -O2 -ffp-contract=off and without -ffast-math: every fp32 step
// below is a single IEEE-754 round-to-nearest-even operation, evaluated in the
// order written. Attention is computed in double.
//
// Sources (page title, section):
//   [FT]  "feat(kvcache): add ISO3/ISO4 KV-cache quantization (--kv-cache-iso)",
//         sections "What" and "Correctness".
//   [S8]  "qwen35/q36: --kv - int8 K/V caches (codes + a FP16 scale per 64 values)",
//         sections "What it does" and "Not in this PR".
//   [K4]  "--kv k8v4: hybrid KV cache -- INT8 K + Hadamard-rotated Q4_0 V (816 B/cell)",
//         sections "What", "How" and "Tests".
// The format list follows [S8 "What it does"] (int8 for both stores, or for one store
// with the other unquantized) and [S8 "Not in this PR"] / [K4 "What"] (q4_0 for both
// stores, K and V rotated by the FWHT-256, 576 B per cell at head_dim 256).
// Where the pages leave a step open, the reading taken is stated at the step.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// ---------------------------------------------------------------------------
// Number formats, written from IEEE-754 binary16 / bfloat16 definitions.
// ---------------------------------------------------------------------------

// double -> binary16, round to nearest, ties to even. Finite values whose
// rounded magnitude exceeds the largest finite half give +-inf (sat == 0) or
// +-65504 (sat == 1). NaN maps to a quiet NaN.
uint16_t half_from_double(double v, int sat) {
    uint16_t sign = std::signbit(v) ? 0x8000 : 0;
    if (std::isnan(v)) return 0x7e00;
    double a = std::fabs(v);
    if (std::isinf(a)) return sign | (sat ? 0x7bff : 0x7c00);
    if (a == 0.0) return sign;
    int e2;
    std::frexp(a, &e2);           // a = f * 2^e2, f in [0.5, 1)
    int E = e2 - 1;               // a in [2^E, 2^(E+1))
    if (E < -14) E = -14;         // subnormal range: quantum is 2^-24
    double scaled = std::ldexp(a, 10 - E);  // exact
    double r = std::nearbyint(scaled);      // default mode: ties to even
    uint32_t ri = (uint32_t)r;
    if (E == -14 && ri < 1024) return sign | (uint16_t)ri;   // subnormal (or zero)
    if (ri == 2048) { ri = 1024; E += 1; }
    if (E > 15) return sign | (sat ? 0x7bff : 0x7c00);
    return sign | (uint16_t)(((E + 15) << 10) | (ri - 1024));
}

double double_from_half(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0) v = std::ldexp((double)m, -24);
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = std::ldexp((double)(m | 0x400), e - 25);
    return sign ? -v : v;
}

float float_from_half(uint16_t h) { return (float)double_from_half(h); }

float float_from_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

// fp32 -> bfloat16, round to nearest, ties to even (the top 16 bits of the
// binary32 encoding after rounding away the low 16); NaN stays a quiet NaN.
uint16_t bf16_from_float(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40);
    const uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7fffu + lsb) >> 16);
}

// ---------------------------------------------------------------------------
// Format geometry. [S8 "What it does"]: int8 codes + one fp16 scale per 64
// values. [K4 "What"]: q4_0 V in 32-value blocks, fp16 d + 16 B of nibbles.
// [FT "What"]: ISO3 50 B and ISO4 68 B per 128-value block.
// Reading (pages silent on memory order): planar storage, codes in one plane and
// scales in another, each indexed [page][kv_head][slot][row bytes]. The ISO4
// block's two bytes beyond code nibbles + fp16 norm are a reserved fp16 written
// as zero, stored after the norm in the scale plane.
// The unquantized store of the one-store formats [S8 "What it does": "k8v32 /
// k32v8 quantize one store only"] keeps the input values as they arrive: the
// pages' engine holds FP32 activations and keeps that store in FP32; here K and V
// arrive as bf16, so the store holds the bf16 values unchanged (2 bytes per value,
// no scale row). Reading the store back gives exactly the input.
// ---------------------------------------------------------------------------

enum { FMT_INT8 = 0, FMT_K8V4 = 1, FMT_ISO3 = 2, FMT_ISO4 = 3, FMT_Q4 = 4, FMT_K8 = 5, FMT_V8 = 6 };
enum { ENC_INT8 = 0, ENC_Q4 = 1, ENC_ISO3 = 2, ENC_ISO4 = 3, ENC_BF16 = 4 };

int store_encoding(int fmt, int store /*0 = K, 1 = V*/) {
    switch (fmt) {
        case FMT_INT8: return ENC_INT8;
        case FMT_K8V4: return store == 0 ? ENC_INT8 : ENC_Q4;
        case FMT_ISO3: return ENC_ISO3;
        case FMT_ISO4: return ENC_ISO4;
        case FMT_Q4: return ENC_Q4;                              // K and V rotated, q4_0
        case FMT_K8: return store == 0 ? ENC_INT8 : ENC_BF16;    // int8 K, V unquantized
        case FMT_V8: return store == 0 ? ENC_BF16 : ENC_INT8;    // K unquantized, int8 V
    }
    return -1;
}

// bytes of codes and of scales for one head vector of length D
void row_bytes(int enc, int D, int* code_b, int* scale_b) {
    switch (enc) {
        case ENC_INT8: *code_b = D;            *scale_b = (D / 64) * 2;  break;
        case ENC_Q4:   *code_b = D / 2;        *scale_b = (D / 32) * 2;  break;
        case ENC_ISO3: *code_b = (D / 128) * 48; *scale_b = (D / 128) * 2; break;
        case ENC_ISO4: *code_b = (D / 128) * 64; *scale_b = (D / 128) * 4; break;
        case ENC_BF16: *code_b = 2 * D;        *scale_b = 0;             break;
        default: *code_b = *scale_b = 0;
    }
}

// ---------------------------------------------------------------------------
// int8 group quantizer [S8 "What it does"; K4 "Tests": INT8 rules with ties to
// even]. Per 64 values: amax = max|x|, d = amax/127 (fp32), d16 = fp16(d)
// saturated, code = clamp(round_half_even(x / d16), -127, 127).
// Reading: the codes are computed against the stored fp16 scale d16 (so the
// dequantized value d16*code is within d16/2 of x), with an IEEE division.
// ---------------------------------------------------------------------------
void quant_int8_group(const float* x, int8_t* q, uint16_t* d16_out) {
    float amax = 0.0f;
    for (int i = 0; i < 64; ++i) amax = std::fmax(amax, std::fabs(x[i]));
    float d = amax / 127.0f;
    uint16_t h = half_from_double((double)d, 1);
    float dh = float_from_half(h);
    for (int i = 0; i < 64; ++i) {
        if (dh == 0.0f) { q[i] = 0; continue; }
        float r = std::nearbyint(x[i] / dh);   // ties to even (default mode)
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q[i] = (int8_t)r;
    }
    *d16_out = h;
}

// ---------------------------------------------------------------------------
// FWHT-256 [S8 "Not in this PR"; K4 "How"]: Walsh-Hadamard transform over the
// head dimension, normalised by 1/16 (orthonormal, self-inverse). Sylvester
// (natural) order; in-place fp32 butterflies at strides 1, 2, ..., 128, each
// (a, b) -> (a + b, a - b) with a the lower index; then an exact *1/16.
// ---------------------------------------------------------------------------
void fwht256_f32(float* x) {
    for (int h = 1; h < 256; h <<= 1)
        for (int i = 0; i < 256; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                float a = x[j], b = x[j + h];
                x[j] = a + b;
                x[j + h] = a - b;
            }
    for (int i = 0; i < 256; ++i) x[i] = x[i] * 0.0625f;
}

void fwht256_f64(double* x) {
    for (int h = 1; h < 256; h <<= 1)
        for (int i = 0; i < 256; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                double a = x[j], b = x[j + h];
                x[j] = a + b;
                x[j + h] = a - b;
            }
    for (int i = 0; i < 256; ++i) x[i] *= 0.0625;
}

// ---------------------------------------------------------------------------
// q4_0 block quantizer on the rotated vector [K4 "What": rotated q4_0].
// Per 32 values: m = the value of largest magnitude (first index on ties),
// d = m / -8, d16 = fp16(d) saturated, code = min(15, trunc(x/d16 + 8.5)),
// all fp32. Reading: codes use the stored d16 and an IEEE division; a lower
// clamp at 0 is kept as a guard (x/d16 >= -8 up to rounding, so it never binds).
// Packing: byte j (j < 16) holds element j in its low nibble and element j+16
// in its high nibble.
// ---------------------------------------------------------------------------
void quant_q4_block(const float* x, uint8_t* nib, uint16_t* d16_out) {
    float amax = 0.0f, m = 0.0f;
    for (int i = 0; i < 32; ++i) {
        float a = std::fabs(x[i]);
        if (a > amax) { amax = a; m = x[i]; }
    }
    float d = m / -8.0f;
    uint16_t h = half_from_double((double)d, 1);
    float dh = float_from_half(h);
    int q[32];
    for (int i = 0; i < 32; ++i) {
        if (dh == 0.0f) { q[i] = 8; continue; }
        float t = x[i] / dh;
        t = t + 8.5f;
        int qi = (int)std::trunc(t);
        if (qi > 15) qi = 15;
        if (qi < 0) qi = 0;
        q[i] = qi;
    }
    for (int j = 0; j < 16; ++j) nib[j] = (uint8_t)(q[j] | (q[j + 16] << 4));
    *d16_out = h;
}

// ---------------------------------------------------------------------------
// Lloyd-Max quantizer for N(0, sigma^2) [FT "What": nearest Lloyd-Max centroid;
// the table is the optimal N-level scalar quantizer of one coordinate of a
// random unit vector in 128 dimensions, approximated by N(0, 1/128)].
// Lloyd iteration in double: boundaries are midpoints of neighbouring levels;
// each level is the conditional mean of its cell,
//   E[Z | a < Z < b] = (phi(a) - phi(b)) / (Phi(b) - Phi(a))   (Z ~ N(0,1)),
// started from the cell quantiles (j + 1/2)/N and iterated to a fixed point.
// ---------------------------------------------------------------------------
double npdf(double z) { return std::isinf(z) ? 0.0 : std::exp(-0.5 * z * z) / std::sqrt(2.0 * M_PI); }
double ncdf(double z) { return 0.5 * std::erfc(-z / std::sqrt(2.0)); }

double ninv(double p) {  // quantile by bisection (start values only)
    double lo = -40.0, hi = 40.0;
    for (int it = 0; it < 200; ++it) {
        double mid = 0.5 * (lo + hi);
        if (ncdf(mid) < p) lo = mid; else hi = mid;
    }
    return 0.5 * (lo + hi);
}

void cell_means(int N, const double* z, double* out) {
    for (int j = 0; j < N; ++j) {
        double a = (j == 0) ? -INFINITY : 0.5 * (z[j - 1] + z[j]);
        double b = (j == N - 1) ? INFINITY : 0.5 * (z[j] + z[j + 1]);
        out[j] = (npdf(a) - npdf(b)) / (ncdf(b) - ncdf(a));
    }
}

// ISO block quantizer helpers --------------------------------------------

// Sum of squares of 128 fp32 values with a fixed evaluation order: 32 partial
// sums over consecutive groups of four (left to right), then pairwise sums at
// lane distances 16, 8, 4, 2, 1 (a butterfly; fp32 addition is commutative so
// every partner pair gets the same value).
float sumsq128(const float* v) {
    float lane[32];
    for (int l = 0; l < 32; ++l) {
        float s = v[4 * l] * v[4 * l];
        s = s + v[4 * l + 1] * v[4 * l + 1];
        s = s + v[4 * l + 2] * v[4 * l + 2];
        s = s + v[4 * l + 3] * v[4 * l + 3];
        lane[l] = s;
    }
    for (int off = 16; off >= 1; off >>= 1) {
        float nl[32];
        for (int l = 0; l < 32; ++l) nl[l] = lane[l] + lane[l ^ off];
        std::memcpy(lane, nl, sizeof(lane));
    }
    return lane[0];
}

// Hamilton product p (x) v of quaternions stored (w, x, y, z), fp32, each
// component evaluated left to right from the textbook expansion.
void qmul_f32(const float* p, const float* v, float* y) {
    float r0 = p[0] * v[0]; r0 = r0 - p[1] * v[1]; r0 = r0 - p[2] * v[2]; r0 = r0 - p[3] * v[3];
    float r1 = p[0] * v[1]; r1 = r1 + p[1] * v[0]; r1 = r1 + p[2] * v[3]; r1 = r1 - p[3] * v[2];
    float r2 = p[0] * v[2]; r2 = r2 - p[1] * v[3]; r2 = r2 + p[2] * v[0]; r2 = r2 + p[3] * v[1];
    float r3 = p[0] * v[3]; r3 = r3 + p[1] * v[2]; r3 = r3 - p[2] * v[1]; r3 = r3 + p[3] * v[0];
    y[0] = r0; y[1] = r1; y[2] = r2; y[3] = r3;
}

void qmul_f64(const double* p, const double* v, double* y) {
    y[0] = p[0] * v[0] - p[1] * v[1] - p[2] * v[2] - p[3] * v[3];
    y[1] = p[0] * v[1] + p[1] * v[0] + p[2] * v[3] - p[3] * v[2];
    y[2] = p[0] * v[2] - p[1] * v[3] + p[2] * v[0] + p[3] * v[1];
    y[3] = p[0] * v[3] + p[1] * v[2] - p[2] * v[1] + p[3] * v[0];
}

struct IsoTables { float c[16]; float b[15]; int N; };

IsoTables iso_tables(int bits);

// [FT "What"]: per 128-value block, L2-normalise, rotate each 4-D group by one
// fixed unit quaternion, code each value to the nearest Lloyd-Max centroid,
// store the corrected norm ||x|| / ||centroids||.
// Readings: the rotation is left multiplication q (x) v; a zero block codes
// y = 0 and stores norm 0; nearest-centroid ties go to the lower level (code =
// number of midpoints strictly below y); the norm is stored as fp16 (saturated).
void quant_iso_block(int bits, const float* x, const float* quat, int* codes,
                     uint16_t* s16_out, float* y_dbg, float* n_dbg, float* cn_dbg) {
    IsoTables T = iso_tables(bits);
    float ss = sumsq128(x);
    float n = std::sqrt(ss);
    float y[128];
    for (int g = 0; g < 32; ++g) {
        float v[4];
        for (int e = 0; e < 4; ++e) v[e] = (n == 0.0f) ? 0.0f : x[4 * g + e] / n;
        qmul_f32(quat, v, &y[4 * g]);
    }
    float cv[128];
    for (int i = 0; i < 128; ++i) {
        int k = 0;
        for (int j = 0; j < T.N - 1; ++j) if (y[i] > T.b[j]) ++k;
        codes[i] = k;
        cv[i] = T.c[k];
    }
    float cn = std::sqrt(sumsq128(cv));
    float s = n / cn;
    *s16_out = half_from_double((double)s, 1);
    if (y_dbg) std::memcpy(y_dbg, y, sizeof(y));
    if (n_dbg) *n_dbg = n;
    if (cn_dbg) *cn_dbg = cn;
}

void pack_iso(int bits, const int* codes, uint8_t* out) {
    if (bits == 3) {
        std::memset(out, 0, 48);
        for (int i = 0; i < 128; ++i) {
            out[i / 4] |= (uint8_t)((codes[i] & 3) << (2 * (i % 4)));
            out[32 + i / 8] |= (uint8_t)(((codes[i] >> 2) & 1) << (i % 8));
        }
    } else {
        std::memset(out, 0, 64);
        for (int i = 0; i < 128; ++i) out[i / 2] |= (uint8_t)((codes[i] & 15) << (4 * (i % 2)));
    }
}

void unpack_iso(int bits, const uint8_t* in, int* codes) {
    for (int i = 0; i < 128; ++i) {
        if (bits == 3)
            codes[i] = ((in[i / 4] >> (2 * (i % 4))) & 3) | (((in[32 + i / 8] >> (i % 8)) & 1) << 2);
        else
            codes[i] = (in[i / 2] >> (4 * (i % 2))) & 15;
    }
}

// ---------------------------------------------------------------------------
// Whole-vector quantize / dequantize for one store encoding.
// x: D fp32 values (the bf16 inputs widened). Output: code and scale rows.
// Dequantized values are returned in the original (unrotated) domain, in double.
// ---------------------------------------------------------------------------
void quant_vector(int enc, int D, const float* x, const float* quat, uint8_t* code, uint8_t* scale) {
    if (enc == ENC_BF16) {
        // unquantized store: the bf16 value itself (x holds bf16 inputs, so this is exact)
        for (int i = 0; i < D; ++i) {
            uint16_t b = bf16_from_float(x[i]);
            std::memcpy(code + 2 * i, &b, 2);
        }
    } else if (enc == ENC_INT8) {
        for (int g = 0; g < D / 64; ++g) {
            uint16_t h;
            quant_int8_group(x + 64 * g, (int8_t*)code + 64 * g, &h);
            std::memcpy(scale + 2 * g, &h, 2);
        }
    } else if (enc == ENC_Q4) {
        float r[256];
        std::memcpy(r, x, sizeof(r));
        fwht256_f32(r);
        for (int g = 0; g < 8; ++g) {
            uint16_t h;
            quant_q4_block(r + 32 * g, code + 16 * g, &h);
            std::memcpy(scale + 2 * g, &h, 2);
        }
    } else {
        int bits = (enc == ENC_ISO3) ? 3 : 4;
        int cb = (bits == 3) ? 48 : 64;
        for (int blk = 0; blk < D / 128; ++blk) {
            int codes[128];
            uint16_t h;
            quant_iso_block(bits, x + 128 * blk, quat, codes, &h, nullptr, nullptr, nullptr);
            pack_iso(bits, codes, code + cb * blk);
            if (bits == 3) {
                std::memcpy(scale + 2 * blk, &h, 2);
            } else {
                uint16_t zero = 0;
                std::memcpy(scale + 4 * blk, &h, 2);
                std::memcpy(scale + 4 * blk + 2, &zero, 2);
            }
        }
    }
}

void dequant_vector(int enc, int D, const uint8_t* code, const uint8_t* scale, const float* quat, double* out) {
    if (enc == ENC_BF16) {
        for (int i = 0; i < D; ++i) {
            uint16_t b;
            std::memcpy(&b, code + 2 * i, 2);
            out[i] = (double)float_from_bf16(b);
        }
    } else if (enc == ENC_INT8) {
        for (int g = 0; g < D / 64; ++g) {
            uint16_t h;
            std::memcpy(&h, scale + 2 * g, 2);
            double d = double_from_half(h);
            for (int i = 0; i < 64; ++i) out[64 * g + i] = d * (double)((const int8_t*)code)[64 * g + i];
        }
    } else if (enc == ENC_Q4) {
        double r[256];
        for (int g = 0; g < 8; ++g) {
            uint16_t h;
            std::memcpy(&h, scale + 2 * g, 2);
            double d = double_from_half(h);
            for (int j = 0; j < 16; ++j) {
                int lo = code[16 * g + j] & 15, hi = code[16 * g + j] >> 4;
                r[32 * g + j] = d * (double)(lo - 8);
                r[32 * g + j + 16] = d * (double)(hi - 8);
            }
        }
        fwht256_f64(r);  // H/16 is its own inverse: back to the original domain
        std::memcpy(out, r, sizeof(r));
    } else {
        int bits = (enc == ENC_ISO3) ? 3 : 4;
        int cb = (bits == 3) ? 48 : 64;
        int sb = (bits == 3) ? 2 : 4;
        IsoTables T = iso_tables(bits);
        double qc[4] = {quat[0], -(double)quat[1], -(double)quat[2], -(double)quat[3]};
        for (int blk = 0; blk < D / 128; ++blk) {
            int codes[128];
            unpack_iso(bits, code + cb * blk, codes);
            uint16_t h;
            std::memcpy(&h, scale + sb * blk, 2);
            double s = double_from_half(h);
            for (int g = 0; g < 32; ++g) {
                double c[4], y[4];
                for (int e = 0; e < 4; ++e) c[e] = T.c[codes[4 * g + e]];
                qmul_f64(qc, c, y);   // conjugate quaternion undoes the rotation
                for (int e = 0; e < 4; ++e) out[128 * blk + 4 * g + e] = s * y[e];
            }
        }
    }
}

IsoTables iso_tables(int bits) {
    static bool ready[2] = {false, false};
    static IsoTables cache[2];
    int k = (bits == 3) ? 0 : 1;
    if (!ready[k]) {
        IsoTables T;
        T.N = (bits == 3) ? 8 : 16;
        double z[16], m[16];
        for (int j = 0; j < T.N; ++j) z[j] = ninv((j + 0.5) / T.N);
        for (int it = 0; it < 200000; ++it) {
            cell_means(T.N, z, m);
            double chg = 0.0;
            for (int j = 0; j < T.N; ++j) { chg = std::fmax(chg, std::fabs(m[j] - z[j])); z[j] = m[j]; }
            if (chg < 1e-15) break;
        }
        double sigma = 1.0 / std::sqrt(128.0);
        // Spec choice: each level rounded to fp16 (kept as fp32), so levels are
        // exact half-precision operands; midpoints of the rounded levels.
        for (int j = 0; j < T.N; ++j) T.c[j] = float_from_half(half_from_double(sigma * z[j], 0));
        for (int j = 0; j < T.N - 1; ++j) T.b[j] = (T.c[j] + T.c[j + 1]) * 0.5f;
        cache[k] = T;
        ready[k] = true;
    }
    return cache[k];
}

// head vector address in a plane
inline size_t row_index(int page, int head, int slot, int Hkv, int P) {
    return ((size_t)page * Hkv + head) * P + slot;
}

int lookup_page(const int32_t* page_table, int max_pages, int b, int pos, int P, int num_pages) {
    int pg = page_table[(size_t)b * max_pages + pos / P];
    if (pg < 0 || pg >= num_pages) return -1;
    return pg;
}

// Dequantize token `pos` of sequence b, all KV heads, for one store: out[Hkv][D].
int dequant_token(int fmt, int store, int num_pages, int Hkv, int D, int P,
                  const uint8_t* codes, const uint8_t* scales, const int32_t* page_table, int max_pages,
                  int b, int pos, const float* quat, double* out) {
    int enc = store_encoding(fmt, store);
    int cb, sb;
    row_bytes(enc, D, &cb, &sb);
    int pg = lookup_page(page_table, max_pages, b, pos, P, num_pages);
    if (pg < 0) return -1;
    for (int h = 0; h < Hkv; ++h) {
        size_t r = row_index(pg, h, pos % P, Hkv, P);
        dequant_vector(enc, D, codes + r * cb, scales + r * sb, quat, out + (size_t)h * D);
    }
    return 0;
}

// Softmax-weighted sum in double, with max subtraction.
void attend(int D, int n, const double* s, const double* const* vrows, double* o) {
    double mx = -INFINITY;
    for (int t = 0; t < n; ++t) mx = std::fmax(mx, s[t]);
    double l = 0.0;
    for (int i = 0; i < D; ++i) o[i] = 0.0;
    for (int t = 0; t < n; ++t) {
        double p = std::exp(s[t] - mx);
        l += p;
        for (int i = 0; i < D; ++i) o[i] += p * vrows[t][i];
    }
    for (int i = 0; i < D; ++i) o[i] = (n > 0) ? o[i] / l : 0.0;
}

}  // namespace

extern "C" {

// ---- number formats (for pins against library converters) ----
void orc_half_from_f64_array(const double* x, uint16_t* out, int64_t n, int sat) {
    for (int64_t i = 0; i < n; ++i) out[i] = half_from_double(x[i], sat);
}
void orc_f64_from_half_array(const uint16_t* h, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = double_from_half(h[i]);
}
void orc_f32_from_bf16_array(const uint16_t* b, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = float_from_bf16(b[i]);
}

// ---- format geometry ----
int orc_row_bytes(int fmt, int store, int D, int* code_b, int* scale_b) {
    int enc = store_encoding(fmt, store);
    if (enc < 0) return -1;
    row_bytes(enc, D, code_b, scale_b);
    return 0;
}

// ---- Lloyd-Max ----
// Unrounded levels for N(0, sigma^2) plus the largest centroid-condition
// residual |c_j - E[X | cell j]| after convergence and the iteration count.
int orc_lloyd_max(int N, double sigma, double* levels, double* resid, int* iters) {
    if (N < 2 || N > 16) return -1;
    double z[16], m[16];
    for (int j = 0; j < N; ++j) z[j] = ninv((j + 0.5) / N);
    int it = 0;
    for (; it < 200000; ++it) {
        cell_means(N, z, m);
        double chg = 0.0;
        for (int j = 0; j < N; ++j) { chg = std::fmax(chg, std::fabs(m[j] - z[j])); z[j] = m[j]; }
        if (chg < 1e-15) break;
    }
    cell_means(N, z, m);
    double r = 0.0;
    for (int j = 0; j < N; ++j) r = std::fmax(r, std::fabs(m[j] - z[j]));
    for (int j = 0; j < N; ++j) levels[j] = sigma * z[j];
    *resid = sigma * r;
    *iters = it;
    return 0;
}

// fp16-rounded ISO levels (as fp32) and their midpoints.
int orc_iso_table(int bits, float* levels, float* mids) {
    if (bits != 3 && bits != 4) return -1;
    IsoTables T = iso_tables(bits);
    for (int j = 0; j < T.N; ++j) levels[j] = T.c[j];
    for (int j = 0; j < T.N - 1; ++j) mids[j] = T.b[j];
    return T.N;
}

// ---- single-block primitives ----
void orc_quant_int8(const float* x, int n, int8_t* codes, uint16_t* scales) {
    for (int g = 0; g < n / 64; ++g) quant_int8_group(x + 64 * g, codes + 64 * g, scales + g);
}
void orc_fwht256(float* x) { fwht256_f32(x); }
void orc_fwht256_f64(double* x) { fwht256_f64(x); }
void orc_quant_q4(const float* x, int n, uint8_t* nib, uint16_t* d) {
    for (int g = 0; g < n / 32; ++g) quant_q4_block(x + 32 * g, nib + 16 * g, d + g);
}
void orc_qmul(const float* p, const float* v, float* y) { qmul_f32(p, v, y); }
float orc_sumsq128(const float* v) { return sumsq128(v); }

// One ISO block with intermediates: y (rotated unit vector), codes, n, ||c||.
int orc_quant_iso_block(int bits, const float* x, const float* quat, int* codes, uint16_t* s16,
                        float* y, float* n, float* cn) {
    if (bits != 3 && bits != 4) return -1;
    quant_iso_block(bits, x, quat, codes, s16, y, n, cn);
    return 0;
}
void orc_pack_iso(int bits, const int* codes, uint8_t* out) { pack_iso(bits, codes, out); }
void orc_unpack_iso(int bits, const uint8_t* in, int* codes) { unpack_iso(bits, in, codes); }

// Whole head vector (D values) for one store encoding of a format.
int orc_quant_vector(int fmt, int store, int D, const float* x, const float* quat, uint8_t* code, uint8_t* scale) {
    int enc = store_encoding(fmt, store);
    if (enc < 0) return -1;
    quant_vector(enc, D, x, quat, code, scale);
    return 0;
}
int orc_dequant_vector(int fmt, int store, int D, const uint8_t* code, const uint8_t* scale, const float* quat, double* out) {
    int enc = store_encoding(fmt, store);
    if (enc < 0) return -1;
    dequant_vector(enc, D, code, scale, quat, out);
    return 0;
}

// ---- paged append (quantize-on-write) ----
// For each new token n: sequence seq_id[n], position pos[n]; the page is
// page_table[seq_id[n] * max_pages + pos[n] / P], the slot pos[n] % P. Each KV
// head's K and V vectors are quantized and written to their planes.
// Returns the number of tokens skipped for an out-of-range page entry.
int orc_append(int fmt, int num_pages, int Hkv, int D, int P,
               uint8_t* kc, uint8_t* ks, uint8_t* vc, uint8_t* vs,
               const uint16_t* k_bf16, const uint16_t* v_bf16, int n_tokens,
               const int32_t* seq_id, const int32_t* pos, const int32_t* page_table, int max_pages,
               const float* quat) {
    int bad = 0;
    std::vector<float> x(D);
    for (int n = 0; n < n_tokens; ++n) {
        int pg = lookup_page(page_table, max_pages, seq_id[n], pos[n], P, num_pages);
        if (pg < 0) { ++bad; continue; }
        for (int st = 0; st < 2; ++st) {
            int enc = store_encoding(fmt, st);
            int cb, sb;
            row_bytes(enc, D, &cb, &sb);
            const uint16_t* src = st == 0 ? k_bf16 : v_bf16;
            uint8_t* cp = st == 0 ? kc : vc;
            uint8_t* sp = st == 0 ? ks : vs;
            for (int h = 0; h < Hkv; ++h) {
                for (int i = 0; i < D; ++i) x[i] = float_from_bf16(src[((size_t)n * Hkv + h) * D + i]);
                size_t r = row_index(pg, h, pos[n] % P, Hkv, P);
                quant_vector(enc, D, x.data(), quat, cp + r * cb, sp + r * sb);
            }
        }
    }
    return bad;
}

// ---- gather + dequantize one sequence: k_out, v_out [L][Hkv][D] (original domain) ----
int orc_gather_dequant(int fmt, int num_pages, int Hkv, int D, int P,
                       const uint8_t* kc, const uint8_t* ks, const uint8_t* vc, const uint8_t* vs,
                       const int32_t* page_table, int max_pages, int b, int L, const float* quat,
                       double* k_out, double* v_out) {
    for (int t = 0; t < L; ++t) {
        if (dequant_token(fmt, 0, num_pages, Hkv, D, P, kc, ks, page_table, max_pages, b, t, quat,
                          k_out + (size_t)t * Hkv * D)) return -1;
        if (dequant_token(fmt, 1, num_pages, Hkv, D, P, vc, vs, page_table, max_pages, b, t, quat,
                          v_out + (size_t)t * Hkv * D)) return -1;
    }
    return 0;
}

// ---- decode attention ----
// For sequence b and query head h (KV head h / (Hq/Hkv)): scores
// s_t = scale * <q_h, k_t> over t < seq_lens[b], softmax, o = sum_t p_t v_t,
// with K/V dequantized from the pool through the page table ("attention over
// the dequantized tensors" [FT "Correctness"; K4 "Tests"]). Output [B][Hq][D].
// An empty sequence gives a zero output.
int orc_decode(int fmt, int num_pages, int Hkv, int D, int P,
               const uint8_t* kc, const uint8_t* ks, const uint8_t* vc, const uint8_t* vs,
               const uint16_t* q_bf16, int B, int Hq, const int32_t* page_table, int max_pages,
               const int32_t* seq_lens, float scale, const float* quat, double* out) {
    if (Hq % Hkv) return -2;
    int G = Hq / Hkv;
    for (int b = 0; b < B; ++b) {
        int L = seq_lens[b];
        std::vector<double> K((size_t)L * Hkv * D), V((size_t)L * Hkv * D);
        if (orc_gather_dequant(fmt, num_pages, Hkv, D, P, kc, ks, vc, vs, page_table, max_pages, b, L, quat,
                               K.data(), V.data())) return -1;
        std::vector<double> s(L);
        std::vector<const double*> vr(L);
        for (int h = 0; h < Hq; ++h) {
            int g = h / G;
            const uint16_t* q = q_bf16 + ((size_t)b * Hq + h) * D;
            for (int t = 0; t < L; ++t) {
                double acc = 0.0;
                const double* k = &K[((size_t)t * Hkv + g) * D];
                for (int i = 0; i < D; ++i) acc += (double)float_from_bf16(q[i]) * k[i];
                s[t] = (double)scale * acc;
                vr[t] = &V[((size_t)t * Hkv + g) * D];
            }
            attend(D, L, s.data(), vr.data(), out + ((size_t)b * Hq + h) * D);
        }
    }
    return 0;
}

// Same attention computed as independent partial softmaxes over the token
// ranges [bounds[j], bounds[j+1]) followed by the partial-softmax merge
// M = max_j m_j, o = sum_j e^{m_j - M} o_j / sum_j e^{m_j - M} l_j.
// Sequence 0 only; out [Hq][D]. Used to pin the merge rule.
int orc_decode_split(int fmt, int num_pages, int Hkv, int D, int P,
                     const uint8_t* kc, const uint8_t* ks, const uint8_t* vc, const uint8_t* vs,
                     const uint16_t* q_bf16, int Hq, const int32_t* page_table, int max_pages,
                     int L, float scale, const float* quat, const int32_t* bounds, int nsplit, double* out) {
    int G = Hq / Hkv;
    std::vector<double> K((size_t)L * Hkv * D), V((size_t)L * Hkv * D);
    if (orc_gather_dequant(fmt, num_pages, Hkv, D, P, kc, ks, vc, vs, page_table, max_pages, 0, L, quat,
                           K.data(), V.data())) return -1;
    for (int h = 0; h < Hq; ++h) {
        int g = h / G;
        const uint16_t* q = q_bf16 + (size_t)h * D;
        std::vector<double> m(nsplit, -INFINITY), l(nsplit, 0.0), o((size_t)nsplit * D, 0.0);
        for (int j = 0; j < nsplit; ++j) {
            for (int t = bounds[j]; t < bounds[j + 1]; ++t) {
                double acc = 0.0;
                for (int i = 0; i < D; ++i) acc += (double)float_from_bf16(q[i]) * K[((size_t)t * Hkv + g) * D + i];
                m[j] = std::fmax(m[j], (double)scale * acc);
            }
            for (int t = bounds[j]; t < bounds[j + 1]; ++t) {
                double acc = 0.0;
                for (int i = 0; i < D; ++i) acc += (double)float_from_bf16(q[i]) * K[((size_t)t * Hkv + g) * D + i];
                double p = std::exp((double)scale * acc - m[j]);
                l[j] += p;
                for (int i = 0; i < D; ++i) o[(size_t)j * D + i] += p * V[((size_t)t * Hkv + g) * D + i];
            }
        }
        double M = -INFINITY;
        for (int j = 0; j < nsplit; ++j) M = std::fmax(M, m[j]);
        double Lsum = 0.0;
        for (int j = 0; j < nsplit; ++j) if (l[j] > 0) Lsum += std::exp(m[j] - M) * l[j];
        for (int i = 0; i < D; ++i) {
            double acc = 0.0;
            for (int j = 0; j < nsplit; ++j) if (l[j] > 0) acc += std::exp(m[j] - M) * o[(size_t)j * D + i];
            out[(size_t)h * D + i] = acc / Lsum;
        }
    }
    return 0;
}

// ---- verify window (several decode queries per sequence) ----
// [S8 "What it does": the verify windows go through the decode kernels; K4
// "Tests": the batched forms with per-query step arrays]. Sequence b has
// W = cu[b+1] - cu[b] queries (rows cu[b] .. cu[b+1]-1 of q) for its last W
// positions: query j sits at position seq_lens[b] - W + j and attends
// positions [0, seq_lens[b] - W + j + 1), all read back from the pool (the
// window's tokens were packed when they were appended). This is decode, run
// once per query with its own length. Returns -3 if W > seq_lens[b].
int orc_verify(int fmt, int num_pages, int Hkv, int D, int P,
               const uint8_t* kc, const uint8_t* ks, const uint8_t* vc, const uint8_t* vs,
               const uint16_t* q_bf16, int B, int Hq, const int32_t* cu, const int32_t* page_table, int max_pages,
               const int32_t* seq_lens, float scale, const float* quat, double* out) {
    for (int b = 0; b < B; ++b) {
        int W = cu[b + 1] - cu[b];
        if (W > seq_lens[b]) return -3;
        for (int j = 0; j < W; ++j) {
            int row = cu[b] + j;
            int len = seq_lens[b] - W + j + 1;
            int rc = orc_decode(fmt, num_pages, Hkv, D, P, kc, ks, vc, vs, q_bf16 + (size_t)row * Hq * D, 1, Hq,
                                page_table + (size_t)b * max_pages, max_pages, &len, scale, quat,
                                out + (size_t)row * Hq * D);
            if (rc) return rc;
        }
    }
    return 0;
}

// ---- extend (prefill-chunk) attention ----
// [FT "What"]: the chunk attends the packed prefix plus the bf16 new tokens,
// which are packed only after attention (prefill never reads its own quantized
// KV). For sequence b with new tokens [cu[b], cu[b+1]) and prefix length
// prefix_lens[b], new token i attends the dequantized prefix positions
// [0, prefix_lens[b]) followed by the raw new tokens j <= i (causal) or all new
// tokens (causal == 0). `rows` lists which global new-token indices to compute
// (nrows of them; rows == NULL computes all, nrows = cu[B]); out [nrows][Hq][D].
int orc_extend(int fmt, int num_pages, int Hkv, int D, int P,
               const uint8_t* kc, const uint8_t* ks, const uint8_t* vc, const uint8_t* vs,
               const uint16_t* q_bf16, const uint16_t* k_new, const uint16_t* v_new, int Hq,
               const int32_t* cu, const int32_t* prefix_lens, int B,
               const int32_t* page_table, int max_pages, float scale, int causal, const float* quat,
               const int32_t* rows, int nrows, double* out) {
    if (Hq % Hkv) return -2;
    int G = Hq / Hkv;
    int total = cu[B];
    if (!rows) nrows = total;
    for (int b = 0; b < B; ++b) {
        int L0 = prefix_lens[b], T0 = cu[b], T1 = cu[b + 1];
        bool any = false;
        for (int r = 0; r < nrows; ++r) {
            int i = rows ? rows[r] : r;
            if (i >= T0 && i < T1) { any = true; break; }
        }
        if (!any) continue;
        std::vector<double> K((size_t)L0 * Hkv * D), V((size_t)L0 * Hkv * D);
        if (orc_gather_dequant(fmt, num_pages, Hkv, D, P, kc, ks, vc, vs, page_table, max_pages, b, L0, quat,
                               K.data(), V.data())) return -1;
        int nmax = L0 + (T1 - T0);
        std::vector<double> s(nmax), vnew((size_t)(T1 - T0) * Hkv * D);
        for (size_t i = 0; i < vnew.size(); ++i) vnew[i] = float_from_bf16(v_new[(size_t)T0 * Hkv * D + i]);
        std::vector<const double*> vr(nmax);
        for (int r = 0; r < nrows; ++r) {
            int i = rows ? rows[r] : r;
            if (i < T0 || i >= T1) continue;
            int nk = L0 + (causal ? (i - T0 + 1) : (T1 - T0));
            for (int h = 0; h < Hq; ++h) {
                int g = h / G;
                const uint16_t* q = q_bf16 + ((size_t)i * Hq + h) * D;
                for (int t = 0; t < nk; ++t) {
                    double acc = 0.0;
                    if (t < L0) {
                        const double* k = &K[((size_t)t * Hkv + g) * D];
                        for (int d = 0; d < D; ++d) acc += (double)float_from_bf16(q[d]) * k[d];
                        vr[t] = &V[((size_t)t * Hkv + g) * D];
                    } else {
                        int j = T0 + (t - L0);
                        const uint16_t* k = k_new + ((size_t)j * Hkv + g) * D;
                        for (int d = 0; d < D; ++d) acc += (double)float_from_bf16(q[d]) * (double)float_from_bf16(k[d]);
                        vr[t] = &vnew[((size_t)(j - T0) * Hkv + g) * D];
                    }
                    s[t] = (double)scale * acc;
                }
                attend(D, nk, s.data(), vr.data(), out + ((size_t)r * Hq + h) * D);
            }
        }
    }
    return 0;
}

}  // extern "C"
