// quant_rows.cuh -- one warp quantizes one head vector (one row of a plane):
// int8 groups, FWHT-256 + q4_0, and ISO3/ISO4 blocks. Every fp32 step uses an
// explicitly rounded intrinsic in a fixed order, so the packed bytes are a pure
// function of the bf16 input. Used by the append kernel and by the decode
// kernel's fused quantize-on-write.
//
// Methods (page title, section):
//   int8   "qwen35/q36: --kv - int8 K/V caches", "What it does": codes + one fp16
//          scale (group absmax / 127) per 64 values; rounding half to even per
//          "--kv k8v4", "Tests".
//   q4_0   "--kv k8v4: hybrid KV cache", "What"/"How": V rotated by the 1/16-
//          normalised FWHT-256, then q4_0 (d = signed absmax / -8,
//          q = min(15, trunc(x/d + 8.5))).
//   bf16   "qwen35/q36: --kv - int8 K/V caches", "What it does": the one-store
//          formats leave the other store unquantized (here: the bf16 input).
//   ISO    "feat(kvcache): add ISO3/ISO4 KV-cache quantization", "What": per 128
//          values L2-normalise, rotate each 4-D group by a unit quaternion, code
//          to the nearest Lloyd-Max level, store ||x|| / ||levels||.
#pragma once

#include "qkv_device.cuh"

namespace qkv {

// Sum of squares of the warp's 128 values (4 per lane), fixed order: the lane's
// four squares left to right, then a butterfly at distances 16, 8, 4, 2, 1.
__device__ __forceinline__ float warp_sumsq4(const float (&x)[4]) {
    float s = __fmul_rn(x[0], x[0]);
    s = __fadd_rn(s, __fmul_rn(x[1], x[1]));
    s = __fadd_rn(s, __fmul_rn(x[2], x[2]));
    s = __fadd_rn(s, __fmul_rn(x[3], x[3]));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, off));
    return s;
}

// Hamilton product q (x) v, components left to right from the textbook expansion.
__device__ __forceinline__ void quat_left_mul(const float* q, const float (&v)[4], float (&y)[4]) {
    float r0 = __fmul_rn(q[0], v[0]);
    r0 = __fsub_rn(r0, __fmul_rn(q[1], v[1]));
    r0 = __fsub_rn(r0, __fmul_rn(q[2], v[2]));
    r0 = __fsub_rn(r0, __fmul_rn(q[3], v[3]));
    float r1 = __fmul_rn(q[0], v[1]);
    r1 = __fadd_rn(r1, __fmul_rn(q[1], v[0]));
    r1 = __fadd_rn(r1, __fmul_rn(q[2], v[3]));
    r1 = __fsub_rn(r1, __fmul_rn(q[3], v[2]));
    float r2 = __fmul_rn(q[0], v[2]);
    r2 = __fsub_rn(r2, __fmul_rn(q[1], v[3]));
    r2 = __fadd_rn(r2, __fmul_rn(q[2], v[0]));
    r2 = __fadd_rn(r2, __fmul_rn(q[3], v[1]));
    float r3 = __fmul_rn(q[0], v[3]);
    r3 = __fadd_rn(r3, __fmul_rn(q[1], v[2]));
    r3 = __fsub_rn(r3, __fmul_rn(q[2], v[1]));
    r3 = __fadd_rn(r3, __fmul_rn(q[3], v[0]));
    y[0] = r0; y[1] = r1; y[2] = r2; y[3] = r3;
}

template <int D>
__device__ __forceinline__ void load_row_f32(const uint16_t* src, int lane, float (&x)[D / 32]) {
    constexpr int E = D / 32;
    const uint16_t* p = src + lane * E;
    if constexpr (E == 8) {
        uint4 w = *reinterpret_cast<const uint4*>(p);
        uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) { x[2 * i] = bf16_bits_to_f32(ws[i] & 0xffffu); x[2 * i + 1] = bf16_bits_to_f32(ws[i] >> 16); }
    } else {
        uint2 w = *reinterpret_cast<const uint2*>(p);
        uint32_t ws[2] = {w.x, w.y};
#pragma unroll
        for (int i = 0; i < 2; ++i) { x[2 * i] = bf16_bits_to_f32(ws[i] & 0xffffu); x[2 * i + 1] = bf16_bits_to_f32(ws[i] >> 16); }
    }
}

// ---- int8: E = D/32 values per lane, 64/E lanes per 64-value group ----
template <int D>
__device__ void append_int8_row(const uint16_t* src, uint8_t* code, uint8_t* scale, int lane) {
    constexpr int E = D / 32, LPG = 64 / E;
    float x[E];
    load_row_f32<D>(src, lane, x);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < E; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int off = 1; off < LPG; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    float d = __fdiv_rn(amax, 127.0f);
    uint16_t h = f32_to_f16_sat(d);
    float dh = f16_bits_to_f32(h);
    uint32_t packed[E / 4];
#pragma unroll
    for (int w = 0; w < E / 4; ++w) {
        uint32_t acc = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int q = 0;
            if (dh != 0.0f) {
                q = __float2int_rn(__fdiv_rn(x[4 * w + j], dh));
                q = max(-127, min(127, q));
            }
            acc |= ((uint32_t)(q & 0xff)) << (8 * j);
        }
        packed[w] = acc;
    }
    if constexpr (E == 8) *reinterpret_cast<uint2*>(code + lane * 8) = make_uint2(packed[0], packed[1]);
    else *reinterpret_cast<uint32_t*>(code + lane * 4) = packed[0];
    if (lane % LPG == 0) reinterpret_cast<uint16_t*>(scale)[lane / LPG] = h;
}

// ---- q4_0 of the FWHT-256-rotated vector (D = 256, 8 values per lane) ----
__device__ inline void append_q4_row(const uint16_t* src, uint8_t* code, uint8_t* scale, int lane) {
    float x[8];
    load_row_f32<256>(src, lane, x);
    // butterflies at strides 1, 2, 4 inside the lane: (a, b) -> (a + b, a - b)
#pragma unroll
    for (int h = 1; h < 8; h <<= 1)
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if ((j & h) == 0) {
                float a = x[j], b = x[j + h];
                x[j] = __fadd_rn(a, b);
                x[j + h] = __fsub_rn(a, b);
            }
    // strides 8 .. 128 across lanes (lane bit k <-> stride 8 << k)
#pragma unroll
    for (int k = 0; k < 5; ++k) {
        bool upper = (lane >> k) & 1;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float o = __shfl_xor_sync(0xffffffffu, x[j], 1 << k);
            x[j] = upper ? __fsub_rn(o, x[j]) : __fadd_rn(x[j], o);
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = __fmul_rn(x[j], 0.0625f);
    // block of 32 = lanes 4m..4m+3; signed value of largest magnitude, first index on ties
    float amax = 0.0f, m = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float a = fabsf(x[j]);
        if (a > amax) { amax = a; m = x[j]; }
    }
    int src_lane = lane;
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
        float oa = __shfl_xor_sync(0xffffffffu, amax, off);
        float om = __shfl_xor_sync(0xffffffffu, m, off);
        int ol = __shfl_xor_sync(0xffffffffu, src_lane, off);
        if (oa > amax || (oa == amax && ol < src_lane)) { amax = oa; m = om; src_lane = ol; }
    }
    float d = __fdiv_rn(m, -8.0f);
    uint16_t h = f32_to_f16_sat(d);
    float dh = f16_bits_to_f32(h);
    uint32_t nib = 0;  // 8 codes, 4 bits each
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        int q = 8;
        if (dh != 0.0f) {
            float t = __fadd_rn(__fdiv_rn(x[j], dh), 8.5f);
            q = __float2int_rz(t);
            q = max(0, min(15, q));
        }
        nib |= (uint32_t)q << (4 * j);
    }
    // byte j of the block = code j | code (j + 16) << 4: lanes 4m, 4m+1 own the
    // low nibbles, lanes 4m+2, 4m+3 the high ones
    uint32_t hi = __shfl_down_sync(0xffffffffu, nib, 2);
    int sub = lane & 3;
    if (sub < 2) {
        uint32_t b0 = 0, b1 = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            b0 |= (((nib >> (4 * j)) & 15u) | (((hi >> (4 * j)) & 15u) << 4)) << (8 * j);
            b1 |= (((nib >> (4 * (j + 4))) & 15u) | (((hi >> (4 * (j + 4))) & 15u) << 4)) << (8 * j);
        }
        *reinterpret_cast<uint2*>(code + (lane >> 2) * 16 + sub * 8) = make_uint2(b0, b1);
    }
    if (sub == 0) reinterpret_cast<uint16_t*>(scale)[lane >> 2] = h;
}

// ---- ISO3 / ISO4: one 128-value block per pass, 4 values per lane ----
template <int BITS>
__device__ void append_iso_block(const uint16_t* src, uint8_t* code, uint8_t* scale, int lane, const float* quat,
                                 const float* levels, const float* mids) {
    constexpr int NL = BITS == 3 ? 8 : 16;
    float x[4];
    {
        uint2 w = *reinterpret_cast<const uint2*>(src + lane * 4);
        x[0] = bf16_bits_to_f32(w.x & 0xffffu); x[1] = bf16_bits_to_f32(w.x >> 16);
        x[2] = bf16_bits_to_f32(w.y & 0xffffu); x[3] = bf16_bits_to_f32(w.y >> 16);
    }
    float n = __fsqrt_rn(warp_sumsq4(x));
    float v[4], y[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = (n == 0.0f) ? 0.0f : __fdiv_rn(x[e], n);
    quat_left_mul(quat, v, y);
    int k[4];
    float cv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        int c = 0;
#pragma unroll
        for (int j = 0; j < NL - 1; ++j) c += (y[e] > mids[j]) ? 1 : 0;
        k[e] = c;
        cv[e] = levels[c];
    }
    float cn = __fsqrt_rn(warp_sumsq4(cv));
    uint16_t s16 = f32_to_f16_sat(__fdiv_rn(n, cn));
    if constexpr (BITS == 3) {
        uint32_t lo = (uint32_t)((k[0] & 3) | ((k[1] & 3) << 2) | ((k[2] & 3) << 4) | ((k[3] & 3) << 6));
        uint32_t hn = (uint32_t)(((k[0] >> 2) & 1) | (((k[1] >> 2) & 1) << 1) | (((k[2] >> 2) & 1) << 2) | (((k[3] >> 2) & 1) << 3));
        uint32_t hn_next = __shfl_down_sync(0xffffffffu, hn, 1);
        code[lane] = (uint8_t)lo;
        if ((lane & 1) == 0) code[32 + (lane >> 1)] = (uint8_t)(hn | (hn_next << 4));
        if (lane == 0) reinterpret_cast<uint16_t*>(scale)[0] = s16;
    } else {
        uint16_t w = (uint16_t)(k[0] | (k[1] << 4) | (k[2] << 8) | (k[3] << 12));
        reinterpret_cast<uint16_t*>(code)[lane] = w;
        if (lane == 0) { reinterpret_cast<uint16_t*>(scale)[0] = s16; reinterpret_cast<uint16_t*>(scale)[1] = 0; }
    }
}


// One row of store encoding ENC (all D values), written to code/scale.
template <int ENC, int D>
__device__ __forceinline__ void quantize_row(const uint16_t* src, uint8_t* code, uint8_t* scale, int lane,
                                             const float* quat, const float* levels, const float* mids) {
    if constexpr (ENC == ENC_BF16) {
        // the unquantized store: the bf16 input row as it is (D / 8 lanes move 16 bytes each)
        (void)scale;
        if (lane < D / 8) reinterpret_cast<uint4*>(code)[lane] = reinterpret_cast<const uint4*>(src)[lane];
    } else if constexpr (ENC == ENC_INT8) {
        append_int8_row<D>(src, code, scale, lane);
    } else if constexpr (ENC == ENC_Q4) {
        append_q4_row(src, code, scale, lane);
    } else {
        constexpr int BITS = ENC == ENC_ISO3 ? 3 : 4;
#pragma unroll 1
        for (int b = 0; b < D / 128; ++b)
            append_iso_block<BITS>(src + 128 * b, code + b * (BITS == 3 ? 48 : 64), scale + b * (BITS == 3 ? 2 : 4),
                                   lane, quat, levels, mids);
    }
}

}  // namespace qkv
