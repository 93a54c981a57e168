// decode.cu -- paged split-K decode attention over the quantized pool, with an
// optional fused quantize-on-write of each sequence's newest token.
//
// Method (page title, section):
//   "qwen35/q36: --kv - int8 K/V caches", "What it does": decode splits the
//   context ("part" kernels) and dequantizes K/V on the fly.
//   "--kv k8v4: hybrid KV cache", "How": K int8 unrotated (q is not rotated), V
//   in the FWHT-256 domain; the attention output is rotated back.
//   "feat(kvcache): add ISO3/ISO4 KV-cache quantization", "What": dequant is
//   norm * (conjugate rotation of the levels); here the query is rotated once
//   instead, <q, conj(R) c> = <R q, c>, and the output is rotated back once.
//   Quantize-on-write: the decode token is packed when written and read back
//   packed (same page, "What": decode is quantize-on-write).
//
// GB300 design (one CTA of 8 warps per SM):
//   * Work is the list of (sequence, KV-head group, page) units; each CTA takes
//     an equal contiguous share (stream-K style), so any mix of lengths keeps
//     every SM equally busy. A share may span several sequences ("pieces").
//   * Each warp owns a contiguous run of pages and a 3-stage TMA pipeline in
//     shared memory (2-D tiled copies with 128-byte swizzle for int8/q4 code
//     planes, 1-D bulk copies for scales and ISO codes) completing on
//     mbarriers; page ids come through a 32-wide register ring.
//   * The page loop is software-pipelined: one straight-line block holds
//     QK^T of page i + 1, the softmax of page i and PV of page i, which share no
//     data, so each warp carries two independent tensor-core chains.
//   * QK^T and PV are warp-level fp16 tensor-core products (m16n8k16) on exact
//     operands: int8 K codes enter as 1152 + c (exact in fp16; the constant is
//     removed per page and group through the query sums), V codes exactly, q4 and
//     Lloyd-Max levels are exact fp16, the (rotated) query is split into fp16
//     hi + lo rows, per-(token, group) scales multiply fp32 scores (K) or are
//     folded into fp16 hi + lo probabilities (V).
//   * Lazy online softmax (base 2): probabilities use a frame max that moves
//     only when a page exceeds it by 2^8 (checked after each page, a rare
//     warp-uniform branch), with a power-of-two range factor keeping
//     probability x V-scale in the fp16 normal range.
//   * Warps merge in shared memory; CTAs merge through the caller's workspace
//     with the partial-softmax rule, done by the last-arriving CTA of each
//     group of pieces (atomic ticket, no waiting), in two levels.
#include "qkv_device.cuh"
#include "qkv_params.h"
#include "quant_rows.cuh"

namespace qkv {

__device__ unsigned int g_err_decode;
__constant__ float c_dec_levels[2][16];
__constant__ float c_dec_mids[2][16];

constexpr int kNW = 8;          // warps per CTA
constexpr int kMaxBatch = 1024; // sequences per call (prefix table in shared memory)
constexpr int kMaxMerge = 64;   // partials merged by one CTA in one level
constexpr int kThreads = kNW * 32;

// ---------------------------------------------------------------------------
// compile-time geometry: code planes of all stages first (1 KB aligned for the
// swizzle), then the scale planes of all stages
// ---------------------------------------------------------------------------
template <int KENC, int VENC, int D>
struct StageGeo {
    static constexpr int KCB = code_row_bytes(KENC, D), KSB = scale_row_bytes(KENC, D);
    static constexpr int VCB = code_row_bytes(VENC, D), VSB = scale_row_bytes(VENC, D);
    static constexpr bool K_TMA = (KENC == ENC_INT8);      // swizzled 2-D boxes of 16 rows x 128 B
    static constexpr bool V_TMA = (VENC == ENC_INT8 || VENC == ENC_Q4);
    static constexpr int al(int x, int a) { return (x + a - 1) / a * a; }
    static constexpr int OFF_KC = 0;
    static constexpr int OFF_VC = al(kPage * KCB, 1024);
    static constexpr int CODE_BYTES = al(OFF_VC + kPage * VCB, 1024);
    static constexpr int OFF_KS = 0;
    static constexpr int OFF_VS = al(kPage * KSB, 16);
    static constexpr int SCALE_BYTES = al(OFF_VS + kPage * VSB, 16);
    static constexpr int TX = kPage * (KCB + KSB + VCB + VSB);
};

// byte address inside a 128-byte-swizzled tile of 16 rows (box width 128 B)
__device__ __forceinline__ int swz(int row, int byte) {
    return (byte >> 7) * 2048 + row * 128 + ((((byte >> 4) & 7) ^ (row & 7)) << 4) + (byte & 15);
}

template <typename T>
__device__ __forceinline__ T lds(const uint8_t* base, int off) { return *reinterpret_cast<const T*>(base + off); }

// int8 word (4 codes) -> half2(1152 + c0, 1152 + c1), half2(1152 + c2, 1152 + c3), exact
__device__ __forceinline__ void i8x4_to_h2x2_biased(uint32_t w, uint32_t& h01, uint32_t& h23) {
    const uint32_t x = w ^ 0x80808080u;
    h01 = prmt(x, 0x64646464u, 0x4140u);
    h23 = prmt(x, 0x64646464u, 0x4342u);
}
// byte i of a and byte i of b -> half2(1152 + a_i, 1152 + b_i), exact
__device__ __forceinline__ uint32_t i8pair_to_h2_biased(uint32_t a, uint32_t b, int i) {
    const uint32_t sel = (uint32_t)(i | (i << 4) | ((4 + i) << 8) | ((4 + i) << 12));
    return lop3_and_xor(prmt(a, b, sel), 0x00ff00ffu, 0x64806480u);
}

template <int KENC, int VENC, int D, int G>
struct Cfg {
    using Geo = StageGeo<KENC, VENC, D>;
    static constexpr bool KISO = (KENC == ENC_ISO3 || KENC == ENC_ISO4);
    static constexpr bool VISO = (VENC == ENC_ISO3 || VENC == ENC_ISO4);
    static constexpr bool QLO = KISO;               // rotated query needs an fp16 lo part
    static constexpr bool KBIAS = (KENC == ENC_INT8);
    static constexpr int KS = D / 16;               // k-steps over the head dimension
    static constexpr int KSPG = group_size(KENC) / 16;
    static constexpr int NGK = D / group_size(KENC);
    static constexpr int MT = D / 16;               // PV m-tiles (16 dims each)
    static constexpr int MTPG = group_size(VENC) / 16;
    static constexpr int NGV = D / group_size(VENC);
    static constexpr bool ISO_LUT = KISO || VISO;
    static constexpr int LUT_ENTRIES = (KENC == ENC_ISO4 || VENC == ENC_ISO4) ? 256 : 64;
    static constexpr int LUT_BYTES = ISO_LUT ? LUT_ENTRIES * 32 * 4 : 0;
    static constexpr int ROW_BYTES = kNW * 512;              // per-warp scratch for the fused quantize-on-write
    static constexpr int SMALL_BYTES = kNW * 8 * 4 * 2 + kMaxMerge * 8 * 4 + 64;
    static constexpr int FIXED = LUT_BYTES + ROW_BYTES + SMALL_BYTES + kNW * 4 * 8 + (kMaxBatch + 1) * 4;
    static constexpr int BUDGET = 225 * 1024 - FIXED - 1024;  // dynamic bytes for stages
    static constexpr int NS_FIT = BUDGET / (kNW * (Geo::CODE_BYTES + Geo::SCALE_BYTES));
    static constexpr int NS = NS_FIT >= 4 ? 4 : NS_FIT;
    static constexpr int PIPE_CODE = kNW * NS * Geo::CODE_BYTES;
    static constexpr int PIPE_BYTES = PIPE_CODE + kNW * NS * Geo::SCALE_BYTES;
    static constexpr int MERGE_BYTES = kNW * 8 * D * 4;
    static constexpr int AREA = ((PIPE_BYTES > MERGE_BYTES ? PIPE_BYTES : MERGE_BYTES) + 1023) / 1024 * 1024;
    static constexpr int OFF_LUT = AREA;
    static constexpr int OFF_ROW = OFF_LUT + LUT_BYTES;
    static constexpr int OFF_SMALL = OFF_ROW + ROW_BYTES;      // warp m/l + merge weights
    static constexpr int OFF_BAR = OFF_SMALL + SMALL_BYTES;
    static constexpr int OFF_PREF = OFF_BAR + kNW * 4 * 8;
    static constexpr int SMEM = OFF_PREF + (kMaxBatch + 1) * 4;
    static_assert(NS >= 3, "the software pipeline keeps three pages per warp");
    static_assert(SMEM + 1024 + 1536 <= 232448, "shared memory budget (dynamic + alignment slack + static)");
};

// final output row: o [G][D] fp32 in shared memory, already normalised
template <int VENC, int D, int G>
__device__ void write_output(const DecodeParams& p, float* o, int b, int hq0, int tid) {
    if constexpr (VENC == ENC_Q4) {
        // inverse FWHT-256 (the transform is its own inverse) per head, one warp per head
        const int w = tid >> 5, lane = tid & 31;
        for (int h = w; h < G; h += kNW) {
            float x[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) x[j] = o[h * D + lane * 8 + j];
#pragma unroll
            for (int hh = 1; hh < 8; hh <<= 1)
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if ((j & hh) == 0) { float a = x[j], c = x[j + hh]; x[j] = a + c; x[j + hh] = a - c; }
#pragma unroll
            for (int k = 0; k < 5; ++k) {
                bool upper = (lane >> k) & 1;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float ot = __shfl_xor_sync(0xffffffffu, x[j], 1 << k);
                    x[j] = upper ? ot - x[j] : x[j] + ot;
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) o[h * D + lane * 8 + j] = x[j] * 0.0625f;
        }
        __syncthreads();
    } else if constexpr (VENC == ENC_ISO3 || VENC == ENC_ISO4) {
        // undo the rotation: conj(q) (x) o per 4-D group
        const float q0 = p.quat[0], q1 = -p.quat[1], q2 = -p.quat[2], q3 = -p.quat[3];
        for (int i = tid; i < G * D / 4; i += blockDim.x) {
            float* v = o + 4 * i;
            float a = v[0], bb = v[1], c = v[2], d = v[3];
            float y0 = q0 * a - q1 * bb - q2 * c - q3 * d;
            float y1 = q0 * bb + q1 * a + q2 * d - q3 * c;
            float y2 = q0 * c - q1 * d + q2 * a + q3 * bb;
            float y3 = q0 * d + q1 * c - q2 * bb + q3 * a;
            v[0] = y0; v[1] = y1; v[2] = y2; v[3] = y3;
        }
        __syncthreads();
    }
    const size_t base = ((size_t)b * p.Hq + hq0) * D;
    if (p.out_f32) {
        float* out = reinterpret_cast<float*>(p.out) + base;
        for (int i = tid; i < G * D; i += blockDim.x) out[i] = o[i];
    } else {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + base;
        for (int i = tid; i < G * D; i += blockDim.x) out[i] = __float2bfloat16_rn(o[i]);
    }
}

// Merge n partial slots (m[8], l[8], O[8][D]) into either a partial slot `dst`
// or the final output. Partial-softmax rule: M = max m_j,
// O = sum_j 2^(m_j - M) O_j, L = sum_j 2^(m_j - M) l_j (base-2 scores).
template <int VENC, int D, int G>
__device__ void merge_slots(const DecodeParams& p, const float* const* slots, int n, float* dst, bool final_out,
                            int b, int hq0, float* sm_w, float* sm_o, int tid) {
    __shared__ float s_M[8], s_L[8];
    if (tid < G) {
        float M = -INFINITY;
        for (int j = 0; j < n; ++j) M = fmaxf(M, slots[j][tid]);
        float L = 0.0f;
        for (int j = 0; j < n; ++j) {
            float mj = slots[j][tid];
            float w = (mj == -INFINITY) ? 0.0f : exp2f(mj - M);
            sm_w[j * 8 + tid] = w;
            L += w * slots[j][8 + tid];
        }
        s_M[tid] = M;
        s_L[tid] = L;
    }
    __syncthreads();
    for (int i = tid; i < G * D; i += blockDim.x) {
        int h = i / D;
        float acc = 0.0f;
        for (int j = 0; j < n; ++j) acc += sm_w[j * 8 + h] * slots[j][16 + i];
        if (final_out) {
            float L = s_L[h];
            sm_o[i] = (L > 0.0f) ? acc / L : 0.0f;
        } else {
            dst[16 + i] = acc;
        }
    }
    if (!final_out && tid < G) { dst[tid] = s_M[tid]; dst[8 + tid] = s_L[tid]; }
    __syncthreads();
    if (final_out) write_output<VENC, D, G>(p, sm_o, b, hq0, tid);
}

// Per-warp page pipeline state and the three per-page operations. Thread
// (g = lane / 4, t = lane % 4) holds the scores of head g % G for the tokens
// 2t, 2t + 1, 2t + 8, 2t + 9 of a page (the C fragment of the QK^T product).
template <int KENC, int VENC, int D, int G>
struct WarpPipe {
    using K = Cfg<KENC, VENC, D, G>;
    using Geo = typename K::Geo;

    // QK^T over the full head dimension for one page: base-2 logits, masked
    // beyond `valid` tokens.
    static __device__ __forceinline__ void scores(const uint8_t* st, const uint8_t* ss, const uint32_t (&qa)[K::KS][4],
                                                  const float (&qbias)[K::NGK], const uint32_t* lut, int g, int t,
                                                  int valid, float scale_log2, float (&sc)[4]) {
        float ksc[4][K::NGK];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int tok = 2 * t + (j & 1) + 8 * (j >> 1);
            if constexpr (KENC == ENC_INT8 && K::NGK == 4) {
                const uint2 w = lds<uint2>(ss, Geo::OFF_KS + tok * Geo::KSB);
                const float2 a = h2_to_f32x2(w.x), b = h2_to_f32x2(w.y);
                ksc[j][0] = a.x; ksc[j][1] = a.y; ksc[j][2] = b.x; ksc[j][3] = b.y;
            } else if constexpr (KENC == ENC_INT8 && K::NGK == 2) {
                const float2 a = h2_to_f32x2(lds<uint32_t>(ss, Geo::OFF_KS + tok * Geo::KSB));
                ksc[j][0] = a.x; ksc[j][1] = a.y;
            } else {
#pragma unroll
                for (int gg = 0; gg < K::NGK; ++gg)
                    ksc[j][gg] = f16_bits_to_f32(lds<uint16_t>(ss, Geo::OFF_KS + tok * Geo::KSB + (KENC == ENC_ISO4 ? 4 : 2) * gg));
            }
        }
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int gg = 0; gg < K::NGK; ++gg) {
            float cacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int r = g + 8 * nt;
                if constexpr (KENC == ENC_INT8) {
                    const uint4 w = lds<uint4>(st, Geo::OFF_KC + swz(r, 64 * gg + 16 * t));
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        uint32_t b0, b1;
                        i8x4_to_h2x2_biased(ws[u], b0, b1);
                        const int ks = gg * 4 + u;
                        mma_f16_16816(cacc[nt], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
                    }
                } else if constexpr (KENC == ENC_ISO3) {
                    const int rb = Geo::OFF_KC + r * Geo::KCB + 48 * gg;
                    const uint2 lo2 = lds<uint2>(st, rb + 8 * t);
                    const uint32_t hib = lds<uint32_t>(st, rb + 32 + 4 * t);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const uint32_t lb = ((u < 4 ? lo2.x : lo2.y) >> (8 * (u & 3))) & 0xffu;
                        const uint32_t hb = (hib >> (4 * u)) & 0xfu;
                        const uint32_t i0 = (lb & 0xfu) | ((hb & 3u) << 4);
                        const uint32_t i1 = (lb >> 4) | ((hb >> 2) << 4);
                        const int ks = gg * 8 + u;
                        mma_f16_16816(cacc[nt], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], lut[i0 * 32], lut[i1 * 32]);
                    }
                } else {  // ISO4
                    const uint4 w = lds<uint4>(st, Geo::OFF_KC + r * Geo::KCB + 64 * gg + 16 * t);
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const uint32_t wd = ws[u >> 1];
                        const uint32_t i0 = (wd >> (16 * (u & 1))) & 0xffu;
                        const uint32_t i1 = (wd >> (16 * (u & 1) + 8)) & 0xffu;
                        const int ks = gg * 8 + u;
                        mma_f16_16816(cacc[nt], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], lut[i0 * 32], lut[i1 * 32]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int nt = j >> 1, e = j & 1;
                float cv = cacc[nt][e];
                if constexpr (K::QLO) cv += cacc[nt][2 + e];
                if constexpr (K::KBIAS) cv -= qbias[gg];
                acc[j] += ksc[j][gg] * cv;
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int tok = 2 * t + (j & 1) + 8 * (j >> 1);
            sc[j] = (tok < valid) ? acc[j] * scale_log2 : -INFINITY;
        }
    }

    // V scales of one page for this thread's four tokens (zero beyond `valid`)
    // and the largest fp16 exponent field among them over the warp.
    static __device__ __forceinline__ uint32_t vscales(const uint8_t* ss, int t, int valid, float (&sv)[4][K::NGV]) {
        uint32_t vmax = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int tok = 2 * t + (j & 1) + 8 * (j >> 1);
            const bool ok = tok < valid;
#pragma unroll
            for (int gv = 0; gv < K::NGV; ++gv) {
                uint32_t hb = lds<uint16_t>(ss, Geo::OFF_VS + tok * Geo::VSB + (VENC == ENC_ISO4 ? 4 : 2) * gv);
                if (!ok) hb = 0;
                vmax = max(vmax, hb & 0x7fffu);
                sv[j][gv] = f16_bits_to_f32(hb);
            }
        }
        return __reduce_max_sync(0xffffffffu, vmax) >> 10;
    }

    // O^T += V^T P for one page. pe: probabilities times the range factor.
    template <bool PLO>
    static __device__ __forceinline__ void pv(const uint8_t* st, const uint32_t* lut, int g, int t,
                                              const float (&pe)[4], const float (&sv)[4][K::NGV],
                                              float (&oacc)[K::MT][4]) {
        const int part = (G <= 4) ? ((g / G) & 1) : 0;
        const bool colzero = (G <= 4) && (g >= 2 * G);
        const int t0 = 2 * t, t1 = 2 * t + 1, t2 = 2 * t + 8, t3 = 2 * t + 9;
#pragma unroll
        for (int gv = 0; gv < K::NGV; ++gv) {
            const float P0 = pe[0] * sv[0][gv], P1 = pe[1] * sv[1][gv], P2 = pe[2] * sv[2][gv], P3 = pe[3] * sv[3][gv];
            const uint32_t h0 = f32x2_to_h2(P0, P1), h1 = f32x2_to_h2(P2, P3);
            uint32_t l0 = 0, l1 = 0;
            if constexpr (PLO) {
                const float2 f0 = h2_to_f32x2(h0), f1 = h2_to_f32x2(h1);
                l0 = f32x2_to_h2(P0 - f0.x, P1 - f0.y);
                l1 = f32x2_to_h2(P2 - f1.x, P3 - f1.y);
            }
            uint32_t bA0, bA1, bB0 = 0, bB1 = 0;
            if constexpr (G <= 4) {
                bA0 = colzero ? 0u : (part ? l0 : h0);
                bA1 = colzero ? 0u : (part ? l1 : h1);
            } else {
                bA0 = h0; bA1 = h1; bB0 = l0; bB1 = l1;
            }
            if constexpr (VENC == ENC_INT8) {
                const int byte = 64 * gv + 8 * g;
                const uint2 va = lds<uint2>(st, Geo::OFF_VC + swz(t0, byte));
                const uint2 vb = lds<uint2>(st, Geo::OFF_VC + swz(t1, byte));
                const uint2 vc2 = lds<uint2>(st, Geo::OFF_VC + swz(t2, byte));
                const uint2 vd = lds<uint2>(st, Geo::OFF_VC + swz(t3, byte));
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t wa = (u < 2) ? va.x : va.y, wb = (u < 2) ? vb.x : vb.y;
                    const uint32_t wc = (u < 2) ? vc2.x : vc2.y, wd = (u < 2) ? vd.x : vd.y;
                    const int bi = (2 * u) & 3;
                    const uint32_t a0 = hsub2_u32(i8pair_to_h2_biased(wa, wb, bi), 0x64806480u);
                    const uint32_t a1 = hsub2_u32(i8pair_to_h2_biased(wa, wb, bi + 1), 0x64806480u);
                    const uint32_t a2 = hsub2_u32(i8pair_to_h2_biased(wc, wd, bi), 0x64806480u);
                    const uint32_t a3 = hsub2_u32(i8pair_to_h2_biased(wc, wd, bi + 1), 0x64806480u);
                    const int mt = 4 * gv + u;
                    mma_f16_16816(oacc[mt], a0, a1, a2, a3, bA0, bA1);
                    if constexpr (G > 4 && PLO) mma_f16_16816(oacc[mt], a0, a1, a2, a3, bB0, bB1);
                }
            } else if constexpr (VENC == ENC_Q4) {
                const int byte = 16 * gv + 2 * g;
                const uint32_t xa = lds<uint16_t>(st, Geo::OFF_VC + swz(t0, byte));
                const uint32_t xb = lds<uint16_t>(st, Geo::OFF_VC + swz(t1, byte));
                const uint32_t xc = lds<uint16_t>(st, Geo::OFF_VC + swz(t2, byte));
                const uint32_t xd = lds<uint16_t>(st, Geo::OFF_VC + swz(t3, byte));
                const uint32_t X = xa | (xb << 16), Y = xc | (xd << 16);
                const uint32_t X8 = X >> 8, Y8 = Y >> 8;
                // low nibbles -> (q - 8) via 1024 + q - 1032; high nibbles via (1024 + 16 q) / 16 - 72
                const uint32_t kSubLo = 0x64086408u;                   // half2(1032, 1032)
                const uint32_t kMul = 0x2c002c00u, kAdd = 0xd480d480u; // half2(1/16), half2(-72)
                const uint32_t a0 = hsub2_u32((X & 0x000f000fu) | 0x64006400u, kSubLo);
                const uint32_t a1 = hsub2_u32((X8 & 0x000f000fu) | 0x64006400u, kSubLo);
                const uint32_t a2 = hsub2_u32((Y & 0x000f000fu) | 0x64006400u, kSubLo);
                const uint32_t a3 = hsub2_u32((Y8 & 0x000f000fu) | 0x64006400u, kSubLo);
                mma_f16_16816(oacc[2 * gv], a0, a1, a2, a3, bA0, bA1);
                if constexpr (G > 4 && PLO) mma_f16_16816(oacc[2 * gv], a0, a1, a2, a3, bB0, bB1);
                const uint32_t c0 = hfma2_u32((X & 0x00f000f0u) | 0x64006400u, kMul, kAdd);
                const uint32_t c1 = hfma2_u32((X8 & 0x00f000f0u) | 0x64006400u, kMul, kAdd);
                const uint32_t c2 = hfma2_u32((Y & 0x00f000f0u) | 0x64006400u, kMul, kAdd);
                const uint32_t c3 = hfma2_u32((Y8 & 0x00f000f0u) | 0x64006400u, kMul, kAdd);
                mma_f16_16816(oacc[2 * gv + 1], c0, c1, c2, c3, bA0, bA1);
                if constexpr (G > 4 && PLO) mma_f16_16816(oacc[2 * gv + 1], c0, c1, c2, c3, bB0, bB1);
            } else {
                // ISO: m-tile u of block gv: row g <-> dim 16g + 2u, row g + 8 <-> dim 16g + 2u + 1
                uint32_t cw[4][2];
                const int tks[4] = {t0, t1, t2, t3};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int rb = Geo::OFF_VC + tks[j] * Geo::VCB;
                    if constexpr (VENC == ENC_ISO3) {
                        cw[j][0] = lds<uint32_t>(st, rb + 48 * gv + 4 * g);
                        cw[j][1] = lds<uint16_t>(st, rb + 48 * gv + 32 + 2 * g);
                    } else {
                        const uint2 v = lds<uint2>(st, rb + 64 * gv + 8 * g);
                        cw[j][0] = v.x; cw[j][1] = v.y;
                    }
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    uint32_t X[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t idx;
                        if constexpr (VENC == ENC_ISO3) idx = ((cw[j][0] >> (4 * u)) & 0xfu) | (((cw[j][1] >> (2 * u)) & 3u) << 4);
                        else idx = ((u < 4 ? cw[j][0] : cw[j][1]) >> (8 * (u & 3))) & 0xffu;
                        X[j] = lut[idx * 32];
                    }
                    const uint32_t a0 = prmt(X[0], X[1], 0x5410u), a1 = prmt(X[0], X[1], 0x7632u);
                    const uint32_t a2 = prmt(X[2], X[3], 0x5410u), a3 = prmt(X[2], X[3], 0x7632u);
                    const int mt = 8 * gv + u;
                    mma_f16_16816(oacc[mt], a0, a1, a2, a3, bA0, bA1);
                    if constexpr (G > 4 && PLO) mma_f16_16816(oacc[mt], a0, a1, a2, a3, bB0, bB1);
                }
            }
        }
    }
};

template <int KENC, int VENC, int D, int G, bool PLO>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, const DecodeParams p) {
    using K = Cfg<KENC, VENC, D, G>;
    using Geo = typename K::Geo;
    using W = WarpPipe<KENC, VENC, D, G>;
    constexpr int NS = K::NS;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 128-byte TMA swizzle patterns are defined on absolute shared addresses: align the base to 1 KB
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int C = gridDim.x, c = blockIdx.x;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + K::OFF_BAR) + warp * 4;
    int* pref = reinterpret_cast<int*>(smem + K::OFF_PREF);
    float* sm_mw = reinterpret_cast<float*>(smem + K::OFF_SMALL);      // [kNW][8]
    float* sm_lw = sm_mw + kNW * 8;                                    // [kNW][8]
    float* sm_w = sm_lw + kNW * 8;                                     // [kMaxMerge][8]
    uint8_t* rowbuf = smem + K::OFF_ROW + warp * 512;
    __shared__ int s_ticket;
    __shared__ const float* s_slots[kMaxMerge];
    __shared__ float s_pM[8], s_pL[8], s_pw[kNW][8];

    // ---- per-call setup: barriers, ISO pair tables, page-count prefix ----
    if (lane == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    if constexpr (K::ISO_LUT) {
        uint32_t* lutw = reinterpret_cast<uint32_t*>(smem + K::OFF_LUT);
        constexpr int TT = (KENC == ENC_ISO4 || VENC == ENC_ISO4) ? 1 : 0;
        for (int e = tid; e < K::LUT_ENTRIES * 32; e += blockDim.x) {
            int idx = e >> 5;
            int c0, c1;
            if constexpr (TT == 1) { c0 = idx & 15; c1 = idx >> 4; }
            else { c0 = (idx & 3) | (((idx >> 4) & 1) << 2); c1 = ((idx >> 2) & 3) | (((idx >> 5) & 1) << 2); }
            lutw[e] = f32x2_to_h2(c_dec_levels[TT][c0], c_dec_levels[TT][c1]);
        }
    }
    {
        // prefix of page counts over sequences (B <= kMaxBatch): pref[b] = sum_{b' < b} np(b')
        __shared__ int s_wsum[kNW];
        const int per = (p.B + blockDim.x - 1) / blockDim.x;
        const int b0 = tid * per;
        int local = 0;
        for (int i = 0; i < per; ++i) {
            int b = b0 + i;
            if (b < p.B) {
                int L = p.seq_lens[b];
                if (L < 0 || L > p.max_pages * kPage) { atomicOr(&g_err_decode, kErrPos); L = max(0, min(L, p.max_pages * kPage)); }
                local += (L + kPage - 1) / kPage;
            }
        }
        int incl = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        if (lane == 31) s_wsum[warp] = incl;
        __syncthreads();
        int wpre = 0;
        for (int w = 0; w < warp; ++w) wpre += s_wsum[w];
        int run = wpre + incl - local;
        for (int i = 0; i < per; ++i) {
            int b = b0 + i;
            if (b < p.B) {
                int L = max(0, min(p.seq_lens[b], p.max_pages * kPage));
                pref[b] = run;
                run += (L + kPage - 1) / kPage;
            }
        }
        if (b0 < p.B && b0 + per >= p.B) pref[p.B] = run;
        __syncthreads();
    }
    const long long NH = p.NH;
    const long long T = (long long)pref[p.B] * NH;   // total (segment, page) units
    const long long beg = T * c / C, end = T * (c + 1) / C;
    auto cta_of = [&](long long x) -> long long { return ((x + 1) * C + T - 1) / T - 1; };

    // empty sequences: zero rows, written by CTA (s mod C)
    for (long long s = c; s < (long long)p.B * NH; s += C) {
        int b = (int)(s / NH);
        if (pref[b + 1] == pref[b]) {
            int hg = (int)(s % NH);
            int kvh = hg / (p.Gtot / G), hgi = hg % (p.Gtot / G);
            size_t base = ((size_t)b * p.Hq + kvh * p.Gtot + hgi * G) * D;
            for (int i = tid; i < G * D; i += blockDim.x) {
                if (p.out_f32) reinterpret_cast<float*>(p.out)[base + i] = 0.0f;
                else reinterpret_cast<__nv_bfloat16*>(p.out)[base + i] = __float2bfloat16_rn(0.0f);
            }
        }
    }

    const uint32_t* lut = reinterpret_cast<const uint32_t*>(smem + K::OFF_LUT) + lane;
    uint8_t* const code_base = smem + (size_t)warp * NS * Geo::CODE_BYTES;
    uint8_t* const scale_base = smem + K::PIPE_CODE + (size_t)warp * NS * Geo::SCALE_BYTES;
    uint32_t gi = 0;   // pages consumed by this warp so far (stage / parity bookkeeping)
    long long x = beg;
    while (x < end) {
        // ---- locate the piece: sequence b, head group hg, pages [p0, p1) ----
        int lo = 0, hi = p.B;   // largest b with pref[b] * NH <= x
        while (hi - lo > 1) { int mid = (lo + hi) >> 1; if ((long long)pref[mid] * NH <= x) lo = mid; else hi = mid; }
        const int b = lo;
        const int np = pref[b + 1] - pref[b];
        const long long seg0 = (long long)pref[b] * NH;
        const int hg = (int)((x - seg0) / np);
        const long long soff = seg0 + (long long)hg * np;          // first unit of this segment
        const int p0 = (int)(x - soff);
        const long long xe = min(end, soff + np);
        const int p1 = (int)(xe - soff);
        const int L = max(0, min(p.seq_lens[b], p.max_pages * kPage));
        const int kvh = hg / (p.Gtot / G), hgi = hg % (p.Gtot / G);
        const int hq0 = kvh * p.Gtot + hgi * G;
        const long long seg = (long long)b * NH + hg;
        const long long clo = cta_of(soff), chi = cta_of(soff + np - 1);
        const int npieces = (int)(chi - clo + 1);

        // ---- this warp's pages ----
        const int npc = p1 - p0;
        const int wp0 = p0 + (int)((long long)npc * warp / kNW);
        const int wp1 = p0 + (int)((long long)npc * (warp + 1) / kNW);
        const int npg = wp1 - wp0;
        const int32_t* ptrow = p.page_table + (size_t)b * p.max_pages;
        const int last_page = (L - 1) / kPage;

        // query fragments (A operand): rows r < 8 -> head r % G (hi part), rows r + 8 -> lo part
        // (rotated query only); for int8 K, 1152 * the per-group sums of the fp16 query
        uint32_t qa[K::KS][4];
        float qbias[K::NGK];
#pragma unroll
        for (int i = 0; i < K::NGK; ++i) qbias[i] = 0.0f;
        {
            const uint16_t* qrow = p.q + ((size_t)b * p.Hq + hq0 + g % G) * D;
#pragma unroll
            for (int ks = 0; ks < K::KS; ++ks) {
                const int gg = ks / K::KSPG, u = ks % K::KSPG;
                int d0;
                if constexpr (KENC == ENC_INT8) d0 = 64 * gg + 16 * t + 4 * u;
                else d0 = 128 * gg + 32 * t + 4 * u;
                float qv[4];
                const uint2 w = *reinterpret_cast<const uint2*>(qrow + d0);
                const float a = bf16_bits_to_f32(w.x & 0xffffu), bq = bf16_bits_to_f32(w.x >> 16);
                const float cq = bf16_bits_to_f32(w.y & 0xffffu), dq = bf16_bits_to_f32(w.y >> 16);
                if constexpr (!K::KISO) {
                    qv[0] = a; qv[1] = bq; qv[2] = cq; qv[3] = dq;
                } else {
                    // rotated query R q for this 4-D group (d0 is a multiple of 4)
                    const float q0 = p.quat[0], q1 = p.quat[1], q2 = p.quat[2], q3 = p.quat[3];
                    qv[0] = q0 * a - q1 * bq - q2 * cq - q3 * dq;
                    qv[1] = q0 * bq + q1 * a + q2 * dq - q3 * cq;
                    qv[2] = q0 * cq - q1 * dq + q2 * a + q3 * bq;
                    qv[3] = q0 * dq + q1 * cq - q2 * bq + q3 * a;
                }
                const uint32_t h01 = f32x2_to_h2(qv[0], qv[1]), h23 = f32x2_to_h2(qv[2], qv[3]);
                qa[ks][0] = h01;
                qa[ks][2] = h23;
                const float2 f01 = h2_to_f32x2(h01), f23 = h2_to_f32x2(h23);
                if constexpr (K::QLO) {
                    qa[ks][1] = f32x2_to_h2(qv[0] - f01.x, qv[1] - f01.y);
                    qa[ks][3] = f32x2_to_h2(qv[2] - f23.x, qv[3] - f23.y);
                } else {
                    qa[ks][1] = 0u;
                    qa[ks][3] = 0u;
                }
                if constexpr (K::KBIAS) qbias[gg] += (f01.x + f01.y) + (f23.x + f23.y);
            }
            if constexpr (K::KBIAS) {
#pragma unroll
                for (int i = 0; i < K::NGK; ++i) {
                    qbias[i] += __shfl_xor_sync(0xffffffffu, qbias[i], 1);
                    qbias[i] += __shfl_xor_sync(0xffffffffu, qbias[i], 2);
                    qbias[i] *= 1152.0f;
                }
            }
        }

        float oacc[K::MT][4];
#pragma unroll
        for (int i = 0; i < K::MT; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.0f;
        // Lazy softmax frame: probabilities are 2^(s - m_frame) and the frame only moves when
        // a page's max exceeds it by more than 8 (so probabilities stay <= 2^8); the range
        // factor 2^E_frame keeps probability x V-scale inside the fp16 normal range.
        float m_frame = -INFINITY, l_run = 0.0f;
        int E_frame = 1000;   // "unset"

        // page-id ring: pid_cur covers pages [32*bc, 32*bc+32), pid_nxt the next 32
        int bc = 0;
        int pid_cur = (lane < npg) ? ptrow[wp0 + lane] : 0;
        int pid_nxt = (32 + lane < npg) ? ptrow[wp0 + 32 + lane] : 0;
        auto issue = [&](int j) {   // warp-uniform
            if ((j >> 5) > bc) {
                pid_cur = pid_nxt;
                ++bc;
                pid_nxt = (32 * (bc + 1) + lane < npg) ? ptrow[wp0 + 32 * (bc + 1) + lane] : 0;
            }
            int pid = __shfl_sync(0xffffffffu, pid_cur, j & 31);
            if (lane == 0) {
                if (pid < 0 || pid >= p.num_pages) { atomicOr(&g_err_decode, kErrPage); pid = 0; }
                const uint32_t slot = (gi + (uint32_t)j) % NS;
                uint8_t* sc = code_base + slot * Geo::CODE_BYTES;
                uint8_t* ss = scale_base + slot * Geo::SCALE_BYTES;
                uint64_t* bar = &bars[slot];
                fence_proxy_async();
                mbar_arrive_expect_tx(bar, Geo::TX);
                const long long row = ((long long)pid * p.Hkv + kvh) * kPage;
                const uint64_t pol = l2_evict_first_policy();   // pages are read once per launch
                if constexpr (Geo::K_TMA) {
#pragma unroll
                    for (int bx = 0; bx < (Geo::KCB + 127) / 128; ++bx)
                        tma_load_2d_hint(sc + Geo::OFF_KC + bx * 2048, &tmK, bar, bx * 128, (int)row, pol);
                } else {
                    bulk_load_hint(sc + Geo::OFF_KC, p.kc + row * Geo::KCB, kPage * Geo::KCB, bar, pol);
                }
                if constexpr (Geo::V_TMA) {
#pragma unroll
                    for (int bx = 0; bx < (Geo::VCB + 127) / 128; ++bx)
                        tma_load_2d_hint(sc + Geo::OFF_VC + bx * 2048, &tmV, bar, bx * 128, (int)row, pol);
                } else {
                    bulk_load_hint(sc + Geo::OFF_VC, p.vc + row * Geo::VCB, kPage * Geo::VCB, bar, pol);
                }
                bulk_load_hint(ss + Geo::OFF_KS, p.ks + row * Geo::KSB, kPage * Geo::KSB, bar, pol);
                bulk_load_hint(ss + Geo::OFF_VS, p.vs + row * Geo::VSB, kPage * Geo::VSB, bar, pol);
            }
        };
        // wait for page j; if it holds the sequence's newest token and the call carries
        // k_new / v_new, quantize that token into the pool and into the staged copy
        auto land = [&](int j) {
            const uint32_t slot = (gi + (uint32_t)j) % NS;
            if (!mbar_wait_bounded(&bars[slot], ((gi + (uint32_t)j) / NS) & 1u)) {
                // a copy that never lands: flag it and go on (results are garbage, nothing hangs)
                if (lane == 0) atomicOr(&g_err_decode, kErrWait);
            }
            if (p.k_new != nullptr && wp0 + j == last_page) {
                uint8_t* st = code_base + slot * Geo::CODE_BYTES;
                uint8_t* ss = scale_base + slot * Geo::SCALE_BYTES;
                const int slot_tok = (L - 1) % kPage;
                const int pid = max(0, min(ptrow[wp0 + j], p.num_pages - 1));
                const float qv[4] = {p.quat[0], p.quat[1], p.quat[2], p.quat[3]};
#pragma unroll
                for (int store = 0; store < 2; ++store) {
                    const uint16_t* src = (store == 0 ? p.k_new : p.v_new) + ((size_t)b * p.Hkv + kvh) * D;
                    if (store == 0) {
                        constexpr int TT = KENC == ENC_ISO4 ? 1 : 0;
                        quantize_row<KENC, D>(src, rowbuf, rowbuf + 256, lane, qv, c_dec_levels[TT], c_dec_mids[TT]);
                    } else {
                        constexpr int TT = VENC == ENC_ISO4 ? 1 : 0;
                        quantize_row<VENC, D>(src, rowbuf, rowbuf + 256, lane, qv, c_dec_levels[TT], c_dec_mids[TT]);
                    }
                    __syncwarp();
                    const int enc = store == 0 ? KENC : VENC;
                    const int cb = code_row_bytes(enc, D), sb = scale_row_bytes(enc, D);
                    const long long grow = ((long long)pid * p.Hkv + kvh) * kPage + slot_tok;
                    uint8_t* gcode = const_cast<uint8_t*>(store == 0 ? p.kc : p.vc) + grow * cb;
                    uint8_t* gscale = const_cast<uint8_t*>(store == 0 ? p.ks : p.vs) + grow * sb;
                    const bool tma_rows = store == 0 ? Geo::K_TMA : Geo::V_TMA;
                    uint8_t* scode = st + (store == 0 ? Geo::OFF_KC : Geo::OFF_VC);
                    uint8_t* sscale = ss + (store == 0 ? Geo::OFF_KS : Geo::OFF_VS);
                    for (int ch = lane; ch < cb / 16; ch += 32) {
                        const uint4 v = *reinterpret_cast<const uint4*>(rowbuf + 16 * ch);
                        *reinterpret_cast<uint4*>(gcode + 16 * ch) = v;
                        const int off = tma_rows ? swz(slot_tok, 16 * ch) : slot_tok * cb + 16 * ch;
                        *reinterpret_cast<uint4*>(scode + off) = v;
                    }
                    for (int e = lane; e < sb / 2; e += 32) {
                        const uint16_t v = reinterpret_cast<const uint16_t*>(rowbuf + 256)[e];
                        reinterpret_cast<uint16_t*>(gscale)[e] = v;
                        reinterpret_cast<uint16_t*>(sscale + slot_tok * sb)[e] = v;
                    }
                    fence_proxy_async();   // these shared writes precede later TMA refills of the stage
                    __syncwarp();
                }
            }
        };
        // end-of-page bookkeeping for page j's scores: move the frame (rare, warp-uniform branch)
        auto frame = [&](const float (&s)[4], int E_page) {
            float pm = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
            pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 1));
            pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 2));
            const bool need = (pm > m_frame + 8.0f) || (E_page < E_frame);
            if (__any_sync(0xffffffffu, need)) {
                const float m_new = (pm > m_frame + 8.0f) ? pm : m_frame;
                const float alpha = (m_new == m_frame) ? 1.0f : fast_exp2(m_frame - m_new);
                const int Enew = min(E_frame, E_page);
                const float ef = (E_frame == 1000) ? 1.0f : __int_as_float((Enew - E_frame + 127) << 23);
                l_run *= alpha;
                const float a0 = __shfl_sync(0xffffffffu, alpha, ((2 * t) % G) * 4);
                const float a1 = __shfl_sync(0xffffffffu, alpha, ((2 * t + 1) % G) * 4);
                const float f0 = a0 * ef, f1 = a1 * ef;
#pragma unroll
                for (int mt = 0; mt < K::MT; ++mt) { oacc[mt][0] *= f0; oacc[mt][1] *= f1; oacc[mt][2] *= f0; oacc[mt][3] *= f1; }
                m_frame = m_new;
                E_frame = Enew;
            }
        };

        // prologue: pages 0 and 1 in flight, scores of page 0
        for (int j = 0; j < NS - 1 && j < npg; ++j) issue(j);
        float s_cur[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        float sv_cur[4][K::NGV];
        if (npg > 0) {
            land(0);
            const uint32_t slot = gi % NS;
            const int valid = min(kPage, L - wp0 * kPage);
            W::scores(code_base + slot * Geo::CODE_BYTES, scale_base + slot * Geo::SCALE_BYTES, qa, qbias, lut, g, t,
                      valid, p.scale_log2, s_cur);
            const uint32_t e16 = W::vscales(scale_base + slot * Geo::SCALE_BYTES, t, valid, sv_cur);
            frame(s_cur, 20 - max((int)e16, 1));
        }
        for (int i = 0; i < npg; ++i) {
            if (i + NS - 1 < npg) issue(i + NS - 1);   // refills the stage of page i - 1
            const bool has_next = i + 1 < npg;
            if (has_next) land(i + 1);
            const uint32_t slot_i = (gi + (uint32_t)i) % NS, slot_n = (gi + (uint32_t)i + 1) % NS;
            // ---- one straight-line block: QK(i + 1), softmax(i), PV(i) are independent ----
            float s_nxt[4];
            const int valid_n = min(kPage, L - (wp0 + i + 1) * kPage);
            W::scores(code_base + slot_n * Geo::CODE_BYTES, scale_base + slot_n * Geo::SCALE_BYTES, qa, qbias, lut, g, t,
                      valid_n, p.scale_log2, s_nxt);
            float pe[4];
            const float e2 = __int_as_float((E_frame + 127) << 23);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float pj = fast_exp2(s_cur[j] - m_frame);
                l_run += pj;
                pe[j] = pj * e2;
            }
            W::template pv<PLO>(code_base + slot_i * Geo::CODE_BYTES, lut, g, t, pe, sv_cur, oacc);
            // ---- next page's V scales and frame ----
            if (has_next) {
                const uint32_t e16 = W::vscales(scale_base + slot_n * Geo::SCALE_BYTES, t, valid_n, sv_cur);
                frame(s_nxt, 20 - max((int)e16, 1));
#pragma unroll
                for (int j = 0; j < 4; ++j) s_cur[j] = s_nxt[j];
            }
        }
        gi += (uint32_t)npg;

        // ---------------- warp -> CTA merge ----------------
        __syncthreads();   // all warps done with their stages: the area becomes the merge buffer
        {
            float* Ow = reinterpret_cast<float*>(smem) + (size_t)warp * 8 * D;   // [8 cols][D]
            float lq = l_run;
            lq += __shfl_xor_sync(0xffffffffu, lq, 1);
            lq += __shfl_xor_sync(0xffffffffu, lq, 2);
            if (t == 0) { sm_mw[warp * 8 + g] = m_frame; sm_lw[warp * 8 + g] = lq; }
            const float inv = (E_frame == 1000) ? 0.0f : __int_as_float((127 - E_frame) << 23);
#pragma unroll
            for (int mt = 0; mt < K::MT; ++mt) {
                int dA;
                if constexpr (VENC == ENC_INT8) dA = 64 * (mt >> 2) + 8 * g + 2 * (mt & 3);
                else if constexpr (VENC == ENC_Q4) dA = 32 * (mt >> 1) + 2 * g + 16 * (mt & 1);
                else dA = 128 * (mt >> 3) + 16 * g + 2 * (mt & 7);
                Ow[(2 * t) * D + dA] = oacc[mt][0] * inv;
                Ow[(2 * t + 1) * D + dA] = oacc[mt][1] * inv;
                Ow[(2 * t) * D + dA + 1] = oacc[mt][2] * inv;
                Ow[(2 * t + 1) * D + dA + 1] = oacc[mt][3] * inv;
            }
        }
        __syncthreads();
        if (tid < G) {
            float M = -INFINITY;
            for (int w = 0; w < kNW; ++w) M = fmaxf(M, sm_mw[w * 8 + tid]);
            float Ls = 0.0f;
            for (int w = 0; w < kNW; ++w) {
                float mw = sm_mw[w * 8 + tid];
                float wt = (mw == -INFINITY) ? 0.0f : exp2f(mw - M);
                s_pw[w][tid] = wt;
                Ls += wt * sm_lw[w * 8 + tid];
            }
            s_pM[tid] = M;
            s_pL[tid] = Ls;
        }
        __syncthreads();
        // combine warps and the columns belonging to the same head
        constexpr int PER = (8 * D + kThreads - 1) / kThreads;
        float vals[PER];
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const int i = tid + k * kThreads;
            float acc = 0.0f;
            if (i < G * D) {
                const int h = i / D, d = i % D;
#pragma unroll 1
                for (int w = 0; w < kNW; ++w) {
                    const float wt = s_pw[w][h];
                    if (wt == 0.0f) continue;
                    const float* Ow2 = reinterpret_cast<const float*>(smem) + (size_t)w * 8 * D;
                    float cs = 0.0f;
                    for (int n = h; n < 8; n += G) cs += Ow2[n * D + d];
                    acc += wt * cs;
                }
            }
            vals[k] = acc;
        }
        __syncthreads();   // warp rows fully read
        if (npieces == 1) {
            float* o = reinterpret_cast<float*>(smem);
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const int i = tid + k * kThreads;
                if (i < G * D) { const float Lh = s_pL[i / D]; o[i] = (Lh > 0.0f) ? vals[k] / Lh : 0.0f; }
            }
            __syncthreads();
            write_output<VENC, D, G>(p, o, b, hq0, tid);
        } else {
            float* mine = p.part1 + (size_t)(c + seg) * p.slot_floats;
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const int i = tid + k * kThreads;
                if (i < G * D) mine[16 + i] = vals[k];
            }
            if (tid < G) { mine[tid] = s_pM[tid]; mine[8 + tid] = s_pL[tid]; }
            __threadfence();
            __syncthreads();
            // two-level last-arrival merge over the pieces of this segment
            const int j = (int)(c - clo);
            int GS = 1;
            while (GS * GS < npieces) ++GS;
            const int ngroups = (npieces + GS - 1) / GS;
            const int grp = j / GS;
            const int gsize = min(GS, npieces - grp * GS);
            const long long gslot = clo + (long long)grp * GS + seg;
            if (tid == 0) s_ticket = atomicAdd(&p.grp_cnt[gslot], 1);
            __syncthreads();
            if (s_ticket == gsize - 1) {
                __threadfence();
                if (tid == 0) p.grp_cnt[gslot] = 0;
                for (int k = tid; k < gsize; k += blockDim.x)
                    s_slots[k] = p.part1 + (size_t)(clo + (long long)grp * GS + k + seg) * p.slot_floats;
                __syncthreads();
                float* o = reinterpret_cast<float*>(smem);
                if (ngroups == 1) {
                    merge_slots<VENC, D, G>(p, s_slots, gsize, nullptr, true, b, hq0, sm_w, o, tid);
                } else {
                    float* gdst = p.part2 + (size_t)gslot * p.slot_floats;
                    merge_slots<VENC, D, G>(p, s_slots, gsize, gdst, false, b, hq0, sm_w, o, tid);
                    __threadfence();
                    __syncthreads();
                    if (tid == 0) s_ticket = atomicAdd(&p.seg_cnt[seg], 1);
                    __syncthreads();
                    if (s_ticket == ngroups - 1) {
                        __threadfence();
                        if (tid == 0) p.seg_cnt[seg] = 0;
                        for (int k = tid; k < ngroups; k += blockDim.x)
                            s_slots[k] = p.part2 + (size_t)(clo + (long long)k * GS + seg) * p.slot_floats;
                        __syncthreads();
                        merge_slots<VENC, D, G>(p, s_slots, ngroups, nullptr, true, b, hq0, sm_w, o, tid);
                    }
                }
            }
        }
        __syncthreads();
        x = xe;
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
cudaError_t decode_upload_levels(const float* lv3, const float* lv4) {
    float lv[2][16] = {}, mid[2][16] = {};
    for (int j = 0; j < 8; ++j) lv[0][j] = lv3[j];
    for (int j = 0; j < 16; ++j) lv[1][j] = lv4[j];
    for (int j = 0; j < 7; ++j) mid[0][j] = (lv3[j] + lv3[j + 1]) * 0.5f;
    for (int j = 0; j < 15; ++j) mid[1][j] = (lv4[j] + lv4[j + 1]) * 0.5f;
    cudaError_t e = cudaMemcpyToSymbol(c_dec_levels, lv, sizeof(lv));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(c_dec_mids, mid, sizeof(mid));
}

cudaError_t decode_read_error(unsigned* out, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_err_decode, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    unsigned z = 0;
    return cudaMemcpyToSymbol(g_err_decode, &z, sizeof(unsigned));
}

int decode_heads_per_cta(int Gtot) { return Gtot >= 8 ? 8 : Gtot; }
int decode_max_batch() { return kMaxBatch; }

template <int KE, int VE, int D, int G>
static cudaError_t launch_one(int grid, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p, cudaStream_t st) {
    using K = Cfg<KE, VE, D, G>;
    auto fn = decode_kernel<KE, VE, D, G, true>;
    static bool configured = false;   // per instantiation; the attribute is per device context
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, K::SMEM + 1024);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    fn<<<grid, kThreads, K::SMEM + 1024, st>>>(tk, tv, p);
    return cudaGetLastError();
}

template <int KE, int VE, int D>
static cudaError_t launch_g(int G, int grid, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p, cudaStream_t st) {
    switch (G) {
        case 1: return launch_one<KE, VE, D, 1>(grid, tk, tv, p, st);
        case 2: return launch_one<KE, VE, D, 2>(grid, tk, tv, p, st);
        case 4: return launch_one<KE, VE, D, 4>(grid, tk, tv, p, st);
        case 8: return launch_one<KE, VE, D, 8>(grid, tk, tv, p, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t decode_launch(int fmt, int D, int G, int grid, const CUtensorMap& tk, const CUtensorMap& tv,
                          const DecodeParams& p, cudaStream_t st) {
    if (fmt == 0 && D == 256) return launch_g<ENC_INT8, ENC_INT8, 256>(G, grid, tk, tv, p, st);
    if (fmt == 0 && D == 128) return launch_g<ENC_INT8, ENC_INT8, 128>(G, grid, tk, tv, p, st);
    if (fmt == 1 && D == 256) return launch_g<ENC_INT8, ENC_Q4, 256>(G, grid, tk, tv, p, st);
    if (fmt == 2 && D == 128) return launch_g<ENC_ISO3, ENC_ISO3, 128>(G, grid, tk, tv, p, st);
    if (fmt == 2 && D == 256) return launch_g<ENC_ISO3, ENC_ISO3, 256>(G, grid, tk, tv, p, st);
    if (fmt == 3 && D == 128) return launch_g<ENC_ISO4, ENC_ISO4, 128>(G, grid, tk, tv, p, st);
    if (fmt == 3 && D == 256) return launch_g<ENC_ISO4, ENC_ISO4, 256>(G, grid, tk, tv, p, st);
    return cudaErrorInvalidValue;
}

}  // namespace qkv
