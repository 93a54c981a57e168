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
// GB300 design (one CTA of 16 warps per SM):
//   * Work is the list of (sequence, KV-head group, page) units; each CTA takes
//     an equal contiguous share (stream-K style), so any mix of lengths keeps
//     every SM equally busy. A share may span several sequences ("pieces").
//   * Warps work in pairs. A pair owns a contiguous run of pages and an
//     NS-stage TMA pipeline in shared memory (2-D tiled copies with 128-byte
//     swizzle for int8/q4 code planes, 1-D bulk copies for scales and ISO
//     codes), completing on mbarriers. Each warp of the pair takes half of the
//     head dimension: half of the QK^T k-steps (partial scores are exchanged
//     through shared memory) and half of the PV output columns. This halves the
//     per-warp registers (accumulators, query fragments) so 16 warps fit.
//   * QK^T and PV are warp-level fp16 tensor-core products (m16n8k16) on exact
//     operands: int8 K codes enter as 1152 + c (exact in fp16; the constant is
//     removed per page and group through the query sums), V codes exactly, q4 and
//     Lloyd-Max levels are exact fp16, the (rotated) query is split into fp16
//     hi + lo rows, per-(token, group) scales multiply fp32 scores (K) or are
//     folded into fp16 hi + lo probabilities (V). Online softmax in fp32 (base
//     2); a warp-uniform exponent keeps scaled probabilities in the fp16
//     normal range.
//   * Pairs merge in shared memory; CTAs merge through the caller's workspace
//     with the partial-softmax rule, done by the last-arriving CTA of each
//     group of pieces (atomic ticket, no waiting), in two levels.
#include "qkv_device.cuh"
#include "qkv_params.h"
#include "quant_rows.cuh"

namespace qkv {

__device__ unsigned int g_err_decode;
__constant__ float c_dec_levels[2][16];
__constant__ float c_dec_mids[2][16];

constexpr int kNW = 16;         // warps per CTA
constexpr int kNP = kNW / 2;    // warp pairs
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
    // V codes enter exactly (c, not 1152 + c): O accumulates over a whole page run, and a
    // removed offset would amplify the accumulation rounding by ~1152 / |mean code|.
    static constexpr bool VBIAS = false;
    static constexpr int KS = D / 16;               // k-steps over the head dimension
    static constexpr int KSH = KS / 2;              // per warp of a pair
    static constexpr int KSPG = group_size(KENC) / 16;
    static constexpr int MT = D / 16;               // PV m-tiles (16 dims each)
    static constexpr int MTH = MT / 2;              // per warp of a pair
    static constexpr int MTPG = group_size(VENC) / 16;
    static constexpr int NGV = D / group_size(VENC);
    static constexpr int NGVH = (MTH + MTPG - 1) / MTPG;  // V groups a warp touches
    static constexpr int NGK = D / group_size(KENC);
    static constexpr int NGKH = (KSH + KSPG - 1) / KSPG;  // K groups a warp touches
    static constexpr int MPER = MTH < MTPG ? MTH : MTPG;  // m-tiles per touched V group
    static constexpr bool ISO_LUT = KISO || VISO;
    static constexpr int LUT_ENTRIES = (KENC == ENC_ISO4 || VENC == ENC_ISO4) ? 256 : 64;
    static constexpr int LUT_BYTES = ISO_LUT ? LUT_ENTRIES * 32 * 4 : 0;
    static constexpr int XCH_BYTES = kNP * 2 * 2 * 32 * 16;   // [pair][parity][role][lane] float4
    static constexpr int SMALL_BYTES = kNP * 8 * 4 * 2 + kMaxMerge * 8 * 4 + 64;
    static constexpr int FIXED = LUT_BYTES + XCH_BYTES + SMALL_BYTES + kNP * 4 * 8 + (kMaxBatch + 1) * 4;
    static constexpr int BUDGET = 225 * 1024 - FIXED - 1024;  // dynamic bytes for stages
    static constexpr int NS_FIT = BUDGET / (kNP * (Geo::CODE_BYTES + Geo::SCALE_BYTES));
    static constexpr int NS = NS_FIT >= 4 ? 4 : NS_FIT;
    static constexpr int PIPE_CODE = kNP * NS * Geo::CODE_BYTES;
    static constexpr int PIPE_BYTES = PIPE_CODE + kNP * NS * Geo::SCALE_BYTES;
    static constexpr int MERGE_BYTES = kNP * 8 * D * 4;
    static constexpr int AREA = ((PIPE_BYTES > MERGE_BYTES ? PIPE_BYTES : MERGE_BYTES) + 1023) / 1024 * 1024;
    static constexpr int OFF_LUT = AREA;
    static constexpr int OFF_XCH = OFF_LUT + LUT_BYTES;
    static constexpr int OFF_SMALL = OFF_XCH + XCH_BYTES;      // pair m/l + merge weights
    static constexpr int OFF_BAR = OFF_SMALL + SMALL_BYTES;
    static constexpr int OFF_PREF = OFF_BAR + kNP * 4 * 8;
    static constexpr int SMEM = OFF_PREF + (kMaxBatch + 1) * 4;
    static_assert(NS >= 2, "pipeline needs at least two stages");
    static_assert(SMEM + 1024 + 1536 <= 232448, "shared memory budget (dynamic + alignment slack + static)");
    static_assert(KS % 2 == 0 && MT % 2 == 0, "pair split");
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

// the two warps of a pair meet on named barrier 1 + pair
__device__ __forceinline__ void pair_sync(int pair) {
    asm volatile("bar.sync %0, 64;" ::"r"(pair + 1) : "memory");
}

template <int KENC, int VENC, int D, int G, bool PLO>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, const DecodeParams p) {
    using K = Cfg<KENC, VENC, D, G>;
    using Geo = typename K::Geo;
    constexpr int NS = K::NS;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 128-byte TMA swizzle patterns are defined on absolute shared addresses: align the base to 1 KB
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int pair = warp >> 1, role = warp & 1;
    const int g = lane >> 2, t = lane & 3;
    const int C = gridDim.x, c = blockIdx.x;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + K::OFF_BAR) + pair * 4;
    int* pref = reinterpret_cast<int*>(smem + K::OFF_PREF);
    float* sm_mw = reinterpret_cast<float*>(smem + K::OFF_SMALL);      // [kNP][8]
    float* sm_lw = sm_mw + kNP * 8;                                    // [kNP][8]
    float* sm_w = sm_lw + kNP * 8;                                     // [kMaxMerge][8]
    float4* xch = reinterpret_cast<float4*>(smem + K::OFF_XCH) + pair * 2 * 2 * 32;   // [parity][role][lane]
    __shared__ int s_ticket;
    __shared__ const float* s_slots[kMaxMerge];
    __shared__ float s_pM[8], s_pL[8], s_pw[kNP][8];

    // ---- per-call setup: barriers, ISO pair tables, page-count prefix ----
    if (role == 0 && lane == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    if constexpr (K::ISO_LUT) {
        uint32_t* lutw = reinterpret_cast<uint32_t*>(smem + K::OFF_LUT);
        constexpr int T = (KENC == ENC_ISO4 || VENC == ENC_ISO4) ? 1 : 0;
        for (int e = tid; e < K::LUT_ENTRIES * 32; e += blockDim.x) {
            int idx = e >> 5;
            int c0, c1;
            if constexpr (T == 1) { c0 = idx & 15; c1 = idx >> 4; }
            else { c0 = (idx & 3) | (((idx >> 4) & 1) << 2); c1 = ((idx >> 2) & 3) | (((idx >> 5) & 1) << 2); }
            lutw[e] = f32x2_to_h2(c_dec_levels[T][c0], c_dec_levels[T][c1]);
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
    uint32_t gi = 0;   // pages consumed by this pair so far (stage / parity bookkeeping)
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

        // ---- this pair's pages ----
        const int npc = p1 - p0;
        const int wp0 = p0 + (int)((long long)npc * pair / kNP);
        const int wp1 = p0 + (int)((long long)npc * (pair + 1) / kNP);
        const int npg = wp1 - wp0;
        const int32_t* ptrow = p.page_table + (size_t)b * p.max_pages;

        // query fragments (A operand) for this warp's k-steps: rows r < 8 -> head r % G (hi part),
        // rows r + 8 -> lo part (rotated query only); plus, for int8 K, the per-group sums of the
        // fp16 query that remove the +1152 code offset
        const int hh = g % G;
        uint32_t qa[K::KSH][4];
        float qbias[K::NGKH];   // indexed by this warp's local K group
#pragma unroll
        for (int i = 0; i < K::NGKH; ++i) qbias[i] = 0.0f;
        {
            const uint16_t* qrow = p.q + ((size_t)b * p.Hq + hq0 + hh) * D;
#pragma unroll
            for (int kk = 0; kk < K::KSH; ++kk) {
                const int ks = role * K::KSH + kk;
                const int gg = ks / K::KSPG, u = ks % K::KSPG;
                int d0;
                if constexpr (KENC == ENC_INT8) d0 = 64 * gg + 16 * t + 4 * u;
                else d0 = 128 * gg + 32 * t + 4 * u;
                float qv[4];
                uint2 w = *reinterpret_cast<const uint2*>(qrow + d0);
                float a = bf16_bits_to_f32(w.x & 0xffffu), bq = bf16_bits_to_f32(w.x >> 16);
                float cq = bf16_bits_to_f32(w.y & 0xffffu), dq = bf16_bits_to_f32(w.y >> 16);
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
                qa[kk][0] = h01;
                qa[kk][2] = h23;
                if constexpr (K::QLO) {
                    const float2 f01 = h2_to_f32x2(h01), f23 = h2_to_f32x2(h23);
                    qa[kk][1] = f32x2_to_h2(qv[0] - f01.x, qv[1] - f01.y);
                    qa[kk][3] = f32x2_to_h2(qv[2] - f23.x, qv[3] - f23.y);
                } else {
                    qa[kk][1] = 0u;
                    qa[kk][3] = 0u;
                }
                if constexpr (K::KBIAS) {
                    const float2 f01 = h2_to_f32x2(h01), f23 = h2_to_f32x2(h23);
                    qbias[kk / K::KSPG] += (f01.x + f01.y) + (f23.x + f23.y);
                }
            }
            if constexpr (K::KBIAS) {
#pragma unroll
                for (int i = 0; i < K::NGKH; ++i) {
                    qbias[i] += __shfl_xor_sync(0xffffffffu, qbias[i], 1);
                    qbias[i] += __shfl_xor_sync(0xffffffffu, qbias[i], 2);
                    qbias[i] *= 1152.0f;
                }
            }
        }

        float oacc[K::MTH][4];
#pragma unroll
        for (int i = 0; i < K::MTH; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.0f;
        float rsum[K::NGVH];   // sum of the probabilities fed to each V group (removes the +1152 offset)
#pragma unroll
        for (int i = 0; i < K::NGVH; ++i) rsum[i] = 0.0f;
        float m_run = -INFINITY, l_run = 0.0f;
        int E_run = 1000;   // "unset"

        // page-id ring (role 0 issues): pid_cur covers pages [32*bc, 32*bc+32), pid_nxt the next 32
        int bc = 0;
        int pid_cur = 0, pid_nxt = 0;
        if (role == 0) {
            pid_cur = (lane < npg) ? ptrow[wp0 + lane] : 0;
            pid_nxt = (32 + lane < npg) ? ptrow[wp0 + 32 + lane] : 0;
        }
        auto issue = [&](int j) {   // called by role-0 warps only, warp-uniformly
            if ((j >> 5) > bc) {
                pid_cur = pid_nxt;
                ++bc;
                pid_nxt = (32 * (bc + 1) + lane < npg) ? ptrow[wp0 + 32 * (bc + 1) + lane] : 0;
            }
            int pid = __shfl_sync(0xffffffffu, pid_cur, j & 31);
            if (lane == 0) {
                if (pid < 0 || pid >= p.num_pages) { atomicOr(&g_err_decode, kErrPage); pid = 0; }
                const uint32_t slot = (gi + (uint32_t)j) % NS;
                uint8_t* sc = smem + (size_t)(pair * NS + slot) * Geo::CODE_BYTES;
                uint8_t* ss = smem + K::PIPE_CODE + (size_t)(pair * NS + slot) * Geo::SCALE_BYTES;
                uint64_t* bar = &bars[slot];
                fence_proxy_async();
                mbar_arrive_expect_tx(bar, Geo::TX);
                const long long row = ((long long)pid * p.Hkv + kvh) * kPage;
                if constexpr (Geo::K_TMA) {
#pragma unroll
                    for (int bx = 0; bx < (Geo::KCB + 127) / 128; ++bx) tma_load_2d(sc + Geo::OFF_KC + bx * 2048, &tmK, bar, bx * 128, (int)row);
                } else {
                    bulk_load(sc + Geo::OFF_KC, p.kc + row * Geo::KCB, kPage * Geo::KCB, bar);
                }
                if constexpr (Geo::V_TMA) {
#pragma unroll
                    for (int bx = 0; bx < (Geo::VCB + 127) / 128; ++bx) tma_load_2d(sc + Geo::OFF_VC + bx * 2048, &tmV, bar, bx * 128, (int)row);
                } else {
                    bulk_load(sc + Geo::OFF_VC, p.vc + row * Geo::VCB, kPage * Geo::VCB, bar);
                }
                bulk_load(ss + Geo::OFF_KS, p.ks + row * Geo::KSB, kPage * Geo::KSB, bar);
                bulk_load(ss + Geo::OFF_VS, p.vs + row * Geo::VSB, kPage * Geo::VSB, bar);
            }
        };
        if (role == 0)
            for (int j = 0; j < NS - 1 && j < npg; ++j) issue(j);

        for (int i = 0; i < npg; ++i) {
            const uint32_t slot = (gi + (uint32_t)i) % NS;
            const uint32_t parity = ((gi + (uint32_t)i) / NS) & 1u;
            uint8_t* st = smem + (size_t)(pair * NS + slot) * Geo::CODE_BYTES;
            uint8_t* ss = smem + K::PIPE_CODE + (size_t)(pair * NS + slot) * Geo::SCALE_BYTES;
            if (!mbar_wait_bounded(&bars[slot], parity)) {
                // a copy that never lands: flag it and go on (results are garbage, nothing hangs)
                if (lane == 0) atomicOr(&g_err_decode, kErrWait);
            }
            const int pg = wp0 + i;
            const int valid = min(kPage, L - pg * kPage);

            // ---- fused quantize-on-write of the newest token (position L - 1) ----
            if (p.k_new != nullptr && pg == (L - 1) / kPage) {
                const int slot_tok = (L - 1) % kPage;
                const int enc = role == 0 ? KENC : VENC;
                const uint16_t* src = (role == 0 ? p.k_new : p.v_new) + ((size_t)b * p.Hkv + kvh) * D;
                uint8_t* rowbuf = reinterpret_cast<uint8_t*>(xch + (i & 1) * 64 + role * 32);   // 512 B scratch
                const float qv[4] = {p.quat[0], p.quat[1], p.quat[2], p.quat[3]};
                if (role == 0) {
                    constexpr int TT = KENC == ENC_ISO4 ? 1 : 0;
                    quantize_row<KENC, D>(src, rowbuf, rowbuf + 256, lane, qv, c_dec_levels[TT], c_dec_mids[TT]);
                } else {
                    constexpr int TT = VENC == ENC_ISO4 ? 1 : 0;
                    quantize_row<VENC, D>(src, rowbuf, rowbuf + 256, lane, qv, c_dec_levels[TT], c_dec_mids[TT]);
                }
                __syncwarp();
                const int cb = code_row_bytes(enc, D), sb = scale_row_bytes(enc, D);
                const int pid = ptrow[pg];
                const long long grow = ((long long)max(0, min(pid, p.num_pages - 1)) * p.Hkv + kvh) * kPage + slot_tok;
                uint8_t* gcode = const_cast<uint8_t*>(role == 0 ? p.kc : p.vc) + grow * cb;
                uint8_t* gscale = const_cast<uint8_t*>(role == 0 ? p.ks : p.vs) + grow * sb;
                const bool tma_rows = role == 0 ? Geo::K_TMA : Geo::V_TMA;
                uint8_t* scode = st + (role == 0 ? Geo::OFF_KC : Geo::OFF_VC);
                uint8_t* sscale = ss + (role == 0 ? Geo::OFF_KS : Geo::OFF_VS);
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
                pair_sync(pair);
            }

            // ---------------- partial scores over this warp's k-steps ----------------
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int gsub = 0; gsub < (K::KSH + K::KSPG - 1) / K::KSPG; ++gsub) {
                // this warp's k-steps that fall in one K group
                const int ks_first = role * K::KSH + gsub * K::KSPG;
                const int gg = ks_first / K::KSPG;
                constexpr int NKS = K::KSH < K::KSPG ? K::KSH : K::KSPG;
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
                            const int kk = gsub * 4 + u;
                            mma_f16_16816(cacc[nt], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
                        }
                    } else if constexpr (KENC == ENC_ISO3) {
                        // k-steps u in [u0, u0 + NKS) of block gg; thread t owns dims 32t + 4u + {0..3}
                        const int u0 = ks_first % K::KSPG;
                        const int rb = Geo::OFF_KC + r * Geo::KCB + 48 * gg;
                        uint32_t lw[2];
                        if constexpr (NKS == 8) { const uint2 v = lds<uint2>(st, rb + 8 * t); lw[0] = v.x; lw[1] = v.y; }
                        else { lw[0] = lds<uint32_t>(st, rb + 8 * t + u0); lw[1] = 0; }
                        uint32_t hib;
                        if constexpr (NKS == 8) hib = lds<uint32_t>(st, rb + 32 + 4 * t);
                        else hib = lds<uint16_t>(st, rb + 32 + 4 * t + u0 / 2);
#pragma unroll
                        for (int uu = 0; uu < NKS; ++uu) {
                            const uint32_t lb = (lw[uu >> 2] >> (8 * (uu & 3))) & 0xffu;
                            const uint32_t hb = (hib >> (4 * uu)) & 0xfu;
                            const uint32_t i0 = (lb & 0xfu) | ((hb & 3u) << 4);
                            const uint32_t i1 = (lb >> 4) | ((hb >> 2) << 4);
                            const int kk = gsub * K::KSPG + uu;
                            mma_f16_16816(cacc[nt], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], lut[i0 * 32], lut[i1 * 32]);
                        }
                    } else {  // ISO4
                        const int u0 = ks_first % K::KSPG;
                        const int rb = Geo::OFF_KC + r * Geo::KCB + 64 * gg + 16 * t + 2 * u0;
                        uint32_t ws[4];
                        if constexpr (NKS == 8) { const uint4 v = lds<uint4>(st, rb); ws[0] = v.x; ws[1] = v.y; ws[2] = v.z; ws[3] = v.w; }
                        else { const uint2 v = lds<uint2>(st, rb); ws[0] = v.x; ws[1] = v.y; ws[2] = ws[3] = 0; }
#pragma unroll
                        for (int uu = 0; uu < NKS; ++uu) {
                            const uint32_t wd = ws[uu >> 1];
                            const uint32_t i0 = (wd >> (16 * (uu & 1))) & 0xffu;
                            const uint32_t i1 = (wd >> (16 * (uu & 1) + 8)) & 0xffu;
                            const int kk = gsub * K::KSPG + uu;
                            mma_f16_16816(cacc[nt], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], lut[i0 * 32], lut[i1 * 32]);
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int tok = 2 * t + (j & 1) + 8 * (j >> 1);
                    float ks;
                    if constexpr (KENC == ENC_INT8) ks = f16_bits_to_f32(lds<uint16_t>(ss, Geo::OFF_KS + tok * Geo::KSB + 2 * gg));
                    else ks = f16_bits_to_f32(lds<uint16_t>(ss, Geo::OFF_KS + tok * Geo::KSB + (KENC == ENC_ISO4 ? 4 : 2) * gg));
                    const int nt = j >> 1, e = j & 1;
                    float cv = cacc[nt][e];
                    if constexpr (K::QLO) cv += cacc[nt][2 + e];
                    if constexpr (K::KBIAS) cv -= qbias[gsub];
                    sc[j] += ks * cv;
                }
            }
            // exchange partial scores inside the pair
            xch[(i & 1) * 64 + role * 32 + lane] = make_float4(sc[0], sc[1], sc[2], sc[3]);
            pair_sync(pair);
            {
                const float4 o = xch[(i & 1) * 64 + (role ^ 1) * 32 + lane];
                sc[0] += o.x; sc[1] += o.y; sc[2] += o.z; sc[3] += o.w;
            }
            // both warps of the pair are past page i - 1: its stage can be refilled
            if (role == 0 && i + NS - 1 < npg) issue(i + NS - 1);
#pragma unroll
            for (int j = 0; j < 4; ++j) sc[j] = ((2 * t + (j & 1) + 8 * (j >> 1)) < valid) ? sc[j] * p.scale_log2 : -INFINITY;

            // ---------------- V scales of this warp's groups, fp16 range exponent ----------------
            float sv[4][K::NGVH];
            uint32_t vmax = 0;
            {
                const int gv0 = (role * K::MTH) / K::MTPG;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const bool ok = (2 * t + (j & 1) + 8 * (j >> 1)) < valid;
#pragma unroll
                    for (int q = 0; q < K::NGVH; ++q) {
                        uint32_t hb = lds<uint16_t>(ss, Geo::OFF_VS + (2 * t + (j & 1) + 8 * (j >> 1)) * Geo::VSB + (VENC == ENC_ISO4 ? 4 : 2) * (gv0 + q));
                        if (!ok) hb = 0;
                        vmax = max(vmax, hb & 0x7fffu);
                        sv[j][q] = f16_bits_to_f32(hb);
                    }
                }
            }
            vmax = __reduce_max_sync(0xffffffffu, vmax);
            const int Epage = 28 - max((int)(vmax >> 10), 1);

            // ---------------- online softmax ----------------
            float pm = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
            pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 1));
            pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 2));
            const float m_new = fmaxf(m_run, pm);
            const bool need = (m_new > m_run) || (Epage < E_run);
            if (__any_sync(0xffffffffu, need)) {
                const float alpha = (m_new == m_run) ? 1.0f : fast_exp2(m_run - m_new);
                const int Enew = min(E_run, Epage);
                const float ef = (E_run == 1000) ? 1.0f : __int_as_float((Enew - E_run + 127) << 23);
                l_run *= alpha;
#pragma unroll
                for (int q = 0; q < K::NGVH; ++q) rsum[q] *= alpha * ef;
                const float a0 = __shfl_sync(0xffffffffu, alpha, ((2 * t) % G) * 4);
                const float a1 = __shfl_sync(0xffffffffu, alpha, ((2 * t + 1) % G) * 4);
                const float f0 = a0 * ef, f1 = a1 * ef;
#pragma unroll
                for (int mt = 0; mt < K::MTH; ++mt) { oacc[mt][0] *= f0; oacc[mt][1] *= f1; oacc[mt][2] *= f0; oacc[mt][3] *= f1; }
                m_run = m_new;
                E_run = Enew;
            }
            float pr[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) { pr[j] = fast_exp2(sc[j] - m_run); l_run += pr[j]; }
            const float e2 = __int_as_float((E_run + 127) << 23);
#pragma unroll
            for (int j = 0; j < 4; ++j) pr[j] *= e2;

            // ---------------- O^T += V^T P over this warp's m-tiles ----------------
            const int part = (G <= 4) ? ((g / G) & 1) : 0;
            const bool colzero = (G <= 4) && (g >= 2 * G);
#pragma unroll
            for (int q = 0; q < K::NGVH; ++q) {
                const int gv = (role * K::MTH) / K::MTPG + q;
                const float P0 = pr[0] * sv[0][q], P1 = pr[1] * sv[1][q], P2 = pr[2] * sv[2][q], P3 = pr[3] * sv[3][q];
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
                if constexpr (K::VBIAS) {
                    const float2 x0 = h2_to_f32x2(bA0), x1 = h2_to_f32x2(bA1);
                    float fed = (x0.x + x0.y) + (x1.x + x1.y);
                    if constexpr (G > 4 && PLO) {
                        const float2 y0 = h2_to_f32x2(bB0), y1 = h2_to_f32x2(bB1);
                        fed += (y0.x + y0.y) + (y1.x + y1.y);
                    }
                    rsum[q] += fed;
                }
                // m-tiles of group gv inside this warp's half
                constexpr int MPER = K::MPER;
                const int mt0 = (role * K::MTH > gv * K::MTPG ? role * K::MTH : gv * K::MTPG);
                if constexpr (VENC == ENC_INT8) {
                    const int byte = 64 * gv + 8 * g;
                    const uint2 va = lds<uint2>(st, Geo::OFF_VC + swz((2 * t), byte));
                    const uint2 vb = lds<uint2>(st, Geo::OFF_VC + swz((2 * t + 1), byte));
                    const uint2 vc2 = lds<uint2>(st, Geo::OFF_VC + swz((2 * t + 8), byte));
                    const uint2 vd = lds<uint2>(st, Geo::OFF_VC + swz((2 * t + 9), byte));
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint32_t wa = (u < 2) ? va.x : va.y, wb = (u < 2) ? vb.x : vb.y;
                        const uint32_t wc = (u < 2) ? vc2.x : vc2.y, wd = (u < 2) ? vd.x : vd.y;
                        const int bi = (2 * u) & 3;
                        const uint32_t a0 = hsub2_u32(i8pair_to_h2_biased(wa, wb, bi), 0x64806480u);
                        const uint32_t a1 = hsub2_u32(i8pair_to_h2_biased(wa, wb, bi + 1), 0x64806480u);
                        const uint32_t a2 = hsub2_u32(i8pair_to_h2_biased(wc, wd, bi), 0x64806480u);
                        const uint32_t a3 = hsub2_u32(i8pair_to_h2_biased(wc, wd, bi + 1), 0x64806480u);
                        const int ml = q * 4 + u;
                        mma_f16_16816(oacc[ml], a0, a1, a2, a3, bA0, bA1);
                        if constexpr (G > 4 && PLO) mma_f16_16816(oacc[ml], a0, a1, a2, a3, bB0, bB1);
                    }
                } else if constexpr (VENC == ENC_Q4) {
                    const int byte = 16 * gv + 2 * g;
                    const uint32_t xa = lds<uint16_t>(st, Geo::OFF_VC + swz((2 * t), byte));
                    const uint32_t xb = lds<uint16_t>(st, Geo::OFF_VC + swz((2 * t + 1), byte));
                    const uint32_t xc = lds<uint16_t>(st, Geo::OFF_VC + swz((2 * t + 8), byte));
                    const uint32_t xd = lds<uint16_t>(st, Geo::OFF_VC + swz((2 * t + 9), byte));
                    const uint32_t X = xa | (xb << 16), Y = xc | (xd << 16);
                    const uint32_t X8 = X >> 8, Y8 = Y >> 8;
                    // low nibbles -> (q - 8) via 1024 + q - 1032; high nibbles via (1024 + 16 q) / 16 - 72
                    const uint32_t kSubLo = 0x64086408u;                   // half2(1032, 1032)
                    const uint32_t kMul = 0x2c002c00u, kAdd = 0xd480d480u; // half2(1/16), half2(-72)
                    const uint32_t a0 = hsub2_u32((X & 0x000f000fu) | 0x64006400u, kSubLo);
                    const uint32_t a1 = hsub2_u32((X8 & 0x000f000fu) | 0x64006400u, kSubLo);
                    const uint32_t a2 = hsub2_u32((Y & 0x000f000fu) | 0x64006400u, kSubLo);
                    const uint32_t a3 = hsub2_u32((Y8 & 0x000f000fu) | 0x64006400u, kSubLo);
                    const int ml = 2 * q;
                    mma_f16_16816(oacc[ml], a0, a1, a2, a3, bA0, bA1);
                    if constexpr (G > 4 && PLO) mma_f16_16816(oacc[ml], a0, a1, a2, a3, bB0, bB1);
                    const uint32_t c0 = hfma2_u32((X & 0x00f000f0u) | 0x64006400u, kMul, kAdd);
                    const uint32_t c1 = hfma2_u32((X8 & 0x00f000f0u) | 0x64006400u, kMul, kAdd);
                    const uint32_t c2 = hfma2_u32((Y & 0x00f000f0u) | 0x64006400u, kMul, kAdd);
                    const uint32_t c3 = hfma2_u32((Y8 & 0x00f000f0u) | 0x64006400u, kMul, kAdd);
                    mma_f16_16816(oacc[ml + 1], c0, c1, c2, c3, bA0, bA1);
                    if constexpr (G > 4 && PLO) mma_f16_16816(oacc[ml + 1], c0, c1, c2, c3, bB0, bB1);
                } else {
                    // ISO: this warp's m-tiles u in [u0, u0 + MPER) of block gv; row g <-> dim 16g + 2u (+1)
                    const int u0 = mt0 - gv * K::MTPG;
                    uint32_t cw[4][2];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int rb = Geo::OFF_VC + (2 * t + (j & 1) + 8 * (j >> 1)) * Geo::VCB;
                        if constexpr (VENC == ENC_ISO3) {
                            if constexpr (MPER == 8) { cw[j][0] = lds<uint32_t>(st, rb + 48 * gv + 4 * g); cw[j][1] = lds<uint16_t>(st, rb + 48 * gv + 32 + 2 * g); }
                            else { cw[j][0] = lds<uint16_t>(st, rb + 48 * gv + 4 * g + u0 / 2); cw[j][1] = lds<uint8_t>(st, rb + 48 * gv + 32 + 2 * g + u0 / 4); }
                        } else {
                            if constexpr (MPER == 8) { const uint2 v = lds<uint2>(st, rb + 64 * gv + 8 * g); cw[j][0] = v.x; cw[j][1] = v.y; }
                            else { cw[j][0] = lds<uint32_t>(st, rb + 64 * gv + 8 * g + u0); cw[j][1] = 0; }
                        }
                    }
#pragma unroll
                    for (int uu = 0; uu < MPER; ++uu) {
                        uint32_t X[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint32_t idx;
                            if constexpr (VENC == ENC_ISO3) idx = ((cw[j][0] >> (4 * uu)) & 0xfu) | (((cw[j][1] >> (2 * uu)) & 3u) << 4);
                            else idx = ((uu < 4 ? cw[j][0] : cw[j][1]) >> (8 * (uu & 3))) & 0xffu;
                            X[j] = lut[idx * 32];
                        }
                        const uint32_t a0 = prmt(X[0], X[1], 0x5410u), a1 = prmt(X[0], X[1], 0x7632u);
                        const uint32_t a2 = prmt(X[2], X[3], 0x5410u), a3 = prmt(X[2], X[3], 0x7632u);
                        const int ml = q * K::MPER + uu;
                        mma_f16_16816(oacc[ml], a0, a1, a2, a3, bA0, bA1);
                        if constexpr (G > 4 && PLO) mma_f16_16816(oacc[ml], a0, a1, a2, a3, bB0, bB1);
                    }
                }
            }
        }
        gi += (uint32_t)npg;

        // ---------------- pair -> CTA merge ----------------
        __syncthreads();   // all pairs done with their stages: the area becomes the merge buffer
        {
            float* Ow = reinterpret_cast<float*>(smem) + (size_t)pair * 8 * D;   // [8 cols][D]
            float lq = l_run;
            lq += __shfl_xor_sync(0xffffffffu, lq, 1);
            lq += __shfl_xor_sync(0xffffffffu, lq, 2);
            if (role == 0 && t == 0) { sm_mw[pair * 8 + g] = m_run; sm_lw[pair * 8 + g] = lq; }
            // remove the +1152 code offset: O -= 1152 * (sum of fed probabilities) per V group and column
            float rs[K::NGVH][2];
#pragma unroll
            for (int q = 0; q < K::NGVH; ++q) {
                float r = 0.0f;
                if constexpr (K::VBIAS) {
                    r = rsum[q];
                    r += __shfl_xor_sync(0xffffffffu, r, 1);
                    r += __shfl_xor_sync(0xffffffffu, r, 2);
                }
                rs[q][0] = __shfl_sync(0xffffffffu, r, (2 * t) * 4) * 1152.0f;
                rs[q][1] = __shfl_sync(0xffffffffu, r, (2 * t + 1) * 4) * 1152.0f;
            }
            const float inv = (E_run == 1000) ? 0.0f : __int_as_float((127 - E_run) << 23);
#pragma unroll
            for (int ml = 0; ml < K::MTH; ++ml) {
                const int mt = role * K::MTH + ml;
                constexpr int QI = 0;
                const int q = ml / K::MPER + QI;
                int dA;
                if constexpr (VENC == ENC_INT8) dA = 64 * (mt >> 2) + 8 * g + 2 * (mt & 3);
                else if constexpr (VENC == ENC_Q4) dA = 32 * (mt >> 1) + 2 * g + 16 * (mt & 1);
                else dA = 128 * (mt >> 3) + 16 * g + 2 * (mt & 7);
                Ow[(2 * t) * D + dA] = (oacc[ml][0] - rs[q][0]) * inv;
                Ow[(2 * t + 1) * D + dA] = (oacc[ml][1] - rs[q][1]) * inv;
                Ow[(2 * t) * D + dA + 1] = (oacc[ml][2] - rs[q][0]) * inv;
                Ow[(2 * t + 1) * D + dA + 1] = (oacc[ml][3] - rs[q][1]) * inv;
            }
        }
        __syncthreads();
        if (tid < G) {
            float M = -INFINITY;
            for (int w = 0; w < kNP; ++w) M = fmaxf(M, sm_mw[w * 8 + tid]);
            float Ls = 0.0f;
            for (int w = 0; w < kNP; ++w) {
                float mw = sm_mw[w * 8 + tid];
                float wt = (mw == -INFINITY) ? 0.0f : exp2f(mw - M);
                s_pw[w][tid] = wt;
                Ls += wt * sm_lw[w * 8 + tid];
            }
            s_pM[tid] = M;
            s_pL[tid] = Ls;
        }
        __syncthreads();
        // combine pairs and the columns belonging to the same head
        constexpr int PER = (8 * D + kThreads - 1) / kThreads;
        float vals[PER];
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const int i = tid + k * kThreads;
            float acc = 0.0f;
            if (i < G * D) {
                const int h = i / D, d = i % D;
#pragma unroll 1
                for (int w = 0; w < kNP; ++w) {
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
        __syncthreads();   // pair rows fully read
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
