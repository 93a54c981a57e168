// extend.cu -- prefill-chunk (extend) attention over a packed int8 prefix plus
// the chunk's own bf16 K/V, on tcgen05 tensor cores with TMEM accumulators.
//
// Method (page title, section): "feat(kvcache): add ISO3/ISO4 KV-cache
// quantization", "What": extend attends the packed prefix plus the bf16 new
// tokens and packs them only after attention (prefill never consumes its own
// quantized KV); "qwen35/q36: --kv - int8 K/V caches", "What it does": prompt
// chunks dequantize the int8 cache on the fly.
//
// GB300 design: one CTA per tile of 128 (token, query head) rows of one KV-head
// group (GQA packing: 128/G tokens x G heads share every K/V tile), 9 warps:
//   * warps 0-3 (softmax): thread r owns TMEM lane r = row r. It combines the
//     per-group partial scores, applies the online softmax (lazy rescale: the
//     running max only moves when it grows by more than 2^8), writes P (fp16)
//     to shared memory and rescales the O row in TMEM when the max moves.
//   * warps 4-7 (producer): fill double-buffered K and V^T tiles of 64 keys in
//     the UMMA K-major, 128-byte-swizzled layout. Prefix keys come through the
//     page table as int8 codes (exact fp16 1152 + c for K, fp16(c * scale) for
//     V); new tokens are bf16 (converted to fp16).
//   * warp 8 (MMA): owns the 512 TMEM columns and issues tcgen05.mma:
//     S_g = Q_g K_g^T per 64-dim group g into 4 x 64 TMEM columns (so the
//     per-(key, group) K scales stay exact and are applied in fp32 by the
//     softmax threads), and O += P V^T into 256 columns.
//   QK of tile j+1 is issued as soon as the softmax threads have pulled S(j)
//   into registers, so it overlaps the softmax of tile j; PV(j) follows P(j).
#include "qkv_device.cuh"
#include "qkv_params.h"
#include "tcgen05.cuh"

namespace qkv {

__device__ unsigned int g_err_extend;

constexpr int kXT = 64;          // keys per KV tile
constexpr int kXThreads = 288;   // 4 softmax warps, 4 producer warps, 1 MMA warp

// shared-memory map (bytes from a 1 KB aligned base)
template <int D>
struct XGeo {
    static constexpr int NA = D / 64;                    // 64-dim atoms (= K scale groups)
    static constexpr int OFF_Q = 0;                      // NA atoms x 128 rows x 128 B
    static constexpr int Q_BYTES = NA * 128 * 128;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;        // 2 buffers x NA atoms x 64 rows x 128 B
    static constexpr int K_BYTES = NA * 64 * 128;
    static constexpr int OFF_V = OFF_K + 2 * K_BYTES;    // 2 buffers x D rows x 128 B
    static constexpr int V_BYTES = D * 128;
    static constexpr int OFF_P = OFF_V + 2 * V_BYTES;    // 128 rows x 128 B
    static constexpr int OFF_SIG = OFF_P + 128 * 128;    // 2 x 64 keys x NA floats
    static constexpr int OFF_BAR = OFF_SIG + 2 * 64 * 4 * 4;
    static constexpr int OFF_TMEM = OFF_BAR + 16 * 8;
    static constexpr int SMEM = OFF_TMEM + 16;
    static constexpr int S_COLS = NA * 64;               // TMEM columns of the group scores
    static constexpr int TMEM_COLS = 512;
    static_assert(S_COLS + D <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM + 1024 <= 232448 - 1024, "shared memory budget");
};

enum { B_Q = 0, B_KVF0 = 1, B_KVF1 = 2, B_KVE0 = 3, B_KVE1 = 4, B_SFULL = 5, B_SFREE = 6, B_PFULL = 7, B_PVDONE = 8 };

__device__ __forceinline__ uint32_t bf16x2_to_h2(uint32_t w) {
    return f32x2_to_h2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

template <int D, int G>
__global__ void __launch_bounds__(kXThreads, 1) extend_kernel(const ExtendParams p) {
    using X = XGeo<D>;
    constexpr int NA = X::NA;
    constexpr int TPT = 128 / G;   // tokens per tile
    extern __shared__ __align__(1024) uint8_t xsmem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(xsmem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.z, hg = blockIdx.y;
    const int cu0 = p.cu[b], T = p.cu[b + 1] - cu0;
    const int tok0 = blockIdx.x * TPT;
    if (T <= 0 || tok0 >= T) return;   // whole CTA, before any allocation
    int L0 = p.prefix_lens[b];
    if (L0 < 0 || L0 > p.max_pages * kPage) {
        if (tid == 0) atomicOr(&g_err_extend, kErrPos);
        L0 = max(0, min(L0, p.max_pages * kPage));
    }
    const int kvh = hg / (p.Gtot / G), hq0 = kvh * p.Gtot + (hg % (p.Gtot / G)) * G;
    const int tok_last = min(T, tok0 + TPT) - 1;
    const int NTP = (L0 + kXT - 1) / kXT;
    const int NTN = p.causal ? (tok_last + kXT) / kXT : (T + kXT - 1) / kXT;
    const int NT = NTP + NTN;
    const int32_t* ptrow = p.page_table + (size_t)b * p.max_pages;

    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + X::OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + X::OFF_TMEM);
    float* sig = reinterpret_cast<float*>(sm + X::OFF_SIG);   // [2][64][4]

    if (warp == 8) tmem_alloc(tmem_slot, X::TMEM_COLS);
    if (tid == 0) {
        mbar_init(&bars[B_Q], 128);
        mbar_init(&bars[B_KVF0], 128);
        mbar_init(&bars[B_KVF1], 128);
        mbar_init(&bars[B_KVE0], 1);
        mbar_init(&bars[B_KVE1], 1);
        mbar_init(&bars[B_SFULL], 1);
        mbar_init(&bars[B_SFREE], 128);
        mbar_init(&bars[B_PFULL], 128);
        mbar_init(&bars[B_PVDONE], 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_S = tmem, tmem_O = tmem + X::S_COLS;
    bool ok = true;
    auto wait = [&](int bi, uint32_t parity) {
        if (!mbar_wait_bounded(&bars[bi], parity)) {
            if (ok) atomicOr(&g_err_extend, kErrWait);
            ok = false;
        }
    };

    if (warp >= 4 && warp < 8) {
        // =========================== producer ===========================
        const int pt = tid - 128;
        {
            // Q tile: row r = (token r / G, head r % G), bf16 -> fp16
            const int r = pt, tok = tok0 + r / G;
            uint8_t* qs = sm + X::OFF_Q;
            const uint16_t* qrow = p.q + ((size_t)(cu0 + min(tok, T - 1)) * p.Hq + hq0 + r % G) * D;
#pragma unroll 4
            for (int c = 0; c < D / 8; ++c) {
                uint4 o = make_uint4(0, 0, 0, 0);
                if (tok < T) {
                    const uint4 w = *reinterpret_cast<const uint4*>(qrow + 8 * c);
                    o = make_uint4(bf16x2_to_h2(w.x), bf16x2_to_h2(w.y), bf16x2_to_h2(w.z), bf16x2_to_h2(w.w));
                }
                *reinterpret_cast<uint4*>(qs + (c >> 3) * 16384 + sw_off(r, c & 7)) = o;
            }
            fence_proxy_async();
            mbar_arrive(&bars[B_Q]);
        }
        for (int j = 0; j < NT && ok; ++j) {
            const int buf = j & 1;
            if (j >= 2) wait(B_KVE0 + buf, ((j - 2) >> 1) & 1);
            uint8_t* ksm = sm + X::OFF_K + buf * X::K_BYTES;
            uint8_t* vsm = sm + X::OFF_V + buf * X::V_BYTES;
            float* sg = sig + buf * 64 * 4;
            const bool prefix = j < NTP;
            // ---- K tile: thread -> (key kk, half hf of the head dim) ----
            {
                constexpr int HALF = D / 2;
                const int kk = pt >> 1, hf = pt & 1;
                if (prefix) {
                    const int pos = kXT * j + kk;
                    int page = -1;
                    if (pos < L0) {
                        page = ptrow[pos >> 4];
                        if (page < 0 || page >= p.num_pages) { atomicOr(&g_err_extend, kErrPage); page = -1; }
                    }
                    const long long row = ((long long)max(page, 0) * p.Hkv + kvh) * kPage + (pos & 15);
                    const uint8_t* src = p.kc + row * D + HALF * hf;
#pragma unroll
                    for (int c = 0; c < HALF / 16; ++c) {
                        uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
                        if (page >= 0) {
                            const uint4 w = *reinterpret_cast<const uint4*>(src + 16 * c);
                            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
                            uint32_t h[8];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const uint32_t x = ws[u] ^ 0x80808080u;   // 1152 + code, exact in fp16
                                h[2 * u] = prmt(x, 0x64646464u, 0x4140u);
                                h[2 * u + 1] = prmt(x, 0x64646464u, 0x4342u);
                            }
                            o0 = make_uint4(h[0], h[1], h[2], h[3]);
                            o1 = make_uint4(h[4], h[5], h[6], h[7]);
                        }
                        const int d0 = HALF * hf + 16 * c;
                        uint8_t* atom = ksm + (d0 >> 6) * 8192;
                        const int cc = (d0 & 63) >> 3;
                        *reinterpret_cast<uint4*>(atom + sw_off(kk, cc)) = o0;
                        *reinterpret_cast<uint4*>(atom + sw_off(kk, cc + 1)) = o1;
                    }
#pragma unroll
                    for (int gq = 0; gq < NA / 2; ++gq) {
                        const int gidx = (NA / 2) * hf + gq;
                        float sv = 0.0f;
                        if (page >= 0) sv = f16_bits_to_f32(reinterpret_cast<const uint16_t*>(p.ks + row * (D / 32))[gidx]);
                        sg[kk * 4 + gidx] = sv;
                    }
                } else {
                    const int n = kXT * (j - NTP) + kk;
                    const uint16_t* src = p.k_new + ((size_t)(cu0 + min(n, T - 1)) * p.Hkv + kvh) * D + HALF * hf;
#pragma unroll
                    for (int c = 0; c < HALF / 8; ++c) {
                        uint4 o = make_uint4(0, 0, 0, 0);
                        if (n < T) {
                            const uint4 w = *reinterpret_cast<const uint4*>(src + 8 * c);
                            o = make_uint4(bf16x2_to_h2(w.x), bf16x2_to_h2(w.y), bf16x2_to_h2(w.z), bf16x2_to_h2(w.w));
                        }
                        const int d0 = HALF * hf + 8 * c;
                        *reinterpret_cast<uint4*>(ksm + (d0 >> 6) * 8192 + sw_off(kk, (d0 & 63) >> 3)) = o;
                    }
#pragma unroll
                    for (int gq = 0; gq < NA / 2; ++gq) sg[kk * 4 + (NA / 2) * hf + gq] = 1.0f;
                }
            }
            // ---- V^T tile: warp -> 64 dims (one scale group), lane -> keys 2l, 2l+1 ----
            {
                const int wv = pt >> 5;                // 0..3
                for (int dblk = wv; dblk < D / 64; dblk += 4) {
                    uint32_t hv[2][32];                 // [key][dim pair] half2 of (dim 2m, 2m+1)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int kk = 2 * lane + e;
                        if (prefix) {
                            const int pos = kXT * j + kk;
                            int page = -1;
                            if (pos < L0) {
                                page = ptrow[pos >> 4];
                                if (page < 0 || page >= p.num_pages) page = -1;
                            }
                            const long long row = ((long long)max(page, 0) * p.Hkv + kvh) * kPage + (pos & 15);
                            uint32_t sv2 = 0;
                            if (page >= 0) {
                                const uint32_t sb = reinterpret_cast<const uint16_t*>(p.vs + row * (D / 32))[dblk];
                                sv2 = sb | (sb << 16);
                            }
                            const uint8_t* src = p.vc + row * D + 64 * dblk;
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                uint4 w = make_uint4(0, 0, 0, 0);
                                if (page >= 0) w = *reinterpret_cast<const uint4*>(src + 16 * c);
                                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                                for (int u = 0; u < 4; ++u) {
                                    const uint32_t x = ws[u] ^ 0x80808080u;
                                    const uint32_t c01 = hsub2_u32(prmt(x, 0x64646464u, 0x4140u), 0x64806480u);
                                    const uint32_t c23 = hsub2_u32(prmt(x, 0x64646464u, 0x4342u), 0x64806480u);
                                    // fp16(code * scale): one correctly rounded fp16 product
                                    hv[e][8 * c + 2 * u] = hfma2_u32(c01, sv2, 0u);
                                    hv[e][8 * c + 2 * u + 1] = hfma2_u32(c23, sv2, 0u);
                                }
                            }
                        } else {
                            const int n = kXT * (j - NTP) + kk;
                            const uint16_t* src = p.v_new + ((size_t)(cu0 + min(n, T - 1)) * p.Hkv + kvh) * D + 64 * dblk;
#pragma unroll
                            for (int c = 0; c < 8; ++c) {
                                uint4 w = make_uint4(0, 0, 0, 0);
                                if (n < T) w = *reinterpret_cast<const uint4*>(src + 8 * c);
                                hv[e][4 * c + 0] = bf16x2_to_h2(w.x);
                                hv[e][4 * c + 1] = bf16x2_to_h2(w.y);
                                hv[e][4 * c + 2] = bf16x2_to_h2(w.z);
                                hv[e][4 * c + 3] = bf16x2_to_h2(w.w);
                            }
                        }
                    }
                    // V^T row d = 64 dblk + dd holds keys along K: (key 2l, key 2l + 1) -> 4 bytes
                    const int kc = (2 * lane) >> 3, kb = ((2 * lane) & 7) * 2;
#pragma unroll
                    for (int m = 0; m < 32; ++m) {
                        const int d = 64 * dblk + 2 * m;
                        const uint32_t lo = prmt(hv[0][m], hv[1][m], 0x5410u);   // dim 2m of both keys
                        const uint32_t hi = prmt(hv[0][m], hv[1][m], 0x7632u);   // dim 2m + 1
                        *reinterpret_cast<uint32_t*>(vsm + sw_off(d, kc) + kb) = lo;
                        *reinterpret_cast<uint32_t*>(vsm + sw_off(d + 1, kc) + kb) = hi;
                    }
                }
            }
            fence_proxy_async();
            mbar_arrive(&bars[B_KVF0 + buf]);
        }
    } else if (warp == 8) {
        // =========================== MMA issue ===========================
        if (lane == 0) {
            const uint32_t qs = smem_addr(sm + X::OFF_Q);
            constexpr uint32_t IDQK = idesc_f16(128, 64), IDPV = idesc_f16(128, D);
            auto issue_qk = [&](int j) {
                const int buf = j & 1;
                wait(B_KVF0 + buf, (j >> 1) & 1);
                if (j >= 1) wait(B_SFREE, (j - 1) & 1);
                tc_fence_after();
                const uint32_t ks = smem_addr(sm + X::OFF_K + buf * X::K_BYTES);
#pragma unroll
                for (int g = 0; g < NA; ++g)
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        umma_f16(tmem_S + 64 * g, sw128_desc(qs + g * 16384 + 32 * u), sw128_desc(ks + g * 8192 + 32 * u),
                                 IDQK, u > 0);
                umma_commit(&bars[B_SFULL]);
            };
            wait(B_Q, 0);
            if (NT > 0) issue_qk(0);
            for (int j = 0; j < NT && ok; ++j) {
                if (j + 1 < NT) issue_qk(j + 1);
                wait(B_PFULL, j & 1);
                tc_fence_after();
                const uint32_t ps = smem_addr(sm + X::OFF_P);
                const uint32_t vs = smem_addr(sm + X::OFF_V + (j & 1) * X::V_BYTES);
#pragma unroll
                for (int u = 0; u < kXT / 16; ++u)
                    umma_f16(tmem_O, sw128_desc(ps + 32 * u), sw128_desc(vs + 32 * u), IDPV, (j > 0 || u > 0));
                umma_commit(&bars[B_KVE0 + (j & 1)]);
                umma_commit(&bars[B_PVDONE]);
            }
        }
        __syncwarp();
    } else {
        // =========================== softmax ===========================
        const int r = tid;   // TMEM lane and tile row
        const int tok = tok0 + r / G, hq = hq0 + r % G;
        const bool rvalid = tok < T;
        const int tokc = min(tok, T - 1);
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        // 1152 * sum of the fp16 query over each 64-dim group removes the K code offset
        float bias[NA];
        {
            const uint16_t* qrow = p.q + ((size_t)(cu0 + tokc) * p.Hq + hq) * D;
#pragma unroll
            for (int g = 0; g < NA; ++g) {
                float s = 0.0f;
#pragma unroll 4
                for (int c = 0; c < 8; ++c) {
                    const uint4 w = *reinterpret_cast<const uint4*>(qrow + 64 * g + 8 * c);
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float2 f = h2_to_f32x2(bf16x2_to_h2(ws[u]));
                        s += f.x + f.y;
                    }
                }
                bias[g] = 1152.0f * s;
            }
        }
        float m_used = -INFINITY, l = 0.0f;
        uint8_t* psm = sm + X::OFF_P;
        for (int j = 0; j < NT && ok; ++j) {
            const int buf = j & 1;
            const bool prefix = j < NTP;
            const float* sg = sig + buf * 64 * 4;
            wait(B_KVF0 + buf, (j >> 1) & 1);   // the producers' key scales of this tile
            wait(B_SFULL, j & 1);
            tc_fence_after();
            float s[kXT];
#pragma unroll
            for (int c = 0; c < kXT / 16; ++c) {
                float acc[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) acc[e] = 0.0f;
#pragma unroll
                for (int g = 0; g < NA; ++g) {
                    float v[16];
                    tmem_ld16(tmem_S + lane_base + 64 * g + 16 * c, v);
                    const float bg = prefix ? bias[g] : 0.0f;
#pragma unroll
                    for (int e = 0; e < 16; ++e) acc[e] += sg[(16 * c + e) * 4 + g] * (v[e] - bg);
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) s[16 * c + e] = acc[e] * p.scale_log2;
            }
            tc_fence_before();
            mbar_arrive(&bars[B_SFREE]);   // S(j) is in registers: QK(j + 1) may overwrite it
            float rmax = -INFINITY;
#pragma unroll
            for (int kk = 0; kk < kXT; ++kk) {
                bool vis;
                if (prefix) vis = (kXT * j + kk) < L0;
                else {
                    const int n = kXT * (j - NTP) + kk;
                    vis = n < T && (!p.causal || n <= tokc);
                }
                if (!vis) s[kk] = -INFINITY;
                rmax = fmaxf(rmax, s[kk]);
            }
            // PV(j - 1) must be done before P is overwritten and before O is rescaled
            if (j >= 1) wait(B_PVDONE, (j - 1) & 1);
            tc_fence_after();
            // frame update per row; the TMEM rescale of O is a whole-warp operation
            // (tcgen05.ld/st are .sync.aligned), so it runs warp-uniformly with
            // factor 1 for rows whose frame did not move
            const bool move = rmax > m_used + 8.0f;
            float alpha = 1.0f;
            if (move) {
                alpha = (m_used == -INFINITY) ? 0.0f : fast_exp2(m_used - rmax);
                l *= alpha;
                m_used = rmax;
            }
            if (j >= 1 && __any_sync(0xffffffffu, move)) {
#pragma unroll 1
                for (int c = 0; c < D / 16; ++c) {
                    float v[16];
                    tmem_ld16(tmem_O + lane_base + 16 * c, v);
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] *= alpha;
                    tmem_st16(tmem_O + lane_base + 16 * c, v);
                }
            }
            const float mref = (m_used == -INFINITY) ? 0.0f : m_used;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint32_t h[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float p0 = fast_exp2(s[8 * c + 2 * u] - mref), p1 = fast_exp2(s[8 * c + 2 * u + 1] - mref);
                    h[u] = f32x2_to_h2(p0, p1);
                    const float2 f = h2_to_f32x2(h[u]);
                    l += f.x + f.y;
                }
                *reinterpret_cast<uint4*>(psm + sw_off(r, c)) = make_uint4(h[0], h[1], h[2], h[3]);
            }
            fence_proxy_async();
            tc_fence_before();
            mbar_arrive(&bars[B_PFULL]);
        }
        if (NT > 0) wait(B_PVDONE, (NT - 1) & 1);
        tc_fence_after();
        const float inv = (l > 0.0f) ? 1.0f / l : 0.0f;
        const size_t obase = ((size_t)(cu0 + tokc) * p.Hq + hq) * D;
#pragma unroll 1
        for (int c = 0; c < D / 16; ++c) {
            float v[16];
            tmem_ld16(tmem_O + lane_base + 16 * c, v);
            if (rvalid) {
                if (p.out_f32) {
                    float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + obase + 16 * c);
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[e] = make_float4(v[4 * e] * inv, v[4 * e + 1] * inv, v[4 * e + 2] * inv, v[4 * e + 3] * inv);
                } else {
                    uint32_t h[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        __nv_bfloat162 bb = __floats2bfloat162_rn(v[2 * e] * inv, v[2 * e + 1] * inv);
                        h[e] = *reinterpret_cast<uint32_t*>(&bb);
                    }
                    uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + obase + 16 * c);
                    o[0] = make_uint4(h[0], h[1], h[2], h[3]);
                    o[1] = make_uint4(h[4], h[5], h[6], h[7]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem, X::TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
cudaError_t extend_read_error(unsigned* out, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_err_extend, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    unsigned z = 0;
    return cudaMemcpyToSymbol(g_err_extend, &z, sizeof(unsigned));
}

template <int D, int G>
static cudaError_t xlaunch(dim3 grid, const ExtendParams& p, cudaStream_t st) {
    auto fn = extend_kernel<D, G>;
    constexpr int smem = XGeo<D>::SMEM + 1024;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    fn<<<grid, kXThreads, smem, st>>>(p);
    return cudaGetLastError();
}

// int8 pools; returns cudaErrorInvalidValue for shapes this kernel does not cover
cudaError_t extend_launch(int fmt, int D, int G, int max_q_len, int NH, int B, const ExtendParams& p, cudaStream_t st) {
    if (fmt != 0) return cudaErrorInvalidValue;
    const int tpt = 128 / G;
    dim3 grid((unsigned)((max_q_len + tpt - 1) / tpt), (unsigned)NH, (unsigned)B);
    if (D == 256) {
        switch (G) {
            case 1: return xlaunch<256, 1>(grid, p, st);
            case 2: return xlaunch<256, 2>(grid, p, st);
            case 4: return xlaunch<256, 4>(grid, p, st);
            case 8: return xlaunch<256, 8>(grid, p, st);
        }
    } else if (D == 128) {
        switch (G) {
            case 1: return xlaunch<128, 1>(grid, p, st);
            case 2: return xlaunch<128, 2>(grid, p, st);
            case 4: return xlaunch<128, 4>(grid, p, st);
            case 8: return xlaunch<128, 8>(grid, p, st);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace qkv
