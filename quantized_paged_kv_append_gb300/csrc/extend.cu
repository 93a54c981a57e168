// extend.cu -- prefill-chunk (extend) attention over a packed int8 prefix plus
// the chunk's own bf16 K/V, on tcgen05 tensor cores with TMEM accumulators.
//
// Method (page title, section): "feat(kvcache): add ISO3/ISO4 KV-cache
// quantization", "What": extend attends the packed prefix plus the bf16 new
// tokens and packs them only after attention (prefill never consumes its own
// quantized KV); "qwen35/q36: --kv - int8 K/V caches", "What it does": prompt
// chunks dequantize the int8 cache on the fly.
//
// GB300 design. A prep kernel dequantizes the keys once per call into the
// caller's workspace (L2-resident at prefill sizes): per (sequence, KV head),
// K' rows in fp16 (the exact code c for the packed prefix, the bf16 new tokens
// converted to fp16) with fp32 key scales beside them (the prefix's K scale per
// 64-dim group, 1 for new tokens, both times the softmax scale), and V^T in
// fp16 (c * scale rounded once for the prefix, the new tokens converted), keys
// padded to 64 so that prefix and new tokens never share a tile. The attention
// kernel then streams 64-key tiles of K' and V^T with TMA (128-byte swizzle,
// exactly the UMMA operand layouts): one CTA per tile of 128 (token, query
// head) rows of one KV-head group (GQA packing: 128/G tokens x G heads share
// every K/V tile), 6 warps:
//   * warps 0-15 (softmax): row r = TMEM lane r is shared by four threads, one
//     per 16 of the 64 keys (warps w, w + 4, w + 8, w + 12). Each combines its
//     keys' per-group partial scores (4 FMAs a key), the four exchange their row
//     maxima once per tile, and all apply the same online-softmax frame (lazy
//     rescale: the running max only moves when it grows by more than 2^8);
//     each writes its part of P (fp16) and rescales its part of the O row.
//   * warps 16 and 17 (producers, one thread each): TMA of the K' + key-scale
//     tiles and of the V^T tiles, double-buffered on separate barriers (a K slot
//     is free once the softmax threads hold the tile's scores and key scales,
//     long before PV of the tile).
//   * warp 18 (MMA): owns the 512 TMEM columns and issues tcgen05.mma:
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
constexpr int kXSplit = 4;                 // threads per row: each takes 64 / kXSplit keys of a tile
constexpr int kXSoft = 128 * kXSplit;      // softmax warps: row r = lane + 32 (w % 4), key part w / 4
constexpr int kXThreads = kXSoft + 96;     // + 2 producer warps (K, V) + 1 MMA warp
constexpr int kXProd = kXSoft / 32, kXMma = kXProd + 2;

// shared-memory map (bytes from a 1 KB aligned base). ISO prefix tiles take the rotated
// query as two fp16 tiles: hi in the query region (which holds the plain query once the
// prefix is done) and the fp16 remainder lo in one more tile after the rest.
// XM: the kind of prefix tile. 0: plain keys; 1: ISO (raw levels against the rotated query,
// fp16 hi + lo); 2: two key planes, fp16 hi + lo, against the plain query (q4 keys rotated
// back to the original domain).
template <int D, int XM = 0>
struct XGeo {
    static constexpr bool ISO = XM == 1;
    static constexpr int NA = D / 64;                    // 64-dim atoms (= K scale groups)
    static constexpr int OFF_Q = 0;                      // NA atoms x 128 rows x 128 B
    static constexpr int Q_BYTES = NA * 128 * 128;
    // K and V staging depth: two tiles, one at head_dim 256 when the prefix tiles need an extra
    // tile (ISO: the rotated query's lo part; XM 2: the lo key plane), which takes the room of
    // the second K and V buffers
    static constexpr int NB = (XM != 0 && D == 256) ? 1 : 2;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;        // NB buffers x NA atoms x 64 rows x 128 B
    static constexpr int K_BYTES = NA * 64 * 128;
    static constexpr int OFF_V = OFF_K + NB * K_BYTES;   // NB buffers x D rows x 128 B
    static constexpr int V_BYTES = D * 128;
    static constexpr int OFF_P = OFF_V + NB * V_BYTES;   // 128 rows x 128 B
    static constexpr int KS_BYTES = kXT * NA * 4;        // fp32 K scales x softmax scale of a tile [64][NA]
    static constexpr int OFF_KS = OFF_P + 128 * 128;     // NB buffers
    static constexpr int OFF_RED = OFF_KS + NB * KS_BYTES;   // [2 tiles][kXSplit parts][128 rows] row-max / row-sum exchange
    static constexpr int OFF_BAR = OFF_RED + 2 * kXSplit * 128 * 4;
    static constexpr int OFF_TMEM = OFF_BAR + 24 * 8;
    static constexpr int OFF_QR = (OFF_TMEM + 16 + 1023) / 1024 * 1024;   // the extra tile: lo query (ISO) or lo keys
    static constexpr int SMEM = XM ? OFF_QR + Q_BYTES : OFF_TMEM + 16;
    static_assert(K_BYTES <= Q_BYTES, "a lo key tile fits the extra tile");
    static constexpr int S_COLS = NA * 64;               // TMEM columns of the group scores
    static constexpr int TMEM_COLS = 512;
    static_assert(S_COLS + D <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM + 1024 <= 232448 - 1024, "shared memory budget");
};

enum {
    B_Q = 0,
    B_KF = 1,     // [2] K' tile + key scales landed (1 + tx)
    B_VF = 3,     // [2] V^T tile landed (1 + tx)
    B_KE = 5,     // [2] K slot free: every softmax thread has the tile's scores and key scales
                  //     (after SFULL, so Q K^T of the tile has completed too)
    B_VE = 7,     // [2] PV of the tile complete: V slot free (commit)
    B_SFULL = 9, B_SFREE = 10, B_PFULL = 11, B_PVDONE = 12,
    B_RMX = 13,   // [2] row maxima of every key part written (all softmax threads)
    B_RSUM = 15,  // row sums of every part written
    B_DRAIN = 16, // every MMA of the CTA complete (commit), before TMEM is released
    B_QPLAIN = 17 // ISO: the plain query replaced the rotated hi tile (all softmax threads)
};

__device__ __forceinline__ uint32_t bf16x2_to_h2(uint32_t w) {
    return f32x2_to_h2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// ---------------------------------------------------------------------------
// prep: dequantize the keys of one 64-key tile of one (sequence, KV head) into
// the workspace planes. Tile t < NTP covers prefix positions 64 t .. 64 t + 63
// (read through the page table), tile NTP + u covers new tokens 64 u .. 64 u + 63.
// Positions past the prefix or the chunk are zero (their scores are masked and
// their P is 0, so V must be finite). Thread (i, qd): position i, dims
// [qd D/4, (qd + 1) D/4). V^T goes through a transposed shared tile.
// What the prefix rows hold, per format (FMT = qkv_format):
//   0 int8 : K' = the exact code c, key scale = the fp16 group scale;
//            V = fp16(c * scale), one rounding.
//   1 k8v4 : K as int8. V: the q4_0 values (q - 8) * d of the FWHT-rotated row,
//            rotated back with the same transform (H / 16 is its own inverse) in
//            fp32 across the four threads of the row, then rounded to fp16 once.
//   2, 3 ISO3 / ISO4 (head_dim 128 or 256): K' = the Lloyd-Max levels c (exact in
//            fp16) with the block's fp16 norm as the key scale of both its
//            64-dim groups; the attention kernel rotates the query for these
//            tiles. V: each 4-D group rotated back, u = conj(q) (x) c in fp32,
//            then fp16(norm * u), one rounding.
// V reaches the attention kernel in the original domain, so the output needs
// no inverse transform.
// ---------------------------------------------------------------------------
__constant__ float c_x_levels[2][16];   // [0] ISO3 (8 levels), [1] ISO4 (16 levels)

// conj(q) (x) c for one 4-D group (q = (w, x, y, z) unit quaternion)
__device__ __forceinline__ void quat_conj_mul(const float* q, float a, float b, float c, float d, float (&u)[4]) {
    u[0] = q[0] * a + q[1] * b + q[2] * c + q[3] * d;
    u[1] = q[0] * b - q[1] * a - q[2] * d + q[3] * c;
    u[2] = q[0] * c + q[1] * d - q[2] * a - q[3] * b;
    u[3] = q[0] * d - q[1] * c + q[2] * b - q[3] * a;
}

// FWHT-256 x 1/16 of one row held by its four threads (64 values each, thread qd owns
// dims [64 qd, 64 qd + 64)): butterflies at distances 1 .. 32 inside the thread, 64 and
// 128 across the threads (lanes qd ^ 1, qd ^ 2). Every lane of the warp must call it.
__device__ __forceinline__ void fwht256_rows4(float (&x)[64], int qd) {
#pragma unroll
    for (int h = 1; h < 64; h <<= 1) {
#pragma unroll
        for (int e = 0; e < 64; ++e) {
            if (e & h) continue;
            const float a = x[e], c = x[e + h];
            x[e] = a + c;
            x[e + h] = a - c;
        }
    }
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
        const bool upper = (qd & m) != 0;
#pragma unroll
        for (int e = 0; e < 64; ++e) {
            const float o = __shfl_xor_sync(0xffffffffu, x[e], m);
            x[e] = upper ? o - x[e] : x[e] + o;
        }
    }
#pragma unroll
    for (int e = 0; e < 64; ++e) x[e] *= 0.0625f;
}

// the q4_0 values (q - 8) * d of blocks 2 qd and 2 qd + 1 of a rotated row (x: 64 values)
__device__ __forceinline__ void q4_blocks2(const uint8_t* code_row, const uint8_t* scale_row, int qd, float (&x)[64]) {
    const uint8_t* src = code_row + 32 * qd;
    const uint16_t* sc = reinterpret_cast<const uint16_t*>(scale_row);
#pragma unroll
    for (int lb = 0; lb < 2; ++lb) {
        const float d16 = f16_bits_to_f32(sc[2 * qd + lb]);
        const uint4 v4 = *reinterpret_cast<const uint4*>(src + 16 * lb);
        const uint32_t w4[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const uint32_t byte = (w4[j >> 2] >> (8 * (j & 3))) & 0xffu;
            x[32 * lb + j] = (float)((int)(byte & 15u) - 8) * d16;
            x[32 * lb + j + 16] = (float)((int)(byte >> 4) - 8) * d16;
        }
    }
}

template <int D, int FMT>
__global__ void __launch_bounds__(256) extend_prep_kernel(const ExtendParams p) {
    constexpr int NA = D / 64, QD = D / 4;
    constexpr bool ISO = FMT == 2 || FMT == 3;
    constexpr bool KI8 = FMT == 0 || FMT == 1 || FMT == 5, VI8 = FMT == 0 || FMT == 6;
    constexpr bool KQ4 = FMT == 4, VQ4 = FMT == 1 || FMT == 4;
    constexpr bool KB16 = FMT == 6, VB16 = FMT == 5;
    __shared__ __align__(16) uint16_t vt[D][kXT + 8];
    const int b = blockIdx.z, kvh = blockIdx.y, t = blockIdx.x;
    const int cu0 = p.cu[b], T = max(0, p.cu[b + 1] - cu0);
    int L0 = p.prefix_lens[b];
    if (L0 < 0 || L0 > p.max_pages * kPage) L0 = max(0, min(L0, p.max_pages * kPage));   // flagged by the attention kernel
    const int NTP = (L0 + kXT - 1) / kXT, NTN = (T + kXT - 1) / kXT;
    if (t >= NTP + NTN) return;
    const int tid = threadIdx.x, i = tid >> 2, qd = tid & 3;
    const bool prefix = t < NTP;
    const size_t krow = ((size_t)b * p.Hkv + kvh) * p.Lmax + (size_t)kXT * t + i;
    uint32_t kw[QD / 2], vw[QD / 2], kl[KQ4 ? QD / 2 : 1];
    float ksv[NA];
    // q4 V (and K): the thread's 64 rotated values; zero for rows past the prefix, so that the
    // cross-thread butterflies below run on every lane of the warp
    float xr[VQ4 ? 64 : 1], xk[KQ4 ? 64 : 1];
#pragma unroll
    for (int e = 0; e < (VQ4 ? 64 : 1); ++e) xr[e] = 0.0f;
#pragma unroll
    for (int e = 0; e < (KQ4 ? 64 : 1); ++e) xk[e] = 0.0f;
#pragma unroll
    for (int k = 0; k < (KQ4 ? QD / 2 : 1); ++k) kl[k] = 0u;
#pragma unroll
    for (int g = 0; g < NA; ++g) ksv[g] = 0.0f;
#pragma unroll
    for (int k = 0; k < QD / 2; ++k) kw[k] = vw[k] = 0u;
    if (prefix) {
        const int pos = kXT * t + i;
        int page = -1;
        if (pos < L0) {
            page = p.page_table[(size_t)b * p.max_pages + (pos >> 4)];
            if (page < 0 || page >= p.num_pages) {
                atomicOr(&g_err_extend, kErrPage);
                page = -1;
            }
        }
        if (page >= 0) {
            const long long row = ((long long)page * p.Hkv + kvh) * kPage + (pos & 15);
            if constexpr (KB16) {
                // the unquantized bf16 K: fp16 (exact in fp16's normal range), key scale 1
                const uint4* ksrc = reinterpret_cast<const uint4*>(p.kc + row * 2 * D) + (QD * qd) / 8;
#pragma unroll
                for (int c = 0; c < QD / 8; ++c) {
                    const uint4 kx = ksrc[c];
                    kw[4 * c + 0] = bf16x2_to_h2(kx.x);
                    kw[4 * c + 1] = bf16x2_to_h2(kx.y);
                    kw[4 * c + 2] = bf16x2_to_h2(kx.z);
                    kw[4 * c + 3] = bf16x2_to_h2(kx.w);
                }
                if (qd == 0) {
#pragma unroll
                    for (int g = 0; g < NA; ++g) ksv[g] = p.scale_log2;
                }
            } else if constexpr (KQ4) {
                // q4 K: (q - 8) * d of the rotated row; rotated back and split into fp16 hi + lo
                // below, where every lane of the warp takes part
                q4_blocks2(p.kc + row * (D / 2), p.ks + row * (D / 16), qd, xk);
                if (qd == 0) {
#pragma unroll
                    for (int g = 0; g < NA; ++g) ksv[g] = p.scale_log2;
                }
            } else if constexpr (KI8) {
                // int8 K: exact codes, fp32 group scales
                const uint8_t* ksrc = p.kc + row * D + QD * qd;
#pragma unroll
                for (int c = 0; c < QD / 16; ++c) {
                    const uint4 kx = *reinterpret_cast<const uint4*>(ksrc + 16 * c);
                    const uint32_t ks4[4] = {kx.x, kx.y, kx.z, kx.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint32_t x = ks4[u] ^ 0x80808080u;   // 1152 + code, then the exact code
                        kw[8 * c + 2 * u] = hsub2_u32(prmt(x, 0x64646464u, 0x4140u), 0x64806480u);
                        kw[8 * c + 2 * u + 1] = hsub2_u32(prmt(x, 0x64646464u, 0x4342u), 0x64806480u);
                    }
                }
                if (qd == 0) {
#pragma unroll
                    for (int g = 0; g < NA; ++g)
                        ksv[g] = f16_bits_to_f32(reinterpret_cast<const uint16_t*>(p.ks + row * NA * 2)[g]) * p.scale_log2;
                }
            }
            if constexpr (VB16) {
                // the unquantized bf16 V: fp16 (exact in fp16's normal range)
                const uint4* vsrc = reinterpret_cast<const uint4*>(p.vc + row * 2 * D) + (QD * qd) / 8;
#pragma unroll
                for (int c = 0; c < QD / 8; ++c) {
                    const uint4 vx = vsrc[c];
                    vw[4 * c + 0] = bf16x2_to_h2(vx.x);
                    vw[4 * c + 1] = bf16x2_to_h2(vx.y);
                    vw[4 * c + 2] = bf16x2_to_h2(vx.z);
                    vw[4 * c + 3] = bf16x2_to_h2(vx.w);
                }
            } else if constexpr (VI8) {
                const uint8_t* vsrc = p.vc + row * D + QD * qd;
                const uint32_t vsb = reinterpret_cast<const uint16_t*>(p.vs + row * NA * 2)[(QD * qd) / 64];
                const uint32_t sv2 = vsb | (vsb << 16);
#pragma unroll
                for (int c = 0; c < QD / 16; ++c) {
                    const uint4 vx = *reinterpret_cast<const uint4*>(vsrc + 16 * c);
                    const uint32_t vs4[4] = {vx.x, vx.y, vx.z, vx.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint32_t y = vs4[u] ^ 0x80808080u;
                        const uint32_t c01 = hsub2_u32(prmt(y, 0x64646464u, 0x4140u), 0x64806480u);
                        const uint32_t c23 = hsub2_u32(prmt(y, 0x64646464u, 0x4342u), 0x64806480u);
                        vw[8 * c + 2 * u] = hfma2_u32(c01, sv2, 0u);       // fp16(code * scale), rounded once
                        vw[8 * c + 2 * u + 1] = hfma2_u32(c23, sv2, 0u);
                    }
                }
            } else if constexpr (VQ4) {
                // q4_0 V, blocks 2 qd and 2 qd + 1 of the rotated row (16 code bytes + one fp16 d each)
                static_assert(D == 256, "q4 V is FWHT-256 rotated");
                q4_blocks2(p.vc + row * (D / 2), p.vs + row * (D / 16), qd, xr);
                // rotated back after this branch, where every lane of the warp takes part
            } else {
                // ISO3 / ISO4: dims [QD qd, QD qd + QD) lie in block nb at offset j0
                constexpr int RB = FMT == 2 ? 48 : 64, SB = FMT == 2 ? 2 : 4;
                constexpr int TT = FMT == 3 ? 1 : 0;
                const int nb = (QD * qd) / 128, j0 = (QD * qd) % 128;
                const float qv[4] = {p.quat[0], p.quat[1], p.quat[2], p.quat[3]};
#pragma unroll
                for (int s2 = 0; s2 < 2; ++s2) {
                    const uint8_t* cb = (s2 ? p.vc : p.kc) + row * (RB * D / 128) + RB * nb;
                    const uint16_t* sc = reinterpret_cast<const uint16_t*>((s2 ? p.vs : p.ks) + row * (SB * D / 128));
                    const float nrm = f16_bits_to_f32(sc[nb * (SB / 2)]);
                    if (s2 == 0 && qd == 0) {
#pragma unroll
                        for (int g = 0; g < NA; ++g) ksv[g] = f16_bits_to_f32(sc[(g >> 1) * (SB / 2)]) * p.scale_log2;
                    }
#pragma unroll
                    for (int g4 = 0; g4 < QD / 4; ++g4) {
                        int code[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = j0 + 4 * g4 + e;
                            if constexpr (FMT == 3) {
                                code[e] = (cb[j >> 1] >> (4 * (j & 1))) & 15;
                            } else {
                                code[e] = ((cb[j >> 2] >> (2 * (j & 3))) & 3) | (((cb[32 + (j >> 3)] >> (j & 7)) & 1) << 2);
                            }
                        }
                        const float c0 = c_x_levels[TT][code[0]], c1 = c_x_levels[TT][code[1]];
                        const float c2 = c_x_levels[TT][code[2]], c3 = c_x_levels[TT][code[3]];
                        if (s2 == 0) {
                            // K': the levels themselves (exact in fp16); the attention kernel rotates
                            // the query instead
                            kw[2 * g4] = f32x2_to_h2(c0, c1);
                            kw[2 * g4 + 1] = f32x2_to_h2(c2, c3);
                        } else {
                            float u[4];
                            quat_conj_mul(qv, c0, c1, c2, c3, u);
                            vw[2 * g4] = f32x2_to_h2(nrm * u[0], nrm * u[1]);
                            vw[2 * g4 + 1] = f32x2_to_h2(nrm * u[2], nrm * u[3]);
                        }
                    }
                }
            }
        }
        if constexpr (VQ4) {
            // q4 V back to the original domain: the FWHT-256 (x 1/16) is its own inverse.
            // `prefix` is uniform over the block, so every lane of the warp reaches the shuffles;
            // rows past the prefix carry zeros and stay zero.
            fwht256_rows4(xr, qd);
#pragma unroll
            for (int k = 0; k < 32; ++k) vw[k] = f32x2_to_h2(xr[2 * k], xr[2 * k + 1]);
        }
        if constexpr (KQ4) {
            // q4 K back to the original domain, as fp16 hi + the fp16 remainder lo (two key planes:
            // one fp16 rounding of the rotated-back key would move scores by more than the bound)
            fwht256_rows4(xk, qd);
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                kw[k] = f32x2_to_h2(xk[2 * k], xk[2 * k + 1]);
                const float2 f = h2_to_f32x2(kw[k]);
                kl[k] = f32x2_to_h2(xk[2 * k] - f.x, xk[2 * k + 1] - f.y);
            }
        }
    } else {
        const int n = kXT * (t - NTP) + i;
        if (n < T) {
            const uint16_t* ksrc = p.k_new + ((size_t)(cu0 + n) * p.Hkv + kvh) * D + QD * qd;
            const uint16_t* vsrc = p.v_new + ((size_t)(cu0 + n) * p.Hkv + kvh) * D + QD * qd;
#pragma unroll
            for (int c = 0; c < QD / 8; ++c) {
                const uint4 kx = *reinterpret_cast<const uint4*>(ksrc + 8 * c);
                const uint4 vx = *reinterpret_cast<const uint4*>(vsrc + 8 * c);
                kw[4 * c + 0] = bf16x2_to_h2(kx.x);
                kw[4 * c + 1] = bf16x2_to_h2(kx.y);
                kw[4 * c + 2] = bf16x2_to_h2(kx.z);
                kw[4 * c + 3] = bf16x2_to_h2(kx.w);
                vw[4 * c + 0] = bf16x2_to_h2(vx.x);
                vw[4 * c + 1] = bf16x2_to_h2(vx.y);
                vw[4 * c + 2] = bf16x2_to_h2(vx.z);
                vw[4 * c + 3] = bf16x2_to_h2(vx.w);
            }
#pragma unroll
            for (int g = 0; g < NA; ++g) ksv[g] = p.scale_log2;   // the new tokens carry no K scale
        }
    }
    uint4* kdst = reinterpret_cast<uint4*>(p.xk + krow * D + QD * qd);
#pragma unroll
    for (int c = 0; c < QD / 8; ++c) kdst[c] = make_uint4(kw[4 * c], kw[4 * c + 1], kw[4 * c + 2], kw[4 * c + 3]);
    if constexpr (KQ4) {
        // the lo key plane (zero for the chunk's new tokens, which are exact in the hi plane)
        uint4* ldst = reinterpret_cast<uint4*>(p.xklo + krow * D + QD * qd);
#pragma unroll
        for (int c = 0; c < QD / 8; ++c) ldst[c] = make_uint4(kl[4 * c], kl[4 * c + 1], kl[4 * c + 2], kl[4 * c + 3]);
    }
    if (qd == 0) {
#pragma unroll
        for (int g = 0; g < NA; ++g) p.xs[krow * NA + g] = ksv[g];
    }
#pragma unroll
    for (int k = 0; k < QD / 2; ++k) {
        vt[QD * qd + 2 * k][i] = (uint16_t)(vw[k] & 0xffffu);
        vt[QD * qd + 2 * k + 1][i] = (uint16_t)(vw[k] >> 16);
    }
    __syncthreads();
    for (int d = tid; d < D; d += 256) {
        uint4* dst = reinterpret_cast<uint4*>(p.xv + (((size_t)b * p.Hkv + kvh) * D + d) * p.Lmax + (size_t)kXT * t);
        const uint4* src = reinterpret_cast<const uint4*>(&vt[d][0]);
#pragma unroll
        for (int c = 0; c < kXT / 8; ++c) dst[c] = src[c];
    }
}

// ISO: the prefix keys are the raw Lloyd-Max levels (exact fp16) with the block norm as
// key scale, and the prefix tiles take the query rotated per 4-D group (<q_h, conj(R) c>
// = <R q_h, c>), held as fp16 hi + lo so that Q K^T sees the fp32 rotated query; the
// bf16 new tokens take the plain query.
template <int D, int G, int XM>
__global__ void __launch_bounds__(kXThreads, 1)
    extend_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, const ExtendParams p) {
    using X = XGeo<D, XM>;
    constexpr bool ISO = XM == 1, KLO = XM == 2;
    static_assert(!KLO || D == 256, "two key planes: q4 keys, head_dim 256");
    constexpr int NA = X::NA;
    constexpr int TPT = 128 / G;   // tokens per tile
    extern __shared__ __align__(1024) uint8_t xsmem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(xsmem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5;
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
    int NTN = p.causal ? (tok_last + kXT) / kXT : (T + kXT - 1) / kXT;
    if (NTP + NTN > p.Lmax / kXT) {   // more new tokens than max_q_len promised
        if (tid == 0) atomicOr(&g_err_extend, kErrPos);
        NTN = max(0, p.Lmax / kXT - NTP);
    }
    const int NT = NTP + NTN;

    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + X::OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + X::OFF_TMEM);

    if (warp == kXMma) tmem_alloc(tmem_slot, X::TMEM_COLS);
    if (tid == 0) {
        mbar_init(&bars[B_Q], kXSoft);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[B_KF + i], 1);
            mbar_init(&bars[B_VF + i], 1);
            mbar_init(&bars[B_KE + i], kXSoft);
            mbar_init(&bars[B_VE + i], 1);
        }
        mbar_init(&bars[B_SFULL], 1);
        mbar_init(&bars[B_SFREE], kXSoft);
        mbar_init(&bars[B_PFULL], kXSoft);
        mbar_init(&bars[B_PVDONE], 1);
        mbar_init(&bars[B_RMX], kXSoft);
        mbar_init(&bars[B_RMX + 1], kXSoft);
        mbar_init(&bars[B_RSUM], kXSoft);
        mbar_init(&bars[B_DRAIN], 1);
        mbar_init(&bars[B_QPLAIN], kXSoft);
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

    if (warp == kXProd || warp == kXProd + 1) {
        // ================= producers: K' + key scales (warp kXProd), V^T (warp kXProd + 1) =================
        // A K slot is refilled as soon as Q K^T of its tile completes, well before PV of the
        // same tile, so the K stream runs about a tile further ahead than the V stream.
        if ((tid & 31) == 0) {
            const bool isk = warp == kXProd;
            const int hrow = b * p.Hkv + kvh;
            const int full0 = isk ? B_KF : B_VF, empty0 = isk ? B_KE : B_VE;
            int j = 0;
            for (; j < NT && ok; ++j) {
                const int buf = j % X::NB;
                if (j >= X::NB) wait(empty0 + buf, ((j - X::NB) / X::NB) & 1);
                uint64_t* bar = &bars[full0 + buf];
                const int krow0 = hrow * p.Lmax + kXT * j;
                if (isk) {
                    const bool lo = KLO && j < NTP;   // prefix tile with a lo key plane
                    mbar_arrive_expect_tx(bar, X::K_BYTES * (lo ? 2 : 1) + X::KS_BYTES);
#pragma unroll
                    for (int g = 0; g < NA; ++g)
                        tma_load_2d(sm + X::OFF_K + buf * X::K_BYTES + g * 8192, &tmK, bar, 64 * g, krow0);
                    if (lo) {
                        // the lo plane follows the hi plane in the workspace (rows + B Hkv Lmax)
                        const int lrow0 = krow0 + p.B * p.Hkv * p.Lmax;
#pragma unroll
                        for (int g = 0; g < NA; ++g) tma_load_2d(sm + X::OFF_QR + g * 8192, &tmK, bar, 64 * g, lrow0);
                    }
                    bulk_load(sm + X::OFF_KS + buf * X::KS_BYTES, p.xs + (size_t)krow0 * NA, X::KS_BYTES, bar);
                } else {
                    mbar_arrive_expect_tx(bar, X::V_BYTES);
                    tma_load_2d(sm + X::OFF_V + buf * X::V_BYTES, &tmV, bar, kXT * j, hrow * D);
                }
            }
            // every copy issued above has landed before the CTA exits
            for (int t = (j >= X::NB ? j - X::NB : 0); t < j; ++t) wait(full0 + t % X::NB, (t / X::NB) & 1);
        }
        __syncwarp();
    } else if (warp == kXMma) {
        // =========================== MMA issue ===========================
        if ((tid & 31) == 0) {
            const uint32_t qs = smem_addr(sm + X::OFF_Q);
            constexpr uint32_t IDQK = idesc_f16(128, 64), IDPV = idesc_f16(128, D);
            auto issue_qk = [&](int j) {
                const int buf = j % X::NB;
                wait(B_KF + buf, (j / X::NB) & 1);
                if (j >= 1) wait(B_SFREE, (j - 1) & 1);
                tc_fence_after();
                const uint32_t ks = smem_addr(sm + X::OFF_K + buf * X::K_BYTES);
                if (KLO && j < NTP) {
                    // prefix tile: the plain query against the hi and then the lo key plane
                    const uint32_t kl = smem_addr(sm + X::OFF_QR);
#pragma unroll
                    for (int g = 0; g < NA; ++g)
#pragma unroll
                        for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                            for (int u = 0; u < 4; ++u)
                                umma_f16(tmem_S + 64 * g, sw128_desc(qs + g * 16384 + 32 * u),
                                         sw128_desc((hl ? kl : ks) + g * 8192 + 32 * u), IDQK, (hl | u) > 0);
                } else if (ISO && j < NTP) {
                    // prefix tile: rotated query, hi (query region) then lo into the same accumulator
                    const uint32_t qr = smem_addr(sm + X::OFF_QR);
#pragma unroll
                    for (int g = 0; g < NA; ++g)
#pragma unroll
                        for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                            for (int u = 0; u < 4; ++u)
                                umma_f16(tmem_S + 64 * g, sw128_desc((hl ? qr : qs) + g * 16384 + 32 * u),
                                         sw128_desc(ks + g * 8192 + 32 * u), IDQK, (hl | u) > 0);
                } else {
                    // ISO: the first chunk tile needs the plain query back in the query region
                    if (ISO && j == NTP && NTP > 0) {
                        wait(B_QPLAIN, 0);
                        tc_fence_after();
                    }
#pragma unroll
                    for (int g = 0; g < NA; ++g)
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            umma_f16(tmem_S + 64 * g, sw128_desc(qs + g * 16384 + 32 * u),
                                     sw128_desc(ks + g * 8192 + 32 * u), IDQK, u > 0);
                }
                umma_commit(&bars[B_SFULL]);
            };
            wait(B_Q, 0);
            if (NT > 0) issue_qk(0);
            for (int j = 0; j < NT && ok; ++j) {
                if (j + 1 < NT) issue_qk(j + 1);
                wait(B_PFULL, j & 1);
                wait(B_VF + j % X::NB, (j / X::NB) & 1);
                tc_fence_after();
                const uint32_t ps = smem_addr(sm + X::OFF_P);
                const uint32_t vs = smem_addr(sm + X::OFF_V + (j % X::NB) * X::V_BYTES);
#pragma unroll
                for (int u = 0; u < kXT / 16; ++u)
                    umma_f16(tmem_O, sw128_desc(ps + 32 * u), sw128_desc(vs + 32 * u), IDPV, (j > 0 || u > 0));
                umma_commit(&bars[B_VE + j % X::NB]);
                umma_commit(&bars[B_PVDONE]);
            }
            // A wait that ran out ends the loop early, possibly with MMAs still in flight:
            // every MMA issued above completes before the CTA releases TMEM and exits.
            if (NT > 0) {
                umma_commit(&bars[B_DRAIN]);
                if (!mbar_wait_bounded(&bars[B_DRAIN], 0)) atomicOr(&g_err_extend, kErrWait);
            }
        }
        __syncwarp();
    } else {
        // =========================== softmax ===========================
        constexpr int KP = kXT / kXSplit;              // keys per thread and tile
        const int part = warp >> 2;                    // keys [KP part, KP part + KP) of every tile
        const int r = 32 * (warp & 3) + (tid & 31);    // TMEM lane and tile row
        const int tok = tok0 + r / G, hq = hq0 + r % G;
        const bool rvalid = tok < T;
        const int tokc = min(tok, T - 1);
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        float* red = reinterpret_cast<float*>(sm + X::OFF_RED);   // [2][128]
        // Q tile row r = (token r / G, head r % G), bf16 -> fp16; this thread: a part of the dims.
        // ISO with a prefix: the rotated query's fp16 hi part goes to the query region and its lo
        // part to the extra tile; the plain query replaces hi once the prefix tiles are done.
        const uint16_t* qrow = p.q + ((size_t)(cu0 + tokc) * p.Hq + hq) * D;
        auto write_query = [&](bool rotated) {
            uint8_t* qs = sm + X::OFF_Q;
#pragma unroll 4
            for (int c = part * (D / 8 / kXSplit); c < (part + 1) * (D / 8 / kXSplit); ++c) {
                uint4 o = make_uint4(0, 0, 0, 0);
                uint4 olo = o;
                if (rvalid) {
                    const uint4 w = *reinterpret_cast<const uint4*>(qrow + 8 * c);
                    o = make_uint4(bf16x2_to_h2(w.x), bf16x2_to_h2(w.y), bf16x2_to_h2(w.z), bf16x2_to_h2(w.w));
                    if (ISO && rotated) {
                        // R q_h per 4-D group (left Hamilton product by the pool quaternion) in fp32,
                        // then hi = fp16(v), lo = fp16(v - hi)
                        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
                        float v[8], y[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(e & 1 ? ww[e >> 1] & 0xffff0000u : ww[e >> 1] << 16);
                        const float q0 = p.quat[0], q1 = p.quat[1], q2 = p.quat[2], q3 = p.quat[3];
#pragma unroll
                        for (int g4 = 0; g4 < 2; ++g4) {
                            const float a = v[4 * g4], b = v[4 * g4 + 1], cc = v[4 * g4 + 2], d = v[4 * g4 + 3];
                            y[4 * g4] = q0 * a - q1 * b - q2 * cc - q3 * d;
                            y[4 * g4 + 1] = q0 * b + q1 * a + q2 * d - q3 * cc;
                            y[4 * g4 + 2] = q0 * cc - q1 * d + q2 * a + q3 * b;
                            y[4 * g4 + 3] = q0 * d + q1 * cc - q2 * b + q3 * a;
                        }
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            hi[k] = f32x2_to_h2(y[2 * k], y[2 * k + 1]);
                            const float2 f = h2_to_f32x2(hi[k]);
                            lo[k] = f32x2_to_h2(y[2 * k] - f.x, y[2 * k + 1] - f.y);
                        }
                        o = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        olo = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    }
                }
                *reinterpret_cast<uint4*>(qs + (c >> 3) * 16384 + sw_off(r, c & 7)) = o;
                if (ISO && rotated)
                    *reinterpret_cast<uint4*>(sm + X::OFF_QR + (c >> 3) * 16384 + sw_off(r, c & 7)) = olo;
            }
            fence_proxy_async();
        };
        write_query(ISO && NTP > 0);
        mbar_arrive(&bars[B_Q]);
        float m_used = -INFINITY, l = 0.0f;
        uint8_t* psm = sm + X::OFF_P;
        for (int j = 0; j < NT && ok; ++j) {
            const int kb = j % X::NB, buf = j & 1;   // K staging slot; row-exchange buffer
            const float* ksc = reinterpret_cast<const float*>(sm + X::OFF_KS + kb * X::KS_BYTES);   // [64][NA]
            wait(B_KF + kb, (j / X::NB) & 1);   // this tile's key scales
            wait(B_SFULL, j & 1);
            tc_fence_after();
            // ---- my KP keys: s = sum_g (K scale x softmax scale)_g * S_g, base 2 ----
            static_assert(KP == 16, "one TMEM load of 16 keys x 4 groups per thread and tile");
            float s[KP];
            {
                const int k0 = KP * part;
                uint32_t raw[64];
                const uint32_t a0 = tmem_S + lane_base + k0;
                if constexpr (NA == 4) tmem_ld16x4(a0, a0 + 64, a0 + 128, a0 + 192, raw);
                else tmem_ld16x4(a0, a0 + 64, a0, a0 + 64, raw);
                tc_fence_before();
                mbar_arrive(&bars[B_SFREE]);   // S(j) is in registers: QK(j + 1) may overwrite it
                if (ISO && j == NTP - 1) {
                    // Q K^T of the last prefix tile has completed: the plain query for the chunk tiles
                    write_query(false);
                    mbar_arrive(&bars[B_QPLAIN]);
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float acc;
                    if constexpr (NA == 4) {
                        const float4 w = reinterpret_cast<const float4*>(ksc)[k0 + e];
                        acc = w.x * __uint_as_float(raw[e]);
                        acc = fmaf(w.y, __uint_as_float(raw[16 + e]), acc);
                        acc = fmaf(w.z, __uint_as_float(raw[32 + e]), acc);
                        acc = fmaf(w.w, __uint_as_float(raw[48 + e]), acc);
                    } else {
                        const float2 w = reinterpret_cast<const float2*>(ksc)[k0 + e];
                        acc = fmaf(w.y, __uint_as_float(raw[16 + e]), w.x * __uint_as_float(raw[e]));
                    }
                    s[e] = acc;
                }
            }
            mbar_arrive(&bars[B_KE + kb]);   // the key scales are read: K(j + NB) may land
            // ---- masking (only tiles that reach past the prefix, the chunk or the causal edge) ----
            const int kbase = j < NTP ? kXT * j : kXT * (j - NTP);
            const int klim = j < NTP ? L0 : (p.causal ? min(T, tokc + 1) : T);   // keys < klim are visible
            if (kbase + KP * part + KP > klim) {
#pragma unroll
                for (int e = 0; e < KP; ++e)
                    if (kbase + KP * part + e >= klim) s[e] = -INFINITY;
            }
            float rmax = s[0];
#pragma unroll
            for (int e = 1; e < KP; ++e) rmax = fmaxf(rmax, s[e]);
            // ---- the row max over all parts (an mbarrier, so that every wait is bounded) ----
            red[(buf * kXSplit + part) * 128 + r] = rmax;
            mbar_arrive(&bars[B_RMX + buf]);
            wait(B_RMX + buf, (j >> 1) & 1);
#pragma unroll
            for (int q = 0; q < kXSplit; ++q) rmax = fmaxf(rmax, red[(buf * kXSplit + q) * 128 + r]);
            // PV(j - 1) must be done before P is overwritten and before O is rescaled
            if (j >= 1) wait(B_PVDONE, (j - 1) & 1);
            tc_fence_after();
            // frame update per row (both halves decide alike); the TMEM rescale of O is a
            // whole-warp operation, run warp-uniformly with factor 1 for rows that keep their frame
            const bool move = rmax > m_used + 8.0f;
            float alpha = 1.0f;
            if (move) {
                alpha = (m_used == -INFINITY) ? 0.0f : fast_exp2(m_used - rmax);
                l *= alpha;
                m_used = rmax;
            }
            if (j >= 1 && __any_sync(0xffffffffu, move)) {
#pragma unroll 1
                for (int c = part * (D / 16 / kXSplit); c < (part + 1) * (D / 16 / kXSplit); ++c) {
                    float v[16];
                    tmem_ld16(tmem_O + lane_base + 16 * c, v);
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] *= alpha;
                    tmem_st16(tmem_O + lane_base + 16 * c, v);
                }
            }
            const float mref = (m_used == -INFINITY) ? 0.0f : m_used;
#pragma unroll
            for (int c = 0; c < KP / 8; ++c) {
                uint32_t h[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float p0 = fast_exp2(s[8 * c + 2 * u] - mref), p1 = fast_exp2(s[8 * c + 2 * u + 1] - mref);
                    h[u] = f32x2_to_h2(p0, p1);
                    const float2 f = h2_to_f32x2(h[u]);
                    l += f.x + f.y;
                }
                *reinterpret_cast<uint4*>(psm + sw_off(r, (KP / 8) * part + c)) = make_uint4(h[0], h[1], h[2], h[3]);
            }
            fence_proxy_async();
            tc_fence_before();
            mbar_arrive(&bars[B_PFULL]);
        }
        if (NT > 0) wait(B_PVDONE, (NT - 1) & 1);
        tc_fence_after();
        // ---- row sum over all parts, then this thread's part of the O row ----
        const int eb = (NT & 1) * kXSplit;   // the exchange buffer the last tile did not use
        red[(eb + part) * 128 + r] = l;
        mbar_arrive(&bars[B_RSUM]);
        wait(B_RSUM, 0);
        float lt = 0.0f;
#pragma unroll
        for (int q = 0; q < kXSplit; ++q) lt += red[(eb + q) * 128 + r];
        const float inv = (lt > 0.0f) ? 1.0f / lt : 0.0f;
        const size_t obase = ((size_t)(cu0 + tokc) * p.Hq + hq) * D;
        constexpr int OC = D / 16 / kXSplit;   // 16-column chunks of O per thread (4 at D = 256, 2 at 128)
        {
            uint32_t raw[64];
            const uint32_t a0 = tmem_O + lane_base + 16 * OC * part;
            if constexpr (OC == 4) tmem_ld16x4(a0, a0 + 16, a0 + 32, a0 + 48, raw);
            else tmem_ld16x4(a0, a0 + 16, a0, a0 + 16, raw);
#pragma unroll
            for (int cc = 0; cc < OC; ++cc) {
                const int c = OC * part + cc;
                float v[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(raw[16 * cc + e]);
                if (rvalid) {
                    if (p.out_f32) {
                        float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + obase + 16 * c);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            o[e] = make_float4(v[4 * e] * inv, v[4 * e + 1] * inv, v[4 * e + 2] * inv, v[4 * e + 3] * inv);
                    } else {
                        uint32_t hb[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            __nv_bfloat162 bb = __floats2bfloat162_rn(v[2 * e] * inv, v[2 * e + 1] * inv);
                            hb[e] = *reinterpret_cast<uint32_t*>(&bb);
                        }
                        uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + obase + 16 * c);
                        o[0] = make_uint4(hb[0], hb[1], hb[2], hb[3]);
                        o[1] = make_uint4(hb[4], hb[5], hb[6], hb[7]);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kXMma) {
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

template <int D, int G, int XM>
static cudaError_t xlaunch(dim3 grid, const CUtensorMap& tk, const CUtensorMap& tv, const ExtendParams& p,
                           cudaStream_t st) {
    auto fn = extend_kernel<D, G, XM>;
    constexpr int smem = XGeo<D, XM>::SMEM + 1024;
    static bool configured[kMaxDevices];   // this instantiation's attribute, per device
    {
        cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(fn), smem, configured);
        if (e != cudaSuccess) return e;
    }
    fn<<<grid, kXThreads, smem, st>>>(tk, tv, p);
    return cudaGetLastError();
}

cudaError_t extend_upload_levels(const float* lv3, const float* lv4) {
    float lv[2][16] = {};
    for (int j = 0; j < 8; ++j) lv[0][j] = lv3[j];
    for (int j = 0; j < 16; ++j) lv[1][j] = lv4[j];
    return cudaMemcpyToSymbol(c_x_levels, lv, sizeof(lv));
}

// Every format (qkv_format) at D 128 or 256 (k8v4: 256); returns cudaErrorInvalidValue
// for shapes this kernel does not cover. Two launches: the prep kernel (one block per
// 64-key tile of every sequence and KV head) writes the workspace planes, the attention
// kernel reads them.
cudaError_t extend_launch(int fmt, int D, int G, int max_q_len, int NH, int B, const CUtensorMap& tk,
                          const CUtensorMap& tv, const ExtendParams& p, cudaStream_t st) {
    if (fmt < 0 || fmt > 6 || (D != 128 && D != 256) || ((fmt == 1 || fmt == 4) && D != 256) ||
        !(G == 1 || G == 2 || G == 4 || G == 8))
        return cudaErrorInvalidValue;
    const dim3 pgrid((unsigned)(p.Lmax / kXT), (unsigned)p.Hkv, (unsigned)B);
    switch (fmt * 1000 + D) {
        case 256: extend_prep_kernel<256, 0><<<pgrid, 256, 0, st>>>(p); break;
        case 128: extend_prep_kernel<128, 0><<<pgrid, 256, 0, st>>>(p); break;
        case 1256: extend_prep_kernel<256, 1><<<pgrid, 256, 0, st>>>(p); break;
        case 2128: extend_prep_kernel<128, 2><<<pgrid, 256, 0, st>>>(p); break;
        case 3128: extend_prep_kernel<128, 3><<<pgrid, 256, 0, st>>>(p); break;
        case 2256: extend_prep_kernel<256, 2><<<pgrid, 256, 0, st>>>(p); break;
        case 3256: extend_prep_kernel<256, 3><<<pgrid, 256, 0, st>>>(p); break;
        case 4256: extend_prep_kernel<256, 4><<<pgrid, 256, 0, st>>>(p); break;
        case 5128: extend_prep_kernel<128, 5><<<pgrid, 256, 0, st>>>(p); break;
        case 5256: extend_prep_kernel<256, 5><<<pgrid, 256, 0, st>>>(p); break;
        case 6128: extend_prep_kernel<128, 6><<<pgrid, 256, 0, st>>>(p); break;
        case 6256: extend_prep_kernel<256, 6><<<pgrid, 256, 0, st>>>(p); break;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int tpt = 128 / G;
    dim3 grid((unsigned)((max_q_len + tpt - 1) / tpt), (unsigned)NH, (unsigned)B);
    // prefix tile kind: ISO -> rotated query (1), q4 -> two key planes (2), else plain (0)
    const int xm = (fmt == 2 || fmt == 3) ? 1 : fmt == 4 ? 2 : 0;
#define QKV_XL(DD, XMM)                                                     \
    switch (G) {                                                           \
        case 1: return xlaunch<DD, 1, XMM>(grid, tk, tv, p, st);           \
        case 2: return xlaunch<DD, 2, XMM>(grid, tk, tv, p, st);           \
        case 4: return xlaunch<DD, 4, XMM>(grid, tk, tv, p, st);           \
        case 8: return xlaunch<DD, 8, XMM>(grid, tk, tv, p, st);           \
    }
    if (xm == 1 && D == 128) { QKV_XL(128, 1) }
    else if (xm == 1) { QKV_XL(256, 1) }
    else if (xm == 2) { QKV_XL(256, 2) }
    else if (D == 256) { QKV_XL(256, 0) }
    else { QKV_XL(128, 0) }
#undef QKV_XL
    return cudaErrorInvalidValue;
}

}  // namespace qkv
