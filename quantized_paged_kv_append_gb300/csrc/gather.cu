// gather.cu -- the dequantized K and V of one sequence, read through its page
// table into dense fp32 rows: one warp per (token, KV head, store).
//
// Method (page title, section): "qwen35/q36: --kv - int8 K/V caches", "What it
// does" (the prompt-chunk path turns the int8 cache back into a dense buffer
// before a library GEMM); "feat(kvcache): add ISO3/ISO4 KV-cache quantization",
// "What" (the extend fast path unpacks ISO blocks into a scratch buffer);
// "--kv k8v4: hybrid KV cache", "How" (V is stored rotated; the rotation is its
// own inverse). Values come back in the original domain:
//   int8 : c * d16;
//   q4_0 : (q - 8) * d16 per 32-value block, then the FWHT-256 x 1/16 over the
//          row (butterflies at distances 1, 2, 4 inside a lane, 8 .. 128 by lane
//          shuffles that every lane of the warp executes);
//   ISO  : s16 * (conj(q) (x) c) per 4-D group of levels c;
//   bf16 : the unquantized store's values as they are.
#include "qkv_device.cuh"
#include "qkv_params.h"

namespace qkv {

__device__ unsigned int g_err_gather;
__constant__ float c_g_levels[2][16];   // [0] ISO3 (8 levels), [1] ISO4 (16 levels)

template <int ENC, int D>
__device__ __forceinline__ void dequant_row(const uint8_t* code, const uint8_t* scale, int lane, const float* qv,
                                            float (&x)[D / 32]) {
    constexpr int E = D / 32;   // values per lane: dims [E lane, E lane + E)
    const int d0 = E * lane;
    if constexpr (ENC == ENC_BF16) {
        (void)scale;
#pragma unroll
        for (int e = 0; e < E; ++e) x[e] = bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(code)[d0 + e]);
    } else if constexpr (ENC == ENC_INT8) {
        const float d16 = f16_bits_to_f32(reinterpret_cast<const uint16_t*>(scale)[d0 / 64]);
#pragma unroll
        for (int e = 0; e < E; ++e) x[e] = (float)(int8_t)code[d0 + e] * d16;
    } else if constexpr (ENC == ENC_Q4) {
        static_assert(D == 256, "q4 V rows are FWHT-256 rotated");
        const int b = d0 / 32, j0 = d0 % 32;   // block, first index inside it
        const float d16 = f16_bits_to_f32(reinterpret_cast<const uint16_t*>(scale)[b]);
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int j = j0 + e;
            const uint32_t byte = code[16 * b + (j & 15)];
            x[e] = (float)((int)((j < 16 ? byte : byte >> 4) & 15u) - 8) * d16;
        }
#pragma unroll
        for (int h = 1; h < E; h <<= 1) {
#pragma unroll
            for (int e = 0; e < E; ++e) {
                if (e & h) continue;
                const float a = x[e], c = x[e + h];
                x[e] = a + c;
                x[e + h] = a - c;
            }
        }
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const bool upper = (lane & m) != 0;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float o = __shfl_xor_sync(0xffffffffu, x[e], m);
                x[e] = upper ? o - x[e] : x[e] + o;
            }
        }
#pragma unroll
        for (int e = 0; e < E; ++e) x[e] *= 0.0625f;
    } else {
        constexpr int RB = ENC == ENC_ISO3 ? 48 : 64, SB = ENC == ENC_ISO3 ? 2 : 4;
        constexpr int TT = ENC == ENC_ISO4 ? 1 : 0;
        const int nb = d0 / 128, j0 = d0 % 128;
        const uint8_t* cb = code + RB * nb;
        const float nrm = f16_bits_to_f32(reinterpret_cast<const uint16_t*>(scale)[nb * (SB / 2)]);
        float c[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int j = j0 + e;
            int k;
            if constexpr (ENC == ENC_ISO4) k = (cb[j >> 1] >> (4 * (j & 1))) & 15;
            else k = ((cb[j >> 2] >> (2 * (j & 3))) & 3) | (((cb[32 + (j >> 3)] >> (j & 7)) & 1) << 2);
            c[e] = c_g_levels[TT][k];
        }
#pragma unroll
        for (int g = 0; g < E / 4; ++g) {
            const float a = c[4 * g], b = c[4 * g + 1], cc = c[4 * g + 2], d = c[4 * g + 3];
            x[4 * g] = nrm * (qv[0] * a + qv[1] * b + qv[2] * cc + qv[3] * d);
            x[4 * g + 1] = nrm * (qv[0] * b - qv[1] * a - qv[2] * d + qv[3] * cc);
            x[4 * g + 2] = nrm * (qv[0] * cc + qv[1] * d - qv[2] * a - qv[3] * b);
            x[4 * g + 3] = nrm * (qv[0] * d - qv[1] * cc + qv[2] * b - qv[3] * a);
        }
    }
}

template <int KENC, int VENC, int D>
__global__ void __launch_bounds__(256) gather_kernel(const GatherParams p) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const long long wid = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (wid >= (long long)p.length * p.Hkv * 2) return;   // whole warps
    const int store = (int)(wid & 1);
    const long long th = wid >> 1;
    const int head = (int)(th % p.Hkv);
    const int t = (int)(th / p.Hkv);
    float* dst = (store ? p.v_out : p.k_out) + ((long long)t * p.Hkv + head) * D + E * lane;
    const int page = p.page_row[t / kPage];
    float x[E];
    if (page < 0 || page >= p.num_pages) {
        if (lane == 0) atomicOr(&g_err_gather, kErrPage);
#pragma unroll
        for (int e = 0; e < E; ++e) x[e] = 0.0f;
    } else {
        const long long row = ((long long)page * p.Hkv + head) * kPage + (t % kPage);
        const float qv[4] = {p.quat[0], p.quat[1], p.quat[2], p.quat[3]};
        if (store == 0) {
            dequant_row<KENC, D>(p.kc + row * code_row_bytes(KENC, D), p.ks + row * scale_row_bytes(KENC, D), lane, qv, x);
        } else {
            dequant_row<VENC, D>(p.vc + row * code_row_bytes(VENC, D), p.vs + row * scale_row_bytes(VENC, D), lane, qv, x);
        }
    }
    // `page` is the same for the whole warp, so the shuffles above run on all lanes
#pragma unroll
    for (int e = 0; e < E; e += 4) *reinterpret_cast<float4*>(dst + e) = make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
cudaError_t gather_upload_levels(const float* lv3, const float* lv4) {
    float lv[2][16] = {};
    for (int j = 0; j < 8; ++j) lv[0][j] = lv3[j];
    for (int j = 0; j < 16; ++j) lv[1][j] = lv4[j];
    return cudaMemcpyToSymbol(c_g_levels, lv, sizeof(lv));
}

cudaError_t gather_read_error(unsigned* out, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_err_gather, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    unsigned z = 0;
    return cudaMemcpyToSymbol(g_err_gather, &z, sizeof(unsigned));
}

// fmt: 0 int8, 1 k8v4, 2 iso3, 3 iso4
cudaError_t gather_launch(int fmt, int D, const GatherParams& p, cudaStream_t st) {
    const long long warps = (long long)p.length * p.Hkv * 2;
    if (warps == 0) return cudaSuccess;
    dim3 grid((unsigned)((warps + 7) / 8)), block(256);
#define QKV_GATHER(KE, VE, DD) gather_kernel<KE, VE, DD><<<grid, block, 0, st>>>(p)
    if (fmt == 0 && D == 256) QKV_GATHER(ENC_INT8, ENC_INT8, 256);
    else if (fmt == 0 && D == 128) QKV_GATHER(ENC_INT8, ENC_INT8, 128);
    else if (fmt == 1 && D == 256) QKV_GATHER(ENC_INT8, ENC_Q4, 256);
    else if (fmt == 2 && D == 128) QKV_GATHER(ENC_ISO3, ENC_ISO3, 128);
    else if (fmt == 2 && D == 256) QKV_GATHER(ENC_ISO3, ENC_ISO3, 256);
    else if (fmt == 3 && D == 128) QKV_GATHER(ENC_ISO4, ENC_ISO4, 128);
    else if (fmt == 3 && D == 256) QKV_GATHER(ENC_ISO4, ENC_ISO4, 256);
    else if (fmt == 4 && D == 256) QKV_GATHER(ENC_Q4, ENC_Q4, 256);
    else if (fmt == 5 && D == 128) QKV_GATHER(ENC_INT8, ENC_BF16, 128);
    else if (fmt == 5 && D == 256) QKV_GATHER(ENC_INT8, ENC_BF16, 256);
    else if (fmt == 6 && D == 128) QKV_GATHER(ENC_BF16, ENC_INT8, 128);
    else if (fmt == 6 && D == 256) QKV_GATHER(ENC_BF16, ENC_INT8, 256);
    else return cudaErrorInvalidValue;
#undef QKV_GATHER
    return cudaGetLastError();
}

}  // namespace qkv
