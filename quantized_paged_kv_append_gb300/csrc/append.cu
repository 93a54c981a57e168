// append.cu -- quantize-on-write of new K/V tokens into the paged pool: one
// warp per (token, KV head, store), the row quantizers of quant_rows.cuh.
#include "qkv_device.cuh"
#include "qkv_params.h"
#include "quant_rows.cuh"

namespace qkv {

__device__ unsigned int g_err_append;
__constant__ float c_app_levels[2][16];  // [0]: 8 ISO3 levels, [1]: 16 ISO4 levels
__constant__ float c_app_mids[2][16];    // midpoints of neighbouring levels

template <int KENC, int VENC, int D>
__global__ void __launch_bounds__(256) append_kernel(const AppendParams p) {
    const int lane = threadIdx.x & 31;
    const long long wid = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const long long total = (long long)p.n_tokens * p.Hkv * 2;
    if (wid >= total) return;
    const int store = (int)(wid & 1);
    const long long th = wid >> 1;
    const int head = (int)(th % p.Hkv);
    const int n = (int)(th / p.Hkv);
    const int sid = p.seq_id[n], ps = p.pos[n];
    if (sid < 0 || sid >= p.num_seqs || ps < 0 || ps >= p.max_pages * kPage) {
        if (lane == 0) atomicOr(&g_err_append, kErrPos);
        return;
    }
    const int page = p.page_table[(long long)sid * p.max_pages + ps / kPage];
    if (page < 0 || page >= p.num_pages) {
        if (lane == 0) atomicOr(&g_err_append, kErrPage);
        return;
    }
    const long long row = ((long long)page * p.Hkv + head) * kPage + (ps % kPage);
    const uint16_t* src = p.src[store] + ((long long)n * p.Hkv + head) * D;
    const int enc = store == 0 ? KENC : VENC;
    const float qv[4] = {p.quat[0], p.quat[1], p.quat[2], p.quat[3]};
    uint8_t* code = p.codes[store] + row * code_row_bytes(enc, D);
    uint8_t* scale = p.scales[store] + row * scale_row_bytes(enc, D);
    if (store == 0) {
        constexpr int T = KENC == ENC_ISO4 ? 1 : 0;
        quantize_row<KENC, D>(src, code, scale, lane, qv, c_app_levels[T], c_app_mids[T]);
    } else {
        constexpr int T = VENC == ENC_ISO4 ? 1 : 0;
        quantize_row<VENC, D>(src, code, scale, lane, qv, c_app_levels[T], c_app_mids[T]);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
cudaError_t append_upload_levels(const float* lv3, const float* lv4) {
    float lv[2][16] = {}, mid[2][16] = {};
    for (int j = 0; j < 8; ++j) lv[0][j] = lv3[j];
    for (int j = 0; j < 16; ++j) lv[1][j] = lv4[j];
    for (int j = 0; j < 7; ++j) mid[0][j] = (lv3[j] + lv3[j + 1]) * 0.5f;
    for (int j = 0; j < 15; ++j) mid[1][j] = (lv4[j] + lv4[j + 1]) * 0.5f;
    cudaError_t e = cudaMemcpyToSymbol(c_app_levels, lv, sizeof(lv));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(c_app_mids, mid, sizeof(mid));
}

cudaError_t append_read_error(unsigned* out, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_err_append, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    unsigned z = 0;
    return cudaMemcpyToSymbol(g_err_append, &z, sizeof(unsigned));
}

// fmt: 0 int8, 1 k8v4, 2 iso3, 3 iso4, 4 q4 (both stores), 5 int8 K + bf16 V, 6 bf16 K + int8 V
cudaError_t append_launch(int fmt, int D, const AppendParams& p, cudaStream_t st) {
    long long warps = (long long)p.n_tokens * p.Hkv * 2;
    if (warps == 0) return cudaSuccess;
    dim3 grid((unsigned)((warps + 7) / 8)), block(256);
#define QKV_APPEND(KE, VE, DD) append_kernel<KE, VE, DD><<<grid, block, 0, st>>>(p)
    if (fmt == 0 && D == 256) QKV_APPEND(ENC_INT8, ENC_INT8, 256);
    else if (fmt == 0 && D == 128) QKV_APPEND(ENC_INT8, ENC_INT8, 128);
    else if (fmt == 1 && D == 256) QKV_APPEND(ENC_INT8, ENC_Q4, 256);
    else if (fmt == 2 && D == 128) QKV_APPEND(ENC_ISO3, ENC_ISO3, 128);
    else if (fmt == 2 && D == 256) QKV_APPEND(ENC_ISO3, ENC_ISO3, 256);
    else if (fmt == 3 && D == 128) QKV_APPEND(ENC_ISO4, ENC_ISO4, 128);
    else if (fmt == 3 && D == 256) QKV_APPEND(ENC_ISO4, ENC_ISO4, 256);
    else if (fmt == 4 && D == 256) QKV_APPEND(ENC_Q4, ENC_Q4, 256);
    else if (fmt == 5 && D == 128) QKV_APPEND(ENC_INT8, ENC_BF16, 128);
    else if (fmt == 5 && D == 256) QKV_APPEND(ENC_INT8, ENC_BF16, 256);
    else if (fmt == 6 && D == 128) QKV_APPEND(ENC_BF16, ENC_INT8, 128);
    else if (fmt == 6 && D == 256) QKV_APPEND(ENC_BF16, ENC_INT8, 256);
    else return cudaErrorInvalidValue;
#undef QKV_APPEND
    return cudaGetLastError();
}

}  // namespace qkv
