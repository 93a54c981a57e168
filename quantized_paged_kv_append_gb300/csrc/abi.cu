// abi.cu -- the C ABI of libqkv.so: argument validation, per-device set-up,
// workspace sizing, TMA descriptor encoding and kernel dispatch by format.
// Declared in include/qkv.h.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/qkv.h"
#include "qkv_device.cuh"

#include "qkv_params.h"

using namespace qkv;

namespace {

thread_local int g_last_cuda = 0;

int cuda_fail(cudaError_t e) {
    g_last_cuda = (int)e;
    return QKV_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Lloyd-Max levels for N(0, 1/128), computed by this library's host code.
// Normalised levels z_j solve the Lloyd conditions for a standard normal:
// cell edges are midpoints, each level is its cell's conditional mean
// (pdf(a) - pdf(b)) / (cdf(b) - cdf(a)). Iterated from an even spacing on
// [-2.5, 2.5] until the largest move is below 1e-15; then scaled by
// 1/sqrt(128) and rounded to fp16 (round to nearest even).
// ---------------------------------------------------------------------------
double std_pdf(double z) { return std::isinf(z) ? 0.0 : 0.3989422804014327 * std::exp(-0.5 * z * z); }
double std_cdf_upper(double z) { return 0.5 * std::erfc(z * 0.7071067811865476); }  // P(Z > z)

void lloyd_levels(int n, double* z) {
    for (int j = 0; j < n; ++j) z[j] = -2.5 + 5.0 * j / (n - 1);
    for (int it = 0; it < 500000; ++it) {
        double nz[16], move = 0.0;
        for (int j = 0; j < n; ++j) {
            double a = j == 0 ? -INFINITY : 0.5 * (z[j - 1] + z[j]);
            double b = j == n - 1 ? INFINITY : 0.5 * (z[j] + z[j + 1]);
            double mass = std_cdf_upper(a) - std_cdf_upper(b);
            nz[j] = (std_pdf(a) - std_pdf(b)) / mass;
            move = std::max(move, std::fabs(nz[j] - z[j]));
        }
        for (int j = 0; j < n; ++j) z[j] = nz[j];
        if (move < 1e-15) break;
    }
}

// double -> binary16 bits, round to nearest even, from the IEEE-754 double encoding
uint16_t half_bits_rne(double v) {
    uint64_t u;
    std::memcpy(&u, &v, 8);
    uint16_t sign = (uint16_t)((u >> 48) & 0x8000);
    int e = (int)((u >> 52) & 0x7ff) - 1023;
    uint64_t mant = (u & ((1ull << 52) - 1)) | (1ull << 52);  // 53-bit significand (normal doubles only)
    if (((u >> 52) & 0x7ff) == 0) return sign;               // zero / double subnormal -> 0
    int shift;        // bits to drop from the 53-bit significand
    int hexp;         // biased half exponent of the result before rounding carry
    if (e >= -14) { shift = 42; hexp = e + 15; }
    else { shift = 42 + (-14 - e); hexp = 0; }
    if (shift > 63) return sign;
    uint64_t keep = mant >> shift, rem = mant & ((1ull << shift) - 1), halfway = 1ull << (shift - 1);
    if (rem > halfway || (rem == halfway && (keep & 1))) ++keep;
    uint32_t bits;
    if (hexp == 0) bits = (uint32_t)keep;                     // subnormal (keep may reach 0x400 = min normal)
    else {
        if (keep == (1ull << 11)) { keep >>= 1; ++hexp; }
        if (hexp >= 31) return (uint16_t)(sign | 0x7c00);
        bits = ((uint32_t)hexp << 10) | (uint32_t)(keep & 0x3ff);
    }
    return (uint16_t)(sign | bits);
}

float half_bits_to_float(uint16_t h) {
    int e = (h >> 10) & 0x1f, m = h & 0x3ff;
    float v = e == 0 ? std::ldexp((float)m, -24) : std::ldexp((float)(m | 0x400), e - 25);
    return (h & 0x8000) ? -v : v;
}

struct Levels { float l3[8]; float l4[16]; };

const Levels& levels() {
    static Levels L;
    static std::once_flag once;
    std::call_once(once, [] {
        const double sigma = 1.0 / std::sqrt(128.0);
        double z[16];
        lloyd_levels(8, z);
        for (int j = 0; j < 8; ++j) L.l3[j] = half_bits_to_float(half_bits_rne(sigma * z[j]));
        lloyd_levels(16, z);
        for (int j = 0; j < 16; ++j) L.l4[j] = half_bits_to_float(half_bits_rne(sigma * z[j]));
    });
    return L;
}

// ---------------------------------------------------------------------------
// per-device set-up (constant tables, SM count), done once per device with that
// device current
// ---------------------------------------------------------------------------
std::mutex g_dev_mu;
bool g_dev_ready[kMaxDevices];
int g_dev_sms[kMaxDevices];

std::mutex g_attr_mu;

int device_setup(int* dev_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return QKV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_dev_ready[dev]) {
        const Levels& L = levels();
        if ((e = append_upload_levels(L.l3, L.l4)) != cudaSuccess) return cuda_fail(e);
        if ((e = decode_tc_upload_levels(L.l3, L.l4)) != cudaSuccess) return cuda_fail(e);
        if ((e = extend_upload_levels(L.l3, L.l4)) != cudaSuccess) return cuda_fail(e);
        if ((e = gather_upload_levels(L.l3, L.l4)) != cudaSuccess) return cuda_fail(e);
        int sms = 0;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return cuda_fail(e);
        g_dev_sms[dev] = sms;
        g_dev_ready[dev] = true;
    }
    *dev_out = dev;
    return QKV_OK;
}

// ---------------------------------------------------------------------------
// TMA descriptors for the int8 / q4 code planes: 2-D [rows][row bytes] uint8,
// box 16 rows x 128 bytes, 128-byte swizzle.
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

int make_code_map(CUtensorMap* map, const void* base, long long rows, int row_bytes) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cuda_fail(cudaErrorNotSupported);
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {128u, 16u};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
    return QKV_OK;
}

// fp16 plane of `rows` rows x `inner` elements, boxes of 64 elements (128 B) x box_rows rows
int make_f16_map(CUtensorMap* map, const void* base, long long rows, long long inner, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cuda_fail(cudaErrorNotSupported);
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
    cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
    return QKV_OK;
}

// ---------------------------------------------------------------------------
// validation
// ---------------------------------------------------------------------------
bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int check_desc(const qkv_cache_desc* d) {
    if (!d) return QKV_ERR_ARG;
    if (d->format < QKV_INT8 || d->format > QKV_KBF16_V8) return QKV_ERR_FORMAT;
    if (d->page_size != kPage || d->num_pages <= 0 || d->num_kv_heads <= 0) return QKV_ERR_ARG;
    const int D = d->head_dim;
    switch (d->format) {
        case QKV_K8V4:
        case QKV_Q4: if (D != 256) return QKV_ERR_HEAD_DIM; break;
        default: if (D != 128 && D != 256) return QKV_ERR_HEAD_DIM; break;
    }
    // the unquantized (bf16) store has no scale plane: its scale pointer may be null
    const bool ks_none = d->format == QKV_KBF16_V8, vs_none = d->format == QKV_K8_VBF16;
    if (!d->k_codes || !d->v_codes || (!d->k_scales && !ks_none) || (!d->v_scales && !vs_none)) return QKV_ERR_ARG;
    if (!aligned16(d->k_codes) || !aligned16(d->k_scales) || !aligned16(d->v_codes) || !aligned16(d->v_scales))
        return QKV_ERR_ARG;
    return QKV_OK;
}

int enc_of(int fmt, int store) {
    switch (fmt) {
        case QKV_INT8: return ENC_INT8;
        case QKV_K8V4: return store == 0 ? ENC_INT8 : ENC_Q4;
        case QKV_ISO3: return ENC_ISO3;
        case QKV_ISO4: return ENC_ISO4;
        case QKV_Q4: return ENC_Q4;
        case QKV_K8_VBF16: return store == 0 ? ENC_INT8 : ENC_BF16;
        case QKV_KBF16_V8: return store == 0 ? ENC_BF16 : ENC_INT8;
    }
    return -1;
}

struct DecodeLayout {
    int G;          // query columns (virtual heads) of a head group
    int Gv;         // virtual query heads per KV head: window x (num_q_heads / num_kv_heads)
    int NH;         // head groups per sequence
    int S;          // segments
    int Cmax;       // CTA upper bound
    int slot_floats;
    size_t bytes;
};

// window: queries per sequence (1 for decode; a verify window attends as window x Gtot
// virtual heads per KV head, query w's heads after query w - 1's)
int decode_layout(const qkv_cache_desc* d, int batch, int num_q_heads, int window, int sms, DecodeLayout* L) {
    if (num_q_heads <= 0 || num_q_heads % d->num_kv_heads) return QKV_ERR_GQA;
    const int Gtot = num_q_heads / d->num_kv_heads;
    if (!(Gtot == 1 || Gtot == 2 || Gtot == 4 || Gtot % 8 == 0)) return QKV_ERR_GQA;
    if (window < 1) return QKV_ERR_ARG;
    L->Gv = window * Gtot;
    L->G = decode_heads_per_cta(L->Gv, d->format);
    L->NH = d->num_kv_heads * (L->Gv / L->G);
    L->S = batch * L->NH;
    L->Cmax = sms;
    L->slot_floats = 2 * (L->G > 8 ? 16 : 8) + L->G * d->head_dim;   // m, l, O of one piece
    // partial slots (m, l, O) of the pieces: piece (CTA c, segment s) uses slot c + s
    const size_t slots = (size_t)L->Cmax + L->S;
    auto al = [](size_t x) { return (x + 255) / 256 * 256; };
    L->bytes = al(slots * L->slot_floats * sizeof(float));
    return QKV_OK;
}

// Extend workspace: per (sequence, KV head) Lmax keys (the prefix padded to 64,
// then the chunk padded to 64) of fp16 K' rows, fp16 V^T rows and fp32 key scales.
struct ExtendLayout {
    long long Lmax;
    size_t off_v, off_s, bytes;
};

int extend_layout(const qkv_cache_desc* d, int batch, int max_q_len, int max_pages_per_seq, ExtendLayout* L) {
    if (batch < 0 || max_q_len < 0 || max_pages_per_seq <= 0) return QKV_ERR_ARG;
    auto r64 = [](long long x) { return (x + 63) / 64 * 64; };
    auto al = [](size_t x) { return (x + 255) / 256 * 256; };
    L->Lmax = r64((long long)max_pages_per_seq * kPage) + r64(max_q_len);
    if (L->Lmax > (1LL << 30)) return QKV_ERR_ARG;
    const size_t heads = (size_t)batch * d->num_kv_heads;
    const size_t plane = al(heads * (size_t)L->Lmax * d->head_dim * 2);
    // K' rows (hi plane; the q4 format adds the lo plane right after it), V^T rows, key scales
    const size_t kplanes = d->format == QKV_Q4 ? 2 : 1;
    L->off_v = kplanes * plane;
    L->off_s = L->off_v + plane;
    L->bytes = L->off_s + al(heads * (size_t)L->Lmax * (d->head_dim / 64) * 4);
    return QKV_OK;
}

}  // namespace

cudaError_t qkv::smem_attr_once(const void* fn, int bytes, bool (&done)[kMaxDevices]) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (!done[dev]) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        done[dev] = true;
    }
    return cudaSuccess;
}

extern "C" {

int qkv_row_bytes(int format, int store, int head_dim, int* code_bytes, int* scale_bytes) {
    if (format < QKV_INT8 || format > QKV_KBF16_V8) return QKV_ERR_FORMAT;
    if ((store != 0 && store != 1) || head_dim <= 0 || !code_bytes || !scale_bytes) return QKV_ERR_ARG;
    const int enc = enc_of(format, store);
    if (head_dim % group_size(enc) || (enc == ENC_Q4 && head_dim != 256)) return QKV_ERR_HEAD_DIM;
    *code_bytes = code_row_bytes(enc, head_dim);
    *scale_bytes = scale_row_bytes(enc, head_dim);
    return QKV_OK;
}

int qkv_iso_levels(int bits, float* out) {
    if (!out || (bits != 3 && bits != 4)) return QKV_ERR_ARG;
    const Levels& L = levels();
    if (bits == 3) { std::memcpy(out, L.l3, sizeof(L.l3)); return 8; }
    std::memcpy(out, L.l4, sizeof(L.l4));
    return 16;
}

int iso_kv_append(const qkv_cache_desc* cache, const void* k, const void* v, int n_tokens, const int32_t* seq_id,
                  const int32_t* pos, const int32_t* page_table, int num_seqs, int max_pages_per_seq, void* stream) {
    int rc = check_desc(cache);
    if (rc) return rc;
    if (n_tokens < 0) return QKV_ERR_ARG;
    if (n_tokens == 0) return QKV_OK;
    if (!k || !v || !seq_id || !pos || !page_table || num_seqs <= 0 || max_pages_per_seq <= 0) return QKV_ERR_ARG;
    if (!aligned16(k) || !aligned16(v)) return QKV_ERR_ARG;
    int dev;
    if ((rc = device_setup(&dev))) return rc;
    AppendParams p;
    p.codes[0] = (uint8_t*)cache->k_codes;
    p.codes[1] = (uint8_t*)cache->v_codes;
    p.scales[0] = (uint8_t*)cache->k_scales;
    p.scales[1] = (uint8_t*)cache->v_scales;
    p.src[0] = (const uint16_t*)k;
    p.src[1] = (const uint16_t*)v;
    p.seq_id = seq_id;
    p.pos = pos;
    p.page_table = page_table;
    p.n_tokens = n_tokens;
    p.Hkv = cache->num_kv_heads;
    p.num_pages = cache->num_pages;
    p.num_seqs = num_seqs;
    p.max_pages = max_pages_per_seq;
    for (int i = 0; i < 4; ++i) p.quat[i] = cache->quat[i];
    cudaError_t e = append_launch(cache->format, cache->head_dim, p, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e);
    return QKV_OK;
}

size_t kv_decode_workspace_size(const qkv_cache_desc* cache, int batch, int num_q_heads, int max_seq_len) {
    (void)max_seq_len;
    if (check_desc(cache) || batch < 0) return 0;
    int dev;
    if (device_setup(&dev)) return 0;
    DecodeLayout L;
    if (decode_layout(cache, batch, num_q_heads, 1, g_dev_sms[dev], &L)) return 0;
    return L.bytes;
}

// decode of `window` queries per sequence (1: kv_decode_attn; more: the fixed verify window)
static int decode_common(const qkv_cache_desc* cache, const void* q, const void* k_new, const void* v_new, int batch,
                         int window, int num_q_heads, const int32_t* page_table, int max_pages_per_seq,
                         const int32_t* seq_lens, int max_seq_len, float scale, void* out, int out_dtype,
                         void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_desc(cache);
    if (rc) return rc;
    if (batch < 0 || max_seq_len < 0) return QKV_ERR_ARG;
    if (batch == 0) return QKV_OK;
    if (batch > decode_max_batch()) return QKV_ERR_UNSUPPORTED;
    if (!q || !page_table || !seq_lens || !out || max_pages_per_seq <= 0) return QKV_ERR_ARG;
    if (out_dtype != QKV_OUT_BF16 && out_dtype != QKV_OUT_F32) return QKV_ERR_ARG;
    if (!aligned16(q) || !aligned16(out)) return QKV_ERR_ARG;
    if ((k_new == nullptr) != (v_new == nullptr)) return QKV_ERR_ARG;
    if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return QKV_ERR_ARG;
    if (!std::isfinite(scale)) return QKV_ERR_ARG;
    int dev;
    if ((rc = device_setup(&dev))) return rc;
    DecodeLayout L;
    if ((rc = decode_layout(cache, batch, num_q_heads, window, g_dev_sms[dev], &L))) return rc;
    if (!workspace || workspace_bytes < L.bytes || !aligned16(workspace)) return QKV_ERR_WORKSPACE;

    const int D = cache->head_dim;
    const long long rows = (long long)cache->num_pages * cache->num_kv_heads * kPage;
    CUtensorMap tk, tv;
    std::memset(&tk, 0, sizeof(tk));
    std::memset(&tv, 0, sizeof(tv));
    const int kenc = enc_of(cache->format, 0), venc = enc_of(cache->format, 1);
    // tensor maps for the planes staged by 128-byte TMA boxes (int8, q4 and bf16 rows; ISO rows go by bulk copies)
    auto tma_plane = [](int enc) { return enc == ENC_INT8 || enc == ENC_Q4 || enc == ENC_BF16; };
    if (tma_plane(kenc) && (rc = make_code_map(&tk, cache->k_codes, rows, code_row_bytes(kenc, D)))) return rc;
    if (tma_plane(venc) && (rc = make_code_map(&tv, cache->v_codes, rows, code_row_bytes(venc, D)))) return rc;

    // grid: at most one CTA per SM, and about 8 pages (one per warp) or more per CTA
    const long long max_pages_hint = ((long long)std::min(max_seq_len, max_pages_per_seq * kPage) + kPage - 1) / kPage;
    const long long units = (long long)L.S * std::max(1LL, max_pages_hint);
    const int grid = (int)std::max(1LL, std::min<long long>(L.Cmax, (units + 7) / 8));

    DecodeParams p;
    p.kc = (const uint8_t*)cache->k_codes;
    p.ks = (const uint8_t*)cache->k_scales;
    p.vc = (const uint8_t*)cache->v_codes;
    p.vs = (const uint8_t*)cache->v_scales;
    p.num_pages = cache->num_pages;
    p.Hkv = cache->num_kv_heads;
    p.q = (const uint16_t*)q;
    p.B = batch;
    p.Hq = num_q_heads;
    p.Gtot = num_q_heads / cache->num_kv_heads;
    p.W = window;
    p.Gv = L.Gv;
    p.NH = L.NH;
    p.page_table = page_table;
    p.max_pages = max_pages_per_seq;
    p.seq_lens = seq_lens;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.out = out;
    p.out_f32 = out_dtype == QKV_OUT_F32;
    for (int i = 0; i < 4; ++i) p.quat[i] = cache->quat[i];
    uint8_t* ws = (uint8_t*)workspace;
    p.part1 = (float*)ws;
    p.slot_floats = L.slot_floats;
    p.k_new = (const uint16_t*)k_new;
    p.v_new = (const uint16_t*)v_new;
    cudaError_t e = decode_tc_launch(D, L.G, grid, cache->format, tk, tv, p, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e);
    return QKV_OK;
}

int kv_decode_attn(const qkv_cache_desc* cache, const void* q, const void* k_new, const void* v_new, int batch,
                   int num_q_heads, const int32_t* page_table, int max_pages_per_seq, const int32_t* seq_lens,
                   int max_seq_len, float scale, void* out, int out_dtype, void* workspace, size_t workspace_bytes,
                   void* stream) {
    return decode_common(cache, q, k_new, v_new, batch, 1, num_q_heads, page_table, max_pages_per_seq, seq_lens,
                         max_seq_len, scale, out, out_dtype, workspace, workspace_bytes, stream);
}

size_t kv_extend_workspace_size(const qkv_cache_desc* cache, int batch, int max_q_len, int max_pages_per_seq) {
    if (check_desc(cache)) return 0;
    ExtendLayout L;
    if (extend_layout(cache, batch, max_q_len, max_pages_per_seq, &L)) return 0;
    return L.bytes;
}

int kv_extend_attn(const qkv_cache_desc* cache, const void* q, const void* k_new, const void* v_new, int num_q_heads,
                   const int32_t* cu_seqlens, const int32_t* prefix_lens, int batch, int max_q_len,
                   const int32_t* page_table, int max_pages_per_seq, float scale, int causal, void* out,
                   int out_dtype, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_desc(cache);
    if (rc) return rc;
    if (batch < 0 || max_q_len < 0) return QKV_ERR_ARG;
    if (batch == 0 || max_q_len == 0) return QKV_OK;
    if (!q || !k_new || !v_new || !cu_seqlens || !prefix_lens || !page_table || !out || max_pages_per_seq <= 0)
        return QKV_ERR_ARG;
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(out)) return QKV_ERR_ARG;
    if (out_dtype != QKV_OUT_BF16 && out_dtype != QKV_OUT_F32) return QKV_ERR_ARG;
    if (!std::isfinite(scale)) return QKV_ERR_ARG;
    if (num_q_heads <= 0 || num_q_heads % cache->num_kv_heads) return QKV_ERR_GQA;
    const int Gtot = num_q_heads / cache->num_kv_heads;
    if (!(Gtot == 1 || Gtot == 2 || Gtot == 4 || Gtot % 8 == 0)) return QKV_ERR_GQA;
    ExtendLayout XL;
    if ((rc = extend_layout(cache, batch, max_q_len, max_pages_per_seq, &XL))) return rc;
    if (!workspace || workspace_bytes < XL.bytes || ((uintptr_t)workspace & 255u)) return QKV_ERR_WORKSPACE;
    int dev;
    if ((rc = device_setup(&dev))) return rc;
    const int G = Gtot >= 8 ? 8 : Gtot;
    const int D = cache->head_dim;
    uint8_t* ws = (uint8_t*)workspace;
    const long long heads = (long long)batch * cache->num_kv_heads;
    CUtensorMap tk, tv;
    std::memset(&tk, 0, sizeof(tk));
    std::memset(&tv, 0, sizeof(tv));
    const long long kplanes = cache->format == QKV_Q4 ? 2 : 1;
    if ((rc = make_f16_map(&tk, ws, kplanes * heads * XL.Lmax, D, 64))) return rc;
    if ((rc = make_f16_map(&tv, ws + XL.off_v, heads * D, XL.Lmax, D))) return rc;
    ExtendParams p;
    p.kc = (const uint8_t*)cache->k_codes;
    p.ks = (const uint8_t*)cache->k_scales;
    p.vc = (const uint8_t*)cache->v_codes;
    p.vs = (const uint8_t*)cache->v_scales;
    p.num_pages = cache->num_pages;
    p.Hkv = cache->num_kv_heads;
    p.q = (const uint16_t*)q;
    p.k_new = (const uint16_t*)k_new;
    p.v_new = (const uint16_t*)v_new;
    p.Hq = num_q_heads;
    p.Gtot = Gtot;
    p.cu = cu_seqlens;
    p.prefix_lens = prefix_lens;
    p.B = batch;
    p.page_table = page_table;
    p.max_pages = max_pages_per_seq;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.causal = causal != 0;
    p.out = out;
    p.out_f32 = out_dtype == QKV_OUT_F32;
    p.Lmax = (int)XL.Lmax;
    p.xk = (uint16_t*)ws;
    p.xv = (uint16_t*)(ws + XL.off_v);
    p.xklo = (uint16_t*)ws + (size_t)heads * XL.Lmax * D;
    p.xs = (float*)(ws + XL.off_s);
    for (int i = 0; i < 4; ++i) p.quat[i] = cache->quat[i];
    const int NH = cache->num_kv_heads * (Gtot / G);
    cudaError_t e = extend_launch(cache->format, D, G, max_q_len, NH, batch, tk, tv, p, (cudaStream_t)stream);
    if (e == cudaErrorInvalidValue) return QKV_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return cuda_fail(e);
    return QKV_OK;
}

// verify workspace: the expanded page-table rows, the per-query lengths, then a decode
// workspace for total_q rows
static int verify_layout(const qkv_cache_desc* cache, int num_q_heads, int total_q, int max_pages_per_seq,
                         size_t* off_lens, size_t* off_dec, size_t* bytes) {
    int dev;
    int rc = device_setup(&dev);
    if (rc) return rc;
    DecodeLayout L;
    if ((rc = decode_layout(cache, total_q, num_q_heads, 1, g_dev_sms[dev], &L))) return rc;
    auto al = [](size_t x) { return (x + 255) / 256 * 256; };
    *off_lens = al((size_t)total_q * max_pages_per_seq * sizeof(int32_t));
    *off_dec = *off_lens + al((size_t)total_q * sizeof(int32_t));
    *bytes = *off_dec + L.bytes;
    return QKV_OK;
}

size_t kv_verify_workspace_size(const qkv_cache_desc* cache, int num_q_heads, int total_q, int max_pages_per_seq) {
    if (check_desc(cache) || total_q < 0 || max_pages_per_seq <= 0) return 0;
    size_t a, b, n;
    if (verify_layout(cache, num_q_heads, total_q, max_pages_per_seq, &a, &b, &n)) return 0;
    return n;
}

int kv_verify_attn(const qkv_cache_desc* cache, const void* q, int batch, int num_q_heads, const int32_t* cu_seqlens,
                   const int32_t* seq_lens, int total_q, const int32_t* page_table, int max_pages_per_seq,
                   int max_seq_len, float scale, void* out, int out_dtype, void* workspace, size_t workspace_bytes,
                   void* stream) {
    int rc = check_desc(cache);
    if (rc) return rc;
    if (batch < 0 || total_q < 0 || max_seq_len < 0) return QKV_ERR_ARG;
    if (batch == 0 || total_q == 0) return QKV_OK;
    if (total_q > decode_max_batch()) return QKV_ERR_UNSUPPORTED;
    if (!q || !cu_seqlens || !seq_lens || !page_table || !out || max_pages_per_seq <= 0) return QKV_ERR_ARG;
    if (num_q_heads <= 0 || num_q_heads % cache->num_kv_heads) return QKV_ERR_GQA;
    size_t off_lens, off_dec, need;
    if ((rc = verify_layout(cache, num_q_heads, total_q, max_pages_per_seq, &off_lens, &off_dec, &need))) return rc;
    if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255u)) return QKV_ERR_WORKSPACE;
    uint8_t* ws = (uint8_t*)workspace;
    VerifyParams vp;
    vp.cu = cu_seqlens;
    vp.W_fixed = 0;
    vp.seq_lens = seq_lens;
    vp.page_table = page_table;
    vp.B = batch;
    vp.max_pages = max_pages_per_seq;
    vp.table_rep = (int32_t*)ws;
    vp.lens_rep = (int32_t*)(ws + off_lens);
    cudaError_t e = verify_expand_launch(vp, total_q, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e);
    return kv_decode_attn(cache, q, nullptr, nullptr, total_q, num_q_heads, vp.table_rep, max_pages_per_seq,
                          vp.lens_rep, max_seq_len, scale, out, out_dtype, ws + off_dec, workspace_bytes - off_dec,
                          stream);
}

// The fixed window in one pass is the int8 decode kernel's verify instantiation; the other
// formats expand the window into one decode row per query (the kv_verify_attn path).
size_t kv_verify_fixed_workspace_size(const qkv_cache_desc* cache, int batch, int window, int num_q_heads,
                                      int max_pages_per_seq) {
    if (check_desc(cache) || batch < 0 || window < 1 || max_pages_per_seq <= 0) return 0;
    if ((long long)batch * window > decode_max_batch()) return 0;
    if (cache->format != QKV_INT8) return kv_verify_workspace_size(cache, num_q_heads, batch * window, max_pages_per_seq);
    int dev;
    if (device_setup(&dev)) return 0;
    DecodeLayout L;
    if (decode_layout(cache, batch, num_q_heads, window, g_dev_sms[dev], &L)) return 0;
    return L.bytes;
}

int kv_verify_attn_fixed(const qkv_cache_desc* cache, const void* q, int batch, int window, int num_q_heads,
                         const int32_t* seq_lens, const int32_t* page_table, int max_pages_per_seq, int max_seq_len,
                         float scale, void* out, int out_dtype, void* workspace, size_t workspace_bytes,
                         void* stream) {
    int rc = check_desc(cache);
    if (rc) return rc;
    if (window < 1 || batch < 0) return QKV_ERR_ARG;
    if ((long long)batch * window > decode_max_batch()) return QKV_ERR_UNSUPPORTED;
    if (cache->format == QKV_INT8)
        return decode_common(cache, q, nullptr, nullptr, batch, window, num_q_heads, page_table, max_pages_per_seq,
                             seq_lens, max_seq_len, scale, out, out_dtype, workspace, workspace_bytes, stream);
    if (batch == 0) return QKV_OK;
    if (!q || !seq_lens || !page_table || !out || max_pages_per_seq <= 0) return QKV_ERR_ARG;
    if (num_q_heads <= 0 || num_q_heads % cache->num_kv_heads) return QKV_ERR_GQA;
    const int total_q = batch * window;
    size_t off_lens, off_dec, need;
    if ((rc = verify_layout(cache, num_q_heads, total_q, max_pages_per_seq, &off_lens, &off_dec, &need))) return rc;
    if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255u)) return QKV_ERR_WORKSPACE;
    uint8_t* ws = (uint8_t*)workspace;
    VerifyParams vp;
    vp.cu = nullptr;
    vp.W_fixed = window;
    vp.seq_lens = seq_lens;
    vp.page_table = page_table;
    vp.B = batch;
    vp.max_pages = max_pages_per_seq;
    vp.table_rep = (int32_t*)ws;
    vp.lens_rep = (int32_t*)(ws + off_lens);
    cudaError_t e = verify_expand_launch(vp, total_q, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e);
    return kv_decode_attn(cache, q, nullptr, nullptr, total_q, num_q_heads, vp.table_rep, max_pages_per_seq,
                          vp.lens_rep, max_seq_len, scale, out, out_dtype, ws + off_dec, workspace_bytes - off_dec,
                          stream);
}

int kv_gather_dequant(const qkv_cache_desc* cache, const int32_t* page_row, int length, float* k_out, float* v_out,
                      void* stream) {
    int rc = check_desc(cache);
    if (rc) return rc;
    if (length < 0) return QKV_ERR_ARG;
    if (length == 0) return QKV_OK;
    if (!page_row || !k_out || !v_out || !aligned16(k_out) || !aligned16(v_out)) return QKV_ERR_ARG;
    int dev;
    if ((rc = device_setup(&dev))) return rc;
    GatherParams p;
    p.kc = (const uint8_t*)cache->k_codes;
    p.ks = (const uint8_t*)cache->k_scales;
    p.vc = (const uint8_t*)cache->v_codes;
    p.vs = (const uint8_t*)cache->v_scales;
    p.num_pages = cache->num_pages;
    p.Hkv = cache->num_kv_heads;
    p.page_row = page_row;
    p.length = length;
    p.k_out = k_out;
    p.v_out = v_out;
    for (int i = 0; i < 4; ++i) p.quat[i] = cache->quat[i];
    cudaError_t e = gather_launch(cache->format, cache->head_dim, p, (cudaStream_t)stream);
    if (e == cudaErrorInvalidValue) return QKV_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return cuda_fail(e);
    return QKV_OK;
}

const char* qkv_strerror(int code) {
    switch (code) {
        case QKV_OK: return "ok";
        case QKV_ERR_ARG: return "invalid argument (null pointer, negative size, misalignment or bad page size)";
        case QKV_ERR_HEAD_DIM: return "head_dim not supported for this format";
        case QKV_ERR_GQA: return "num_q_heads must be a supported multiple of num_kv_heads";
        case QKV_ERR_WORKSPACE: return "workspace missing or smaller than the required size";
        case QKV_ERR_FORMAT: return "unknown KV format";
        case QKV_ERR_CUDA: return "CUDA runtime error (see qkv_last_cuda_error)";
        case QKV_ERR_DEVICE: return "device-side range check fired";
        case QKV_ERR_UNSUPPORTED: return "request outside what this build implements";
    }
    return "unknown error code";
}

int qkv_last_cuda_error(void) { return g_last_cuda; }

int qkv_device_error(int clear) {
    unsigned a = 0;
    cudaError_t e = append_read_error(&a, clear != 0);
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned x = 0, t = 0;
    e = extend_read_error(&x, clear != 0);
    if (e != cudaSuccess) return cuda_fail(e);
    e = decode_tc_read_error(&t, clear != 0);
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned g = 0, v = 0;
    e = gather_read_error(&g, clear != 0);
    if (e != cudaSuccess) return cuda_fail(e);
    e = verify_read_error(&v, clear != 0);
    if (e != cudaSuccess) return cuda_fail(e);
    return (int)(a | x | t | g | v);
}

}  // extern "C"
