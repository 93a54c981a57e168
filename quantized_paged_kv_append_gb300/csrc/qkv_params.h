// qkv_params.h -- kernel parameter blocks and the host-side entry points of the
// kernel translation units (append.cu, decode_tc.cu, extend.cu, gather.cu, verify.cu), shared with abi.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qkv {

struct AppendParams {
    uint8_t* codes[2];       // [store]: 0 = K, 1 = V
    uint8_t* scales[2];
    const uint16_t* src[2];  // bf16 [n][Hkv][D]
    const int32_t* seq_id;
    const int32_t* pos;
    const int32_t* page_table;
    int n_tokens, Hkv, num_pages, num_seqs, max_pages;
    float quat[4];
};

struct DecodeParams {
    const uint8_t* kc;
    const uint8_t* ks;
    const uint8_t* vc;
    const uint8_t* vs;
    int num_pages, Hkv;
    const uint16_t* q;   // bf16 [B * W][Hq][D]
    int B, Hq, Gtot;     // Gtot = Hq / Hkv
    int W;               // queries per sequence: 1 (decode) or a verify window; query w of sequence b
                         // is row b * W + w, at position seq_lens[b] - W + w
    int Gv;              // virtual query heads per KV head = W * Gtot (virtual head w * Gtot + h)
    int NH;              // head groups per sequence = Hkv * Gv / G
    const int32_t* page_table;
    int max_pages;
    const int32_t* seq_lens;
    float scale_log2;    // softmax scale * log2(e)
    void* out;
    int out_f32;
    float quat[4];
    float* part1;        // (C + S) partial slots: m[ML], l[ML], O[G][D] per piece (ML = 8, or 16 when G = 16)
    int slot_floats;     // 2 ML + G D
    int rec_by_seg;      // merge blocks indexed by segment (when segments <= CTAs), else by the closing CTA
    int ctas;            // CTAs of the decode grid (the split of the units follows from it and seq_lens)
    const uint16_t* k_new;   // optional bf16 [B][Hkv][D]: quantize-on-write of position seq_lens[b] - 1
    const uint16_t* v_new;
};

struct ExtendParams {
    const uint8_t* kc;
    const uint8_t* ks;
    const uint8_t* vc;
    const uint8_t* vs;
    int num_pages, Hkv;
    const uint16_t* q;       // bf16 [Tsum][Hq][D]
    const uint16_t* k_new;   // bf16 [Tsum][Hkv][D]
    const uint16_t* v_new;
    int Hq, Gtot;
    const int32_t* cu;           // [B + 1] new-token offsets
    const int32_t* prefix_lens;  // [B]
    int B;
    const int32_t* page_table;
    int max_pages;
    float scale_log2;
    int causal;
    void* out;
    int out_f32;
    int Lmax;            // keys per (sequence, KV head) in the workspace planes (multiple of 64)
    uint16_t* xk;        // workspace: fp16 K' [B * Hkv][Lmax][D]
    uint16_t* xklo;      // workspace (q4 format): the fp16 remainder of K', right after xk
    uint16_t* xv;        // workspace: fp16 V^T [B * Hkv][D][Lmax]
    float* xs;           // workspace: fp32 key scales x softmax scale [B * Hkv][Lmax][D / 64]
    float quat[4];       // ISO formats: the pool's unit quaternion (w, x, y, z)
};

struct GatherParams {
    const uint8_t* kc;
    const uint8_t* ks;
    const uint8_t* vc;
    const uint8_t* vs;
    int num_pages, Hkv;
    const int32_t* page_row;   // the sequence's page-table row: page of position t = page_row[t / 16]
    int length;                // positions [0, length)
    float* k_out;              // fp32 [length][Hkv][D]
    float* v_out;
    float quat[4];
};

struct VerifyParams {
    const int32_t* cu;          // [B + 1] query rows of each sequence's window, or null: W_fixed rows each
    int W_fixed;
    const int32_t* seq_lens;    // [B]
    const int32_t* page_table;  // [B][max_pages]
    int B, max_pages;
    int32_t* table_rep;         // workspace: [total_q][max_pages], row r = the page-table row of its sequence
    int32_t* lens_rep;          // workspace: [total_q], the query's own length
};

// Devices the library keeps per-device state for (device ordinals 0 .. kMaxDevices - 1).
constexpr int kMaxDevices = 64;

// Raises kernel `fn`'s dynamic shared-memory limit to `bytes` on the current
// device the first time it is asked there. The attribute belongs to the device's
// context, so `done` (one flag per device, owned by the caller: one array per
// kernel) records where it has been set; a process-wide mutex guards the flags.
cudaError_t smem_attr_once(const void* fn, int bytes, bool (&done)[kMaxDevices]);

cudaError_t append_upload_levels(const float* lv3, const float* lv4);
cudaError_t append_read_error(unsigned* out, bool clear);
cudaError_t append_launch(int fmt, int D, const AppendParams& p, cudaStream_t st);

// query heads per CTA of the decode kernel, and the largest batch of one decode call
int decode_heads_per_cta(int Gv, int fmt);   // Gv = virtual query heads per KV head
int decode_max_batch();
// decode on tcgen05 tensor cores (decode_tc.cu): every format, D 128 or 256, G in {1, 2, 4, 8}
cudaError_t decode_tc_launch(int D, int G, int grid, int fmt, const CUtensorMap& tk, const CUtensorMap& tv,
                             const DecodeParams& p, cudaStream_t st);
cudaError_t decode_tc_upload_levels(const float* lv3, const float* lv4);
cudaError_t decode_tc_read_error(unsigned* out, bool clear);

cudaError_t extend_read_error(unsigned* out, bool clear);
cudaError_t extend_upload_levels(const float* lv3, const float* lv4);

cudaError_t gather_upload_levels(const float* lv3, const float* lv4);
cudaError_t gather_read_error(unsigned* out, bool clear);
cudaError_t gather_launch(int fmt, int D, const GatherParams& p, cudaStream_t st);

cudaError_t verify_read_error(unsigned* out, bool clear);
cudaError_t verify_expand_launch(const VerifyParams& p, int total_q, cudaStream_t st);
cudaError_t extend_launch(int fmt, int D, int G, int max_q_len, int NH, int B, const CUtensorMap& tk,
                          const CUtensorMap& tv, const ExtendParams& p, cudaStream_t st);

}  // namespace qkv
