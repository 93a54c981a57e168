/*
 * qkv.h -- C ABI of the GB300 quantized paged KV-cache library (libqkv.so).
 *
 * Three operations make up the path:
 *   iso_kv_append   quantize-on-write of new K/V tokens into a paged pool
 *   kv_decode_attn  paged split-K decode attention with on-the-fly dequant
 *                   and the partial-softmax merge
 *   kv_extend_attn  prefill-chunk attention over a packed prefix plus the
 *                   chunk's own bf16 K/V (packed afterwards by iso_kv_append)
 *
 * Sources (page title, section):
 *   [FT] "feat(kvcache): add ISO3/ISO4 KV-cache quantization (--kv-cache-iso)":
 *        "What" (ISO3/ISO4 blocks, quantize-on-write decode, deferred packing in
 *        extend), "Caveats" (bf16 KV input, head_dim % 128 == 0, validated at
 *        configuration time).
 *   [S8] "qwen35/q36: --kv - int8 K/V caches (codes + a FP16 scale per 64
 *        values)": "What it does" (int8 codes + one fp16 scale per 64 values,
 *        separate code and scale buffers, head_dim a multiple of 64, a format
 *        dispatcher, decode splits and on-the-fly dequant).
 *   [K4] "--kv k8v4: hybrid KV cache -- INT8 K + Hadamard-rotated Q4_0 V": "What",
 *        "How" (separate K/V pointers, V and the output Hadamard-rotated, q not),
 *        "Tests" (non-identity page table, ties-to-even int8 rules).
 *
 * Conventions common to every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller. The library
 *     allocates no memory and never synchronizes the stream. `stream` is a
 *     cudaStream_t (NULL = legacy default stream).
 *   - Arguments are validated on the host before any launch; an invalid call
 *     returns a negative QKV_ERR_* code and launches nothing. No C++ exception
 *     crosses this interface. Device-side range checks (page-table entries,
 *     positions) never trap: the offending token or page is skipped and a bit
 *     is set in a device error word read by qkv_device_error().
 *   - bf16 tensors are little-endian IEEE bfloat16; fp16 scales are IEEE
 *     binary16.
 *   - Page size is 16 tokens. A token at position `pos` of sequence `b` lives
 *     in physical page page_table[b * max_pages_per_seq + pos / 16], slot
 *     pos % 16. page_table is int32, row-major [batch][max_pages_per_seq].
 */
#ifndef QKV_H_
#define QKV_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QKV_API __attribute__((visibility("default")))
#else
#define QKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* KV formats [S8 "What it does", "Not in this PR"; K4 "What"; FT "What"]. */
typedef enum {
    QKV_INT8 = 0,     /* K and V: int8 codes + fp16 scale (group absmax/127) per 64 values     */
    QKV_K8V4 = 1,     /* K as QKV_INT8; V: FWHT-256 (x1/16) then q4_0 per 32 values; D = 256   */
    QKV_ISO3 = 2,     /* K and V: per 128 values, 3-bit Lloyd-Max codes (48 B) + fp16 norm    */
    QKV_ISO4 = 3,     /* K and V: per 128 values, 4-bit codes (64 B) + fp16 norm + 2 B reserved */
    QKV_Q4 = 4,       /* K and V as the V of QKV_K8V4 (FWHT-256 then q4_0; 576 B per cell at
                         2 KV heads); D = 256. The query is rotated in the kernels            */
    QKV_K8_VBF16 = 5, /* K as QKV_INT8; V unquantized: the bf16 input values, no scales       */
    QKV_KBF16_V8 = 6  /* K unquantized (bf16 input values, no scales); V as QKV_INT8          */
} qkv_format;

typedef enum { QKV_OUT_BF16 = 0, QKV_OUT_F32 = 1 } qkv_out_dtype;

enum {
    QKV_OK = 0,
    QKV_ERR_ARG = -1,        /* null pointer, negative size, bad page size, ...          */
    QKV_ERR_HEAD_DIM = -2,   /* head_dim not supported by the format                     */
    QKV_ERR_GQA = -3,        /* num_q_heads not a supported multiple of num_kv_heads     */
    QKV_ERR_WORKSPACE = -4,  /* workspace pointer null or smaller than *_workspace_size   */
    QKV_ERR_FORMAT = -5,     /* unknown format enum                                       */
    QKV_ERR_CUDA = -6,       /* a CUDA runtime call failed; see qkv_last_cuda_error()     */
    QKV_ERR_DEVICE = -7,     /* a device-side range check fired (qkv_device_error)        */
    QKV_ERR_UNSUPPORTED = -8 /* valid request outside what this build implements          */
};

/*
 * Pool descriptor. The four planes are caller-owned device buffers laid out
 * [num_pages][num_kv_heads][page_size][row bytes] with the row bytes of
 * qkv_row_bytes(). Plane contents per format (element order within a row):
 *   int8 codes : int8, one per value; scales: fp16 per 64 values.
 *   q4 codes   : per 32-value block 16 bytes, byte j = value j (low nibble) |
 *                value j+16 (high nibble); scales: signed fp16 d per block.
 *   iso3 codes : per 128-value block 48 bytes: bytes 0..31 hold the low two
 *                code bits (value i at byte i/4, bits 2*(i%4)); bytes 32..47
 *                the high bit (value i at byte 32 + i/8, bit i%8);
 *                scales: fp16 corrected norm per block.
 *   iso4 codes : per block 64 bytes, value i at byte i/2 (low nibble if i even);
 *                scales: per block fp16 corrected norm followed by a reserved
 *                fp16 written as 0 (68 B per block in total).
 *   bf16 codes : the unquantized store of QKV_K8_VBF16 / QKV_KBF16_V8: the bf16
 *                input values, two bytes each; that store has no scale plane
 *                (0 scale bytes per row; its scale pointer may be NULL).
 * `quat` is the fixed unit quaternion (w, x, y, z) of the ISO formats; it is
 * ignored by the other formats. Buffers must be 16-byte aligned.
 */
typedef struct {
    int32_t format;       /* qkv_format                                  */
    int32_t num_pages;    /* physical pages in the pool                  */
    int32_t page_size;    /* must be 16                                  */
    int32_t num_kv_heads;
    int32_t head_dim;     /* k8v4, q4: 256; the other formats: 128 or 256 */
    int32_t reserved0;
    void* k_codes;
    void* k_scales;
    void* v_codes;
    void* v_scales;
    float quat[4];
} qkv_cache_desc;

/* Bytes of codes and of scales in one row (one token, one KV head) of store
 * `store` (0 = K, 1 = V) for a format and head_dim. Host only. */
QKV_API int qkv_row_bytes(int format, int store, int head_dim, int* code_bytes, int* scale_bytes);

/* The fp16-rounded Lloyd-Max levels (ascending, as fp32) that this library
 * uses for ISO3 (bits = 3, 8 levels) or ISO4 (bits = 4, 16 levels), computed by
 * its own host code for N(0, 1/128). Returns the level count. Host only. */
QKV_API int qkv_iso_levels(int bits, float* levels);

/*
 * iso_kv_append -- quantize-on-write [FT "What"; S8 "What it does"].
 * k, v: bf16 [n_tokens][num_kv_heads][head_dim]. seq_id, pos: int32
 * [n_tokens]. Token n is quantized per the descriptor's format and written to
 * page_table[seq_id[n] * max_pages_per_seq + pos[n] / 16], slot pos[n] % 16,
 * for every KV head, K and V. page_table has num_seqs rows. A token whose
 * seq_id is outside [0, num_seqs), whose pos is outside
 * [0, 16 * max_pages_per_seq), or whose page entry is outside [0, num_pages)
 * is skipped and flags the device error word. n_tokens == 0 is a no-op.
 * The bytes written are a deterministic function of the bf16 inputs (fixed
 * fp32 operation order, IEEE division and square root, no contraction).
 */
QKV_API int iso_kv_append(const qkv_cache_desc* cache, const void* k, const void* v, int n_tokens,
                  const int32_t* seq_id, const int32_t* pos, const int32_t* page_table,
                  int num_seqs, int max_pages_per_seq, void* stream);

/*
 * kv_decode_attn -- decode attention, one query per sequence [S8 "What it
 * does"; K4 "How"], with optional quantize-on-write of the step's own token
 * [FT "What": decode is quantize-on-write].
 * q: bf16 [batch][num_q_heads][head_dim]; query head h reads KV head
 * h / (num_q_heads / num_kv_heads). Sequence b attends positions
 * [0, seq_lens[b]) (seq_lens: int32 device [batch]).
 * k_new, v_new: NULL, or bf16 [batch][num_kv_heads][head_dim]: before
 * attending, position seq_lens[b] - 1 of every sequence is quantized from them
 * and written to the pool (the same bytes iso_kv_append writes), and the
 * attention reads it back packed. With num_q_heads / num_kv_heads > 8 several
 * blocks write the same row with identical bytes. Without them the caller
 * appends the current token first.
 * max_seq_len: host-side upper bound on seq_lens used to size the schedule.
 * out: [batch][num_q_heads][head_dim] in bf16 or fp32. scale is the softmax
 * scale (usually 1/sqrt(head_dim)). An empty sequence gives a zero row.
 * workspace: device scratch of at least kv_decode_workspace_size() bytes (the
 * partial results of sequences split across thread blocks and the records of
 * their merge), 16-byte aligned; no initialization needed: every call writes
 * what it later reads. Calls sharing a workspace must not overlap in time.
 * batch <= 1024; num_q_heads / num_kv_heads in {1, 2, 4} or a multiple of 8.
 */
QKV_API size_t kv_decode_workspace_size(const qkv_cache_desc* cache, int batch, int num_q_heads, int max_seq_len);

QKV_API int kv_decode_attn(const qkv_cache_desc* cache, const void* q, const void* k_new, const void* v_new,
                           int batch, int num_q_heads, const int32_t* page_table, int max_pages_per_seq,
                           const int32_t* seq_lens, int max_seq_len, float scale, void* out, int out_dtype,
                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * kv_extend_attn -- extend (prefill-chunk) attention [FT "What": extend attends
 * the packed prefix plus the bf16 new tokens and packs them after attention;
 * S8 "What it does": prompt chunks dequantize the cache on the fly].
 * For sequence b the chunk's new tokens are rows [cu_seqlens[b],
 * cu_seqlens[b+1]) of q (bf16 [total][num_q_heads][head_dim]) and of k_new /
 * v_new (bf16 [total][num_kv_heads][head_dim]); its packed prefix is positions
 * [0, prefix_lens[b]) of the pool. New token i attends the dequantized prefix
 * and the raw bf16 new tokens 0..i (causal != 0) or all of them (causal == 0).
 * cu_seqlens (int32 [batch + 1]) and prefix_lens (int32 [batch]) are device
 * arrays; max_q_len is a host upper bound on the per-sequence new-token count.
 * out: [total][num_q_heads][head_dim], bf16 or fp32. The caller packs the new
 * tokens afterwards with iso_kv_append (deferred packing).
 * workspace: device scratch of at least kv_extend_workspace_size() bytes,
 * 256-byte aligned, no initialization needed (smaller or misaligned:
 * QKV_ERR_WORKSPACE). The call first dequantizes the prefix and the chunk's new
 * keys and values into it (fp16 planes, read by the attention kernel with TMA);
 * calls sharing a workspace must not overlap in time. A chunk longer than
 * max_q_len sets the position bit of qkv_device_error and is cut at max_q_len.
 * Formats: int8 (head_dim 128 or 256), k8v4 (256), ISO3 / ISO4 (128 or 256),
 * with num_q_heads / num_kv_heads in {1, 2, 4} or a multiple of 8. V is dequantized into the original domain first (k8v4
 * rotated back by the FWHT-256, ISO by the conjugate quaternion), so the output
 * needs no transform; ISO keys stay as their levels and the prefix tiles take
 * the query rotated by the pool quaternion.
 */
QKV_API size_t kv_extend_workspace_size(const qkv_cache_desc* cache, int batch, int max_q_len, int max_pages_per_seq);

QKV_API int kv_extend_attn(const qkv_cache_desc* cache, const void* q, const void* k_new, const void* v_new,
                           int num_q_heads, const int32_t* cu_seqlens, const int32_t* prefix_lens, int batch,
                           int max_q_len, const int32_t* page_table, int max_pages_per_seq, float scale, int causal,
                           void* out, int out_dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * kv_verify_attn -- the verify window of speculative decoding: several decode
 * queries per sequence [S8 "What it does": the verify windows go through the
 * decode kernels; K4 "Tests": batched forms with per-query step arrays].
 * Sequence b owns query rows [cu_seqlens[b], cu_seqlens[b+1]) of q (bf16
 * [total_q][num_q_heads][head_dim]); with W = cu_seqlens[b+1] - cu_seqlens[b],
 * its query j sits at position seq_lens[b] - W + j and attends positions
 * [0, seq_lens[b] - W + j + 1), all read from the pool (the window's tokens were
 * appended, and packed, before the call). cu_seqlens (int32 [batch + 1]) and
 * seq_lens (int32 [batch]) are device arrays; total_q = cu_seqlens[batch] is
 * given on the host too, total_q <= 1024. out: [total_q][num_q_heads][head_dim],
 * bf16 or fp32. Every format; num_q_heads / num_kv_heads as for decode.
 * workspace: at least kv_verify_workspace_size() bytes, 256-byte aligned, no
 * initialization needed. The call expands the window into one decode row per
 * query in the workspace (the sequence's page-table row and the query's own
 * length), then runs kv_decode_attn on those rows: each query reads its own
 * prefix. A window longer than its sequence sets the position bit of the device
 * error word; its queries that would sit before position 0 give zero rows.
 */
QKV_API size_t kv_verify_workspace_size(const qkv_cache_desc* cache, int num_q_heads, int total_q,
                                        int max_pages_per_seq);

QKV_API int kv_verify_attn(const qkv_cache_desc* cache, const void* q, int batch, int num_q_heads,
                           const int32_t* cu_seqlens, const int32_t* seq_lens, int total_q, const int32_t* page_table,
                           int max_pages_per_seq, int max_seq_len, float scale, void* out, int out_dtype,
                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * kv_verify_attn_fixed -- the verify window in one pass, for windows of the same
 * length W = window in every sequence (the MTP draft length of a step)
 * [S8 "What it does": verify windows; K4 "Tests": batched forms with per-query
 * step arrays]. q: bf16 [batch * window][num_q_heads][head_dim]; row
 * b * window + w is query w of sequence b, at position seq_lens[b] - window + w,
 * and attends positions [0, seq_lens[b] - window + w + 1), all from the pool.
 * out: [batch * window][num_q_heads][head_dim], bf16 or fp32;
 * batch * window <= 1024. For the int8 format the window's queries share each
 * K/V tile read: the window x (num_q_heads / num_kv_heads) queries of a KV head
 * attend as up to 16 columns of the same tile pass (with the V scales folded into
 * the fp16 V tile, one rounding), so a window of W costs about
 * ceil(W x (num_q_heads / num_kv_heads) / 16) decode passes rather than W. The
 * other formats expand the window into one decode row per query, as
 * kv_verify_attn does. workspace: at least kv_verify_fixed_workspace_size()
 * bytes, 256-byte aligned, no initialization needed. A sequence shorter than the
 * window sets the position bit of the device error word; its queries that would
 * sit before position 0 give zero rows. Errors as kv_decode_attn.
 */
QKV_API size_t kv_verify_fixed_workspace_size(const qkv_cache_desc* cache, int batch, int window, int num_q_heads,
                                              int max_pages_per_seq);

QKV_API int kv_verify_attn_fixed(const qkv_cache_desc* cache, const void* q, int batch, int window, int num_q_heads,
                                 const int32_t* seq_lens, const int32_t* page_table, int max_pages_per_seq,
                                 int max_seq_len, float scale, void* out, int out_dtype, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * kv_gather_dequant -- the dequantized K and V of one sequence as dense fp32
 * rows [S8 "What it does": the prompt-chunk path turns the int8 cache back into
 * a dense buffer before a library GEMM; FT "What": the extend fast path unpacks
 * ISO blocks into a scratch buffer; K4 "How": V is stored FWHT-rotated].
 * page_row: int32 device array, the sequence's page-table row: position t lives
 * in page page_row[t / 16], slot t % 16 (pass page_table + b * max_pages_per_seq).
 * k_out, v_out: fp32 device [length][num_kv_heads][head_dim], 16-byte aligned,
 * caller-owned. Values are in the original domain, computed in fp32: int8
 * c * d; k8v4 V (q - 8) * d per block, rotated back by the FWHT-256 (x 1/16);
 * ISO s * (conj(q) (x) c) per 4-D group of levels. A page entry outside
 * [0, num_pages) gives zero rows and sets bit 0 of the device error word.
 * length == 0 is a no-op. A debug / interoperability call, not on the
 * attention path.
 */
QKV_API int kv_gather_dequant(const qkv_cache_desc* cache, const int32_t* page_row, int length, float* k_out,
                              float* v_out, void* stream);

/*
 * kv_decode_attn_noalloc -- kv_decode_attn without a caller-provided workspace.
 * The reference pages have no counterpart to this entry point; it exists for
 * callers that cannot allocate device memory: code running while a stream is
 * captured into a CUDA graph (allocation is not allowed during capture), hosts
 * whose device memory is owned by another pool or framework, and loops that
 * must never allocate. The library allocates nothing here either: it uses a
 * fixed 8 MiB scratch array in static device memory, reserved on every GPU that
 * loads the library until the process exits.
 * Arguments and results are those of kv_decode_attn. A request whose workspace
 * (kv_decode_workspace_size) exceeds 8 MiB returns QKV_ERR_WORKSPACE and
 * launches nothing. Each call clears the scratch span it uses on `stream`
 * first. All calls on a device share the one array, so calls that can overlap
 * on the GPU (different streams, or threads without ordering) race and must
 * not be issued. The first call on each device resolves the array's device
 * address (cudaGetSymbolAddress); make that first call before any stream
 * capture.
 */
QKV_API int kv_decode_attn_noalloc(const qkv_cache_desc* cache, const void* q, const void* k_new, const void* v_new,
                                   int batch, int num_q_heads, const int32_t* page_table, int max_pages_per_seq,
                                   const int32_t* seq_lens, int max_seq_len, float scale, void* out, int out_dtype,
                                   void* stream);

/* Human-readable text for a QKV_* return code. */
QKV_API const char* qkv_strerror(int code);

/* The cudaError_t of the last failed CUDA call made by this library. */
QKV_API int qkv_last_cuda_error(void);

/* Reads (and if `clear`, resets) the device error word: bit 0 = page-table
 * entry out of range, bit 1 = bad position / sequence index, bit 2 = a bounded
 * wait gave up. Synchronizes the device. Returns the word, or a negative
 * QKV_ERR_CUDA. */
QKV_API int qkv_device_error(int clear);

#ifdef __cplusplus
}
#endif

#endif /* QKV_H_ */
