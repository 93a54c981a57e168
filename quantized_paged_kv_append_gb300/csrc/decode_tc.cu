// decode_tc.cu -- paged decode attention over a quantized KV cache (int8, k8v4,
// ISO3, ISO4, q4_0 for both stores, one-store int8 with the other store bf16) on
// tcgen05 tensor cores (TMEM accumulators), with the newest token's
// quantize-on-write fused in, and the verify window of speculative decoding.
//
// Method (page title, section): "qwen35/q36: --kv - int8 K/V caches", "What it
// does" (int8 K/V planes, one fp16 absmax/127 scale per 64 values, dequantized on
// the fly by the partial-attention decode kernels); "--kv k8v4: hybrid KV cache",
// "How" (q4_0 V in the FWHT-rotated domain, output rotated back); "feat(kvcache):
// add ISO3/ISO4 KV-cache quantization", "What" (ISO blocks; decode quantizes the
// new token into its page before attending). The partial results of a sequence
// split across CTAs are merged with the log-sum-exp rule (the pages name the
// partial kernels but do not print the rule; it is the standard one).
//
// GB300 design (one CTA of 15 warps per SM, persistent over an equal share of
// the (sequence, KV-head group, page) units -- stream-K):
//   * tile = 8 pages = 128 tokens of one (sequence, head group);
//   * warps 12 (K) and 14 (V) stage the int8 code planes of each tile with
//     2-D TMA (128-byte swizzle) and the scale rows with bulk copies, two tiles
//     deep, each on its own schedule; they also quantize the newest token into
//     the pool and the staged copy;
//   * warps 4-11 (converters) turn int8 codes into exact fp16: K as 1152 + c
//     straight into TMEM (the A operand of Q K^T, one token per TMEM lane), V
//     as c into an MN-major shared-memory tile (the B operand of P'^T V'); K of
//     tile T is converted before V of tile T - 1, so Q K^T runs a tile ahead
//     (the bf16 K of format 6 is copied in two k-step halves, each released by
//     its own commit);
//   * warp 13 (one thread) issues tcgen05.mma: S_g = K'_g Q_g^T per 64-dim
//     scale group g (M = 128 tokens, N = 16 query columns; 16 MMAs per tile at
//     D = 256) and O += P'^T V' (M = 64 P' columns: 16 per scale group = 8
//     heads hi + lo, N = D, K = 16 tokens; 8 MMAs per tile). An MMA costs at
//     least ~52 cycles of tensor pipe whatever its N (N <= 64) or M, so the
//     tile is laid out to need as few instructions as possible;
//   * warps 0-3 (softmax) own one token each: they combine the group scores in
//     fp32 with the exact K scales (removing the 1152 offset through the query
//     sums), run a lazy online softmax (the frame max moves only when a score
//     exceeds it by 2^8; all four warps agree on it once per tile), and write P'
//     = p * V-scale * 2^E as fp16 hi + lo parts;
//   * the other formats reuse the same roles: k8v4 converts its q4_0 V into
//     fp16((q - 8) * d) (the block scale folded into V', so P' carries none)
//     and rotates each piece's O back by the FWHT-256; ISO turns code pairs into
//     fp16 level pairs through a per-lane table, takes the query rotated by the
//     pool quaternion as fp16 hi + lo columns, and rotates O back per 4-D group;
//   * int8 with 16 query columns (16 heads per KV head, or a verify window's
//     queries as "virtual heads"): all N = 16 columns of the query tile are
//     heads, the V scales are folded into V' as for k8v4, and P' holds 16 heads
//     hi + lo; the verify window (VW) is a template flag with its own
//     instantiations (per-column causal lengths, query rows b W + w);
//   * pieces that do not cover a whole sequence write a partial slot (m, l, O) to
//     the caller's workspace; a second kernel (decode_tc_combine), launched with
//     programmatic stream serialization, merges them.
#include "qkv_device.cuh"
#include "qkv_params.h"
#include "quant_rows.cuh"
#include "tcgen05.cuh"

namespace qkv {

__device__ unsigned int g_err_dtc;
// Lloyd-Max levels and decision midpoints: [0] ISO3 (8 levels), [1] ISO4 (16 levels)
__constant__ float c_tc_levels[2][16];
__constant__ float c_tc_mids[2][16];

namespace {

constexpr int kTok = 128;                   // tokens per tile
constexpr int kTP = kTok / kPage;           // pages per tile
constexpr int kSoftW = 4, kConvW = 8;
constexpr int kWProd = kSoftW + kConvW;     // producer warp of the K planes
constexpr int kWMma = kWProd + 1;           // MMA warp
constexpr int kWProdV = kWMma + 1;          // producer warp of the V planes
constexpr int kThr = (kWProdV + 1) * 32;    // 480 threads

// Formats (the ABI's qkv_format): 0 int8 K and V; 1 k8v4 (int8 K, q4_0 codes of the
// FWHT-rotated V); 2 / 3 ISO3 / ISO4 (K and V: Lloyd-Max codes of the rotated unit
// vector per 128 values, one fp16 norm scale per block); 4 q4_0 for both stores (K
// rotated like V; the query is rotated by the same FWHT); 5 int8 K with the bf16 V
// unquantized; 6 the bf16 K unquantized with int8 V.
template <int D, int FMT>
struct TG {
    static constexpr bool ISO = FMT == 2 || FMT == 3;
    static constexpr bool KQ = FMT == 4;                 // K: q4_0 of the rotated row
    static constexpr bool VQ = FMT == 1 || FMT == 4;     // V: q4_0 of the rotated row (output rotated back)
    static constexpr bool KB = FMT == 6, VB = FMT == 5;  // the unquantized bf16 K / V
    static constexpr bool QHL = ISO || KQ;               // transformed query: fp16 hi (rows 0..7) + lo (8..15)
    static constexpr int ISO_RB = FMT == 2 ? 48 : 64;             // ISO code bytes per 128 values
    static constexpr int ISO_SB = FMT == 2 ? 2 : 4;               // ISO scale bytes per 128 values
    static constexpr int NA = D / 64;             // 64-dim atoms (Q tile, K' and V' tiles)
    static constexpr int NKG = ISO ? D / 128 : KQ ? D / 32 : D / 64;   // K scale groups = score accumulators
    static constexpr int KROW = ISO ? ISO_RB * D / 128 : KQ ? D / 2 : KB ? 2 * D : D;   // K code bytes of one row
    static constexpr int KSROW = ISO ? ISO_SB * D / 128 : KQ ? 2 * (D / 32) : KB ? 0 : 2 * NA;   // K scale bytes
    static constexpr int VROW = ISO ? KROW : VQ ? D / 2 : VB ? 2 * D : D;
    static constexpr int VSROW = ISO ? KSROW : VQ ? 2 * (D / 32) : VB ? 0 : 2 * NA;
    static constexpr int VG = ISO ? D / 128 : (VQ ? D / 32 : D / 64);   // V scale groups (q4, bf16: scale 1)
    static constexpr int PG = 4;                  // P' column groups of 16 (8 heads hi + lo)
    static constexpr int PM = 16 * PG;            // M of the PV MMA: 64
    static constexpr int PAGE_B = KROW * kPage;   // staged K codes of one page
    static constexpr int VPAGE_B = VROW * kPage;  // staged V codes of one page
    static constexpr int KBOX = KB ? 2 * D / 128 : KQ ? 1 : D / 128;   // 128-byte TMA boxes per K page (not ISO)
    static constexpr int VBOX = VPAGE_B / 2048;   // 128-byte TMA boxes per V page (not ISO)
    static constexpr int SC_B = kPage * KSROW;    // staged K scales of one page
    static constexpr int VSC_B = kPage * VSROW;   // staged V scales of one page
    static constexpr int KSTB = KB ? 1 : 2;       // K staging tiles (bf16 K: one, for shared-memory room)
    static constexpr int VSTB = VB ? 0 : 2;       // V staging tiles (bf16 V lands in V' itself)
    static constexpr int VPB = VB ? 2 : 1;        // V' tiles
    static constexpr int NSB = KQ ? 1 : 2;        // TMEM score buffers (q4 K: 8 accumulators, one buffer)
    static constexpr int QT = 1;                  // query tile (QHL: hi rows 0..7, lo rows 8..15)
    static constexpr int SACC = ISO ? 2 : 1;      // score accumulators per K scale group (ISO: even / odd k-steps)
    static constexpr int SBUF = NKG * SACC * 16;  // TMEM columns of one score buffer
    static constexpr int LUT_N = FMT == 2 ? 64 : FMT == 3 ? 256 : 0;   // code pair -> fp16 level pair
    static constexpr int KE_N = kConvW + (KB ? 0 : kSoftW);   // arrivals that free a K slot
    static constexpr int VE_N = VB ? 1 : kConvW + kSoftW;     // arrivals that free a V slot (bf16 V: the PV commit)
    static constexpr int OFF_KST = 0;                               // [KSTB][8][PAGE_B]
    static constexpr int OFF_VST = OFF_KST + KSTB * kTP * PAGE_B;   // [VSTB][8][VPAGE_B]
    static constexpr int OFF_VP = OFF_VST + VSTB * kTP * VPAGE_B;   // V' [VPB][NA][128 rows][128 B]
    static constexpr int OFF_PP = OFF_VP + VPB * NA * 16384;        // P' [PM / 64][128 rows][128 B]
    static constexpr int OFF_Q = OFF_PP + (PM / 64) * 16384;        // Q [QT][NA][16 rows][128 B]
    static constexpr int OFF_LUT = OFF_Q + QT * NA * 2048;          // per-lane level pairs [LUT_N][32]
    static constexpr int OFF_KSC = OFF_LUT + LUT_N * 32 * 4;        // [KSTB][8][SC_B]
    static constexpr int OFF_VSC = OFF_KSC + KSTB * kTP * SC_B;     // [2][8][VSC_B]
    static constexpr int OFF_BIAS = OFF_VSC + 2 * kTP * VSC_B;      // float [NA][8]
    static constexpr int OFF_RED = OFF_BIAS + 256;                  // softmax-warp reductions
    static constexpr int OFF_ROW = OFF_RED + 1024;                  // quantize-on-write rows [2][512]
    static constexpr int OFF_BAR = OFF_ROW + 1024;
    static constexpr int OFF_MISC = OFF_BAR + 32 * 8;
    static constexpr int SMEM = OFF_MISC + 64;
    static constexpr int KCOL = 0;                     // K' columns: D / 2 (16-bit pairs)
    static constexpr int SCOL = D / 2;                 // NSB score buffers of SBUF columns
    static constexpr int OCOL = SCOL + NSB * SBUF;     // O (M = 64 rows in lanes 32 (r / 16) + r % 16, N = D)
    static constexpr int TCOLS = (OCOL + D) <= 256 ? 256 : 512;
    static_assert(OCOL + D <= 512, "TMEM budget");
    static_assert(SMEM + 1024 <= 232448 - 1024, "shared memory budget");
    static_assert(2 * kTP * SC_B <= 4096 && 2 * kTP * VSC_B <= 4096, "scale staging");
    static_assert(!VQ || D == 256, "q4 V is FWHT-256 rotated");
    static_assert(!KQ || D == 256, "q4 K is FWHT-256 rotated");
    static_assert(OFF_VP % 1024 == 0 && OFF_PP % 1024 == 0 && OFF_Q % 1024 == 0, "UMMA operand alignment");
    static_assert(PAGE_B % 16 == 0 && VPAGE_B % 16 == 0 && SC_B % 16 == 0 && VSC_B % 16 == 0, "bulk copies");
    static_assert(KROW * kPage <= 2048 * 4 && VROW * kPage <= 2048 * 4, "TMA boxes per page");
};

enum {
    B_KF = 0,    // [2] K codes + K scales of a tile landed (2 arrivals + tx)
    B_KE = 2,    // [2] K slot free (8 converter warps + 4 softmax warps)
    B_VF = 4,    // [2]
    B_VE = 6,    // [2]
    B_KCV = 8,   // K' written to TMEM (8 converter warps; bf16 K: the 4 warps of k-step half 0)
    B_VCV = 9,   // V' written (8 converter warps)
    B_QKD = 10,  // [2] QK^T of a tile complete (commit)
    B_PVD = 12,  // [2] PV of a tile complete (commit)
    B_SF = 16,   // [2] score buffer read (4 softmax warps)
    B_PFL = 18,  // P' written (4 softmax warps)
    B_QRD = 19,  // query tile of a piece written (1)
    B_PAT = 20,  // [kind] producer: the newest token's page landed (1 + tx)
    B_DRN = 22,  // every MMA of the CTA complete (commit), before TMEM is released
    B_KCV1 = 23, // bf16 K: K' of k-step half 1 written (its 4 converter warps)
    B_QKH = 24,  // [2] bf16 K: the Q K^T MMAs of k-step half 0 of a tile complete (commit)
    B_N = 26
};
static_assert(B_N <= 32, "barrier area holds 32 barriers");

__device__ __forceinline__ void soft_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ float exp2i(int n) { return __int_as_float((n + 127) << 23); }
// position inside an aligned group of 4 <-> dimension: the converters emit (d0, d2), (d1, d3)
__device__ __forceinline__ int perm4(int e) { return (e & ~3) | ((e & 1) << 1) | ((e >> 1) & 1); }

// Warp-wide max (MAX) or sum of each of 8 per-lane values with 9 shuffles instead of
// 40: every step halves the values a lane carries. On return, lane l holds the result
// for value (l >> 2) & 7 (all four lanes of a quad hold the same one).
template <bool MAX>
__device__ __forceinline__ float warp_reduce8(const float (&v)[8], int lane) {
    auto op = [](float a, float b) { return MAX ? fmaxf(a, b) : a + b; };
    float a[4], b2[2];
    const bool u4 = (lane & 16) != 0, u3 = (lane & 8) != 0, u2 = (lane & 4) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float r = __shfl_xor_sync(0xffffffffu, u4 ? v[i] : v[i + 4], 16);
        a[i] = op(u4 ? v[i + 4] : v[i], r);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const float r = __shfl_xor_sync(0xffffffffu, u3 ? a[j] : a[j + 2], 8);
        b2[j] = op(u3 ? a[j + 2] : a[j], r);
    }
    float c1 = op(u2 ? b2[1] : b2[0], __shfl_xor_sync(0xffffffffu, u2 ? b2[0] : b2[1], 4));
    c1 = op(c1, __shfl_xor_sync(0xffffffffu, c1, 2));
    return op(c1, __shfl_xor_sync(0xffffffffu, c1, 1));
}

__device__ __forceinline__ int seq_len_clamped(const DecodeParams& p, int b) {
    return max(0, min(p.seq_lens[b], p.max_pages * kPage));
}
// The same from an L2-only load (ld.global.cg: nothing is kept in L1), for the
// speculative read before the dependency wait.
__device__ __forceinline__ int seq_len_clamped_cg(const DecodeParams& p, int b) {
    return max(0, min(__ldcg(p.seq_lens + b), p.max_pages * kPage));
}
__device__ __forceinline__ void prefetch_l1(const void* a) { asm volatile("prefetch.global.L1 [%0];" ::"l"(a)); }
// bytes (a multiple of 16) at a 16-byte aligned global address into L2; no data is returned
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

struct Piece {
    int b, hg, p0, p1, L;
    long long soff, np;
};

// The CTA's pieces, in order: contiguous page ranges of one (sequence, head group).
struct Walker {
    int b;
    long long pref, x, end;
    template <bool CG = false>
    __device__ bool next(const DecodeParams& p, Piece& pc) {
        while (x < end && b < p.B) {
            const int L = CG ? seq_len_clamped_cg(p, b) : seq_len_clamped(p, b);
            const long long np = (L + kPage - 1) / kPage;
            const long long seg0 = pref * p.NH;
            if (np == 0 || x >= seg0 + np * p.NH) {
                pref += np;
                ++b;
                continue;
            }
            const int hg = (int)((x - seg0) / np);
            const long long soff = seg0 + (long long)hg * np;
            const long long xe = min(end, soff + np);
            pc.b = b;
            pc.hg = hg;
            pc.p0 = (int)(x - soff);
            pc.p1 = (int)(xe - soff);
            pc.L = L;
            pc.soff = soff;
            pc.np = np;
            x = xe;
            return true;
        }
        return false;
    }
};

// Bounded wait on an mbarrier phase. A wait that runs out sets the device error
// bit and the CTA-wide abort flag; every later wait of the CTA then returns at
// once, so a broken launch ends after one time-out instead of one per wait
// (its results are garbage and the error word says so).
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    for (uint32_t i = 0; i < (1u << 20); ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63) == 63 && *abort_flag) return false;
    }
    atomicOr(&g_err_dtc, kErrWait);
    *abort_flag = 1;
    return false;
}

// Virtual head gv of KV head kvh (gv = w * Gtot + h): query row b * W + w, query head kvh * Gtot + h.
// VW: the kernel runs a verify window (W > 1); otherwise W = 1 and gv is the head's index in
// its KV group.
template <bool VW>
__device__ __forceinline__ size_t qrow_index(const DecodeParams& p, int b, int kvh, int gv) {
    if constexpr (!VW) return (size_t)b * p.Hq + (size_t)kvh * p.Gtot + gv;
    const int w = gv / p.Gtot, h = gv - w * p.Gtot;
    return ((size_t)b * p.W + w) * p.Hq + (size_t)kvh * p.Gtot + h;
}
// element d of the output row whose first element is at orow (= qrow_index(...) * D)
__device__ __forceinline__ void write_row(const DecodeParams& p, size_t orow, int d, float v) {
    const size_t o = orow + d;
    if (p.out_f32) reinterpret_cast<float*>(p.out)[o] = v;
    else reinterpret_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(v);
}
// element i of the head group's output (i = column * D + dim; column = virtual head gv0 + i / D)
template <int D, int G, bool VW>
__device__ void write_out(const DecodeParams& p, int b, int kvh, int gv0, int i, float v) {
    const size_t o = qrow_index<VW>(p, b, kvh, gv0 + i / D) * D + (i % D);
    if (p.out_f32) reinterpret_cast<float*>(p.out)[o] = v;
    else reinterpret_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(v);
}

}  // namespace

template <int D, int G, int FMT, bool VW>
__global__ void __launch_bounds__(kThr, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const DecodeParams p) {
    using X = TG<D, FMT>;
    constexpr int NA = X::NA;
    constexpr bool VQ = X::VQ;
    constexpr bool kSplitK = X::KB;   // Q K^T issued in two k-step halves (bf16 K)
    // 16 query columns (int8): the V scales are folded into V' (fp16(c d), one rounding) so that
    // P' holds 16 heads hi + lo in each 16-row slot pair; QH = per-head arrays of the softmax
    constexpr bool VFOLD = G > 8;
    constexpr int QH = G > 8 ? 16 : 8;
    static_assert(G <= 8 || (FMT == 0 && G == 16), "16 query columns: the int8 format only");
    static_assert(!VW || FMT == 0, "the one-pass verify window: the int8 format only");
    extern __shared__ __align__(1024) uint8_t dsm_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int C = gridDim.x, c = blockIdx.x;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + X::OFF_BAR);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + X::OFF_MISC);
    volatile int* s_abort = reinterpret_cast<volatile int*>(sm + X::OFF_MISC + 32);
    auto wait_or_flag = [&](uint64_t* bar, uint32_t parity) { return wait_or_abort(bar, parity, s_abort); };

    // ---------------- set-up: barriers, TMEM, this CTA's share of the units ----------------
    if (tid == 0) {
        mbar_init(&bars[B_KF], 2);
        mbar_init(&bars[B_KF + 1], 2);
        mbar_init(&bars[B_VF], 2);
        mbar_init(&bars[B_VF + 1], 2);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[B_KE + i], X::KE_N);
            mbar_init(&bars[B_VE + i], X::VE_N);
            mbar_init(&bars[B_QKD + i], 1);
            mbar_init(&bars[B_QKH + i], 1);
            mbar_init(&bars[B_PVD + i], 1);
            mbar_init(&bars[B_SF + i], kSoftW);
        }
        mbar_init(&bars[B_KCV], kSplitK ? kConvW / 2 : kConvW);
        mbar_init(&bars[B_KCV1], kConvW / 2);
        mbar_init(&bars[B_VCV], kConvW);
        mbar_init(&bars[B_PFL], kSoftW);
        mbar_init(&bars[B_QRD], 1);
        mbar_init(&bars[B_PAT], 1);
        mbar_init(&bars[B_PAT + 1], 1);
        mbar_init(&bars[B_DRN], 1);
        fence_mbar_init();
        *s_abort = 0;
    }
    if constexpr (X::ISO) {
        // per-lane copies (no bank conflicts) of the fp16 level pair of every pair of codes:
        // ISO4 pair index = c0 | c1 << 4; ISO3 pair index = low 2 bits of c0, c1 | their high bits << 4
        uint32_t* lutw = reinterpret_cast<uint32_t*>(sm + X::OFF_LUT);
        constexpr int TT = FMT == 3 ? 1 : 0;
        for (int e = tid; e < X::LUT_N * 32; e += kThr) {
            const int idx = e >> 5;
            int c0, c1;
            if constexpr (TT == 1) {
                c0 = idx & 15;
                c1 = idx >> 4;
            } else {
                c0 = (idx & 3) | (((idx >> 4) & 1) << 2);
                c1 = ((idx >> 2) & 3) | (((idx >> 5) & 1) << 2);
            }
            lutw[e] = f32x2_to_h2(c_tc_levels[TT][c0], c_tc_levels[TT][c1]);
        }
    }
    if (warp == kWMma) tmem_alloc(tslot, X::TCOLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    // Every warp derives this CTA's share of the (sequence, head group, page) units from
    // seq_lens on its own, so no block-wide barrier follows the dependency wait and the
    // producers reach the page table one global load later.
    auto compute_share = [&](auto len_of, bool flag_errors, int& b0, long long& pref0, long long& Tunits) {
        b0 = p.B;
        pref0 = 0;
        const int per = (p.B + 31) / 32;
        const int b_lo = min(p.B, lane * per), b_hi = min(p.B, b_lo + per);
        long long local = 0;
        for (int b = b_lo; b < b_hi; ++b) {
            const int Lr = len_of(b);
            // a verify window longer than its sequence is flagged too (its early queries see nothing)
            if (flag_errors && warp == 0 && (Lr < 0 || Lr > p.max_pages * kPage || (VW && Lr < p.W)))
                atomicOr(&g_err_dtc, kErrPos);
            local += (max(0, min(Lr, p.max_pages * kPage)) + kPage - 1) / kPage;
        }
        long long incl = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const long long v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        Tunits = __shfl_sync(0xffffffffu, incl, 31) * p.NH;
        const long long beg = Tunits * c / C;
        long long pref = incl - local, fpref = 0;
        int fb = -1;
        for (int b = b_lo; b < b_hi; ++b) {
            const long long np = (max(0, min(len_of(b), p.max_pages * kPage)) + kPage - 1) / kPage;
            if (np > 0 && pref * p.NH <= beg && beg < (pref + np) * p.NH) {
                fb = b;
                fpref = pref;
            }
            pref += np;
        }
        const unsigned found = __ballot_sync(0xffffffffu, fb >= 0);
        if (found) {
            const int src = __ffs(found) - 1;
            b0 = __shfl_sync(0xffffffffu, fb, src);
            pref0 = __shfl_sync(0xffffffffu, fpref, src);
        }
    };
    // Before the dependency wait: the share as seq_lens reads now (L2-only loads; the previous
    // kernel may still change it). It serves addresses only: the producers prefetch the first
    // two tiles' pages into L2 (a prefetch returns no data, so a later write by the previous
    // kernel is still what the copies after the wait read) and, after the wait, load the page
    // ids of the first piece at once; those are kept only if the piece that the share read
    // after the wait gives is the same. Every value the kernel uses is loaded after the wait.
    // The share itself is kept too: with at most 128 sequences every lane holds its (up to 4)
    // seq_lens values as read here, and after the wait the warp compares them with a fresh read;
    // if none changed (and the first piece's own length read agrees), the share and the first
    // piece stand and the post-wait prefix scan and divisions are skipped.
    Piece spc;
    spc.b = -1;
    int spid_cur = 0, spid_nxt = 0;
    const int per_lane = (p.B + 31) / 32;
    const bool sfast = per_lane <= 4;
    int slen[4] = {0, 0, 0, 0};
    int b0s = 0;
    long long pref0s = 0, Tus = 0, begs = 0, ends = 0;
    bool shas = false;
    {
        const int b_lo = min(p.B, lane * per_lane);
        if (sfast) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (i < per_lane && b_lo + i < p.B) slen[i] = __ldcg(p.seq_lens + b_lo + i);
        }
        auto pick = [&](int i) { return i == 0 ? slen[0] : i == 1 ? slen[1] : i == 2 ? slen[2] : slen[3]; };
        if (sfast) compute_share([&](int b) { return pick(b - b_lo); }, false, b0s, pref0s, Tus);
        else compute_share([&](int b) { return __ldcg(p.seq_lens + b); }, false, b0s, pref0s, Tus);
        begs = Tus * c / C;
        ends = Tus * (c + 1) / C;
        if (warp == kWProd || warp == kWProdV || warp < kSoftW) {
            Walker ws{b0s, pref0s, begs, ends};
            shas = ws.template next<true>(p, spc);
        }
        if (shas && (warp == kWProd || warp == kWProdV)) {
            const int kind = warp == kWProdV ? 1 : 0;
            if (lane == 0) prefetch_tensormap(kind ? &tmV : &tmK);
            const int npf = min(2 * kTP, spc.p1 - spc.p0);
            if (lane < npf) {
                const int pid = __ldcg(p.page_table + (size_t)spc.b * p.max_pages + spc.p0 + lane);
                if (pid >= 0 && pid < p.num_pages) {
                    const int rowb = kind ? X::VROW : X::KROW, scrow = kind ? X::VSROW : X::KSROW;
                    const long long prow = ((long long)pid * p.Hkv + spc.hg / (p.Gv / G)) * kPage;
                    bulk_prefetch_l2((kind ? p.vc : p.kc) + prow * rowb, kPage * rowb);
                    if (scrow) bulk_prefetch_l2((kind ? p.vs : p.ks) + prow * scrow, kPage * scrow);
                }
            }
        }
        // inputs may come from the previous kernel in the stream (programmatic dependent launch)
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;");
        if (shas) {
            if (warp == kWProd || warp == kWProdV) {
                const int32_t* row = p.page_table + (size_t)spc.b * p.max_pages + spc.p0;
                const int npc = spc.p1 - spc.p0;
                spid_cur = lane < npc ? row[lane] : 0;
                spid_nxt = 32 + lane < npc ? row[32 + lane] : 0;
            } else if (warp < kSoftW) {
                const int kvh = spc.hg / (p.Gv / G), hgi = spc.hg % (p.Gv / G);
                if (tid < G * D * 2 / 128)   // the query rows of the first piece (2 D bytes a head)
                    prefetch_l1(reinterpret_cast<const uint8_t*>(p.q + qrow_index<VW>(p, spc.b, kvh, hgi * G + tid / (D / 64)) * D) +
                                128 * (tid % (D / 64)));
            }
        } else {
            spc.b = -1;
        }
    }
    // validate the share read before the wait (see above); warp 0 also flags bad lengths here
    bool fast = false;
    // (the verify-window instantiations skip it: their 16-column softmax has no registers to spare)
    if (!VW && sfast && shas && spc.b == b0s) {
        const int b_lo = min(p.B, lane * per_lane);
        bool same = true;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (i < per_lane && b_lo + i < p.B) {
                const int Lr = p.seq_lens[b_lo + i];
                same &= Lr == slen[i];
                if (warp == 0 && (Lr < 0 || Lr > p.max_pages * kPage || (VW && Lr < p.W))) atomicOr(&g_err_dtc, kErrPos);
            }
        fast = __all_sync(0xffffffffu, same) && spc.L == seq_len_clamped(p, spc.b);
    }
    int b0;
    long long pref0, Tunits;
    if (fast) {
        b0 = b0s;
        pref0 = pref0s;
        Tunits = Tus;
    } else {
        compute_share([&](int b) { return p.seq_lens[b]; }, true, b0, pref0, Tunits);
    }
    const long long beg = fast ? begs : Tunits * c / C, end = fast ? ends : Tunits * (c + 1) / C;
    auto cta_of = [&](long long x) -> long long { return ((x + 1) * C + Tunits - 1) / Tunits - 1; };

    // empty sequences: zero rows, written by CTA (s mod C)
    for (long long s = c; s < (long long)p.B * p.NH; s += C) {
        const int b = (int)(s / p.NH);
        if (seq_len_clamped(p, b) == 0) {
            const int hg = (int)(s % p.NH);
            const int kvh = hg / (p.Gv / G), hgi = hg % (p.Gv / G);
            for (int i = tid; i < G * D; i += kThr) write_out<D, G, VW>(p, b, kvh, hgi * G, i, 0.0f);
        }
    }
    // the piece iterator; with a validated share its first piece is spc, already worked out
    Walker walker{b0, pref0, beg, end};
    if (fast) walker = Walker{spc.b, pref0s, spc.soff + spc.p1, end};
    auto first_piece = [&](Piece& pc) -> bool {
        if (fast) {
            pc = spc;
            return true;
        }
        return walker.next(p, pc);
    };

    if (warp == kWProd || warp == kWProdV) {
        // ============================ producers (K, V) ============================
        // One warp per plane, so that the K stream runs ahead of the V stream (PV of a
        // tile comes much later than its Q K^T). Page ids come from a 32-entry ring per
        // lane, refilled a block ahead, so no tile waits for a page-table load.
        const int kind = warp == kWProdV ? 1 : 0;
        uint64_t* const fullb = &bars[kind ? B_VF : B_KF];
        uint64_t* const emptyb = &bars[kind ? B_VE : B_KE];
        const CUtensorMap* tm = kind ? &tmV : &tmK;
        const uint8_t* scl = kind ? p.vs : p.ks;
        const uint16_t* newsrc = kind ? p.v_new : p.k_new;
        // per-plane geometry: V pages of q4 codes are half as wide and carry twice the scales;
        // ISO pages (48 or 64 code bytes per 128 values) are staged row-major by one bulk copy;
        // the unquantized bf16 V goes straight into the V' tile (its 64-dim boxes are the MN-major
        // operand layout), bf16 K into one staging tile
        const int pageb = kind ? X::VPAGE_B : X::PAGE_B, scb = kind ? X::VSC_B : X::SC_B;
        const int nbox = kind ? X::VBOX : X::KBOX, scrow = kind ? X::VSROW : X::KSROW;
        const int nslot = kind ? 2 : X::KSTB;   // staging slots of this plane
        const bool to_vp = X::VB && kind;
        const int rowb = pageb / kPage;   // code bytes of one row
        const uint8_t* codes = kind ? p.vc : p.kc;
        // where box bx of page j of a tile in slot buf lands
        auto dst = [&](int buf, int j, int bx) -> uint8_t* {
            if (to_vp) return sm + X::OFF_VP + buf * NA * 16384 + bx * 16384 + j * 2048;
            return sm + (kind ? X::OFF_VST : X::OFF_KST) + (buf * kTP + j) * pageb + bx * 2048;
        };
        uint32_t T = 0, pat_phase = 0;
        Piece pc;
        bool first = true;
        for (bool have = first_piece(pc); have; have = walker.next(p, pc)) {
            const int kvh = pc.hg / (p.Gv / G);
            const int32_t* ptrow = p.page_table + (size_t)pc.b * p.max_pages;
            const int last_page = (pc.L - 1) / kPage;
            const int npc = pc.p1 - pc.p0;
            int bc = 0;
            int pid_cur, pid_nxt;
            if (first && pc.b == spc.b && pc.p0 == spc.p0 && pc.p1 == spc.p1) {
                // the same addresses as the page ids loaded right after the wait
                pid_cur = spid_cur;
                pid_nxt = spid_nxt;
            } else {
                pid_cur = lane < npc ? ptrow[pc.p0 + lane] : 0;
                pid_nxt = 32 + lane < npc ? ptrow[pc.p0 + 32 + lane] : 0;
            }
            first = false;
            for (int pg0 = pc.p0; pg0 < pc.p1; pg0 += kTP, ++T) {
                const int npg = min(kTP, pc.p1 - pg0);
                const int buf = nslot == 2 ? (int)(T & 1) : 0;
                const uint32_t round = nslot == 2 ? T >> 1 : T;   // uses of this slot so far
                // the page of the sequence's last token is patched after it lands: the newest row
                // (quantize-on-write) and, for the bf16 V tile, zeros in the rows past the end
                const int jp = ((p.k_new != nullptr || to_vp) && last_page >= pg0 && last_page < pg0 + npg) ? last_page - pg0 : -1;
                const int pi = pg0 - pc.p0;   // page index inside the piece (a multiple of 8)
                if ((pi >> 5) > bc) {
                    pid_cur = pid_nxt;
                    ++bc;
                    pid_nxt = 32 * (bc + 1) + lane < npc ? ptrow[pc.p0 + 32 * (bc + 1) + lane] : 0;
                }
                int pid = __shfl_sync(0xffffffffu, pid_cur, (pi & 31) + (lane & 7));
                if (lane < npg && (pid < 0 || pid >= p.num_pages)) {
                    atomicOr(&g_err_dtc, kErrPage);
                    pid = 0;
                }
                const int pid_patch = __shfl_sync(0xffffffffu, pid, jp < 0 ? 0 : jp);
                if (round >= 1) wait_or_flag(emptyb + buf, (round - 1) & 1);
                uint64_t* full = fullb + buf;
                uint8_t* ss = sm + (kind ? X::OFF_VSC : X::OFF_KSC) + buf * kTP * scb;
                const int nload = npg - (jp >= 0 ? 1 : 0);
                if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)nload * (pageb + scb));
                __syncwarp();
                if (lane < npg && lane != jp) {
                    // pages are read once per launch: evict-first in L2
                    const int row = (pid * p.Hkv + kvh) * kPage;
                    const uint64_t pol = l2_evict_first_policy();
                    if constexpr (X::ISO) {
                        bulk_load_hint(dst(buf, lane, 0), codes + (size_t)row * rowb, pageb, full, pol);
                    } else {
                        for (int bx = 0; bx < nbox; ++bx)
                            tma_load_2d_hint(dst(buf, lane, bx), tm, full, bx * 128, row, pol);
                    }
                    if (scb) bulk_load_hint(ss + lane * scb, scl + (size_t)row * scrow, scb, full, pol);
                }
                if (jp >= 0) {
                    // the sequence's newest token: load its page, quantize the new row into the
                    // pool and into the staged copy, then release the tile
                    const int row = (pid_patch * p.Hkv + kvh) * kPage;
                    uint64_t* pb = &bars[B_PAT + kind];
                    if (lane == 0) {
                        mbar_arrive_expect_tx(pb, pageb + scb);
                        if constexpr (X::ISO) {
                            bulk_load(dst(buf, jp, 0), codes + (size_t)row * rowb, pageb, pb);
                        } else {
                            for (int bx = 0; bx < nbox; ++bx) tma_load_2d(dst(buf, jp, bx), tm, pb, bx * 128, row);
                        }
                        if (scb) bulk_load(ss + jp * scb, scl + (size_t)row * scrow, scb, pb);
                    }
                    // after an abort elsewhere, still let this copy land before the row is patched
                    if (!wait_or_flag(pb, pat_phase)) mbar_wait_bounded(pb, pat_phase);
                    pat_phase ^= 1;
                    if (to_vp && (pc.L % kPage) != 0) {
                        // rows past the sequence end hold whatever the pool has there; P' is 0 for
                        // them, but 0 x NaN is not, so they are zeroed
                        const int r0 = pc.L % kPage;
                        for (int e = lane; e < (kPage - r0) * NA * 8; e += 32) {
                            const int rw = r0 + e / (NA * 8), at = (e / 8) % NA, u = e % 8;
                            *reinterpret_cast<uint4*>(dst(buf, jp, at) + rw * 128 + 16 * u) = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                }
                if (jp >= 0 && p.k_new != nullptr) {
                    const int row = (pid_patch * p.Hkv + kvh) * kPage;
                    uint8_t* rowbuf = sm + X::OFF_ROW + kind * 512;
                    const uint16_t* src = newsrc + ((size_t)pc.b * p.Hkv + kvh) * D;
                    if constexpr (X::ISO) {
                        constexpr int TT = FMT == 3 ? 1 : 0;
                        quantize_row<FMT == 3 ? ENC_ISO4 : ENC_ISO3, D>(src, rowbuf, rowbuf + 256, lane, p.quat,
                                                                        c_tc_levels[TT], c_tc_mids[TT]);
                    } else if (kind ? VQ : X::KQ) {
                        quantize_row<ENC_Q4, D>(src, rowbuf, rowbuf + 256, lane, nullptr, nullptr, nullptr);
                    } else if (kind ? X::VB : X::KB) {
                        quantize_row<ENC_BF16, D>(src, rowbuf, rowbuf + 256, lane, nullptr, nullptr, nullptr);
                    } else {
                        quantize_row<ENC_INT8, D>(src, rowbuf, rowbuf + 256, lane, nullptr, nullptr, nullptr);
                    }
                    __syncwarp();
                    const int rr = (pc.L - 1) % kPage;
                    const long long grow = (long long)row + rr;
                    uint8_t* gcode = const_cast<uint8_t*>(codes) + grow * rowb;
                    uint8_t* gscale = const_cast<uint8_t*>(scl) + grow * scrow;
                    if (lane < rowb / 16) {
                        const uint4 v = *reinterpret_cast<const uint4*>(rowbuf + 16 * lane);
                        *reinterpret_cast<uint4*>(gcode + 16 * lane) = v;
                        if constexpr (X::ISO) *reinterpret_cast<uint4*>(dst(buf, jp, 0) + rr * rowb + 16 * lane) = v;
                        else *reinterpret_cast<uint4*>(dst(buf, jp, lane >> 3) + sw_off(rr, lane & 7)) = v;
                    }
                    if (lane < scrow / 2) {
                        const uint16_t v = reinterpret_cast<const uint16_t*>(rowbuf + 256)[lane];
                        reinterpret_cast<uint16_t*>(gscale)[lane] = v;
                        reinterpret_cast<uint16_t*>(ss + jp * scb + rr * scrow)[lane] = v;
                    }
                    __syncwarp();
                }
                if (to_vp && npg < kTP) {
                    // pages the tile does not load: zero V' rows (stale shared memory may hold NaN)
                    for (int e = lane; e < (kTP - npg) * NA * 128; e += 32) {
                        const int pg = npg + e / (NA * 128), at = (e / 128) % NA, u = e % 128;
                        *reinterpret_cast<uint4*>(dst(buf, pg, at) + 16 * u) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                if (jp >= 0 || (to_vp && npg < kTP)) {
                    fence_proxy_async();   // generic writes before the tensor core (and later TMA refills)
                    __syncwarp();
                }
                if (lane == 0) mbar_arrive(full);
            }
        }
        // every copy issued above has landed before the CTA exits (bounded waits that do not
        // stop at the abort flag: the copies of an aborted launch still land in this CTA's memory)
        for (uint32_t t = (T >= (uint32_t)nslot ? T - nslot : 0); t < T; ++t)
            if (!mbar_wait_bounded(fullb + (nslot == 2 ? (t & 1) : 0), (nslot == 2 ? t >> 1 : t) & 1))
                atomicOr(&g_err_dtc, kErrWait);
    } else if (warp == kWMma) {
        // =============================== MMA issue ===============================
        if (lane == 0) {
            constexpr uint32_t IDQK = idesc_f16(128, 16, 0, 0, X::KB ? 1 : 0);      // bf16 K: bf16 operands
            constexpr uint32_t IDPV = idesc_f16(X::PM, D, 1, 1, X::VB ? 1 : 0);     // bf16 V: bf16 P' and V'
            // base descriptors; every MMA adds a compile-time offset (16-byte units) to them
            const uint64_t qd0 = sw128_desc(smem_addr(sm + X::OFF_Q));
            const uint64_t vd0 = sw128_desc_lbo(smem_addr(sm + X::OFF_VP), 16384, 1024);
            const uint64_t pd0 = sw128_desc_lbo(smem_addr(sm + X::OFF_PP), 16384, 1024);
            const uint32_t tk = tmem + X::KCOL, to = tmem + X::OCOL;
            // two cursors over the same tiles. The tensor pipe runs MMAs in issue order; PV sits
            // on the critical path (its V' and P' tiles are single-buffered), so PV goes first and
            // QK^T runs at most one tile ahead of the next PV, overlapping the V' conversion.
            Walker wq = walker, wv = walker;
            Piece pq, pv;
            bool hq = wq.next(p, pq), hv = wv.next(p, pv);
            int tq = 0, tv = 0;           // tile index inside the current piece
            uint32_t Tq = 0, Tv = 0, pieceq = 0;
            int qh = 0;                   // the next Q K^T half of tile Tq
            uint32_t idle = 0;
            while ((hq || hv) && idle < (1u << 22)) {
                if ((idle & 63) == 63 && *s_abort) break;
                bool progressed = false;
                if (hv && Tv < Tq) {
                    bool ready = mbar_test_wait(&bars[B_PFL], Tv & 1);
                    // V' of the tile: converted, or (bf16 V) landed in its own V' tile
                    if (ready) ready = X::VB ? mbar_test_wait(&bars[B_VF + (Tv & 1)], (Tv >> 1) & 1)
                                             : mbar_test_wait(&bars[B_VCV], Tv & 1);
                    if (ready) {
                        tc_fence_after();
                        const uint64_t vdt = vd0 + (uint64_t)(X::VB ? ((Tv & 1) * NA * 16384) >> 4 : 0);
                        // O[64 P' columns][D] += P'^T (MN-major, token rows) x V' (MN-major, token rows)
#pragma unroll
                        for (int u = 0; u < kTok / 16; ++u)
                            umma_f16(to, pd0 + (uint64_t)((u * 2048) >> 4), vdt + (uint64_t)((u * 2048) >> 4), IDPV,
                                     (tv > 0 || u > 0));
                        umma_commit(&bars[B_PVD + (Tv & 1)]);
                        if constexpr (X::VB) umma_commit(&bars[B_VE + (Tv & 1)]);   // the V' tile is free
                        ++Tv;
                        if (pv.p0 + kTP * (tv + 1) < pv.p1) {
                            ++tv;
                        } else {
                            tv = 0;
                            hv = wv.next(p, pv);
                        }
                        progressed = true;
                    }
                }
                // bf16 K: Q K^T of a tile in two halves, k-steps 0-1 and 2-3 of every 64-dim group
                // (the four accumulators stay interleaved in each half). The converters of half h
                // write the K' columns of those k-steps and wait only for the MMAs of half h of the
                // tile before, so K' of the next tile is written while the other half's MMAs still
                // run (53.6 -> 49.5 us at 131072 tokens). The other formats issue the tile at once:
                // there an early half queues ahead of PV in the tensor pipe and PV, whose P' and V'
                // tiles are single-buffered, finishes later (int8: 40.0 -> 42.6 us).
                auto qk_half = [&](int h) {
                    const uint32_t sd = tmem + X::SCOL + (Tq % X::NSB) * X::SBUF;
                    if constexpr (X::KQ) {
                        // q4 K: one accumulator per 32-dim block (its own scale); two k-steps a
                        // block against the rotated query's hi (N columns 0..7) and lo (8..15)
#pragma unroll
                        for (int u = 0; u < 2; ++u)
#pragma unroll
                            for (int g = 0; g < X::NKG; ++g)
                                umma_f16_ta(sd + 16 * g, tk + 8 * (2 * g + u),
                                            qd0 + (uint64_t)(((g >> 1) * 2048 + (g & 1) * 64 + 32 * u) >> 4), IDQK, u > 0);
                    } else if constexpr (X::ISO) {
                        // per 128-dim block: 8 k-steps against the query tile whose N columns hold
                        // the rotated query's fp16 hi (0..7) and lo (8..15) parts; even and odd
                        // k-steps go to two accumulators, so consecutive MMAs are independent
#pragma unroll
                        for (int u = 0; u < 8; ++u)
#pragma unroll
                            for (int gk = 0; gk < X::NKG; ++gk)
                                umma_f16_ta(sd + 32 * gk + 16 * (u & 1), tk + 8 * (8 * gk + u),
                                            qd0 + (uint64_t)(((2 * gk + (u >> 2)) * 2048 + 32 * (u & 3)) >> 4),
                                            IDQK, u > 1);
                    } else {
                        // k-step outer, scale group inner: consecutive MMAs write different
                        // accumulators, so the tensor pipe overlaps them instead of waiting on
                        // each accumulator's previous k-step
#pragma unroll
                        for (int ui = 0; ui < (kSplitK ? 2 : 4); ++ui)
#pragma unroll
                            for (int g = 0; g < NA; ++g) {
                                const int u = kSplitK ? 2 * h + ui : ui;
                                umma_f16_ta(sd + 16 * g, tk + 8 * (4 * g + u), qd0 + (uint64_t)((g * 2048 + 32 * u) >> 4),
                                            IDQK, u > 0);
                            }
                    }
                };
                if (hq && qh == 1) {
                    if (mbar_test_wait(&bars[B_KCV1], Tq & 1)) {
                        tc_fence_after();
                        qk_half(1);
                        umma_commit(&bars[B_QKD + (Tq & 1)]);
                        ++Tq;
                        qh = 0;
                        if (pq.p0 + kTP * (tq + 1) < pq.p1) {
                            ++tq;
                        } else {
                            tq = 0;
                            ++pieceq;
                            hq = wq.next(p, pq);
                        }
                        progressed = true;
                    }
                } else if (hq && (!hv || Tq <= Tv + 1)) {
                    const bool first = tq == 0;
                    bool ready = mbar_test_wait(&bars[B_KCV], Tq & 1);
                    if (ready && Tq >= (uint32_t)X::NSB)
                        ready = mbar_test_wait(&bars[B_SF + Tq % X::NSB], ((Tq / X::NSB) - 1) & 1);
                    if (ready && first) ready = mbar_test_wait(&bars[B_QRD], pieceq & 1);
                    if (ready) {
                        tc_fence_after();
                        qk_half(0);
                        if constexpr (kSplitK) {
                            umma_commit(&bars[B_QKH + (Tq & 1)]);
                            qh = 1;
                        } else {
                            umma_commit(&bars[B_QKD + (Tq & 1)]);
                            ++Tq;
                            if (pq.p0 + kTP * (tq + 1) < pq.p1) {
                                ++tq;
                            } else {
                                tq = 0;
                                ++pieceq;
                                hq = wq.next(p, pq);
                            }
                        }
                        progressed = true;
                    }
                }
                idle = progressed ? 0 : idle + 1;
            }
            if (hq || hv) {
                atomicOr(&g_err_dtc, kErrWait);
                *s_abort = 1;
            }
            // every MMA issued above completes before TMEM is released (after an abort the
            // loop ends with MMAs possibly still in flight)
            if (Tq > 0 || Tv > 0 || qh) {
                umma_commit(&bars[B_DRN]);
                if (!mbar_wait_bounded(&bars[B_DRN], 0)) atomicOr(&g_err_dtc, kErrWait);
            }
        }
        __syncwarp();
    } else if (warp >= kSoftW) {
        // =============================== converters ===============================
        // Eight warps: warp (sub, hf) owns token rows 32 sub .. 32 sub + 31 and half hf of
        // the head dimension. Iteration T converts K of tile T (Q K^T of a tile may run one
        // tile ahead of PV) and then V of tile T - 1, so V' waits for nothing but PV of the
        // tile before it.
        const int cw = warp - kSoftW, sub = cw & 3, hf = cw >> 2;
        const int r = 32 * sub + lane, jpage = r >> 4, rr = r & 15;
        constexpr int NCH = D / 32;   // 16-code chunks per thread (half of the head dimension)
        const uint32_t lb = (uint32_t)(32 * sub) << 16;
        // ISO: the fp16 level pairs of 16 consecutive code pairs p0 .. p0 + 15 (dims 2 p, 2 p + 1)
        // of one staged token row, through the per-lane pair table
        const uint32_t* lut = reinterpret_cast<const uint32_t*>(sm + X::OFF_LUT) + lane;
        auto iso16 = [&](const uint8_t* crow, int p0, uint32_t (&w)[16]) {
            const uint8_t* cb = crow + (p0 >> 6) * X::ISO_RB;   // 64 pairs per 128-value block
            const int q0 = p0 & 63;
            if constexpr (FMT == 3) {
                const uint4 x = *reinterpret_cast<const uint4*>(cb + q0);   // byte q = codes 2q (low), 2q + 1
                const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int i = 0; i < 16; ++i) w[i] = lut[((xs[i >> 2] >> (8 * (i & 3))) & 0xffu) * 32];
            } else {
                // byte l: low 2 bits of codes 4l .. 4l + 3; nibble l of the high-bit bytes: their bit 2
                const int l0 = q0 >> 1;
                const uint2 lo = *reinterpret_cast<const uint2*>(cb + l0);
                const uint32_t hn = *reinterpret_cast<const uint32_t*>(cb + 32 + (l0 >> 1));
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int l = i >> 1, u = i & 1;
                    const uint32_t lob = ((l < 4 ? lo.x : lo.y) >> (8 * (l & 3))) & 0xffu;
                    const uint32_t hnn = (hn >> (4 * l)) & 0xfu;
                    w[i] = lut[(((lob >> (4 * u)) & 0xfu) | (((hnn >> (2 * u)) & 3u) << 4)) * 32];
                }
            }
        };
        int v_npg = 0, v_pos0 = 0, v_len = 0;   // extent of the tile whose V is converted next
        auto convert_v = [&](uint32_t Tc) {
            if constexpr (X::VB) return;   // the bf16 V tile lands in V' itself
            // rows past the sequence end (or of pages the tile did not load) may hold anything in
            // shared memory; the q4 path multiplies by a staged scale, so those rows are zeroed
            const bool vrow_ok = jpage < v_npg && v_pos0 + r < v_len;
            const int buf = Tc & 1;
            wait_or_flag(&bars[B_VF + buf], (Tc >> 1) & 1);
            // V' is free once PV of the tile before read it
            if (Tc >= 1) wait_or_flag(&bars[B_PVD + ((Tc - 1) & 1)], ((Tc - 1) >> 1) & 1);
            const uint8_t* slot = sm + X::OFF_VST + (buf * kTP + jpage) * X::VPAGE_B;
            uint8_t* vp = sm + X::OFF_VP;
            if constexpr (X::ISO) {
                // level pairs in natural dim order: pair p -> V' atom p / 32, 16-byte chunk (p % 32) / 4
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    const int p0 = (D / 4) * hf + 16 * c;
                    uint32_t w[16];
                    iso16(slot + rr * X::VROW, p0, w);
                    uint8_t* atom = vp + (p0 >> 5) * 16384;
                    const int ch = (p0 & 31) >> 2;
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        *reinterpret_cast<uint4*>(atom + sw_off(r, ch + k)) = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
                }
            } else if constexpr (VQ) {
                // q4_0 block b (32 dims: 16 code bytes, byte j = element j low, j + 16 high nibble)
                // -> fp16((q - 8) * d), one rounding (q - 8 is exact in fp16; the block scale d is
                // folded in here, so P' needs no V scale groups). Pairs come out as (4w, 4w + 2),
                // (4w + 1, 4w + 3): the same position <-> dimension permutation (perm4) as the int8 path.
                const uint16_t* vsr = reinterpret_cast<const uint16_t*>(sm + X::OFF_VSC + (buf * kTP + jpage) * X::VSC_B +
                                                                        rr * X::VSROW);
#pragma unroll
                for (int bi = 0; bi < D / 64; ++bi) {
                    const int blk = (D / 64) * hf + bi;
                    const uint4 x = *reinterpret_cast<const uint4*>(slot + sw_off(rr, blk));
                    const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
                    const uint32_t sb = vrow_ok ? (uint32_t)vsr[blk] : 0u, s2 = sb | (sb << 16);
                    uint32_t lo[8], hi[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        lo[2 * k] = hfma2_u32(hsub2_u32((xs[k] & 0x000f000fu) | 0x64006400u, 0x64086408u), s2, 0u);
                        lo[2 * k + 1] = hfma2_u32(hsub2_u32(((xs[k] >> 8) & 0x000f000fu) | 0x64006400u, 0x64086408u), s2, 0u);
                        hi[2 * k] = hfma2_u32(hsub2_u32(((xs[k] >> 4) & 0x000f000fu) | 0x64006400u, 0x64086408u), s2, 0u);
                        hi[2 * k + 1] = hfma2_u32(hsub2_u32(((xs[k] >> 12) & 0x000f000fu) | 0x64006400u, 0x64086408u), s2, 0u);
                    }
                    uint8_t* atom = vp + (blk >> 1) * 16384;
                    const int ch = 4 * (blk & 1);
                    *reinterpret_cast<uint4*>(atom + sw_off(r, ch)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    *reinterpret_cast<uint4*>(atom + sw_off(r, ch + 1)) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
                    *reinterpret_cast<uint4*>(atom + sw_off(r, ch + 2)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4*>(atom + sw_off(r, ch + 3)) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
                }
            } else {
                // 16 query columns: fp16(c d) with the row's scale of the 64-dim group (rows past the
                // sequence end, whose staged scale may be anything, get scale 0)
                const uint16_t* vsr = reinterpret_cast<const uint16_t*>(sm + X::OFF_VSC + (buf * kTP + jpage) * X::VSC_B +
                                                                        rr * X::VSROW);
#pragma unroll
                for (int i = 0; i < NCH; ++i) {
                    const int gc = hf * NCH + i;
                    const uint4 x = *reinterpret_cast<const uint4*>(slot + (gc >> 3) * 2048 + sw_off(rr, gc & 7));
                    const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
                    uint32_t w[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        w[2 * k] = hsub2_u32(lop3_and_xor(xs[k], 0x00ff00ffu, 0x64806480u), 0x64806480u);
                        w[2 * k + 1] = hsub2_u32(lop3_and_xor(xs[k] >> 8, 0x00ff00ffu, 0x64806480u), 0x64806480u);
                    }
                    if constexpr (VFOLD) {
                        const uint32_t sb = vrow_ok ? (uint32_t)vsr[gc >> 2] : 0u, s2 = sb | (sb << 16);
#pragma unroll
                        for (int k = 0; k < 8; ++k) w[k] = hfma2_u32(w[k], s2, 0u);
                    }
                    uint8_t* atom = vp + (gc >> 2) * 16384;
                    const int ch = 2 * (gc & 3);
                    *reinterpret_cast<uint4*>(atom + sw_off(r, ch)) = make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint4*>(atom + sw_off(r, ch + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
                }
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars[B_VCV]);
                mbar_arrive(&bars[B_VE + buf]);
            }
        };
        uint32_t T = 0;
        Piece pc;
        for (bool have = first_piece(pc); have; have = walker.next(p, pc)) {
            for (int pg0 = pc.p0; pg0 < pc.p1; pg0 += kTP, ++T) {
                const int buf = X::KSTB == 2 ? (int)(T & 1) : 0;
                // ---- K of tile T: exact fp16 1152 + c (int8), q - 8 (q4) or the bf16 values, one
                // token per TMEM lane ----
                wait_or_flag(&bars[B_KF + buf], (X::KSTB == 2 ? T >> 1 : T) & 1);
                // the K' columns of half hf are free once the MMAs of tile T - 1 that read them are done
                if (T >= 1)
                    wait_or_flag(&bars[(kSplitK && !hf ? B_QKH : B_QKD) + ((T - 1) & 1)], ((T - 1) >> 1) & 1);
                tc_fence_after();
                if constexpr (X::ISO) {
                    // level pairs of dims 2 p, 2 p + 1 into TMEM column p, one token per lane
                    const uint8_t* crow = sm + X::OFF_KST + (buf * kTP + jpage) * X::PAGE_B + rr * X::KROW;
#pragma unroll
                    for (int c = 0; c < D / 128; ++c) {
                        uint32_t w[32];
                        const int p0 = (D / 4) * hf + 32 * c;
                        uint32_t w0[16], w1[16];
                        iso16(crow, p0, w0);
                        iso16(crow, p0 + 16, w1);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            w[i] = w0[i];
                            w[16 + i] = w1[i];
                        }
                        tmem_st32_nowait(tmem + lb + X::KCOL + p0, w);
                    }
                    tmem_wait_st();
                } else if constexpr (X::KQ) {
                    // q4_0 block b of the rotated row -> exact fp16 q - 8 into TMEM columns 16 b ..
                    // 16 b + 15 (low-nibble pairs, then high-nibble pairs: position p of the block
                    // holds element perm4(p), as in the int8 path)
                    const uint8_t* slot = sm + X::OFF_KST + (buf * kTP + jpage) * X::PAGE_B;
#pragma unroll
                    for (int b2 = 0; b2 < 2; ++b2) {
                        uint32_t w[32];
#pragma unroll
                        for (int bb = 0; bb < 2; ++bb) {
                            const int blk = 4 * hf + 2 * b2 + bb;
                            const uint4 x = *reinterpret_cast<const uint4*>(slot + sw_off(rr, blk));
                            const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                w[16 * bb + 2 * k] = hsub2_u32((xs[k] & 0x000f000fu) | 0x64006400u, 0x64086408u);
                                w[16 * bb + 2 * k + 1] = hsub2_u32(((xs[k] >> 8) & 0x000f000fu) | 0x64006400u, 0x64086408u);
                                w[16 * bb + 8 + 2 * k] = hsub2_u32(((xs[k] >> 4) & 0x000f000fu) | 0x64006400u, 0x64086408u);
                                w[16 * bb + 8 + 2 * k + 1] = hsub2_u32(((xs[k] >> 12) & 0x000f000fu) | 0x64006400u, 0x64086408u);
                            }
                        }
                        tmem_st32_nowait(tmem + lb + X::KCOL + 16 * (4 * hf + 2 * b2), w);
                    }
                    tmem_wait_st();
                } else if constexpr (X::KB) {
                    // bf16 K: the staged values as they are, dims 2 c, 2 c + 1 in TMEM column c; half
                    // hf holds k-steps 2 hf, 2 hf + 1 of every 64-dim group (TMEM columns 32 g + 16 hf ..)
                    const uint8_t* slot = sm + X::OFF_KST + jpage * X::PAGE_B;
#pragma unroll
                    for (int g = 0; g < NA; ++g) {
                        uint32_t w[16];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int gc = 8 * g + 4 * hf + i;   // 16-byte chunk = 8 dims
                            const uint4 x = *reinterpret_cast<const uint4*>(slot + (gc >> 3) * 2048 + sw_off(rr, gc & 7));
                            w[4 * i] = x.x;
                            w[4 * i + 1] = x.y;
                            w[4 * i + 2] = x.z;
                            w[4 * i + 3] = x.w;
                        }
                        tmem_st16_nowait(tmem + lb + X::KCOL + 32 * g + 16 * hf, w);
                    }
                    tmem_wait_st();
                } else {
                    const uint8_t* slot = sm + X::OFF_KST + (buf * kTP + jpage) * X::PAGE_B;
#pragma unroll
                    for (int i0 = 0; i0 < NCH; i0 += 4) {
                        uint32_t w[32];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int gc = hf * NCH + i0 + i;
                            const uint4 x = *reinterpret_cast<const uint4*>(slot + (gc >> 3) * 2048 + sw_off(rr, gc & 7));
                            const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                w[8 * i + 2 * k] = lop3_and_xor(xs[k], 0x00ff00ffu, 0x64806480u);
                                w[8 * i + 2 * k + 1] = lop3_and_xor(xs[k] >> 8, 0x00ff00ffu, 0x64806480u);
                            }
                        }
                        tmem_st32_nowait(tmem + lb + X::KCOL + 8 * (hf * NCH + i0), w);
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bars[kSplitK && hf ? B_KCV1 : B_KCV]);
                    mbar_arrive(&bars[B_KE + buf]);
                }
                // ---- V of tile T - 1 ----
                if (T >= 1) convert_v(T - 1);
                v_npg = min(kTP, pc.p1 - pg0);
                v_pos0 = pg0 * kPage;
                v_len = pc.L;
            }
        }
        if (T >= 1) convert_v(T - 1);
    } else {
        // =============================== softmax ===============================
        const int r = tid;   // token row of the tile = TMEM lane
        const uint32_t lb = (uint32_t)(32 * warp) << 16;
        float* bias_s = reinterpret_cast<float*>(sm + X::OFF_BIAS);
        int* red_flag = reinterpret_cast<int*>(sm + X::OFF_RED);                 // [2][4]
        int* red_e = red_flag + 8;                                               // [2][4]
        float* red_m = reinterpret_cast<float*>(sm + X::OFF_RED + 64);           // [2][4][QH]
        float* red_l = red_m + 8 * QH;                                           // [4][QH]
        float* sML = red_l + 4 * QH;                                             // M[QH], L[QH]
        uint32_t T = 0, piece = 0;
        Piece pc;
        for (bool have = first_piece(pc); have; have = walker.next(p, pc)) {
            const int kvh = pc.hg / (p.Gv / G), gv0 = (pc.hg % (p.Gv / G)) * G;   // KV head, first virtual head
            // ---- query tile (B operand, K-major, dims in converter order) and the offset sums ----
            {
                uint8_t* qsm = sm + X::OFF_Q;
                // q4 K: the query rotated by the FWHT-256 (x 1/16) in fp32 first, in the P' area
                // (free between pieces): thread (head hh, slice q16) takes strides 16 .. 128 on
                // dims q16 + 16 k, then strides 1 .. 8 on dims 16 q16 + i
                float* qrot = reinterpret_cast<float*>(sm + X::OFF_PP);   // [8][D]
                if constexpr (X::KQ) {
                    const int hh = r >> 4, q16 = r & 15;
                    if (hh < G) {
                        const uint16_t* qrow = p.q + qrow_index<VW>(p, pc.b, kvh, gv0 + hh) * D;
                        float x[16];
#pragma unroll
                        for (int k = 0; k < 16; ++k) x[k] = bf16_bits_to_f32(qrow[q16 + 16 * k]);
#pragma unroll
                        for (int st = 1; st < 16; st <<= 1)
#pragma unroll
                            for (int k = 0; k < 16; ++k)
                                if ((k & st) == 0) {
                                    const float a0 = x[k], a1 = x[k + st];
                                    x[k] = a0 + a1;
                                    x[k + st] = a0 - a1;
                                }
#pragma unroll
                        for (int k = 0; k < 16; ++k) qrot[hh * D + q16 + 16 * k] = x[k];
                    }
                    soft_sync();
                    if (hh < G) {
                        float y[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) y[i] = qrot[hh * D + 16 * q16 + i];
#pragma unroll
                        for (int st = 1; st < 16; st <<= 1)
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                if ((i & st) == 0) {
                                    const float a0 = y[i], a1 = y[i + st];
                                    y[i] = a0 + a1;
                                    y[i + st] = a0 - a1;
                                }
#pragma unroll
                        for (int i = 0; i < 16; ++i) qrot[hh * D + 16 * q16 + i] = y[i] * 0.0625f;
                    }
                    soft_sync();
                }
                // ISO and q4 K: rows n < 8 take the transformed query's fp16 hi part, rows 8 + n its lo part
                constexpr int QROWS = X::QHL ? 8 : 16;
                for (int idx = r; idx < QROWS * NA * 8; idx += 128) {
                    const int n = idx / (NA * 8), rem = idx % (NA * 8), a = rem >> 3, cc = rem & 7;
                    uint32_t w[4] = {0u, 0u, 0u, 0u}, wl[4] = {0u, 0u, 0u, 0u};
                    if (n < G) {
                        const uint16_t* qrow = p.q + qrow_index<VW>(p, pc.b, kvh, gv0 + n) * D + 64 * a + 8 * cc;
                        const uint4 raw = *reinterpret_cast<const uint4*>(qrow);
                        const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
                        float v[8];
                        if constexpr (X::KQ) {
                            // positions in the q4 K' order (perm4 inside each group of four)
#pragma unroll
                            for (int e = 0; e < 8; ++e) v[e] = qrot[n * D + 64 * a + 8 * cc + perm4(e)];
                        } else if constexpr (X::ISO) {
                            // natural dim order; each 4-D group rotated: <q, conj(R) c> = <R q, c>
#pragma unroll
                            for (int e = 0; e < 8; ++e) v[e] = bf16_bits_to_f32((rw[e >> 1] >> (16 * (e & 1))) & 0xffffu);
                            const float q0 = p.quat[0], q1 = p.quat[1], q2 = p.quat[2], q3 = p.quat[3];
#pragma unroll
                            for (int g4 = 0; g4 < 2; ++g4) {
                                const float a0 = v[4 * g4], b0 = v[4 * g4 + 1], c0 = v[4 * g4 + 2], d0 = v[4 * g4 + 3];
                                v[4 * g4] = q0 * a0 - q1 * b0 - q2 * c0 - q3 * d0;
                                v[4 * g4 + 1] = q0 * b0 + q1 * a0 + q2 * d0 - q3 * c0;
                                v[4 * g4 + 2] = q0 * c0 - q1 * d0 + q2 * a0 + q3 * b0;
                                v[4 * g4 + 3] = q0 * d0 + q1 * c0 - q2 * b0 + q3 * a0;
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int d = perm4(e);
                                v[e] = bf16_bits_to_f32((rw[d >> 1] >> (16 * (d & 1))) & 0xffffu);
                            }
                        }
#pragma unroll
                        for (int k = 0; k < 4; ++k) w[k] = X::KB ? rw[k] : f32x2_to_h2(v[2 * k], v[2 * k + 1]);   // bf16 K: bf16 query as it is
                        if constexpr (X::QHL) {
                            // the fp16 remainder of the transformed query
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const float2 f = h2_to_f32x2(w[k]);
                                wl[k] = f32x2_to_h2(v[2 * k] - f.x, v[2 * k + 1] - f.y);
                            }
                        }
                    }
                    *reinterpret_cast<uint4*>(qsm + a * 2048 + sw_off(n, cc)) = make_uint4(w[0], w[1], w[2], w[3]);
                    if constexpr (X::QHL)
                        *reinterpret_cast<uint4*>(qsm + a * 2048 + sw_off(8 + n, cc)) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
                }
                // 1152 * (sum of the fp16 query over each 64-dim group): thread -> (head, D / TPH dims)
                constexpr int TPH = 128 / QH, DPT = D / TPH, TPG = 64 / DPT;
                const int h = r / TPH, s0 = (r % TPH) * DPT;
                float part = 0.0f;
                if (h < G) {
                    const uint16_t* qrow = p.q + qrow_index<VW>(p, pc.b, kvh, gv0 + h) * D + s0;
                    for (int d = 0; d < DPT; ++d)
                        part += __half2float(__float2half_rn(bf16_bits_to_f32(qrow[d])));
                }
#pragma unroll
                for (int off = 1; off < TPG; off <<= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
                // only the int8 K' carries the 1152 offset
                constexpr bool KI8 = !X::ISO && !X::KQ && !X::KB;
                if (h < G && (r % TPH) % TPG == 0) bias_s[(s0 / 64) * QH + h] = KI8 ? 1152.0f * part : 0.0f;
            }
            fence_proxy_async();
            soft_sync();
            if (r == 0) mbar_arrive(&bars[B_QRD]);
            // the offset sums in registers (16 columns: read from shared memory each tile, for room)
            constexpr int GB = G > 8 ? 1 : G;
            float bias[NA][GB];
#pragma unroll
            for (int g = 0; g < NA; ++g)
#pragma unroll
                for (int h = 0; h < GB; ++h) bias[g][h] = bias_s[g * QH + h];

            float m[G], l[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                m[h] = -INFINITY;
                l[h] = 0.0f;
            }
            int E = 1000;   // range exponent of the frame ("unset")
            for (int pg0 = pc.p0, t = 0; pg0 < pc.p1; pg0 += kTP, ++t, ++T) {
                const int npg = min(kTP, pc.p1 - pg0);
                const int buf = T & 1;
                const uint32_t ph = (T >> 1) & 1;
                const int jpage = r >> 4;
                const int pos = (pg0 + jpage) * kPage + (r & 15);
                const bool valid = jpage < npg && pos < pc.L;
                // ---- scores ----
                float ks[X::NKG];
                if constexpr (X::KB) {
#pragma unroll
                    for (int g = 0; g < X::NKG; ++g) ks[g] = 1.0f;   // the bf16 K carries no scale
                } else {
                    const int kb = X::KSTB == 2 ? buf : 0;
                    wait_or_flag(&bars[B_KF + kb], (X::KSTB == 2 ? T >> 1 : T) & 1);
                    // one fp16 scale per group (ISO4 rows carry 2 reserved bytes after each)
                    const uint16_t* ksr = reinterpret_cast<const uint16_t*>(sm + X::OFF_KSC + (kb * kTP + jpage) * X::SC_B +
                                                                            (r & 15) * X::KSROW);
#pragma unroll
                    for (int g = 0; g < X::NKG; ++g) ks[g] = f16_bits_to_f32(ksr[g * (X::ISO ? X::ISO_SB / 2 : 1)]);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[B_KE + kb]);
                }
                wait_or_flag(&bars[B_QKD + buf], ph);
                tc_fence_after();
                float s[G];
#pragma unroll
                for (int h = 0; h < G; ++h) s[h] = 0.0f;
                const uint32_t sbuf = tmem + lb + X::SCOL + (T % X::NSB) * X::SBUF;
#pragma unroll
                for (int g = 0; g < X::NKG; ++g) {
                    float v[16];
                    tmem_ld16(sbuf + 16 * X::SACC * g, v);
                    if constexpr (X::KQ) {
                        // hi + lo columns of the rotated query; exact codes q - 8, the block's scale
#pragma unroll
                        for (int h = 0; h < G; ++h) s[h] += ks[g] * (v[h] + v[8 + h]);
                    } else if constexpr (X::ISO) {
                        // hi + lo columns of the even k-steps, then of the odd ones
                        float v2[16];
                        tmem_ld16(sbuf + 16 * X::SACC * g + 16, v2);
#pragma unroll
                        for (int h = 0; h < G; ++h) s[h] += ks[g] * ((v[h] + v[8 + h]) + (v2[h] + v2[8 + h]));
                    } else {
#pragma unroll
                        for (int h = 0; h < G; ++h) s[h] += ks[g] * (v[h] - (G > 8 ? bias_s[g * QH + h] : bias[g][h < GB ? h : 0]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_SF + T % X::NSB]);
#pragma unroll
                for (int h = 0; h < G; ++h) s[h] = valid ? s[h] * p.scale_log2 : -INFINITY;
                // a verify window: query w sees positions < L - W + w + 1, so the last W - 1 rows
                // of the sequence are hidden from the columns of the earlier queries
                if (VW && valid && pos > pc.L - p.W) {
                    // columns of queries w < pos - (L - W) do not see pos: virtual heads below hmin
                    const int hmin = (pos - (pc.L - p.W)) * p.Gtot - gv0;
#pragma unroll
                    for (int h = 0; h < G; ++h)
                        if (h < hmin) s[h] = -INFINITY;
                }
                // ---- V scales ----
                float vsf[X::VG];
                int e_row = 0;
                if constexpr (!X::VB) wait_or_flag(&bars[B_VF + buf], ph);
                if constexpr (VQ || X::VB || VFOLD) {
                    // the q4 block scales (and the int8 scales with 16 columns) are folded into V' by
                    // the converters; the bf16 V has none
#pragma unroll
                    for (int g = 0; g < X::VG; ++g) vsf[g] = 1.0f;
                    e_row = 15;   // the fp16 exponent field of 1.0
                } else {
                    const uint8_t* vsr = sm + X::OFF_VSC + (buf * kTP + jpage) * X::VSC_B + (r & 15) * X::VSROW;
#pragma unroll
                    for (int g = 0; g < X::VG; ++g) {
                        const uint32_t hb = reinterpret_cast<const uint16_t*>(vsr)[g * (X::ISO ? X::ISO_SB / 2 : 1)];
                        vsf[g] = f16_bits_to_f32(hb);
                        e_row = max(e_row, (int)((hb & 0x7fffu) >> 10));
                    }
                }
                if constexpr (!X::VB) {   // the bf16 V tile is released by the PV commit
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[B_VE + buf]);
                }
                if (!valid) e_row = 0;
                // ---- frame: all 128 threads agree on the max and the range exponent ----
                bool need = false;
#pragma unroll
                for (int h = 0; h < G; ++h) need |= s[h] > m[h] + 8.0f;
                need |= valid && (20 - max(e_row, 1)) < E;
                const unsigned any_w = __ballot_sync(0xffffffffu, need);
                if (lane == 0) red_flag[buf * 4 + warp] = any_w != 0;
                soft_sync();
                const bool any = (red_flag[buf * 4] | red_flag[buf * 4 + 1] | red_flag[buf * 4 + 2] | red_flag[buf * 4 + 3]) != 0;
                bool rescale = false;
                float fac[QH];
#pragma unroll
                for (int h = 0; h < QH; ++h) fac[h] = 1.0f;
                if (any) {
#pragma unroll
                    for (int o8 = 0; o8 < QH / 8; ++o8) {   // head octets
                        float v8[8];
#pragma unroll
                        for (int h = 0; h < 8; ++h) v8[h] = 8 * o8 + h < G ? s[8 * o8 + h < G ? 8 * o8 + h : 0] : -INFINITY;
                        const float wm = warp_reduce8<true>(v8, lane);
                        if ((lane & 3) == 0 && 8 * o8 + (lane >> 2) < G)
                            red_m[buf * 4 * QH + warp * QH + 8 * o8 + (lane >> 2)] = wm;
                    }
                    const int ew = __reduce_max_sync(0xffffffffu, (unsigned)e_row);
                    if (lane == 0) red_e[buf * 4 + warp] = ew;
                    soft_sync();
                    const int et = max(max(red_e[buf * 4], red_e[buf * 4 + 1]), max(red_e[buf * 4 + 2], red_e[buf * 4 + 3]));
                    const int Enew = min(E, 20 - max(et, 1));
                    const float ef = (E == 1000) ? 1.0f : exp2i(Enew - E);
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float* rm = red_m + buf * 4 * QH + h;
                        const float M = fmaxf(fmaxf(rm[0], rm[QH]), fmaxf(rm[2 * QH], rm[3 * QH]));
                        const float mn = (M > m[h] + 8.0f) ? M : m[h];
                        const float alpha = (m[h] == -INFINITY) ? 0.0f : (mn == m[h] ? 1.0f : fast_exp2(m[h] - mn));
                        l[h] *= alpha;
                        fac[h] = alpha * ef;
                        m[h] = mn;
                    }
                    rescale = t > 0;
                    E = Enew;
                }
                // ---- probabilities ----
                float pr[G];
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    // (a verify column can be hidden from every row of a tile before its frame is set)
                    pr[h] = (VW ? s[h] != -INFINITY : valid) ? fast_exp2(s[h] - m[h]) : 0.0f;
                    l[h] += pr[h];
                }
                // ---- P' (and the rare rescale of O) once PV of the previous tile is done ----
                if (T >= 1) wait_or_flag(&bars[B_PVD + ((T - 1) & 1)], ((T - 1) >> 1) & 1);
                tc_fence_after();
                // O rows 16 g + j (lane j of warp g: head j % 8, hi / lo) over the dims of group g;
                // ISO V groups are 128 dims, so warp g < VG owns 128 columns
                constexpr int OW = X::ISO ? X::VG : NA, OCW = X::ISO ? 128 : 64;
                if constexpr (VFOLD) {
                    // 16 columns: slot w (warp w) holds heads 8 (w & 1) + j; it is read over the dims
                    // [D / 2 (w >> 1), + D / 2) only, so those are the columns rescaled
                    if (rescale) {
                        const int hw = 8 * (warp & 1) + (lane & 7);
                        float f = fac[0];
#pragma unroll
                        for (int h = 1; h < QH; ++h) f = (hw == h) ? fac[h] : f;
#pragma unroll 1
                        for (int c4 = 0; c4 < D / 32; ++c4) {
                            float v[16];
                            const uint32_t ta = tmem + lb + X::OCOL + (D / 2) * (warp >> 1) + 16 * c4;
                            tmem_ld16(ta, v);
#pragma unroll
                            for (int j = 0; j < 16; ++j) v[j] *= f;
                            tmem_st16(ta, v);
                        }
                    }
                } else if (rescale && warp < OW) {
                    float f = fac[0];
#pragma unroll
                    for (int h = 1; h < 8; ++h) f = ((lane & 7) == h) ? fac[h] : f;
#pragma unroll 1
                    for (int c4 = 0; c4 < OCW / 16; ++c4) {
                        float v[16];
                        const uint32_t ta = tmem + lb + X::OCOL + OCW * warp + 16 * c4;
                        tmem_ld16(ta, v);
#pragma unroll
                        for (int j = 0; j < 16; ++j) v[j] *= f;
                        tmem_st16(ta, v);
                    }
                }
                {
                    const float e2 = (E == 1000) ? 1.0f : exp2i(E);
                    uint8_t* pp = sm + X::OFF_PP;
#pragma unroll
                    for (int g = 0; g < X::PG; ++g) {
                        uint32_t hw[4] = {0u, 0u, 0u, 0u}, lw[4] = {0u, 0u, 0u, 0u};
                        // (16 columns: every slot, since each carries all D dims of its octet)
                        if ((VFOLD || g < X::VG) && valid) {
                            const float sc = vsf[g < X::VG ? g : 0] * e2;
                            // 16 columns: slot g holds heads 8 (g & 1) + h (slots 2, 3 repeat 0, 1)
                            const int hb = G > 8 ? 8 * (g & 1) : 0;
                            float P[8];
#pragma unroll
                            for (int h = 0; h < 8; ++h) P[h] = hb + h < G ? pr[hb + h < G ? hb + h : 0] * sc : 0.0f;
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                if constexpr (X::VB) {
                                    // bf16 V': P' in bf16 hi + lo (the operands of one MMA share a type)
                                    __nv_bfloat162 hb = __floats2bfloat162_rn(P[2 * k], P[2 * k + 1]);
                                    const float2 f = __bfloat1622float2(hb);
                                    __nv_bfloat162 lb2 = __floats2bfloat162_rn(P[2 * k] - f.x, P[2 * k + 1] - f.y);
                                    hw[k] = *reinterpret_cast<uint32_t*>(&hb);
                                    lw[k] = *reinterpret_cast<uint32_t*>(&lb2);
                                } else {
                                    hw[k] = f32x2_to_h2(P[2 * k], P[2 * k + 1]);
                                    const float2 f = h2_to_f32x2(hw[k]);
                                    lw[k] = f32x2_to_h2(P[2 * k] - f.x, P[2 * k + 1] - f.y);
                                }
                            }
                        }
                        uint8_t* pa = pp + (g >> 2) * 16384;   // 64 P' columns (4 groups) per atom
                        *reinterpret_cast<uint4*>(pa + sw_off(r, 2 * (g & 3))) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        *reinterpret_cast<uint4*>(pa + sw_off(r, 2 * (g & 3) + 1)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                    }
                }
                fence_proxy_async();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_PFL]);
            }
            // ---- end of the piece: O out of TMEM, row sums, merge ----
            wait_or_flag(&bars[B_PVD + ((T - 1) & 1)], ((T - 1) >> 1) & 1);
            tc_fence_after();
            // row sums first, then O straight from TMEM to the output (or to the partial slot)
#pragma unroll
            for (int o8 = 0; o8 < QH / 8; ++o8) {   // head octets
                float v8[8];
#pragma unroll
                for (int h = 0; h < 8; ++h) v8[h] = 8 * o8 + h < G ? l[8 * o8 + h < G ? 8 * o8 + h : 0] : 0.0f;
                const float ws = warp_reduce8<false>(v8, lane);
                if ((lane & 3) == 0 && 8 * o8 + (lane >> 2) < G) red_l[warp * QH + 8 * o8 + (lane >> 2)] = ws;
            }
            soft_sync();
            if (r < G) {
                float mr = m[0];
#pragma unroll
                for (int h = 1; h < G; ++h) mr = (r == h) ? m[h] : mr;
                sML[r] = mr;
                sML[QH + r] = red_l[r] + red_l[QH + r] + red_l[2 * QH + r] + red_l[3 * QH + r];
            }
            soft_sync();
            const long long clo = cta_of(pc.soff), chi = cta_of(pc.soff + pc.np - 1);
            const int npieces = (int)(chi - clo + 1);
            const long long seg = (long long)pc.b * p.NH + pc.hg;
            float* mine = p.part1 + (size_t)(c + seg) * p.slot_floats;
            if constexpr (VQ) {
                // q4 V: O in the int8 layout (warp g: lanes h and 8 + h hold the hi and lo rows of
                // head h; P' is the same in every group, so warp g takes the dims of group g). The
                // rotated output goes per head to shared memory (the P' area is free), the inverse
                // rotation (FWHT-256 x 1/16, its own inverse) runs there, then the output or the
                // partial slot is written. The rotation is linear, so the merge of partial slots
                // commutes with it.
                float* ox = reinterpret_cast<float*>(sm + X::OFF_PP);   // [8 heads][D]
                {
                    const float e_inv = (E == 1000) ? 0.0f : exp2i(-E);
                    const float Lh = lane < G ? sML[QH + (lane < G ? lane : 0)] : 0.0f;
                    const float inv = npieces == 1 ? (Lh > 0.0f ? e_inv / Lh : 0.0f) : e_inv;
#pragma unroll 1
                    for (int c4 = 0; c4 < 4; ++c4) {
                        float v[16];
                        tmem_ld16(tmem + lb + X::OCOL + 64 * warp + 16 * c4, v);
#pragma unroll
                        for (int j = 0; j < 16; ++j) v[j] += __shfl_xor_sync(0xffffffffu, v[j], 8);
                        if (lane < G) {
                            const int d0 = 64 * warp + 16 * c4;
#pragma unroll
                            for (int j = 0; j < 16; ++j) ox[lane * D + d0 + perm4(j)] = v[j] * inv;
                        }
                    }
                }
                soft_sync();
                const int hh = r >> 4, q = r & 15;   // thread (head, 16-dim slice)
                if (hh < G) {
                    // strides 16 .. 128: the dims q + 16 k
                    float x[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) x[k] = ox[hh * D + q + 16 * k];
#pragma unroll
                    for (int st = 1; st < 16; st <<= 1)
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            if ((k & st) == 0) {
                                const float a0 = x[k], a1 = x[k + st];
                                x[k] = a0 + a1;
                                x[k + st] = a0 - a1;
                            }
#pragma unroll
                    for (int k = 0; k < 16; ++k) ox[hh * D + q + 16 * k] = x[k];
                }
                soft_sync();
                if (hh < G) {
                    // strides 1 .. 8: the dims 16 q + i
                    float y[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) y[i] = ox[hh * D + 16 * q + i];
#pragma unroll
                    for (int st = 1; st < 16; st <<= 1)
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if ((i & st) == 0) {
                                const float a0 = y[i], a1 = y[i + st];
                                y[i] = a0 + a1;
                                y[i + st] = a0 - a1;
                            }
#pragma unroll
                    for (int i = 0; i < 16; ++i) y[i] *= 0.0625f;
                    if (npieces == 1) {
#pragma unroll
                        {
                            const size_t orow = qrow_index<VW>(p, pc.b, kvh, gv0 + hh) * D;
#pragma unroll
                            for (int i = 0; i < 16; ++i) write_row(p, orow, 16 * q + i, y[i]);
                        }
                    } else {
                        float4* dst = reinterpret_cast<float4*>(mine + 2 * QH + hh * D + 16 * q);
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) dst[q4] = make_float4(y[4 * q4], y[4 * q4 + 1], y[4 * q4 + 2], y[4 * q4 + 3]);
                    }
                }
            } else if constexpr (VFOLD) {
                // 16 columns: slot w (warp w) holds heads 8 (w & 1) + j, hi in lane j, lo in lane 8 + j,
                // each over all D dims (V' carries the scales); warp w writes the dims
                // [D / 2 (w >> 1), + D / 2) of its heads, in converter order inside each aligned 4
                const int head = 8 * (warp & 1) + (lane & 7);
                const float e_inv = (E == 1000) ? 0.0f : exp2i(-E);
                const float Lh = sML[QH + head];
                const float inv = npieces == 1 ? (Lh > 0.0f ? e_inv / Lh : 0.0f) : e_inv;
                const size_t orow = qrow_index<VW>(p, pc.b, kvh, gv0 + head) * D;
#pragma unroll 1
                for (int c4 = 0; c4 < D / 32; ++c4) {
                    float v[16];
                    const int d0 = (D / 2) * (warp >> 1) + 16 * c4;
                    tmem_ld16(tmem + lb + X::OCOL + d0, v);
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] += __shfl_xor_sync(0xffffffffu, v[j], 8);
                    if (lane < 8 && head < G) {
                        float o[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) o[perm4(j)] = v[j] * inv;
                        if (npieces == 1) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) write_row(p, orow, d0 + j, o[j]);
                        } else {
                            float4* dst = reinterpret_cast<float4*>(mine + 2 * QH + head * D + d0);
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) dst[q4] = make_float4(o[4 * q4], o[4 * q4 + 1], o[4 * q4 + 2], o[4 * q4 + 3]);
                        }
                    }
                }
            } else if (warp < (X::ISO ? X::VG : NA)) {
                // warp g: lanes h and 8 + h hold the hi and lo rows of head h over the dims of group g
                // (64 dims in converter order for int8; 128 dims in natural order for ISO, where each
                // 4-D group is rotated back: conj(q) (x) o)
                constexpr int OCW = X::ISO ? 128 : 64;
                const float e_inv = (E == 1000) ? 0.0f : exp2i(-E);
                const float Lh = lane < G ? sML[QH + lane] : 0.0f;
                const float inv = npieces == 1 ? (Lh > 0.0f ? e_inv / Lh : 0.0f) : e_inv;
                const size_t orow = qrow_index<VW>(p, pc.b, kvh, gv0 + (lane < G ? lane : 0)) * D;
#pragma unroll 1
                for (int c4 = 0; c4 < OCW / 16; ++c4) {
                    float v[16];
                    tmem_ld16(tmem + lb + X::OCOL + OCW * warp + 16 * c4, v);
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] += __shfl_xor_sync(0xffffffffu, v[j], 8);
                    if (lane < G) {
                        const int d0 = OCW * warp + 16 * c4;
                        float o[16];
                        if constexpr (X::ISO) {
                            const float q0 = p.quat[0], q1 = p.quat[1], q2 = p.quat[2], q3 = p.quat[3];
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const float a0 = v[4 * k], b0 = v[4 * k + 1], c0 = v[4 * k + 2], dd = v[4 * k + 3];
                                o[4 * k] = (q0 * a0 + q1 * b0 + q2 * c0 + q3 * dd) * inv;
                                o[4 * k + 1] = (q0 * b0 - q1 * a0 - q2 * dd + q3 * c0) * inv;
                                o[4 * k + 2] = (q0 * c0 + q1 * dd - q2 * a0 - q3 * b0) * inv;
                                o[4 * k + 3] = (q0 * dd - q1 * c0 + q2 * b0 - q3 * a0) * inv;
                            }
                        } else if constexpr (X::VB) {
                            // the bf16 V' holds dims in natural order
#pragma unroll
                            for (int j = 0; j < 16; ++j) o[j] = v[j] * inv;
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j) o[perm4(j)] = v[j] * inv;
                        }
                        if (npieces == 1) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) write_row(p, orow, d0 + j, o[j]);
                        } else {
                            float4* dst = reinterpret_cast<float4*>(mine + 2 * QH + lane * D + d0);
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) dst[q4] = make_float4(o[4 * q4], o[4 * q4 + 1], o[4 * q4 + 2], o[4 * q4 + 3]);
                        }
                    }
                }
            }
            tc_fence_before();
            if (npieces > 1 && r < G) {
                // the partial slot's frame and row sum; the combine kernel merges the segment's slots
                mine[r] = sML[r];
                mine[QH + r] = sML[QH + r];
            }
            soft_sync();
            ++piece;
        }
    }

    // ---------------- tear-down ----------------
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWMma) tmem_dealloc(tmem, X::TCOLS);
}

// ---------------------------------------------------------------------------
// combine: merge the partial slots of every segment split across CTAs.
// Grid (G * D / 64, R): block (s, y) merges output floats [64 s, 64 s + 64) of
// one segment -- segment y when there are no more segments than decode CTAs,
// else the multi-piece segment that decode CTA y closes (if any) -- with the
// partial-softmax rule M = max m_j, O = sum 2^(m_j - M) O_j / sum 2^(m_j - M) l_j
// (base-2 scores). Which CTAs hold the segment's pieces follows from seq_lens
// alone (the decode grid's split is a pure function of it), so it is worked
// out before the dependency wait and the merge needs one round of loads after it.
// ---------------------------------------------------------------------------
constexpr int kCombThr = 128;
constexpr int kMaxGrid = 256;   // decode CTAs (pieces of one segment) the combine step can merge
constexpr int kMaxBatchDec = 1024;

template <int D, int G, bool VW>
__global__ void __launch_bounds__(kCombThr) decode_tc_combine(const DecodeParams p) {
    __shared__ float s_w[kMaxGrid], s_l[kMaxGrid];
    __shared__ float4 s_acc[8][16];
    __shared__ float s_red[8];
    __shared__ long long s_pref[kMaxBatchDec + 1];   // pages of the sequences before b
    __shared__ long long s_wsum[kCombThr / 32];
    __shared__ int s_info[6];
    const int t = threadIdx.x;
    // The next kernel in the stream may be scheduled now: it does its own set-up while this
    // grid waits, and waits for this grid to complete before it reads anything.
    asm volatile("griddepcontrol.launch_dependents;");
    // ---- before the dependency wait: the segment and its pieces, from seq_lens (an input
    // of the decode grid that it does not write) ----
    {
        const int per = (p.B + kCombThr - 1) / kCombThr;
        const int b_lo = min(p.B, t * per), b_hi = min(p.B, b_lo + per);
        long long loc = 0;
        for (int b = b_lo; b < b_hi; ++b) loc += (seq_len_clamped(p, b) + kPage - 1) / kPage;
        long long incl = loc;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const long long v = __shfl_up_sync(0xffffffffu, incl, off);
            if ((t & 31) >= off) incl += v;
        }
        if ((t & 31) == 31) s_wsum[t >> 5] = incl;
        __syncthreads();
        long long pref = incl - loc, total = 0;
        for (int w = 0; w < kCombThr / 32; ++w) {
            if (w < (t >> 5)) pref += s_wsum[w];
            total += s_wsum[w];
        }
        for (int b = b_lo; b < b_hi; ++b) {
            s_pref[b] = pref;
            pref += (seq_len_clamped(p, b) + kPage - 1) / kPage;
        }
        if (t == 0) s_pref[p.B] = total;
        __syncthreads();
        if (t == 0) {
            const long long Tunits = total * p.NH, C = p.ctas;
            auto cta_of = [&](long long x) -> long long { return ((x + 1) * C + Tunits - 1) / Tunits - 1; };
            int n = 0, clo = 0, seg = 0, hg = 0, b = 0;
            if (p.rec_by_seg) {
                seg = blockIdx.y;
                b = seg / p.NH;
                hg = seg % p.NH;
                const long long np = s_pref[b + 1] - s_pref[b];
                if (np > 0) {
                    const long long soff = s_pref[b] * p.NH + hg * np;
                    clo = (int)cta_of(soff);
                    n = (int)(cta_of(soff + np - 1) - clo + 1);
                }
            } else if (Tunits > 0) {
                // the segment holding this CTA's first unit, if it started in an earlier CTA and
                // ends in this one (a CTA closes at most one multi-piece segment)
                const long long c = blockIdx.y, beg = Tunits * c / C, end = Tunits * (c + 1) / C;
                if (beg < end) {
                    int lo = 0, hi = p.B - 1;   // first b with s_pref[b + 1] * NH > beg
                    while (lo < hi) {
                        const int mid = (lo + hi) >> 1;
                        if (s_pref[mid + 1] * p.NH > beg) hi = mid;
                        else lo = mid + 1;
                    }
                    b = lo;
                    const long long np = s_pref[b + 1] - s_pref[b];
                    hg = (int)((beg - s_pref[b] * p.NH) / np);
                    const long long soff = s_pref[b] * p.NH + (long long)hg * np;
                    if (soff < beg && soff + np <= end) {
                        clo = (int)cta_of(soff);
                        n = (int)(c - clo + 1);
                        seg = b * p.NH + hg;
                    }
                }
            }
            const int kvh = hg / (p.Gv / G), hgi = hg % (p.Gv / G);
            s_info[0] = n;
            s_info[1] = clo;
            s_info[2] = seg;
            s_info[3] = b;
            s_info[4] = hgi * G;
            s_info[5] = kvh;
        }
        __syncthreads();
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the decode grid has completed
    const int n = s_info[0];
    if (n < 2) return;
    const int clo = s_info[1], seg = s_info[2], b = s_info[3], gv0 = s_info[4], kvh = s_info[5];
    const int s = blockIdx.x;
    const int f0 = 64 * s, h = f0 / D;
    auto slot = [&](int j) { return p.part1 + (size_t)(clo + j + seg) * p.slot_floats; };
    constexpr int ML = G > 8 ? 16 : 8;   // m[ML], l[ML], then O
    // O loads first (independent of the weights): thread -> float4 e, slots j = sg, sg + 8, ...
    const int e = t & 15, sg = t >> 4;
    float4 v[20];
#pragma unroll
    for (int k = 0; k < 20; ++k) {
        const int j = sg + 8 * k;
        v[k] = j < n ? *reinterpret_cast<const float4*>(slot(j) + 2 * ML + f0 + 4 * e) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float mloc = -INFINITY;
    for (int j = t; j < n; j += kCombThr) {
        const float mj = slot(j)[h];
        s_w[j] = mj;
        s_l[j] = slot(j)[ML + h];
        mloc = fmaxf(mloc, mj);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, off));
    if ((t & 31) == 0) s_red[t >> 5] = mloc;
    __syncthreads();
    const float M = fmaxf(fmaxf(s_red[0], s_red[1]), fmaxf(s_red[2], s_red[3]));
    float lloc = 0.0f;
    for (int j = t; j < n; j += kCombThr) {
        const float w = s_w[j] == -INFINITY ? 0.0f : exp2f(s_w[j] - M);
        s_w[j] = w;
        lloc += w * s_l[j];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lloc += __shfl_xor_sync(0xffffffffu, lloc, off);
    __syncthreads();
    if ((t & 31) == 0) s_red[4 + (t >> 5)] = lloc;
    __syncthreads();
    const float L = s_red[4] + s_red[5] + s_red[6] + s_red[7];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 20; ++k) {
        const int j = sg + 8 * k;
        if (j < n) {
            const float w = s_w[j];
            acc.x += w * v[k].x;
            acc.y += w * v[k].y;
            acc.z += w * v[k].z;
            acc.w += w * v[k].w;
        }
    }
    for (int j = sg + 160; j < n; j += 8) {   // segments split over more than 160 CTAs
        const float w = s_w[j];
        const float4 x = *reinterpret_cast<const float4*>(slot(j) + 2 * ML + f0 + 4 * e);
        acc.x += w * x.x;
        acc.y += w * x.y;
        acc.z += w * x.z;
        acc.w += w * x.w;
    }
    s_acc[sg][e] = acc;
    __syncthreads();
    if (t < 64) {
        const int q = t >> 2, c4 = t & 3;   // float4 q, component c4
        float a = 0.0f;
#pragma unroll
        for (int g2 = 0; g2 < 8; ++g2) {
            const float4 x = s_acc[g2][q];
            a += c4 == 0 ? x.x : c4 == 1 ? x.y : c4 == 2 ? x.z : x.w;
        }
        write_out<D, G, VW>(p, b, kvh, gv0, f0 + 4 * q + c4, L > 0.0f ? a / L : 0.0f);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
cudaError_t decode_tc_upload_levels(const float* lv3, const float* lv4) {
    float lv[2][16] = {}, mid[2][16] = {};
    for (int j = 0; j < 8; ++j) lv[0][j] = lv3[j];
    for (int j = 0; j < 16; ++j) lv[1][j] = lv4[j];
    for (int j = 0; j < 7; ++j) mid[0][j] = (lv3[j] + lv3[j + 1]) * 0.5f;
    for (int j = 0; j < 15; ++j) mid[1][j] = (lv4[j] + lv4[j + 1]) * 0.5f;
    cudaError_t e = cudaMemcpyToSymbol(c_tc_levels, lv, sizeof(lv));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(c_tc_mids, mid, sizeof(mid));
}

// query columns of a head group: up to 8 (16 for int8: the Q K^T tile has N = 16 columns, and
// with the V scales folded into V' the PV tile holds 16 heads hi + lo)
int decode_heads_per_cta(int Gv, int fmt) {
    if (fmt == 0 && Gv % 16 == 0) return 16;
    for (int G = 8; G > 1; G >>= 1)
        if (Gv % G == 0) return G;
    return 1;
}
int decode_max_batch() { return kMaxBatchDec; }

cudaError_t decode_tc_read_error(unsigned* out, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_err_dtc, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    unsigned z = 0;
    return cudaMemcpyToSymbol(g_err_dtc, &z, sizeof(unsigned));
}

// Both kernels are launched with programmatic stream serialization: each may
// start while its predecessor in the stream drains, and waits for it
// (griddepcontrol.wait) before touching memory.
template <int D, int G, int FMT, bool VW>
static cudaError_t launch_tc(int grid, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p_in,
                             cudaStream_t st) {
    DecodeParams p = p_in;
    p.rec_by_seg = (long long)p.B * p.NH <= grid;
    p.ctas = grid;
    using X = TG<D, FMT>;
    auto fn = decode_tc_kernel<D, G, FMT, VW>;
    static bool configured[kMaxDevices];   // this instantiation's attribute, per device
    {
        cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(fn), X::SMEM + 1024, configured);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThr);
    cfg.dynamicSmemBytes = X::SMEM + 1024;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, fn, tk, tv, p);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(G * D / 64, p.rec_by_seg ? p.B * p.NH : grid);
    cfg.blockDim = dim3(kCombThr);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, decode_tc_combine<D, G, VW>, p);
}

template <int D, int FMT, bool VW = false>
static cudaError_t launch_tc_g(int G, int grid, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                               cudaStream_t st) {
    if constexpr (FMT == 0 && !VW)   // a verify window (int8): its own instantiations
        if (p.W > 1) return launch_tc_g<D, FMT, true>(G, grid, tk, tv, p, st);
    switch (G) {
        case 1: return launch_tc<D, 1, FMT, VW>(grid, tk, tv, p, st);
        case 2: return launch_tc<D, 2, FMT, VW>(grid, tk, tv, p, st);
        case 4: return launch_tc<D, 4, FMT, VW>(grid, tk, tv, p, st);
        case 8: return launch_tc<D, 8, FMT, VW>(grid, tk, tv, p, st);
        case 16:
            if constexpr (FMT == 0) return launch_tc<D, 16, FMT, VW>(grid, tk, tv, p, st);
            break;
    }
    return cudaErrorInvalidValue;
}

// fmt: 0 int8 (head_dim 128 or 256), 1 k8v4 (256), 2 ISO3 and 3 ISO4 (128 or 256), 4 q4 (256),
// 5 int8 K + bf16 V and 6 bf16 K + int8 V (128 or 256); the
// tensor maps are used for int8 and q4 code planes only
cudaError_t decode_tc_launch(int D, int G, int grid, int fmt, const CUtensorMap& tk, const CUtensorMap& tv,
                             const DecodeParams& p, cudaStream_t st) {
    grid = grid < kMaxGrid ? grid : kMaxGrid;
    if (fmt == 1) return D == 256 ? launch_tc_g<256, 1>(G, grid, tk, tv, p, st) : cudaErrorInvalidValue;
    if (fmt == 4) return D == 256 ? launch_tc_g<256, 4>(G, grid, tk, tv, p, st) : cudaErrorInvalidValue;
    if (D != 128 && D != 256) return cudaErrorInvalidValue;
    switch (fmt) {
        case 0: return D == 256 ? launch_tc_g<256, 0>(G, grid, tk, tv, p, st) : launch_tc_g<128, 0>(G, grid, tk, tv, p, st);
        case 5: return D == 256 ? launch_tc_g<256, 5>(G, grid, tk, tv, p, st) : launch_tc_g<128, 5>(G, grid, tk, tv, p, st);
        case 6: return D == 256 ? launch_tc_g<256, 6>(G, grid, tk, tv, p, st) : launch_tc_g<128, 6>(G, grid, tk, tv, p, st);
        case 2: return D == 256 ? launch_tc_g<256, 2>(G, grid, tk, tv, p, st) : launch_tc_g<128, 2>(G, grid, tk, tv, p, st);
        case 3: return D == 256 ? launch_tc_g<256, 3>(G, grid, tk, tv, p, st) : launch_tc_g<128, 3>(G, grid, tk, tv, p, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace qkv
