// Decode attention over a paged KV cache, split-K partitions and their
// log-sum-exp merge, for sm_103a.
//
// The math: for one query token, s_t = scale * <q, K_t>, out = softmax(s) V
// (tutorial chapter 12, Attention(Q_t, K_1:t, V_1:t)), with the streaming
// online softmax m_new = max(m, rowmax S), l = e^(m - m_new) l + rowsum P,
// O = e^(m - m_new) O + P V, one division at the end (vLLM deep dive 06,
// FlashAttention ③).  Long contexts are cut into KV partitions that run on
// different SMs and are merged with the same rescale rule (Flash-Decoding, ⑥;
// LLM-101-CN "推理优化" combine_result).
//
// Kernel design (GB300):
//  * One CTA per (KV head, sequence, partition).  Warp 4 is the producer: one
//    lane issues 4-D TMA tensor loads of 16-token tiles of K and V straight
//    from the paged cache, the physical block id from the block table being
//    the outermost coordinate, into a ring of shared-memory stages guarded by
//    mbarriers.  Warps 0-3 consume stage i = w (mod 4) each.
//  * Per 16-token stage a consumer computes S^T = K Q^T on the tensor cores
//    (mma.sync m16n8k16, M = 16 tokens, N = 8 query heads of the GQA group,
//    K = 16 dims), the online-softmax update in fp32, and O^T += V^T P^T
//    (M = 16 dims, N = 8 heads, K = 16 tokens).  P enters the second product
//    as two 16-bit terms (hi + lo) so the weights keep ~16 significant bits;
//    a single 16-bit P would break the attention tolerance for short contexts.
//    movmatrix turns the S^T fragments into P^T operand fragments in registers.
//  * Every wait on an mbarrier is bounded by %globaltimer: on expiry the CTA
//    flags PKV_EFLAG_TIMEOUT, drains its own TMA copies and returns.
//  * Bad block ids are flagged and their tokens skipped; tokens at or past the
//    context length are masked (their scores are -inf and their V rows are
//    zeroed in registers, so garbage in unused slots never reaches the output).
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <mutex>
#include <type_traits>

#include <cuda_fp8.h>
#include <cudaTypedefs.h>

#include "pkv_common.cuh"
#include "pkv_ptx.cuh"

namespace pkv {

constexpr int kStageTokens = 16;      // tokens per pipeline stage
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxChunkPages = 128;   // pages per partition (block-table slice in smem)
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait before giving up

// Shared-memory geometry of a decode stage: K then V of 16 tokens, as 128-byte
// swizzled rows per column block (64 dims of a 16-bit cache, 128 of an E4M3 one).
template <int D, bool F8 = false>
struct Tile {
    static constexpr int kElemBytes = F8 ? 1 : 2;
    static constexpr int kRegionElems = 128 / kElemBytes;     // elements per 128-byte row
    static constexpr int kRegions = D / kRegionElems;         // column blocks
    static constexpr int kRegionBytes = kStageTokens * 128;   // 16 rows of 128 bytes, swizzled
    static constexpr int kHalfBytes = kRegions * kRegionBytes;  // K (or V) of one stage
    static constexpr int kStageBytes = 2 * kHalfBytes;
    // Ring depth: 64 KB (three CTAs an SM); 48 KB for E4M3 stages, whose
    // kernel (at one 8-column group) holds four CTAs an SM to hide the longer
    // per-stage arithmetic behind more warps.
    static constexpr int kStages = (F8 ? 49152 : 65536) / kStageBytes;
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kSmemBytes = 1024 /*align*/ + kRingBytes + 2 * kStages * 8 +
                                      (kMaxChunkPages + 1) * 4 + 16;
};

// Shared-memory q tile of the two-group (NT = 2) 16-bit kernels: the CTA's
// 16 query columns x D dims, rows of D * 2 bytes with the 16-byte chunks
// XOR-swizzled by the row (column) index mod 8, plus alignment slack.  Each
// k-step's B fragments come from it by one ldmatrix just before the S^T
// products, instead of 32 registers a thread holding q all along: that took
// the GQA-16 kernel's register spills to none and the multi-query one's from
// 100 to 32 bytes (Llama-70B layer verifying 4 tokens, 32 rows: 54.9 -> 57.8 %
// of peak; 17 rows on the Llama-7B layer 63.4 -> 67.0 %).
template <int D, int NT, bool F8>
constexpr int q_tile_bytes() { return (NT == 2 && !F8) ? 128 + NT * 8 * D * 2 : 0; }

struct DecodeParams {
    void* out;
    const void* q;
    const int32_t* block_tables;
    const int32_t* context_lens;
    float* partial_o;    // [B][H_q][num_splits][D] when num_splits > 1
    float* partial_lse;  // [B][H_q][num_splits]
    const void* k_new;     // nullable: fused append of one new token per sequence ([B][H_kv][D])
    const void* v_new;
    float k_scale;         // E4M3 cache: the fused append stores E4M3(k / k_scale) (v: v_scale)
    void* k_cache;         // the caches, for the fused append's stores
    void* v_cache;
    const int2* seq_info;  // nullable: per sequence (shared-prefix tokens, prefix partials written)
    const int2* items;     // nullable: compact list of (unit b*H_kv+g, partition); CTA x takes item x
    const int* item_count;
    int32_t* err_flag;
    int max_blocks_per_seq;
    int num_blocks;
    int block_size;
    int num_q_heads;
    int group;           // query heads per KV head
    int num_splits;
    int chunk_tokens;    // tokens per partition (a multiple of 16)
    int num_kv_heads;
    int max_context_len;
    bool hnd;            // head-major cache layout
    float scale_log2;    // scale * log2(e) (times the K scale of an E4M3 cache)
    float v_scale;       // value of one V unit: 1, or the V scale of an E4M3 cache
    int q_len;           // > 0 (multi-query): columns are (query token, head), causal
    int row_blocks;      // multi-query: CTAs per (sequence, KV head), NT * 8 rows each
    // nullable (shared-prefix calls): per unit (sequence, KV head), the partials
    // still to be written; the CTA that writes a unit's last one merges its rows
    int* unit_left;
};

// Context length of sequence b as the kernels use it: negative or too long
// values are clamped (and flagged by the decode kernel).
__device__ __forceinline__ int clamped_len(int n, int cap) { return n < 0 ? 0 : (n > cap ? cap : n); }

// Partitions of a sequence's suffix of `suffix` tokens (the whole context
// without a shared prefix): partition j covers tokens [j*C, (j+1)*C) of it, C
// = chunk_tokens.  Without a shared prefix (slot0 == 0) an empty context still
// gets one partition, whose CTA writes the zero row; after a prefix, an empty
// suffix has none.
__device__ __forceinline__ int suffix_partitions(int suffix, int slot0, int chunk) {
    if (suffix == 0) return slot0 > 0 ? 0 : 1;
    return (suffix + chunk - 1) / chunk;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, __nv_bfloat16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi, __half) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float2 unpack2(uint32_t x, __nv_bfloat16) {
    return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&x));
}
__device__ __forceinline__ float2 unpack2(uint32_t x, __half) {
    return __half22float2(*reinterpret_cast<__half2*>(&x));
}

// 16-token box of K or V for KV head g at token offset toff of block blk,
// 64-dim region starting at dim c0, in either cache layout.
__device__ __forceinline__ void load_kv_box(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int g, int toff, int blk, bool hnd,
                                            uint64_t policy) {
    if (hnd)
        ptx::tma_load_4d(dst, map, bar, c0, toff, g, blk, policy);
    else
        ptx::tma_load_4d(dst, map, bar, c0, g, toff, blk, policy);
}

// Bounded wait on an mbarrier phase.  Returns false (after raising the CTA's
// abort flag and the device error bit on expiry) if the phase did not complete.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           int32_t* err_flag,
                                           uint64_t limit_ns = kWaitLimitNs) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer() - t0 > limit_ns) {
            *abort_flag = 1;
            flag_error(err_flag, PKV_EFLAG_TIMEOUT);
            return false;
        }
    }
}

#ifdef PKV_DEBUG
// Debug builds (-DPKV_DEBUG) fill ring slots with all-ones bytes, a NaN in
// fp16, bf16 and E4M3 alike, whenever their contents stop being valid: the
// whole ring at the start, and each slot when its stage is released.  A read
// of a slot whose copy has not landed, or of a stage already released, then
// turns the output to NaN instead of passing unnoticed.  `lanes` threads
// (lane index `lane`) share the fill; each makes its writes visible to the
// async proxy, which writes the slot next.
__device__ __forceinline__ void poison_smem(uint8_t* base, int bytes, int lane, int lanes) {
    for (int i = lane; i < bytes / 16; i += lanes)
        reinterpret_cast<uint4*>(base)[i] = make_uint4(~0u, ~0u, ~0u, ~0u);
    ptx::fence_proxy_async_smem();
}
#endif

// Two E4M3 codes (the first in the low byte) as a pair of T, exactly: every
// E4M3 value is an fp16 (and a bf16) value.
__device__ __forceinline__ uint32_t e4m3x2_to(uint32_t v, __half) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(v & 0xffffu), __NV_E4M3);
    return (uint32_t)h.x | ((uint32_t)h.y << 16);
}
__device__ __forceinline__ uint32_t e4m3x2_to(uint32_t v, __nv_bfloat16) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(v & 0xffffu), __NV_E4M3);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
    return pack2(f.x, f.y, __nv_bfloat16());
}

// Scores may exceed a column's softmax reference m by up to this much (base 2)
// before m is moved: e^(s - m) then stays at most 256, far inside fp32 and the
// 16-bit P terms.
constexpr float kLazyLog2 = 8.f;

// One 16-token stage of K and V, staged in shared memory (128-byte swizzled
// rows of 64 dims, K then V), against the query columns held in `qb`:
// S^T = K Q^T on the tensor cores, the base-2 online-softmax update of
// (m, l, O^T), and O^T = alpha * O^T + V^T P^T.  Columns are query rows (the
// heads of a GQA group, or rows of several sequences); `qb`, `o`, `m*`, `l*`
// hold, per 8-column group nt, columns nt*8 + 2*(lane%4) and +1.  Token i
// (0..15) of the stage takes part only when i < nvalid, and, with ROW_LIMITS,
// only for the columns c with tok0 + i < lim[nt][c]; V rows of tokens at
// i >= nvalid are zeroed in registers so unused slots never reach the output.
//
// F8: the stage holds E4M3 codes, one 128-byte row per token (128 dims).  An
// ldmatrix of 16-bit units then yields four consecutive dims of a token per
// register; converted to T pairs they feed the same products with the dims
// of each 16-dim block permuted (k-slots 2tq, 2tq+1 <- dims 4tq, 4tq+1 and
// 2tq+8, 2tq+9 <- 4tq+2, 4tq+3), which qb must follow.  For V, the transposed
// 16-bit units hold a pair of dims for two tokens; split into even and odd
// dims they make the A operand with the rows of each 16-dim block permuted
// (row r <- dim 2r for r < 8, dim 2(r-8)+1 for r >= 8): o comes out in that
// order.
template <typename T, int D, int NT, bool ROW_LIMITS, bool F8 = false, bool QS = false>
__device__ __forceinline__ void stage_update(uint32_t kbase, uint32_t vbase, int nvalid, int tok0,
                                             const int (&lim)[NT][2],
                                             const uint32_t (&qb)[NT][D / 16][2],
                                             float (&o)[NT][D / 16][4], float (&m0)[NT],
                                             float (&m1)[NT], float (&l0)[NT], float (&l1)[NT],
                                             float scale_log2, int lane, uint32_t qaddr = 0) {
    constexpr int KSTEPS = D / 16;
    constexpr int kRegionBytes = kStageTokens * 128;
    const int gq = lane >> 2;
    const int tq = lane & 3;
    // ldmatrix row offsets (the swizzle XORs the 16-byte chunk index with the
    // row index mod 8; rows here are tokens).
    const int mi = lane >> 3;
    const int r8 = lane & 7;
    const int k_tok = (mi & 1) * 8 + r8;   // K: matrices (t0-7,c), (t8-15,c), (t0-7,c+1), (t8-15,c+1)
    const int k_csel = mi >> 1;
    const int v_tok = (mi >> 1) * 8 + r8;  // V: matrices (t0-7,c), (t0-7,c+1), (t8-15,c), (t8-15,c+1)
    const int v_csel = mi & 1;

    // S^T = K Q^T
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) s[nt][c] = 0.f;
    if constexpr (F8) {
        static_assert(D == 128, "an E4M3 stage row holds 128 dims");
        // matrices: (tokens 0-7, block 2j), (8-15, 2j), (0-7, 2j+1), (8-15, 2j+1).
        // Odd 16-dim blocks accumulate apart (s2) to halve the dependent MMA chain.
        const int row = (mi & 1) * 8 + r8;
        float s2[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) s2[nt][c] = 0.f;
#pragma unroll
        for (int j = 0; j < D / 32; ++j) {
            const int chunk = 2 * j + (mi >> 1);
            uint32_t r[4];
            ptx::ldmatrix_x4(r, kbase + row * 128 + ((chunk ^ r8) << 4));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t a[4];
                a[0] = e4m3x2_to(r[2 * h], T());
                a[1] = e4m3x2_to(r[2 * h + 1], T());
                a[2] = e4m3x2_to(r[2 * h] >> 16, T());
                a[3] = e4m3x2_to(r[2 * h + 1] >> 16, T());
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    ptx::mma_16816<T>(h ? s2[nt] : s[nt], a, qb[nt][2 * j + h][0],
                                      qb[nt][2 * j + h][1]);
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) s[nt][c] += s2[nt][c];
    } else {
        // odd k-steps accumulate apart (s2): two dependent MMA chains, not one
        float s2[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) s2[nt][c] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
            const int chunk = ks * 2 + k_csel;
            const uint32_t addr =
                kbase + (chunk >> 3) * kRegionBytes + k_tok * 128 + (((chunk & 7) ^ r8) << 4);
            uint32_t a[4];
            ptx::ldmatrix_x4(a, addr);
            if constexpr (QS) {
                static_assert(NT == 2, "the q tile serves two 8-column groups");
                // matrices (group 0, dims 16ks..+7), (0, +8..15), (1, ..), (1, ..):
                // lane's row = column (mi >> 1) * 8 + r8, chunk 2ks + (mi & 1)
                uint32_t qf[4];
                ptx::ldmatrix_x4(qf, qaddr + ((mi >> 1) * 8 + r8) * (D * 2) +
                                         (((2 * ks + (mi & 1)) ^ r8) << 4));
                ptx::mma_16816<T>((ks & 1) ? s2[0] : s[0], a, qf[0], qf[1]);
                ptx::mma_16816<T>((ks & 1) ? s2[1] : s[1], a, qf[2], qf[3]);
            } else {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    ptx::mma_16816<T>((ks & 1) ? s2[nt] : s[nt], a, qb[nt][ks][0], qb[nt][ks][1]);
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) s[nt][c] += s2[nt][c];
    }

    // Online softmax in base 2.  s[nt][0]: (token gq, column 2tq), [1]: (gq, 2tq+1),
    // [2]: (gq+8, 2tq), [3]: (gq+8, 2tq+1).
    const bool lo_ok = gq < nvalid;
    const bool hi_ok = gq + 8 < nvalid;
    uint32_t pb_hi[NT][2], pb_lo[NT][2];
    float alpha0[NT], alpha1[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int c = 0; c < 4; ++c) s[nt][c] *= scale_log2;
        if (!lo_ok) s[nt][0] = s[nt][1] = -INFINITY;
        if (!hi_ok) s[nt][2] = s[nt][3] = -INFINITY;
        if constexpr (ROW_LIMITS) {
            if (tok0 + gq >= lim[nt][0]) s[nt][0] = -INFINITY;
            if (tok0 + gq >= lim[nt][1]) s[nt][1] = -INFINITY;
            if (tok0 + gq + 8 >= lim[nt][0]) s[nt][2] = -INFINITY;
            if (tok0 + gq + 8 >= lim[nt][1]) s[nt][3] = -INFINITY;
        }
        float mx0 = fmaxf(s[nt][0], s[nt][2]);
        float mx1 = fmaxf(s[nt][1], s[nt][3]);
        // The reference m need not be the exact running maximum: any m with
        // every score at most m + kLazyLog2 keeps each e^(s - m) <= 2^kLazyLog2,
        // and O, l and lse = m + log l come out the same up to rounding.  So
        // while the whole warp's scores of this stage fit under the current
        // references (one vote), they are kept (alpha = 1) and the cross-lane
        // maximum is skipped; otherwise m moves to the exact maximum.  The
        // E4M3 stage keeps the exact maximum every stage: with the lazy
        // reference its Llama-70B GQA-8 layer step measured slower (66.6
        // against 68.0 % of the copy peak), though its other layers ran faster.
        bool keep = false;
        if constexpr (!F8)
            keep = __all_sync(0xffffffffu, mx0 <= m0[nt] + kLazyLog2 && mx1 <= m1[nt] + kLazyLog2);
        if (keep) {
            alpha0[nt] = alpha1[nt] = 1.f;
        } else {
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = fmaxf(m0[nt], mx0);
            const float mn1 = fmaxf(m1[nt], mx1);
            alpha0[nt] = exp2f(m0[nt] - (mn0 == -INFINITY ? 0.f : mn0));
            alpha1[nt] = exp2f(m1[nt] - (mn1 == -INFINITY ? 0.f : mn1));
            m0[nt] = mn0;
            m1[nt] = mn1;
        }
        const float ref0 = m0[nt] == -INFINITY ? 0.f : m0[nt];
        const float ref1 = m1[nt] == -INFINITY ? 0.f : m1[nt];
        const float p0 = exp2f(s[nt][0] - ref0);
        const float p1 = exp2f(s[nt][1] - ref1);
        const float p2 = exp2f(s[nt][2] - ref0);
        const float p3 = exp2f(s[nt][3] - ref1);
        l0[nt] = l0[nt] * alpha0[nt] + (p0 + p2);
        l1[nt] = l1[nt] * alpha1[nt] + (p1 + p3);
        // P as hi + lo 16-bit terms, transposed into P^T operand fragments.
        const uint32_t h01 = pack2(p0, p1, T());
        const uint32_t h23 = pack2(p2, p3, T());
        const float2 r01 = unpack2(h01, T());
        const float2 r23 = unpack2(h23, T());
        const uint32_t l01 = pack2(p0 - r01.x, p1 - r01.y, T());
        const uint32_t l23 = pack2(p2 - r23.x, p3 - r23.y, T());
        pb_hi[nt][0] = ptx::movmatrix_trans(h01);
        pb_hi[nt][1] = ptx::movmatrix_trans(h23);
        pb_lo[nt][0] = ptx::movmatrix_trans(l01);
        pb_lo[nt][1] = ptx::movmatrix_trans(l23);
    }

    // O^T = alpha * O^T + V^T P^T.  The rescale is skipped when no column's max
    // moved (alpha = 1 everywhere, the common case once the max has settled).
    bool moved = false;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) moved |= (alpha0[nt] != 1.f) | (alpha1[nt] != 1.f);
    if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int mt = 0; mt < KSTEPS; ++mt) {
                o[nt][mt][0] *= alpha0[nt];
                o[nt][mt][1] *= alpha1[nt];
                o[nt][mt][2] *= alpha0[nt];
                o[nt][mt][3] *= alpha1[nt];
            }
    }
    // V rows of tokens at i >= nvalid are zeroed in the A fragments (only a
    // ragged stage pays for the masks).
    auto v_pass = [&](auto ragged_tag) {
        constexpr bool RAGGED = decltype(ragged_tag)::value;
        uint32_t vmask_lo = 0xffffffffu, vmask_hi = 0xffffffffu;
        if constexpr (RAGGED) {
            // A fragments of V^T hold tokens 2tq, 2tq+1 (a0, a1) and 2tq+8, 2tq+9 (a2, a3)
            vmask_lo = (2 * tq < nvalid ? 0x0000ffffu : 0u) |
                       (2 * tq + 1 < nvalid ? 0xffff0000u : 0u);
            vmask_hi = (2 * tq + 8 < nvalid ? 0x0000ffffu : 0u) |
                       (2 * tq + 9 < nvalid ? 0xffff0000u : 0u);
        }
        auto accumulate = [&](int mt, uint32_t (&a)[4]) {
            if constexpr (RAGGED) {
                a[0] &= vmask_lo;
                a[1] &= vmask_lo;
                a[2] &= vmask_hi;
                a[3] &= vmask_hi;
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                ptx::mma_16816<T>(o[nt][mt], a, pb_hi[nt][0], pb_hi[nt][1]);
                ptx::mma_16816<T>(o[nt][mt], a, pb_lo[nt][0], pb_lo[nt][1]);
            }
        };
        if constexpr (F8) {
            const int row = (mi & 1) * 8 + r8;
#pragma unroll
            for (int j = 0; j < D / 32; ++j) {
                const int chunk = 2 * j + (mi >> 1);
                uint32_t r[4];
                ptx::ldmatrix_x4_trans(r, vbase + row * 128 + ((chunk ^ r8) << 4));
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    // r[2h]: tokens 2tq, 2tq+1; r[2h+1]: tokens 2tq+8, 2tq+9; bytes (dim 2gq,
                    // token a), (dim 2gq+1, token a), (dim 2gq, token b), (dim 2gq+1, token b)
                    uint32_t a[4];
                    a[0] = e4m3x2_to(__byte_perm(r[2 * h], 0u, 0x0020), T());      // even dim
                    a[1] = e4m3x2_to(__byte_perm(r[2 * h], 0u, 0x0031), T());      // odd dim
                    a[2] = e4m3x2_to(__byte_perm(r[2 * h + 1], 0u, 0x0020), T());
                    a[3] = e4m3x2_to(__byte_perm(r[2 * h + 1], 0u, 0x0031), T());
                    accumulate(2 * j + h, a);
                }
            }
        } else {
#pragma unroll
            for (int mt = 0; mt < KSTEPS; ++mt) {
                const int chunk = mt * 2 + v_csel;
                const uint32_t addr = vbase + (chunk >> 3) * kRegionBytes + v_tok * 128 +
                                      (((chunk & 7) ^ r8) << 4);
                uint32_t a[4];
                ptx::ldmatrix_x4_trans(a, addr);
                accumulate(mt, a);
            }
        }
    };
    if (nvalid < kStageTokens)
        v_pass(std::true_type{});
    else
        v_pass(std::false_type{});
}

// Merge of split partials (log-sum-exp rule): one warp per (row of q, query
// head), four rows per CTA.  Each lane owns float4 columns of the head (lane,
// lane + 32, ...) and weighs every partition itself: w_p = e^(lse_p - m*),
// out = sum_p w_p O_p / sum_p w_p; m* and sum_p w_p come from lane-strided
// sums and shuffles.  No shared memory and no CTA barrier: rows are short,
// and the merge of a call is a few thousand of them.  With context_lens given
// (the decode path), a sequence whose context fitted a single partition was
// written by the decode kernel and is skipped, and only the partitions that
// hold tokens are read.  Multi-query rows (q_len > 0) are merged from the
// partitions of their sequence's context; with mq_direct (the decode kernel's
// multi-query form) a context that fitted one partition was written directly
// and is skipped.  Without context_lens (pkv_merge), every row merges all
// num_splits partials.
struct MergeParams {
    void* out;
    const float* partial_o;
    const float* partial_lse;
    const int32_t* context_lens;  // nullable
    const int2* seq_info;         // nullable: shared-prefix tokens and prefix partials per sequence
    int num_q_heads;
    int num_kv_heads;
    int group;                    // query heads per KV head
    int num_splits;
    int head_dim;                 // a multiple of 4, at most 512
    int chunk_tokens;
    int cap;                      // context clamp, as in the decode kernel
    int q_len;                    // > 0: multi-query rows (sequence, query token)
    int mq_slots;                 // multi-query: partial slots per context partition (1 or 2)
    bool mq_direct;               // multi-query partials of the decode kernel (single ones direct)
    int64_t rows;                 // (row of q, query head) pairs
};

constexpr int kMergeRowsPerCta = 4;
constexpr int kMergeThreads = kMergeRowsPerCta * 32;
constexpr int kMergeMaxHeadDim = 512;

// One row's merge, by one warp (lane = its lane).  The partials are read
// through L2 (ld.global.cg): the kernels that merge a unit's rows as soon as
// its last partial is written read what other CTAs of the same launch, or of
// a launch running beside it, have just written.
template <typename T>
__device__ __forceinline__ void merge_row(const MergeParams& p, int64_t row, int lane) {
    const int b = (int)(row / p.num_q_heads);  // row of q: a sequence, or (sequence, query token)
    int ns = p.num_splits;
    if (p.q_len > 0) {
        // multi-query partials: the partitions of the sequence's context
        const int n = clamped_len(__ldg(p.context_lens + b / p.q_len), p.cap);
        if (p.mq_direct) {
            ns = suffix_partitions(n, 0, p.chunk_tokens);
            if (ns <= 1) return;  // written directly by the decode kernel
        } else {
            ns = (n + p.chunk_tokens - 1) / p.chunk_tokens * p.mq_slots;
        }
    } else if (p.context_lens != nullptr) {
        int start = 0, slot0 = 0;
        if (p.seq_info != nullptr) {
            const int2 si = __ldcg(p.seq_info + b);
            start = si.x;
            slot0 = si.y;
        }
        const int n = clamped_len(__ldg(p.context_lens + b), p.cap);
        ns = slot0 + suffix_partitions(max(0, n - start), slot0, p.chunk_tokens);
        if (slot0 == 0 && ns <= 1) return;  // written directly by the decode kernel
    }
    const float* lse = p.partial_lse + row * p.num_splits;
    // m* = max_p lse_p and 1 / sum_p e^(lse_p - m*)
    float mx = -INFINITY;
    for (int sp = lane; sp < ns; sp += 32) mx = fmaxf(mx, __ldcg(lse + sp));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float den = 0.f;
    if (mx != -INFINITY)
        for (int sp = lane; sp < ns; sp += 32) {
            const float ls = __ldcg(lse + sp);
            if (ls != -INFINITY) den += exp2f((ls - mx) * kLog2e);
        }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
    const float inv = den > 0.f ? 1.f / den : 0.f;
    const int cols = p.head_dim / 4;
    const float* po = p.partial_o + row * p.num_splits * p.head_dim;
    T* out = static_cast<T*>(p.out) + row * p.head_dim;
    // Lane-owned float4 columns c = lane + 32k.  Weights come 32 partitions at
    // a time, one per lane, and reach the other lanes by shuffles; each lane
    // reads its columns of kMergeBatch partials before it adds any of them, so
    // the partials' reads overlap instead of waiting on one another.  A zero
    // weight (an empty partition, whose O may hold anything) adds nothing.
    constexpr int kMergeBatch = 8;
    for (int k = 0; 32 * k < cols; ++k) {
        const int c = lane + 32 * k;
        const bool col_ok = c < cols;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (mx != -INFINITY)
            for (int s0 = 0; s0 < ns; s0 += 32) {
                const int sl = s0 + lane;
                const float ls = sl < ns ? __ldcg(lse + sl) : -INFINITY;
                const float wl = ls == -INFINITY ? 0.f : exp2f((ls - mx) * kLog2e);
                const int nb = min(32, ns - s0);
                for (int u0 = 0; u0 < nb; u0 += kMergeBatch) {
                    float4 v[kMergeBatch];
#pragma unroll
                    for (int u = 0; u < kMergeBatch; ++u)
                        v[u] = (col_ok && u0 + u < nb)
                                   ? __ldcg(reinterpret_cast<const float4*>(
                                         po + (int64_t)(s0 + u0 + u) * p.head_dim + c * 4))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int u = 0; u < kMergeBatch; ++u) {
                        const float wgt = __shfl_sync(0xffffffffu, wl, u0 + u);
                        if (wgt != 0.f) {
                            acc.x = fmaf(wgt, v[u].x, acc.x);
                            acc.y = fmaf(wgt, v[u].y, acc.y);
                            acc.z = fmaf(wgt, v[u].z, acc.z);
                            acc.w = fmaf(wgt, v[u].w, acc.w);
                        }
                    }
                }
            }
        if (col_ok) {
            uint2 packed;
            packed.x = pack2(acc.x * inv, acc.y * inv, T());
            packed.y = pack2(acc.z * inv, acc.w * inv, T());
            *reinterpret_cast<uint2*>(out + c * 4) = packed;
        }
    }
}

// NT = number of 8-column groups (1: up to 8 query rows, 2: up to 16); F8:
// E4M3 cache codes.  MQ: multi-query, the columns are the (query token i,
// query head) rows of a chunk of q_len tokens (row i * group + head in group),
// and row i sees positions < n - q_len + 1 + i; only the stages that reach
// past the first limit of the CTA's rows apply the per-column limits.  With
// row_blocks > 1 the rows of a (sequence, KV head) are split over adjacent
// CTAs of NT * 8 rows each, which read the same context at the same time (the
// second copy mostly from L2).
template <typename T, int D, int NT, bool F8 = false, bool MQ = false>
__global__ void __launch_bounds__(kThreads, (F8 && NT == 1) ? 4 : 3)
decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
              const DecodeParams p) {
    using Cfg = Tile<D, F8>;
    constexpr int S = Cfg::kStages;
    constexpr int KSTEPS = D / 16;   // k-steps of S^T = K Q^T, also m-tiles of O^T

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* ring = smem;
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(ring + Cfg::kRingBytes);
    uint64_t* empty_bar = full_bar + S;
    int* table = reinterpret_cast<int*>(empty_bar + S);
    volatile int* abort_flag = table + kMaxChunkPages + 1;
    constexpr bool QS = q_tile_bytes<D, NT, F8>() > 0;
    uint8_t* q_tile = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(table + kMaxChunkPages + 5) + 127) & ~uintptr_t(127));

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int bs = p.block_size;
    const int bs_shift = __ffs(bs) - 1;  // block sizes are powers of two

    // Let the merge kernel (launched as a programmatic dependent) get scheduled
    // as soon as every CTA of this grid has started; it waits for our results.
    ptx::launch_dependents();
    // Inputs may come from the previous kernel on the stream (the append).
    ptx::grid_dependency_wait();

    int g, b, split;
    if (p.items != nullptr) {
        // A compact work list built on the device: only partitions with tokens
        // get a CTA; grid positions past the end of the list exit at once.
        if ((int)blockIdx.x >= *p.item_count) return;
        const int2 it = p.items[blockIdx.x];
        g = it.x % p.num_kv_heads;
        b = it.x / p.num_kv_heads;
        split = it.y;
    } else {
        // Grid order (KV head fastest, then sequence, then partition): all first
        // partitions run before any second one, so sequences that share physical
        // blocks (a common prompt prefix) read them close together in time and
        // the repeats hit in L2.
        g = MQ ? blockIdx.x / p.row_blocks : blockIdx.x;
        b = blockIdx.y;
        split = blockIdx.z;
    }
    // MQ: the CTA's first row of the (sequence, KV head)'s q_len * group rows
    const int col0 = MQ ? (int)(blockIdx.x % p.row_blocks) * (NT * 8) : 0;

    const int cap = min(p.max_blocks_per_seq * bs, p.max_context_len);
    const int n_raw = __ldg(p.context_lens + b);
    // With a shared prefix (seq_info), the first `start` tokens were attended by
    // the prefix kernel, which wrote this sequence's partials 0 .. slot0-1; the
    // partitions here cover the suffix and write from partial slot0 on.
    int start = 0, slot0 = 0;
    if (p.seq_info != nullptr) {
        const int2 si = __ldcg(p.seq_info + b);
        start = si.x;
        slot0 = si.y;
    }
    // Partition start does not depend on the context length, so the producer
    // warp fetches the block-table slice at the same time as the length.
    const int t_begin = start + split * p.chunk_tokens;
    const int page0 = t_begin / bs;
    // pages a partition can touch: it may start and end mid-page
    const int max_pages = min(p.max_blocks_per_seq - page0, (p.chunk_tokens + bs - 1) / bs + 1);
    const int32_t* row = p.block_tables + (int64_t)b * p.max_blocks_per_seq + page0;
    int blk_r[5] = {-1, -1, -1, -1, -1};  // up to 160 pages: kMaxChunkPages + 1
    static_assert(kMaxChunkPages + 1 <= 5 * 32, "the producer lanes hold the table slice");
    if (warp == kConsumerWarps) {
#pragma unroll
        for (int r = 0; r < 5; ++r)
            if (lane + 32 * r < max_pages) blk_r[r] = __ldg(row + lane + 32 * r);
    }
    if ((n_raw < 0 || n_raw > cap || (MQ && n_raw < p.q_len)) && split == 0 && g == 0 &&
        tid == 0)
        flag_error(p.err_flag, PKV_EFLAG_CONTEXT_LEN);
    const int n = clamped_len(n_raw, cap);
    const int suffix = max(0, n - start);
    const int nsplit = suffix_partitions(suffix, slot0, p.chunk_tokens);
    if (split >= nsplit) return;
    const int t_end = min(n, start + (split + 1) * p.chunk_tokens);
    const int nstages = t_end > t_begin ? (t_end - t_begin + kStageTokens - 1) / kStageTokens : 0;
    const bool direct = slot0 == 0 && nsplit == 1;  // the whole answer is this CTA's

    // Fused append: the one CTA of (sequence, KV head) whose partition holds the
    // last position n-1 first stores the new token's K and V rows of this KV
    // head into that position's slot, then orders the stores before its own
    // TMA reads (no other CTA reads that position).  An E4M3 cache stores the
    // codes pkv_append_fp8 would: E4M3(x / scale), the quotient rounded to fp32
    // and then to the nearest E4M3 value (ties to even), saturating at +-448.
    if (p.k_new != nullptr && n_raw == n && n > 0 && t_begin <= n - 1 && n - 1 < t_end &&
        warp < kConsumerWarps && tid < 2 * (D / 8)) {
        const int pos = n - 1;
        const int blk = __ldg(p.block_tables + (int64_t)b * p.max_blocks_per_seq + pos / bs);
        if (blk >= 0 && blk < p.num_blocks) {
            const bool is_v = tid >= D / 8;
            const int c = tid % (D / 8);  // 16-byte chunk of the row
            const int64_t src = ((int64_t)b * p.num_kv_heads + g) * (D / 8) + c;
            const int64_t dst =
                (p.hnd ? ((int64_t)blk * p.num_kv_heads + g) * bs + pos % bs
                       : ((int64_t)blk * bs + pos % bs) * p.num_kv_heads + g) * (D / 8) + c;
            const uint4 v = __ldg(static_cast<const uint4*>(is_v ? p.v_new : p.k_new) + src);
            if constexpr (F8) {
                // eight 16-bit elements in, eight one-byte codes out
                const float sc = is_v ? p.v_scale : p.k_scale;
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                uint32_t codes[2] = {0u, 0u};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 x = pair_to_float2(w[j], T());
                    const float2 f = make_float2(__fdiv_rn(x.x, sc), __fdiv_rn(x.y, sc));
                    const uint32_t two = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
                    codes[j / 2] |= two << (16 * (j % 2));
                }
                static_cast<uint2*>(is_v ? p.v_cache : p.k_cache)[dst] =
                    make_uint2(codes[0], codes[1]);
            } else {
                static_cast<uint4*>(is_v ? p.v_cache : p.k_cache)[dst] = v;
            }
            ptx::fence_proxy_async_global();
        }
    }

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(ptx::smem_addr(&full_bar[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&empty_bar[s]), 1);
        }
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == kConsumerWarps) {
        // Keep this partition's slice of the block table, validating each id.
        const int npages = t_end > t_begin ? (t_end + bs - 1) / bs - page0 : 0;
#pragma unroll
        for (int r = 0; r < 5; ++r) {
            const int i = lane + 32 * r;
            if (i < npages) {
                int blk = blk_r[r];
                if (blk < 0 || blk >= p.num_blocks) {
                    flag_error(p.err_flag, PKV_EFLAG_BLOCK_ID);
                    blk = -1;
                }
                table[i] = blk;
            }
        }
        if (lane == 0) {
            ptx::prefetch_tensormap(&tm_k);
            ptx::prefetch_tensormap(&tm_v);
        }
    }
#ifdef PKV_DEBUG
    poison_smem(ring, Cfg::kRingBytes, tid, kThreads);
#endif
    if constexpr (QS) {
        // the CTA's query columns (zero rows past the ones in use)
        const int ncols_q = MQ ? min(NT * 8, p.q_len * p.group - col0) : p.group;
        const T* qb0 = static_cast<const T*>(p.q) +
                       ((int64_t)b * (MQ ? p.q_len : 1) * p.num_q_heads + g * p.group) * D;
        for (int idx = tid; idx < NT * 8 * (D / 8); idx += kThreads) {
            const int col = idx / (D / 8), chunk = idx % (D / 8);
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (col < ncols_q) {
                const int cc = MQ ? col0 + col : col;
                const int off = MQ ? (cc / p.group) * p.num_q_heads + cc % p.group : col;
                v = __ldg(reinterpret_cast<const uint4*>(qb0 + (int64_t)off * D) + chunk);
            }
            *reinterpret_cast<uint4*>(q_tile + col * (D * 2) + ((chunk ^ (col & 7)) << 4)) = v;
        }
    }
    __syncthreads();

    const uint32_t ring_addr = ptx::smem_addr(ring);

    // ---------------------------------------------------------------- producer
    // Lane j of the producer warp fills the slots of stages j, j + P, j + 2P, ...
    // (P = kConsumerWarps, the stages consumer warp j takes), so one warp
    // instruction waits for, and issues the copies of, P stages.
    // S a multiple of the consumer warps: every slot then has one consumer warp
    // (and one producer lane), so no warp can wait on a slot's next phase while
    // its current one is still pending (a parity wait would pass at once).
    static_assert(S % kConsumerWarps == 0, "each ring slot has one consumer warp");
    if (warp == kConsumerWarps) {
        if (lane < kConsumerWarps) {
            const uint64_t policy = ptx::l2_policy_evict_first();
            int issued = 0;  // one past this lane's last stage issued
            for (int i = lane; i < nstages; i += kConsumerWarps) {
                const int slot = i % S;
                if (i >= S &&
                    !wait_phase(ptx::smem_addr(&empty_bar[slot]), ((i / S) - 1) & 1, abort_flag,
                                p.err_flag))
                    break;
                const int tok0 = t_begin + i * kStageTokens;
                const int blk = table[(tok0 >> bs_shift) - page0];
                const uint32_t fb = ptx::smem_addr(&full_bar[slot]);
                if (blk >= 0) {
                    const int toff = tok0 & (bs - 1);
                    const uint32_t kdst = ring_addr + slot * Cfg::kStageBytes;
                    ptx::mbar_arrive_expect_tx(fb, Cfg::kStageBytes);
#pragma unroll
                    for (int r = 0; r < Cfg::kRegions; ++r) {
                        load_kv_box(kdst + r * Cfg::kRegionBytes, &tm_k, fb,
                                    r * Cfg::kRegionElems, g, toff, blk, p.hnd, policy);
                        load_kv_box(kdst + Cfg::kHalfBytes + r * Cfg::kRegionBytes, &tm_v, fb,
                                    r * Cfg::kRegionElems, g, toff, blk, p.hnd, policy);
                    }
                } else {
                    ptx::mbar_arrive(fb);  // nothing to load: the consumer masks the stage
                }
                issued = i + 1;
            }
            if (*abort_flag) {
                // Wait (bounded) for this lane's copies still in flight before leaving.
                for (int i = lane; i < issued; i += kConsumerWarps) {
                    if (i < issued - S) continue;
                    const uint32_t fb = ptx::smem_addr(&full_bar[i % S]);
                    const uint64_t t0 = ptx::globaltimer();
                    while (!ptx::mbar_try_wait(fb, (i / S) & 1) &&
                           ptx::globaltimer() - t0 < kWaitLimitNs) {
                    }
                }
            }
        }
    }

    // ---------------------------------------------------------------- consumers
    const int gq = lane >> 2;  // fragment row group
    const int tq = lane & 3;   // fragment column pair
    float o[NT][KSTEPS][4];    // O^T tiles: 16 dims x 8 heads each
    float m0[NT], m1[NT], l0[NT], l1[NT];  // heads 2tq and 2tq+1 of each 8-head group
    if (warp < kConsumerWarps) {
        // Q^T operand fragments (B of S^T = K Q^T): column nt*8 + gq, dims 2tq.. of
        // each k-step (for an E4M3 cache, dims 4tq.. and 4tq+2.., the K fragments'
        // order).  A column is a head of the group, or (MQ) a (query token, head).
        uint32_t qb[NT][KSTEPS][2];
        const int ncols = MQ ? min(NT * 8, p.q_len * p.group - col0) : p.group;
        // the first row of the CTA's block of q: head g*group of the sequence (MQ:
        // of its first query token)
        const T* qbase = static_cast<const T*>(p.q) +
                         ((int64_t)b * (MQ ? p.q_len : 1) * p.num_q_heads + g * p.group) * D;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int col = nt * 8 + gq;
            // rows of q after the first: the column's head, or (MQ) its query
            // token's rows of all heads plus its head
            const int cc = MQ ? col0 + (col >= ncols ? 0 : col) : col;
            const int off = MQ ? (cc / p.group) * p.num_q_heads + cc % p.group : col;
            const uint32_t* qrow = reinterpret_cast<const uint32_t*>(qbase + off * D);
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
                const bool ok = col < ncols;
                const int d0 = F8 ? ks * 16 + 4 * tq : ks * 16 + 2 * tq;
                const int d1 = F8 ? d0 + 2 : d0 + 8;
                if constexpr (!QS) {
                    qb[nt][ks][0] = ok ? __ldg(qrow + d0 / 2) : 0u;
                    qb[nt][ks][1] = ok ? __ldg(qrow + d1 / 2) : 0u;
                } else {
                    qb[nt][ks][0] = qb[nt][ks][1] = 0u;
                }
            }
            m0[nt] = m1[nt] = -INFINITY;
            l0[nt] = l1[nt] = 0.f;
#pragma unroll
            for (int mt = 0; mt < KSTEPS; ++mt)
#pragma unroll
                for (int c = 0; c < 4; ++c) o[nt][mt][c] = 0.f;
        }

        int no_limit[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) no_limit[nt][0] = no_limit[nt][1] = INT_MAX;
        // MQ: the causal limits of this thread's fragment columns 2tq and 2tq+1
        // (columns past the rows in use get the largest limit: their q is zero
        // and their results are not written), and the first position that some
        // column does not see.
        int lim[NT][2];
        int causal0 = INT_MAX;
        if constexpr (MQ) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    lim[nt][k] =
                        max(0, n - p.q_len + 1 + (col0 + nt * 8 + 2 * tq + k) / p.group);
            causal0 = n - p.q_len + 1 + col0 / p.group;
        }

        for (int i = warp; i < nstages; i += kConsumerWarps) {
            const int slot = i % S;
            if (!wait_phase(ptx::smem_addr(&full_bar[slot]), (i / S) & 1, abort_flag, p.err_flag))
                break;
            const int tok0 = t_begin + i * kStageTokens;
            const int blk = table[(tok0 >> bs_shift) - page0];
            const int nvalid = blk >= 0 ? min(kStageTokens, t_end - tok0) : 0;
            if (nvalid > 0) {
                const uint32_t kbase = ring_addr + slot * Cfg::kStageBytes;
                const uint32_t qaddr = ptx::smem_addr(q_tile);
                if (MQ && tok0 + kStageTokens > causal0)
                    stage_update<T, D, NT, true, F8, QS>(kbase, kbase + Cfg::kHalfBytes, nvalid,
                                                         tok0, lim, qb, o, m0, m1, l0, l1,
                                                         p.scale_log2, lane, qaddr);
                else
                    stage_update<T, D, NT, false, F8, QS>(kbase, kbase + Cfg::kHalfBytes, nvalid,
                                                          0, no_limit, qb, o, m0, m1, l0, l1,
                                                          p.scale_log2, lane, qaddr);
            }
            __syncwarp();
#ifdef PKV_DEBUG
            poison_smem(ring + slot * Cfg::kStageBytes, Cfg::kStageBytes, lane, 32);
            __syncwarp();
#endif
            if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&empty_bar[slot]));
        }
    }

    __syncthreads();
    if (*abort_flag) return;

    // ---------------------------------------------------------------- combine the warps
    // Reuses the ring (every copy has landed and been consumed).
    constexpr int HP = NT * 8;        // heads per warp state
    constexpr int OSTRIDE = D + 4;    // padded row of the per-warp O tile (conflict-free writes)
    static_assert((kConsumerWarps * HP * OSTRIDE + 3 * kConsumerWarps * HP + HP) * 4 <=
                      Cfg::kRingBytes,
                  "the combine buffers fit in the ring they reuse");
    float* sm_o = reinterpret_cast<float*>(ring);                 // [warps][HP][OSTRIDE]
    float* sm_m = sm_o + kConsumerWarps * HP * OSTRIDE;           // [warps][HP]
    float* sm_l = sm_m + kConsumerWarps * HP;                     // [warps][HP]
    if (warp < kConsumerWarps) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float a = l0[nt], c = l1[nt];
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                a += __shfl_xor_sync(0xffffffffu, a, off);
                c += __shfl_xor_sync(0xffffffffu, c, off);
            }
            const int h0 = nt * 8 + 2 * tq;
            if (gq == 0) {
                sm_m[warp * HP + h0] = m0[nt];
                sm_m[warp * HP + h0 + 1] = m1[nt];
                sm_l[warp * HP + h0] = a;
                sm_l[warp * HP + h0 + 1] = c;
            }
            float* w0 = sm_o + (warp * HP + h0) * OSTRIDE;
            float* w1 = w0 + OSTRIDE;
#pragma unroll
            for (int mt = 0; mt < KSTEPS; ++mt) {
                // fragment rows gq and gq+8 of block mt are dims gq, gq+8 (16-bit cache)
                // or 2gq, 2gq+1 (E4M3 cache)
                const int da = F8 ? mt * 16 + 2 * gq : mt * 16 + gq;
                const int db = F8 ? da + 1 : da + 8;
                w0[da] = o[nt][mt][0];
                w1[da] = o[nt][mt][1];
                w0[db] = o[nt][mt][2];
                w1[db] = o[nt][mt][3];
            }
        }
        ptx::named_barrier_sync(1, kConsumerWarps * 32);

        // Per-column combine factors, once per column: c_w = e^(m_w - m*) / L with
        // L = sum_w e^(m_w - m*) l_w, and the column's log-sum-exp.
        const int G = MQ ? min(NT * 8, p.q_len * p.group - col0) : p.group;
        float* sm_f = sm_l + kConsumerWarps * HP;   // [HP][warps]
        float* sm_lse = sm_f + HP * kConsumerWarps; // [HP]
        if (tid < G) {
            const int h = tid;
            float mx = -INFINITY;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) mx = fmaxf(mx, sm_m[w * HP + h]);
            float c[kConsumerWarps];
            float den = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float mw = sm_m[w * HP + h];
                c[w] = (mx == -INFINITY || mw == -INFINITY) ? 0.f : exp2f(mw - mx);
                den = fmaf(sm_l[w * HP + h], c[w], den);
            }
            const float inv = den > 0.f ? p.v_scale / den : 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) sm_f[h * kConsumerWarps + w] = c[w] * inv;
            sm_lse[h] = den > 0.f ? (mx + log2f(den)) * kLn2 : -INFINITY;
        }
        ptx::named_barrier_sync(1, kConsumerWarps * 32);

        // Four consecutive dims of one head per thread and iteration.
        for (int idx = tid; idx < G * (D / 4); idx += kConsumerWarps * 32) {
            const int h = idx / (D / 4);
            const int j = (idx - h * (D / 4)) * 4;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float f = sm_f[h * kConsumerWarps + w];
                const float4 v = *reinterpret_cast<const float4*>(sm_o + (w * HP + h) * OSTRIDE + j);
                acc.x = fmaf(v.x, f, acc.x);
                acc.y = fmaf(v.y, f, acc.y);
                acc.z = fmaf(v.z, f, acc.z);
                acc.w = fmaf(v.w, f, acc.w);
            }
            // (row of q, query head) of the column: rows of q are sequences, or
            // (sequence, query token) with MQ
            const int64_t orow =
                MQ ? ((int64_t)b * p.q_len + (col0 + h) / p.group) * p.num_q_heads +
                         g * p.group + (col0 + h) % p.group
                   : (int64_t)b * p.num_q_heads + (g * G + h);
            if (direct) {
                T* out = static_cast<T*>(p.out) + orow * D + j;
                uint2 packed;
                packed.x = pack2(acc.x, acc.y, T());
                packed.y = pack2(acc.z, acc.w, T());
                *reinterpret_cast<uint2*>(out) = packed;
            } else {
                const int64_t prow = orow * p.num_splits + slot0 + split;
                *reinterpret_cast<float4*>(p.partial_o + prow * D + j) = acc;
                if (j == 0) p.partial_lse[prow] = sm_lse[h];
            }
        }
    }

    // Shared-prefix calls (16-bit caches, one query per sequence): the CTA
    // that writes the last of a unit's partials (prefix partitions and suffix
    // partitions alike) merges the unit's rows.
    if (!MQ && !F8 && p.unit_left != nullptr && !direct) {
        __threadfence();  // this thread's partials, before the count below
        __syncthreads();
        int* last = table;  // the table slice is not read after the main loop
        if (tid == 0)
            *last = atomicAdd(p.unit_left + (int64_t)b * p.num_kv_heads + g, -1) == 1;
        __syncthreads();
        if (*last) {
            __threadfence();
            MergeParams mp = {};
            mp.out = p.out;
            mp.partial_o = p.partial_o;
            mp.partial_lse = p.partial_lse;
            mp.context_lens = p.context_lens;
            mp.seq_info = p.seq_info;
            mp.num_q_heads = p.num_q_heads;
            mp.num_kv_heads = p.num_kv_heads;
            mp.group = p.group;
            mp.num_splits = p.num_splits;
            mp.head_dim = D;
            mp.chunk_tokens = p.chunk_tokens;
            mp.cap = cap;
            for (int h = warp; h < p.group; h += kThreads / 32)
                merge_row<T>(mp, (int64_t)b * p.num_q_heads + g * p.group + h, lane);
        }
    }
}

// ---------------------------------------------------------------------------
// Shared-prefix decode: the prefix kernel (5th-generation tensor cores)
// ---------------------------------------------------------------------------
// Sequences come in contiguous groups (group_start); the first prefix_len
// tokens of every member of group p are the same physical blocks (a shared
// prompt, [inference] Copy-on-Write; RadixAttention in [chapter12]).  For one
// (group, KV head) the members' query rows form a dense matrix Q [rows x D]
// (row r is query head g*group + r % group of sequence first + r / group) that
// meets every prefix token once: softmax(Q K^T * scale) V over the prefix is a
// real contraction, so it runs on tcgen05.  One CTA takes 128 query rows and
// one prefix partition, in tiles of 64 tokens:
//   S = Q K^T        tcgen05.mma M=128, N=64, 16-dim steps; S in tensor memory
//   softmax          threads reading their rows of S directly
//   O += P V         M=128, N=D, 16-token steps; P enters as hi + lo 16-bit
//                    terms (as in the decode kernel), written by the softmax
//                    over its S and read as the A operand from tensor memory;
//                    O stays in tensor memory
// In MODE 0 (this path) warp 8 streams K/V tiles by TMA into a 4-stage ring,
// warp 9 owns the tensor memory and one of its lanes issues the MMAs, warps
// 0-7 run the softmax: two threads per query row, one for tokens 0-31 of every
// tile, one for tokens 32-63.  The two halves are independent online softmaxes
// with accumulators O_a and O_b of their own in tensor memory (O_a += P[:, 0:32]
// V[0:32], O_b += P[:, 32:64] V[32:64]); they meet once, at the end, where the
// rows' normalised O and log-sum-exp are combined and written as partials.  S
// (and P over it) is double-buffered, so S of the next tile is computed during
// this tile's softmax.  A half's reference max is raised (and its O rescaled in
// tensor memory) only when its running max exceeds it by more than 2^8; P
// stays below 256 and the final normalisation uses the same references, so
// the result is the same softmax.  Multi-query calls with more than 32 rows per
// (sequence, KV head) use the same kernel in MODES 1 and 2 (one softmax thread
// per tensor-memory lane, two CTAs an SM; see prefix_kernel); smaller ones run
// on the decode kernel.

// ---------------------------------------------------------------------------
// Shared-prefix decode: the plan
// ---------------------------------------------------------------------------
// One CTA writes, for every sequence, its (shared-prefix tokens, prefix
// partials) record, the compact list of the suffix partitions that hold
// tokens, unit by unit ((sequence, KV head) pairs, KV head fastest), and each
// unit's count of partials to come.  The decode grid is sized for the longest
// sequence; with the list, only real partitions get a CTA and the rest of the
// grid exits at once.  The plan is a launch of its own on the caller's stream,
// ahead of both the suffix decode and the prefix kernel (which runs beside the
// decode on a second stream), so neither waits for the other.

constexpr int kPlanThreads = 1024;
constexpr int kPlanStagedGroups = 4096;

struct PlanParams {
    const int32_t* context_lens;
    const int32_t* group_start;
    const int32_t* group_prefix_len;
    int2* seq_info;   // [B] out
    int2* items;      // out: (unit, partition)
    int* item_count;  // out
    int* unit_left;   // out: per unit, the partials (prefix and suffix) still to be written
    int32_t* err_flag;
    int num_seqs;
    int num_kv_heads;
    int num_groups;
    int max_group_size;
    int max_prefix_len;
    int block_size;
    int max_blocks_per_seq;
    int prefix_chunk;
    int chunk_tokens;
    int cap;
    int group;        // query heads per KV head
};

struct PrefixParams {
    const void* q;
    const int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* group_start;       // [num_groups + 1]
    const int32_t* group_prefix_len;  // [num_groups]
    float* partial_o;                 // [B][H_q][num_splits][D]
    float* partial_lse;               // [B][H_q][num_splits]
    int32_t* err_flag;
    int max_blocks_per_seq;
    int num_blocks;
    int block_size;
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int group;            // query heads per KV head
    int num_splits;       // partial slots per (sequence, query head)
    int num_groups;
    int max_group_size;
    int max_prefix_len;
    int prefix_chunk;     // prefix tokens per partition (a multiple of 64 and of block_size)
    int cap;              // context clamp
    int q_len;            // 0: shared prefixes; > 0: multi-query (q_len query tokens per sequence)
    bool hnd;             // head-major cache layout
    float scale_log2;
    // Shared prefixes (MODE 0): the CTA that writes the last partial of a unit
    // (sequence, KV head) merges the unit's rows into out; nullable.
    int* unit_left;
    void* out;
    const int2* seq_info;
    int suffix_chunk;     // tokens per suffix partition
};

// Pages of a tensor-core kernel partition (its block-table slice in shared
// memory): multi-query partitions of up to 4096 tokens at 16-token pages,
// one per (sequence, KV head) on a 4096-token context, measured faster than
// two of 2048 (Llama-70B layer, 8 query tokens: 54.9 -> 60.4 % of peak).
constexpr int kPrefixMaxChunkPages = 256;
constexpr int kPrefixTileRows = 128;     // query rows per CTA (MMA M)
constexpr int kPrefixTileTokens = 64;    // tokens per tile (N of S, K of O)
constexpr int kPrefixStages = 4;
// Multi-query modes: ring stages (Q lives in tensor memory, so the ring takes
// the shared memory two CTAs an SM leave).
template <int D> constexpr int mq_stages() { return D == 64 ? 6 : 3; }
constexpr int kPrefixSoftmaxWarps = 8;   // two threads per query row (token halves)
constexpr int kPrefixThreads = (kPrefixSoftmaxWarps + 2) * 32;
constexpr int kPrefixTmaWarp = kPrefixSoftmaxWarps;
constexpr int kPrefixMmaWarp = kPrefixSoftmaxWarps + 1;
constexpr float kRescaleLog2 = 8.f;      // P values stay below 2^8 between rescales

template <int D, int NSTG = kPrefixStages, bool ONE_ACC = false>
struct PrefixTile {
    static constexpr int kRegions = D / 64;                            // 128-byte column blocks
    static constexpr int kQRegionBytes = kPrefixTileRows * 128;
    // ONE_ACC (multi-query modes): Q is the A operand of S from tensor memory,
    // none of it in shared memory
    static constexpr int kQBytes = ONE_ACC ? 0 : kRegions * kQRegionBytes;
    static constexpr int kKVRegionBytes = kPrefixTileTokens * 128;     // 64 tokens x 64 dims
    static constexpr int kHalfBytes = kRegions * kKVRegionBytes;       // K (or V) of one tile
    static constexpr int kStageBytes = 2 * kHalfBytes;
    static constexpr int kXchBytes = 2 * kPrefixTileRows * 8;  // (m, l) per row and half
    // full[stages], empty[stages], s_full[2], p_ready[2], o_done[2], q_ready, drain
    static constexpr int kBarriers = 2 * NSTG + 8;
    static constexpr int kSmemBytes = 1024 + kQBytes + NSTG * kStageBytes + kXchBytes +
                                      kBarriers * 8 + (kPrefixMaxChunkPages + 1) * 4 + 64;
    // S0, S1 (64 columns each; P of the tile overwrites its S as hi/lo 16-bit
    // pairs), O_a, O_b (D columns each).  ONE_ACC: one S/P buffer, Q as 16-bit
    // pairs (D/2 columns) where S1 would be, and only O_a.
    static constexpr uint32_t kColQ = kPrefixTileTokens;
    static constexpr uint32_t kColOa = 2 * kPrefixTileTokens;
    static constexpr uint32_t kColOb = kColOa + D;
    static constexpr uint32_t kTmemEnd = ONE_ACC ? kColOa + D : kColOb + D;
    static constexpr uint32_t kTmemCols = kTmemEnd <= 256 ? 256 : 512;
    static_assert(kTmemEnd <= kTmemCols, "tensor memory layout");
    static_assert(!ONE_ACC || kColQ + D / 2 <= kColOa, "Q fits between S and O");
};

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator, A and B
// of one 16-bit type (0 = fp16, 1 = bf16), A K-major, B K-major or MN-major.
__host__ __device__ constexpr uint32_t mma_idesc(uint32_t fmt, int m, int n, bool b_mn_major) {
    return (1u << 4) | (fmt << 7) | (fmt << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
template <typename T> struct F16Format;
template <> struct F16Format<__half> { static constexpr uint32_t value = 0; };
template <> struct F16Format<__nv_bfloat16> { static constexpr uint32_t value = 1; };

// A group is used only when its bounds and prefix length are sane; otherwise
// its members are decoded in full by the decode kernel (and the error flagged).
__device__ __forceinline__ bool group_valid(const int32_t* group_start,
                                            const int32_t* group_prefix_len, int grp, int num_seqs,
                                            int max_group_size, int max_prefix_len, int block_size,
                                            int max_blocks_per_seq, int& first, int& last,
                                            int& plen) {
    first = group_start[grp];
    last = group_start[grp + 1];
    plen = group_prefix_len[grp];
    return first >= 0 && first <= last && last <= num_seqs && last - first <= max_group_size &&
           plen >= 0 && plen <= max_prefix_len && plen % block_size == 0 &&
           plen <= max_blocks_per_seq * block_size;
}

__device__ __forceinline__ bool prefix_group_valid(const PrefixParams& p, int grp, int& first,
                                                   int& last, int& plen) {
    return group_valid(p.group_start, p.group_prefix_len, grp, p.num_seqs, p.max_group_size,
                       p.max_prefix_len, p.block_size, p.max_blocks_per_seq, first, last, plen);
}

// A bounded wait whose outcome is the same for the whole warp (a lane that
// gives up raises the CTA's abort flag; the warp then leaves together, so
// warp-collective tensor-memory instructions never run on part of a warp).
__device__ __forceinline__ bool warp_wait_phase(uint32_t bar, uint32_t parity,
                                                volatile int* abort_flag, int32_t* err_flag) {
    const bool ok = wait_phase(bar, parity, abort_flag, err_flag);
    return __all_sync(0xffffffffu, ok);
}

// Two fp32 weights as hi + lo 16-bit terms packed in pairs (element 0 in the
// low half).  bf16: both terms by truncation (a bit mask; hi + lo keeps p to
// 2^-14 relative); fp16: both terms rounded to nearest.
__device__ __forceinline__ void split_hi_lo(float p0, float p1, uint32_t& hi, uint32_t& lo,
                                            __nv_bfloat16) {
    const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
    hi = __byte_perm(b0, b1, 0x7632);
    const float r0 = p0 - __uint_as_float(b0 & 0xffff0000u);
    const float r1 = p1 - __uint_as_float(b1 & 0xffff0000u);
    lo = __byte_perm(__float_as_uint(r0), __float_as_uint(r1), 0x7632);
}
__device__ __forceinline__ void split_hi_lo(float p0, float p1, uint32_t& hi, uint32_t& lo, __half) {
    hi = pack2(p0, p1, __half());
    const float2 back = unpack2(hi, __half());
    lo = pack2(p0 - back.x, p1 - back.y, __half());
}

// The plan of a shared-prefix call, one CTA.  Every
// KV head of a sequence has the same suffix partitions, so one block-wide
// scan over the sequences' partition counts places all the units: unit
// (b, g) starts at H_kv * (partitions of the sequences before b) + g * c_b.
// The group bounds are read into shared memory first (when there are at most
// kPlanStagedGroups groups), so each sequence's search of them costs no
// round trips to memory.
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const PlanParams p) {
    __shared__ int s_start[kPlanStagedGroups + 1];
    __shared__ int s_plen[kPlanStagedGroups];
    __shared__ int warp_sum[kPlanThreads / 32];  // exclusive prefix of the warp totals
    __shared__ int s_base;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    constexpr int kWarps = kPlanThreads / 32;
    ptx::launch_dependents();
    ptx::grid_dependency_wait();  // lengths and groups may come from the previous kernel

    // the first sequences' lengths, read while the group bounds are staged
    int n_raw = tid < p.num_seqs ? __ldg(p.context_lens + tid) : 0;
    const bool staged = p.num_groups > 0 && p.num_groups <= kPlanStagedGroups;
    if (staged) {
        for (int i = tid; i <= p.num_groups; i += kPlanThreads) s_start[i] = p.group_start[i];
        for (int i = tid; i < p.num_groups; i += kPlanThreads) s_plen[i] = p.group_prefix_len[i];
    }
    const int32_t* gs = staged ? s_start : p.group_start;
    const int32_t* gp = staged ? s_plen : p.group_prefix_len;
    if (tid == 0) s_base = 0;
    __syncthreads();

    for (int b0 = 0; b0 < p.num_seqs; b0 += kPlanThreads) {
        const int b = b0 + tid;
        int cnt = 0;  // suffix partitions with tokens, per KV head of sequence b
        const int n_next =
            b + kPlanThreads < p.num_seqs ? __ldg(p.context_lens + b + kPlanThreads) : 0;
        if (b < p.num_seqs) {
            // the sequence's (shared-prefix tokens, prefix partials) record, and
            // the prefix CTAs its rows meet: every prefix partition of each
            // 128-row tile that holds one of them
            int2 info = make_int2(0, 0);
            int tiles = 0;
            if (p.num_groups > 0) {
                int lo = 0, hi = p.num_groups - 1;  // last group with group_start <= b
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (gs[mid] <= b) lo = mid; else hi = mid - 1;
                }
                int first, last, plen;
                if (group_valid(gs, gp, lo, p.num_seqs, p.max_group_size, p.max_prefix_len,
                                p.block_size, p.max_blocks_per_seq, first, last, plen) &&
                    first <= b && b < last) {
                    info = make_int2(plen, (plen + p.prefix_chunk - 1) / p.prefix_chunk);
                    const int r0 = (b - first) * p.group;
                    tiles = (r0 + p.group - 1) / kPrefixTileRows - r0 / kPrefixTileRows + 1;
                } else {
                    flag_error(p.err_flag, PKV_EFLAG_GROUP);
                }
            }
            p.seq_info[b] = info;
            const int n = clamped_len(n_raw, p.cap);
            cnt = suffix_partitions(max(0, n - info.x), info.y, p.chunk_tokens);
            const int left = info.y * tiles + cnt;
            for (int g = 0; g < p.num_kv_heads; ++g)
                p.unit_left[(int64_t)b * p.num_kv_heads + g] = left;
        }
        int incl = cnt;  // inclusive warp scan
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        if (lane == 31) warp_sum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int w = lane < kWarps ? warp_sum[lane] : 0;
            int wi = w;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, wi, off);
                if (lane >= off) wi += v;
            }
            if (lane < kWarps) warp_sum[lane] = wi - w;
        }
        __syncthreads();
        const int before = s_base + warp_sum[warp] + incl - cnt;  // partitions of sequences < b
        if (b < p.num_seqs && cnt > 0) {
            int2* dst = p.items + (int64_t)p.num_kv_heads * before;
            for (int g = 0; g < p.num_kv_heads; ++g)
                for (int j = 0; j < cnt; ++j)
                    dst[g * cnt + j] = make_int2(b * p.num_kv_heads + g, j);
        }
        __syncthreads();
        if (tid == kPlanThreads - 1) s_base = before + cnt;
        __syncthreads();
        n_raw = n_next;
    }
    if (tid == 0) *p.item_count = s_base * p.num_kv_heads;
}

// MODE 0: up to 128 query rows, two softmax threads per row (token halves),
// accumulators O_a and O_b.
// MODE 1 (at most 64 query rows in the CTA): rows 64-127 of the tile repeat
// rows 0-63, so the rows' softmax runs on all four SM sub-partitions (a warp
// reaches only its own quarter of the tensor-memory lanes); lane r's thread
// takes tokens 0-31 of each tile and lane r + 64's tokens 32-63.  P rows 0-63
// carry tokens 0-31 and zeros for 32-63, rows 64-127 the reverse, so one
// accumulator holds two independent partial softmaxes of each row (lanes r
// and r + 64), written as partial slots 2 * partition and 2 * partition + 1.
// MODE 2: up to 128 query rows, one softmax thread per row taking all 64
// tokens of each tile, one accumulator.
// MODES 1 and 2 run four softmax warps and 256 tensor-memory columns (one S/P
// buffer, Q as the A operand of S, one accumulator) and a ring of the shared
// memory left: two CTAs share an SM, so one's start and per-tile chain
// overlap the other's.
template <typename T, int D, int MODE = 0>
__global__ void __launch_bounds__((MODE != 0 ? 4 : kPrefixSoftmaxWarps) * 32 + 64, MODE != 0 ? 2 : 1)
prefix_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
              const PrefixParams p) {
    constexpr bool ONE = MODE != 0;   // one thread per lane, one accumulator, two CTAs an SM
    constexpr bool PAIR = MODE == 1;  // rows 64-127 repeat rows 0-63
    constexpr int SW = ONE ? 4 : kPrefixSoftmaxWarps;  // softmax warps; then the TMA and MMA warps
    constexpr int NS = ONE ? mq_stages<D>() : kPrefixStages;
    constexpr int NSB = ONE ? 1 : 2;  // S/P buffers: tile j uses buffer j % NSB
    using Cfg = PrefixTile<D, NS, ONE>;
    constexpr int R = Cfg::kRegions;
    constexpr int KSTEPS = D / 16;
    constexpr int TT = kPrefixTileTokens;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* sq = smem;                          // Q: [region][128 rows][128 B], swizzled
    uint8_t* ring = sq + Cfg::kQBytes;           // stages of K [region][64][128 B], then V
    float2* xch = reinterpret_cast<float2*>(ring + NS * Cfg::kStageBytes);  // [half][row] (m, l)
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring + NS * Cfg::kStageBytes + Cfg::kXchBytes);
    uint64_t* full_bar = bars;
    uint64_t* empty_bar = bars + NS;
    // MODE 0: tile j uses S/P buffer j % 2 with its own s_full and p_ready
    // barriers (MODES 1-2: the one buffer and barrier 0, S(j) issued after
    // P V(j-1), so S(j) completing implies P V(j-1) has).  MODE 0: a
    // softmax thread passes S(j+1) only after P V(j-1) was issued, i.e. after
    // p_ready of buffer (j+1) % 2 completed for tile j-1, so its arrival for
    // tile j+1 never lands in an earlier tile's phase.
    uint64_t* s_full = bars + 2 * NS;  // [2]
    uint64_t* p_ready = s_full + 2;    // [2]
    uint64_t* o_done = p_ready + 2;  // [2]: O += P V of even / odd tiles done
    uint64_t* q_ready = o_done + 2;
    uint64_t* drain = q_ready + 1;
    int* table = reinterpret_cast<int*>(bars + Cfg::kBarriers);
    volatile int* abort_flag = table + kPrefixMaxChunkPages + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(table + kPrefixMaxChunkPages + 2);
    int* warp_lim = table + kPrefixMaxChunkPages + 3;  // [SW]

    const int rt = blockIdx.x;                     // tile of 128 query rows
    const int g = blockIdx.y % p.num_kv_heads;     // KV head
    const int grp = blockIdx.y / p.num_kv_heads;   // group (shared prefix) or sequence (multi-query)
    const int part = blockIdx.z;                   // partition of the tokens
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int bs = p.block_size;
    const int bs_shift = __ffs(bs) - 1;  // block sizes are powers of two

    ptx::launch_dependents();
    ptx::grid_dependency_wait();

    // The CTA's query rows and tokens.  Shared prefix (q_len == 0): row r is
    // query head g*group + r % group of member first + r / group of group grp,
    // against the group's prefix tokens.  Multi-query (q_len > 0): row r is
    // query head g*group + r % group of query token i = r / group of sequence
    // grp, against the sequence's context, causal within the chunk of q_len
    // new tokens (token i sees positions < n - q_len + 1 + i).
    int first, rows, t_limit, n_seq = 0;
    if (p.q_len == 0) {
        if (grp >= p.num_groups) return;
        int last, plen;
        if (!prefix_group_valid(p, grp, first, last, plen)) return;
        rows = (last - first) * p.group;
        t_limit = plen;
    } else {
        first = grp;
        const int n_raw = __ldg(p.context_lens + first);
        if ((n_raw < 0 || n_raw > p.cap || n_raw < p.q_len) && rt == 0 && g == 0 && part == 0 &&
            threadIdx.x == 0)
            flag_error(p.err_flag, PKV_EFLAG_CONTEXT_LEN);
        n_seq = clamped_len(n_raw, p.cap);
        rows = p.q_len * p.group;
        t_limit = n_seq;
    }
    const int row0 = rt * kPrefixTileRows;
    const int t_begin = part * p.prefix_chunk;
    const int t_chunk_end = min(t_limit, t_begin + p.prefix_chunk);
    if (row0 >= rows || t_begin >= t_chunk_end) return;
    const int page0 = t_begin / bs;

    // This thread's query row (softmax warps): its row of q and of the
    // partials ([rows of q][H_q]), its context limit, and its token half.
    const int srow = 32 * (warp % 4) + lane;  // row within the tile = tensor-memory lane
    const int half = warp / 4;                // tokens 32*half .. 32*half+31 of every tile
    const int dcopy = PAIR ? (srow >> 6) : 0;  // MODE 1: which copy of the row this lane holds
    const int r = row0 + (PAIR ? (srow & 63) : srow);
    const bool row_ok = warp < SW && r < rows;
    const int head = g * p.group + (row_ok ? r % p.group : 0);
    int64_t qrow;
    int lim = 0;
    if (p.q_len == 0) {
        const int seq = first + (row_ok ? r / p.group : 0);
        qrow = (int64_t)seq * p.num_q_heads + head;
        if (row_ok) lim = clamped_len(__ldg(p.context_lens + seq), p.cap);
    } else {
        const int i = row_ok ? r / p.group : 0;
        qrow = ((int64_t)first * p.q_len + i) * p.num_q_heads + head;
        if (row_ok) lim = max(0, n_seq - p.q_len + 1 + i);
    }

    if (tid == 0) {
        for (int st = 0; st < NS; ++st) {
            ptx::mbar_init(ptx::smem_addr(&full_bar[st]), 1);
            ptx::mbar_init(ptx::smem_addr(&empty_bar[st]), 1);
        }
        ptx::mbar_init(ptx::smem_addr(&s_full[0]), 1);
        ptx::mbar_init(ptx::smem_addr(&s_full[1]), 1);
        ptx::mbar_init(ptx::smem_addr(&p_ready[0]), SW * 32);
        ptx::mbar_init(ptx::smem_addr(&p_ready[1]), SW * 32);
        ptx::mbar_init(ptx::smem_addr(&o_done[0]), 1);
        ptx::mbar_init(ptx::smem_addr(&o_done[1]), 1);
        ptx::mbar_init(ptx::smem_addr(q_ready), SW * 32);
        ptx::mbar_init(ptx::smem_addr(drain), 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    // The softmax threads' halves of their query rows, loaded before the barrier
    // below so the load overlaps the block-table read (stored to shared memory
    // after it).
    constexpr int QV = ONE ? D / 8 : D / 16;  // 16-byte pieces per thread (whole row, or half)
    uint4 qv[QV];
    if (warp < SW) {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) + qrow * D);
#pragma unroll
        for (int k = 0; k < QV; ++k)
            qv[k] = row_ok ? __ldg(src + half * QV + k) : make_uint4(0u, 0u, 0u, 0u);
        int m = lim;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (lane == 0) warp_lim[warp] = m;
    } else if (warp == SW) {
        // The partition's slice of the block table (from the first member's row).
        const int npages = (t_chunk_end + bs - 1) / bs - page0;
        const int32_t* trow = p.block_tables + (int64_t)first * p.max_blocks_per_seq + page0;
        for (int i = lane; i < npages; i += 32) {
            int blk = __ldg(trow + i);
            if (blk < 0 || blk >= p.num_blocks) {
                flag_error(p.err_flag, PKV_EFLAG_BLOCK_ID);
                blk = -1;
            }
            table[i] = blk;
        }
        if (lane == 0) {
            ptx::prefetch_tensormap(&tm_k);
            ptx::prefetch_tensormap(&tm_v);
        }
    } else {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), Cfg::kTmemCols);
        ptx::tmem_relinquish_alloc_permit();
    }
#ifdef PKV_DEBUG
    poison_smem(ring, NS * Cfg::kStageBytes, tid, (SW + 2) * 32);
#endif
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // Tokens past every row's context take no part for any row of this CTA: not read.
    int max_lim = 0;
#pragma unroll
    for (int w = 0; w < SW; ++w) max_lim = max(max_lim, warp_lim[w]);
    const int t_end = min(t_chunk_end, max(t_begin, max_lim));
    const int ntiles = (t_end - t_begin + TT - 1) / TT;
    const uint32_t ring_addr = ptx::smem_addr(ring);
    const uint32_t q_addr = ptx::smem_addr(sq);
    auto sbuf = [](int j) { return j % NSB; };          // S/P buffer of tile j
    auto sphase = [](int j) { return (j / NSB) & 1; };  // its barriers' phase parity

    if (warp == SW) {
        // ------------------------------------------------------------ producer
        // The tile's box loads (16-token page box x 64-dim region x K/V) are
        // spread over the warp's lanes: one thread issuing them in turn is the
        // bottleneck of this kernel, several lanes issue them at once.
        constexpr int kBoxes = TT / kStageTokens;
        constexpr int kLoads = kBoxes * R * 2;
        static_assert(kLoads <= 32, "one load per lane");
        const uint64_t policy = ptx::l2_policy_evict_last();  // other row tiles read it too
        const int bx = lane / (R * 2);
        const int rr = (lane / 2) % R;
        const bool is_v = lane & 1;
        int issued = 0;
        for (int j = 0; j < ntiles; ++j) {
            const int slot = j % NS;
            if (j >= NS && !warp_wait_phase(ptx::smem_addr(&empty_bar[slot]), ((j / NS) - 1) & 1,
                                            abort_flag, p.err_flag))
                break;
#ifdef PKV_DEBUG
            // the tensor core has finished reading the slot: nothing may read it again
            // before this tile's copies land
            if (j >= NS) {
                ptx::tc_fence_after_sync();
                poison_smem(ring + slot * Cfg::kStageBytes, Cfg::kStageBytes, lane, 32);
                __syncwarp();
            }
#endif
            const uint32_t kdst = ring_addr + slot * Cfg::kStageBytes;
            const uint32_t fb = ptx::smem_addr(&full_bar[slot]);
            const int tok0 = t_begin + j * TT + bx * kStageTokens;
            const int blk = lane < kLoads && tok0 < t_end ? table[(tok0 >> bs_shift) - page0] : -1;
            const uint32_t loads = __ballot_sync(0xffffffffu, blk >= 0);
            if (lane == 0) {
                if (loads == 0)
                    ptx::mbar_arrive(fb);  // nothing to load: every token of the tile is masked
                else
                    ptx::mbar_arrive_expect_tx(fb, __popc(loads) * kStageTokens * 128);
            }
            __syncwarp();
            if (blk >= 0) {
                const uint32_t off = (is_v ? Cfg::kHalfBytes : 0) + rr * Cfg::kKVRegionBytes +
                                     bx * kStageTokens * 128;
                load_kv_box(kdst + off, is_v ? &tm_v : &tm_k, fb, rr * 64, g, tok0 & (bs - 1), blk,
                            p.hnd, policy);
            }
            issued = j + 1;
        }
        if (lane == 0 && *abort_flag) {
            for (int j = max(0, issued - NS); j < issued; ++j) {
                const uint32_t fb = ptx::smem_addr(&full_bar[j % NS]);
                const uint64_t t0 = ptx::globaltimer();
                while (!ptx::mbar_try_wait(fb, (j / NS) & 1) &&
                       ptx::globaltimer() - t0 < kWaitLimitNs) {
                }
            }
        }
    } else if (warp == (SW + 1)) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t fmt = F16Format<T>::value;
            constexpr uint32_t idesc_s = mma_idesc(fmt, kPrefixTileRows, TT, false);
            constexpr uint32_t idesc_o = mma_idesc(fmt, kPrefixTileRows, D, true);
            bool ok = wait_phase(ptx::smem_addr(q_ready), 0, abort_flag, p.err_flag);
            if (ok) ptx::tc_fence_after_sync();
            // S(j) = Q K(j)^T into S buffer j % 2 (tile j's K/V have landed)
            auto issue_s = [&](int j) {
                const int slot = j % NS;
                ptx::tc_fence_after_sync();
                const uint32_t kb = ring_addr + slot * Cfg::kStageBytes;
#pragma unroll
                for (int ks = 0; ks < KSTEPS; ++ks) {
                    const uint32_t koff = (ks / 4) * Cfg::kQRegionBytes + (ks % 4) * 32;
                    const uint64_t b = ptx::smem_desc_sw128(
                        kb + (ks / 4) * Cfg::kKVRegionBytes + (ks % 4) * 32, 16, 1024);
                    if constexpr (ONE) {
                        // A = Q from tensor memory: 16 dims = 8 columns a step
                        ptx::tc_mma_f16_ts(tmem, tmem + Cfg::kColQ + ks * 8, b, idesc_s,
                                           ks > 0 ? 1u : 0u);
                    } else {
                        const uint64_t a = ptx::smem_desc_sw128(q_addr + koff, 16, 1024);
                        ptx::tc_mma_f16(tmem + (j % 2) * TT, a, b, idesc_s, ks > 0 ? 1u : 0u);
                    }
                }
                ptx::tc_commit(ptx::smem_addr(&s_full[sbuf(j)]));
            };
            // O += P(j) V(j) (the softmax has written P(j))
            auto issue_pv = [&](int j) {
                ptx::tc_fence_after_sync();
                const uint32_t vb = ring_addr + (j % NS) * Cfg::kStageBytes + Cfg::kHalfBytes;
                constexpr int HTK = MODE == 2 ? TT : TT / 2;  // tokens per softmax thread
#pragma unroll
                for (int kt = 0; kt < TT / 16; ++kt) {
                    // tokens 0-31 accumulate into O_a, tokens 32-63 into O_b; MODES 1
                    // and 2: every step into the one accumulator
                    const bool to_a = ONE || kt < TT / 32;
                    const uint32_t acc = tmem + (to_a ? Cfg::kColOa : Cfg::kColOb);
                    const uint32_t keep = (j > 0 || (ONE ? kt > 0 : kt % (TT / 32) > 0)) ? 1u : 0u;
                    const uint64_t b = ptx::smem_desc_sw128(vb + kt * 16 * 128, Cfg::kKVRegionBytes, 1024);
                    // tokens 16kt.. of P: unit u's hi pairs at u*HTK, lo pairs HTK/2 on
                    const int u = kt * 16 / HTK;
                    const uint32_t a_hi = tmem + sbuf(j) * TT + u * HTK + (kt * 16 % HTK) / 2;
                    ptx::tc_mma_f16_ts(acc, a_hi, b, idesc_o, keep);
                    ptx::tc_mma_f16_ts(acc, a_hi + HTK / 2, b, idesc_o, 1u);
                }
                ptx::tc_commit(ptx::smem_addr(&o_done[j % 2]));
                ptx::tc_commit(ptx::smem_addr(&empty_bar[j % NS]));
            };
            if constexpr (ONE) {
                // One thread issues both kinds as their inputs become ready, so
                // a product whose P is written never queues behind an S whose
                // copy is in flight.  S(j) may start once P V(j-1), the last
                // reader of the one S/P buffer, is issued (the tensor core runs
                // them in order).
                int next_s = 0, next_pv = 0;
                uint64_t t_last = ptx::globaltimer();
                while (ok && next_pv < ntiles) {
                    bool moved = false;
                    if (next_pv < next_s &&
                        ptx::mbar_try_wait(ptx::smem_addr(&p_ready[sbuf(next_pv)]), sphase(next_pv))) {
                        issue_pv(next_pv++);
                        moved = true;
                    }
                    if (next_s < ntiles && next_s < next_pv + NSB &&
                        ptx::mbar_try_wait(ptx::smem_addr(&full_bar[next_s % NS]), (next_s / NS) & 1)) {
                        issue_s(next_s++);
                        moved = true;
                    }
                    if (moved) {
                        t_last = ptx::globaltimer();
                    } else if (*abort_flag) {
                        ok = false;
                    } else if (ptx::globaltimer() - t_last > kWaitLimitNs) {
                        *abort_flag = 1;
                        flag_error(p.err_flag, PKV_EFLAG_TIMEOUT);
                        ok = false;
                    }
                }
            } else {
                auto wait_s = [&](int j) {
                    return wait_phase(ptx::smem_addr(&full_bar[j % NS]), (j / NS) & 1, abort_flag,
                                      p.err_flag);
                };
                for (int j = 0; j < 2 && j < ntiles && ok; ++j) {
                    ok = wait_s(j);
                    if (ok) issue_s(j);
                }
                for (int j = 0; j < ntiles && ok; ++j) {
                    if (!wait_phase(ptx::smem_addr(&p_ready[sbuf(j)]), sphase(j), abort_flag,
                                    p.err_flag)) {
                        ok = false;
                        break;
                    }
                    issue_pv(j);
                    if (j + 2 < ntiles) {
                        ok = wait_s(j + 2);
                        if (ok) issue_s(j + 2);
                    }
                }
            }
            // every MMA has completed before the tensor memory is released
            ptx::tc_commit(ptx::smem_addr(drain));
            const uint64_t t0 = ptx::globaltimer();
            while (!ptx::mbar_try_wait(ptx::smem_addr(drain), 0) &&
                   ptx::globaltimer() - t0 < kWaitLimitNs) {
            }
        }
    } else {
        // ------------------------------------------------------------ softmax rows
        constexpr int HT = MODE == 2 ? TT : TT / 2;  // tokens per thread and tile
        constexpr int HB = HT / kStageTokens;         // 16-token boxes per thread
        // this thread's tokens of every tile: unit `unit` of HT tokens
        const int unit = PAIR ? dcopy : MODE == 2 ? 0 : half;
        const uint32_t lane_base = (uint32_t)(32 * (warp % 4)) << 16;
        if constexpr (ONE) {
            // This thread's row of Q into its tensor-memory lane, dims 2c and
            // 2c+1 in column kColQ + c (the A operand layout of S = Q K^T).
            static_assert(QV % 8 == 0, "whole 32-column stores");
#pragma unroll
            for (int h = 0; h < QV / 8; ++h)
                ptx::tmem_st32(tmem + lane_base + Cfg::kColQ + h * 32,
                               *reinterpret_cast<const uint32_t(*)[32]>(qv + h * 8));
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(ptx::smem_addr(q_ready));
        } else {
            // This thread's half of its row of Q into shared memory (16-byte
            // chunk c of a 128-byte row lands at chunk c ^ (row % 8): the
            // 128-byte swizzle of the MMA operand).
#pragma unroll
            for (int k = 0; k < QV; ++k) {
                const int c = half * QV + k;
                *reinterpret_cast<uint4*>(sq + (c / 8) * Cfg::kQRegionBytes + srow * 128 +
                                          (((c % 8) ^ (srow & 7)) << 4)) = qv[k];
            }
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(ptx::smem_addr(q_ready));
        }
        const uint32_t col_o = (half && !ONE) ? Cfg::kColOb : Cfg::kColOa;  // this thread's accumulator
        float m_ref = -INFINITY;  // reference max of this half's P (log2 domain)
        float l = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            if (!warp_wait_phase(ptx::smem_addr(&s_full[sbuf(j)]), sphase(j), abort_flag,
                                 p.err_flag)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after_sync();
            uint32_t sv[HT];
#pragma unroll
            for (int h = 0; h < HT / 32; ++h)
                ptx::tmem_ld32(tmem + lane_base + sbuf(j) * TT + unit * HT + h * 32,
                               *reinterpret_cast<uint32_t(*)[32]>(sv + h * 32));
            const int tile0 = t_begin + j * TT;
            const int h0 = tile0 + unit * HT;  // first token of this thread's unit
            // Tokens present (a valid block, before t_end), per 16-token box of the tile.
            int nvalid[TT / kStageTokens];
#pragma unroll
            for (int bx = 0; bx < TT / kStageTokens; ++bx) {
                const int tok0 = tile0 + bx * kStageTokens;
                nvalid[bx] = (tok0 < t_end && table[(tok0 >> bs_shift) - page0] >= 0)
                                 ? min(kStageTokens, t_end - tok0)
                                 : 0;
            }
            bool complete = h0 + HT <= lim;
#pragma unroll
            for (int bx = 0; bx < HB; ++bx) complete &= nvalid[unit * HB + bx] == kStageTokens;
            float sc[HT];
#pragma unroll
            for (int i = 0; i < HT; ++i) sc[i] = __uint_as_float(sv[i]) * p.scale_log2;
            if (!complete) {
#pragma unroll
                for (int i = 0; i < HT; ++i)
                    if (!((i % kStageTokens) < nvalid[unit * HB + i / kStageTokens] && h0 + i < lim))
                        sc[i] = -INFINITY;
            }
            // max, as a tree
            float red[HT / 2];
#pragma unroll
            for (int i = 0; i < HT / 2; ++i) red[i] = fmaxf(sc[i], sc[i + HT / 2]);
#pragma unroll
            for (int w = HT / 4; w > 0; w >>= 1)
#pragma unroll
                for (int i = 0; i < w; ++i) red[i] = fmaxf(red[i], red[i + w]);
            const float mx = red[0];
            float alpha = 1.f;
            bool rescale = false;
            if (m_ref == -INFINITY) {
                m_ref = mx;  // O and l of this half are still zero for this row
            } else if (mx > m_ref + kRescaleLog2) {
                alpha = ptx::ex2_approx(m_ref - mx);
                m_ref = mx;
                rescale = true;
            }
            const float ref = m_ref == -INFINITY ? 0.f : m_ref;
#pragma unroll
            for (int i = 0; i < HT; ++i) sc[i] = ptx::ex2_approx(sc[i] - ref);
            // sum, as a tree
#pragma unroll
            for (int i = 0; i < HT / 2; ++i) red[i] = sc[i] + sc[i + HT / 2];
#pragma unroll
            for (int w = HT / 4; w > 0; w >>= 1)
#pragma unroll
                for (int i = 0; i < w; ++i) red[i] += red[i + w];
            l = l * alpha + red[0];
            // O is rescaled only once the previous tile's O += P V has completed
            // (o_done alternates between two barriers, so the parity wait can
            // never meet a phase two behind: S(j) completing implies P V(j-2) has).
            if (__any_sync(0xffffffffu, rescale)) {
                if (j > 0 && !warp_wait_phase(ptx::smem_addr(&o_done[(j - 1) % 2]),
                                              ((j - 1) / 2) & 1, abort_flag, p.err_flag)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after_sync();
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t ov[32];
                    const uint32_t ta = tmem + lane_base + col_o + c * 32;
                    ptx::tmem_ld32(ta, ov);
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                    ptx::tmem_st32(ta, ov);
                }
            }
            // P as hi + lo 16-bit terms over this thread's own S columns of the
            // tile's buffer (already read): the HT/2 columns of hi pairs, then
            // the HT/2 of lo pairs; the MMA takes them as its A operand.
            {
                uint32_t pv[HT];
#pragma unroll
                for (int e = 0; e < HT / 2; ++e)
                    split_hi_lo(sc[2 * e], sc[2 * e + 1], pv[e], pv[HT / 2 + e], T());
#pragma unroll
                for (int h = 0; h < HT / 32; ++h)
                    ptx::tmem_st32(tmem + lane_base + sbuf(j) * TT + unit * HT + h * 32,
                                   *reinterpret_cast<const uint32_t(*)[32]>(pv + h * 32));
                if constexpr (PAIR) {
                    // The other copy's half of this lane (S values no thread reads)
                    // must be zero for the steps that bring it into this lane's O.
                    uint32_t z[HT];
#pragma unroll
                    for (int e = 0; e < HT; ++e) z[e] = 0u;
                    ptx::tmem_st32(tmem + lane_base + sbuf(j) * TT + (1 - dcopy) * HT, z);
                }
            }
            // V rows of tokens that were not loaded hold stale or uninitialised
            // bytes: zero them so 0 * V stays 0.
            bool partial = false;
#pragma unroll
            for (int bx = 0; bx < TT / kStageTokens; ++bx) partial |= nvalid[bx] < kStageTokens;
            if (partial) {
                uint8_t* vst = ring + (j % NS) * Cfg::kStageBytes + Cfg::kHalfBytes;
                for (int idx = tid; idx < TT * R * 8; idx += SW * 32) {
                    const int row = idx / (R * 8);
                    const int rem = idx - row * (R * 8);
                    if (row % kStageTokens >= nvalid[row / kStageTokens])
                        *reinterpret_cast<uint4*>(vst + (rem / 8) * Cfg::kKVRegionBytes + row * 128 +
                                                  (rem % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(ptx::smem_addr(&p_ready[sbuf(j)]));
        }
        if (ok && ntiles > 0)
            ok = warp_wait_phase(ptx::smem_addr(&o_done[(ntiles - 1) % 2]), ((ntiles - 1) / 2) & 1,
                                 abort_flag, p.err_flag);
        // The two halves of each row meet: every softmax thread passes this
        // barrier exactly once, aborted or not.
        xch[half * kPrefixTileRows + srow] = make_float2(m_ref, l);
        ptx::named_barrier_sync(1, SW * 32);
        if constexpr (ONE) {
            if (ok && !*abort_flag) {
                // Each lane's partial softmax on its own: O / l and its log-sum-exp,
                // as partial slot part (MODE 1: 2 * part + copy).
                ptx::tc_fence_after_sync();
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const int64_t prow = qrow * p.num_splits + (PAIR ? 2 * part + dcopy : part);
                float* dst = p.partial_o + prow * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t ov[32];
                    if (ntiles > 0) {
                        ptx::tmem_ld32(tmem + lane_base + Cfg::kColOa + c * 32, ov);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] = 0u;
                    }
                    if (row_ok) {
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            float4 v;
                            v.x = __uint_as_float(ov[i]) * inv;
                            v.y = __uint_as_float(ov[i + 1]) * inv;
                            v.z = __uint_as_float(ov[i + 2]) * inv;
                            v.w = __uint_as_float(ov[i + 3]) * inv;
                            *reinterpret_cast<float4*>(dst + c * 32 + i) = v;
                        }
                    }
                }
                if (row_ok)
                    p.partial_lse[prow] = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
            }
        } else if (ok && !*abort_flag) {
            // Epilogue: O = (2^(m_a - M) O_a + 2^(m_b - M) O_b) / L with M the larger
            // reference and L = 2^(m_a - M) l_a + 2^(m_b - M) l_b; this thread
            // writes columns half*D/2 .. half*D/2 + D/2 - 1 of its row, as prefix
            // partial `part`, and (half 0) the log-sum-exp.
            ptx::tc_fence_after_sync();
            const float2 ha = xch[srow];
            const float2 hb = xch[kPrefixTileRows + srow];
            const float mm = fmaxf(ha.x, hb.x);
            const float fa = ha.x == -INFINITY ? 0.f : ptx::ex2_approx(ha.x - mm);
            const float fb = hb.x == -INFINITY ? 0.f : ptx::ex2_approx(hb.x - mm);
            const float L = ha.y * fa + hb.y * fb;
            const float inv = L > 0.f ? 1.f / L : 0.f;
            const int64_t prow = qrow * p.num_splits + part;
            float* dst = p.partial_o + prow * D + half * (D / 2);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t oa[32], ob[32];
                if (ntiles > 0) {
                    const uint32_t cbase = tmem + lane_base + half * (D / 2) + c * 32;
                    ptx::tmem_ld32(cbase + Cfg::kColOa, oa);
                    ptx::tmem_ld32(cbase + Cfg::kColOb, ob);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) oa[i] = ob[i] = 0u;
                }
                if (row_ok) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        float4 v;
                        v.x = L > 0.f ? (__uint_as_float(oa[i]) * fa + __uint_as_float(ob[i]) * fb) * inv : 0.f;
                        v.y = L > 0.f ? (__uint_as_float(oa[i + 1]) * fa + __uint_as_float(ob[i + 1]) * fb) * inv : 0.f;
                        v.z = L > 0.f ? (__uint_as_float(oa[i + 2]) * fa + __uint_as_float(ob[i + 2]) * fb) * inv : 0.f;
                        v.w = L > 0.f ? (__uint_as_float(oa[i + 3]) * fa + __uint_as_float(ob[i + 3]) * fb) * inv : 0.f;
                        *reinterpret_cast<float4*>(dst + c * 32 + i) = v;
                    }
                }
            }
            if (row_ok && half == 0)
                p.partial_lse[prow] = L > 0.f ? (mm + log2f(L)) * kLn2 : -INFINITY;
        }
    }

    if (MODE == 0 && p.unit_left != nullptr) __threadfence();  // partials, before the counts
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == (SW + 1)) {
        __syncwarp();
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, Cfg::kTmemCols);
    }

    // Shared prefixes: the tile's rows are one contribution to each of its
    // members' units; the CTA that makes a unit's last contribution merges the
    // unit's rows (the plan counted P partitions x the tiles a member's rows
    // span, plus the member's suffix partitions).
    if constexpr (MODE == 0) {
        if (p.unit_left != nullptr && !*abort_flag) {
            int* list = table;  // the table slice is not read after the main loop
            const int m_lo = row0 / p.group;
            const int m_hi = (min(rows, row0 + kPrefixTileRows) - 1) / p.group;
            if (tid == 0) list[0] = 0;
            __syncthreads();
            if (tid <= m_hi - m_lo) {
                const int seq = first + m_lo + tid;
                if (atomicAdd(p.unit_left + (int64_t)seq * p.num_kv_heads + g, -1) == 1)
                    list[1 + atomicAdd(&list[0], 1)] = seq;
            }
            __syncthreads();
            const int nm = list[0];
            if (nm > 0) {
                __threadfence();
                MergeParams mp = {};
                mp.out = p.out;
                mp.partial_o = p.partial_o;
                mp.partial_lse = p.partial_lse;
                mp.context_lens = p.context_lens;
                mp.seq_info = p.seq_info;
                mp.num_q_heads = p.num_q_heads;
                mp.num_kv_heads = p.num_kv_heads;
                mp.group = p.group;
                mp.num_splits = p.num_splits;
                mp.head_dim = D;
                mp.chunk_tokens = p.suffix_chunk;
                mp.cap = p.cap;
                for (int k = warp; k < nm * p.group; k += (SW + 2))
                    merge_row<T>(mp, (int64_t)list[1 + k / p.group] * p.num_q_heads +
                                         g * p.group + k % p.group,
                                 lane);
            }
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kMergeThreads)
merge_kernel(const MergeParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kMergeRowsPerCta + (threadIdx.x >> 5);
    ptx::launch_dependents();
    ptx::grid_dependency_wait();
    if (row >= p.rows) return;
    merge_row<T>(p, row, lane);
}

// Self-test of the bounded wait: one warp waits on a barrier phase that
// nothing completes, so the wait must give up after limit_ns, raise
// PKV_EFLAG_TIMEOUT and return.
__global__ void __launch_bounds__(32) wait_timeout_selftest_kernel(int32_t* err_flag,
                                                                   uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_word;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_addr(&bar), 1);
        abort_word = 0;
        ptx::fence_barrier_init();
    }
    __syncwarp();
    wait_phase(ptx::smem_addr(&bar), 0, &abort_word, err_flag, limit_ns);
}

// ---------------------------------------------------------------------------
// Host side: split planning, tensor maps, launches
// ---------------------------------------------------------------------------

static int current_sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    if (dev < 0 || dev >= 64) return -1;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
        cudaGetLastError();
        return -1;
    }
    cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

// The stream on which a shared-prefix call runs its prefix kernel beside the
// suffix decode on the caller's stream, with the events that fork it from the
// caller's stream and join it back: one set per CUDA context, made on the
// context's first such call and kept for the life of the process.  It has the
// highest priority the device offers, so that the prefix CTAs (one an SM)
// are placed first when both grids wait for SMs.  The mutex is held from the
// fork to the join, so calls from several host threads never see one
// another's event records.
struct SideStream {
    unsigned long long ctx_id;
    cudaStream_t stream;
    cudaEvent_t fork, join;
};
constexpr int kMaxSideStreams = 64;
static std::mutex g_side_mutex;
static SideStream g_side[kMaxSideStreams];
static int g_side_count = 0;

// The current context's side stream, made if need be; nullptr when there is
// none to be had (no context id, more contexts than entries, or the runtime
// refused), in which case the caller runs the prefix on its own stream.
// Call with g_side_mutex held.
static const SideStream* side_stream_locked() {
    unsigned long long id = 0;
    if (!current_context_id(&id)) return nullptr;
    for (int i = 0; i < g_side_count; ++i)
        if (g_side[i].ctx_id == id) return &g_side[i];
    if (g_side_count == kMaxSideStreams) return nullptr;
    SideStream e = {id, nullptr, nullptr, nullptr};
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess ||
        cudaStreamCreateWithPriority(&e.stream, cudaStreamNonBlocking, greatest) != cudaSuccess ||
        cudaEventCreateWithFlags(&e.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&e.join, cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        if (e.join) cudaEventDestroy(e.join);
        if (e.fork) cudaEventDestroy(e.fork);
        if (e.stream) cudaStreamDestroy(e.stream);
        cudaGetLastError();
        return nullptr;
    }
    g_side[g_side_count] = e;
    return &g_side[g_side_count++];
}

struct Plan {
    int num_splits;      // partitions per sequence, at most
    int chunk_tokens;
    size_t workspace_bytes;
};

// Validates the shape arguments shared by planning and launching.
static pkv_status check_shapes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                               int block_size, int max_context_len, int num_splits) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || max_context_len < 0 || num_splits < 0 || num_splits > PKV_MAX_SPLITS)
        return PKV_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    if (!supported_head_dim(head_dim) || !supported_block_size(block_size) ||
        num_q_heads / num_kv_heads > kMaxGroup)
        return PKV_ERR_UNSUPPORTED;
    if (num_seqs > 65535 || num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

// Partitions: whole 16-token stages, whatever the page size; the automatic
// plan sizes them from 256 to 2048 tokens by an estimate of the time (see the
// loop).  ctas_per_sm: the decode kernel's resident CTAs an SM (3, or 4 for
// the E4M3 kernel at one 8-column group); unit_mult: CTAs per (sequence, KV
// head) and partition (the multi-query row blocks).
constexpr double kCtaStartTokens = 384.0;  // a CTA's fixed start, in tokens streamed
static pkv_status make_plan(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, int max_context_len, int num_splits, Plan* plan,
                            int ctas_per_sm = 3, int unit_mult = 1) {
    pkv_status st = check_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                 max_context_len, num_splits);
    if (st != PKV_OK) return st;
    // Partitions are whole 16-token stages (a stage box may start anywhere in a
    // page), at most kMaxChunkPages pages long so a partition's slice of the
    // block table, starting mid-page, fits kMaxChunkPages + 1 entries.
    const int max_stages = std::max(1, (max_context_len + kStageTokens - 1) / kStageTokens);
    const int cap_stages = kMaxChunkPages * block_size / kStageTokens;
    int chunk_stages;
    if (num_splits == 0) {
        const int sms = current_sm_count();
        if (sms <= 0) return PKV_ERR_CUDA;
        // From 256 to 2048 tokens.  Equal-length CTAs (at the longest
        // context) run in waves of resident CTAs; every wave costs its
        // partition's tokens plus a CTA's fixed start (context length and
        // block-table reads, the first copy round trip), kCtaStartTokens in
        // tokens streamed.  The count with the least (waves rounded up) x
        // (tokens + start) wins, the fewest partitions among equals.  A
        // partly filled last wave costs less than this counts (fewer CTAs on
        // an SM still draw most of its bandwidth), more waves cost their
        // starts: measured on the Llama-70B layer (32 x 4096 tokens, GQA-8),
        // 5 partitions (2.8 waves) ran at 89.6 % of peak, the 7 of a
        // fill-the-last-wave rule (3.9 waves) at 86.9 %; allowing partitions
        // of up to 2048 tokens (3 partitions, 1.7 waves) 91.7 %.
        const int64_t units = (int64_t)std::max(1, num_seqs) * num_kv_heads * unit_mult;
        const double slots = (double)ctas_per_sm * sms;
        const int min_chunk = 256 / kStageTokens, max_chunk = std::min(2048 / kStageTokens, cap_stages);
        const int lo = std::max(1, (max_stages + max_chunk - 1) / max_chunk);
        const int hi = std::max(lo, std::min(PKV_MAX_SPLITS, (max_stages + min_chunk - 1) / min_chunk));
        // A count whose CTAs do not fill one wave leaves resident slots idle
        // with nothing to come: it is taken only when no count fills one (the
        // E4M3 Llama-70B layer: 2 partitions of 2048 tokens, 0.84 waves, 62.4 %
        // against 66.8 % for 4).
        double best = 0.0, best_fill = 0.0;
        int chunk_fill = 0;
        chunk_stages = (max_stages + lo - 1) / lo;
        for (int s = lo; s <= hi; ++s) {
            const int cs = (max_stages + s - 1) / s;
            const int splits = (max_stages + cs - 1) / cs;
            if (splits != s) continue;  // the same partition as a smaller count
            const double ctas = (double)units * splits;
            const double waves = std::ceil(ctas / slots);
            const double cost = waves * (cs * kStageTokens + kCtaStartTokens);
            if (s == lo || cost < best - 1e-9) {
                best = cost;
                chunk_stages = cs;
            }
            if (ctas >= slots && (chunk_fill == 0 || cost < best_fill - 1e-9)) {
                best_fill = cost;
                chunk_fill = cs;
            }
        }
        if (chunk_fill > 0) chunk_stages = chunk_fill;
    } else {
        chunk_stages = (max_stages + num_splits - 1) / num_splits;
    }
    chunk_stages = std::min(std::max(chunk_stages, 1), cap_stages);
    const int chunk = chunk_stages * kStageTokens;
    const int64_t splits64 = std::max<int64_t>(1, ((int64_t)max_context_len + chunk - 1) / chunk);
    if (splits64 > PKV_MAX_SPLITS) return PKV_ERR_UNSUPPORTED;  // context too long for the plan
    const int splits = (int)splits64;
    plan->num_splits = splits;
    plan->chunk_tokens = chunk;
    plan->workspace_bytes =
        splits > 1 ? (size_t)num_seqs * num_q_heads * splits * (head_dim + 1) * sizeof(float) + 256
                   : 0;
    return PKV_OK;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        else
            cudaGetLastError();
    });
    return fn;
}

// Tensor map over a token-major cache [num_blocks][block_size][H_kv][D]: dims
// (innermost first) D, H_kv, block_size, num_blocks; box 64 dims x 1 head x 16
// tokens x 1 block.  Head major [num_blocks][H_kv][block_size][D]: dims D,
// block_size, H_kv, num_blocks; box 64 dims x 16 tokens x 1 head x 1 block.
// 128-byte swizzle either way, so a box lands as 16 rows of 128 bytes.
//
// Encoded maps are remembered (a few dozen, the oldest replaced first): a map
// is a pure function of its arguments (the base address and the geometry), so
// a remembered map stays right whatever happens to the memory behind it, and
// the calls of a decode loop over the same caches skip the encoding.
struct CacheMapKey {
    const void* base;
    int dtype, num_blocks, block_size, num_kv_heads, head_dim;
    bool hnd, f8;
    bool operator==(const CacheMapKey& o) const {
        return base == o.base && dtype == o.dtype && num_blocks == o.num_blocks &&
               block_size == o.block_size && num_kv_heads == o.num_kv_heads &&
               head_dim == o.head_dim && hnd == o.hnd && f8 == o.f8;
    }
};
constexpr int kCacheMapEntries = 32;
static std::mutex g_map_mutex;
static CacheMapKey g_map_keys[kCacheMapEntries];
static CUtensorMap g_maps[kCacheMapEntries];
static int g_map_count = 0, g_map_next = 0;

static bool encode_cache_map(CUtensorMap* map, const void* base, pkv_dtype dtype, int num_blocks,
                             int block_size, int num_kv_heads, int head_dim, bool hnd, bool f8);

static bool make_cache_map(CUtensorMap* map, const void* base, pkv_dtype dtype, int num_blocks,
                           int block_size, int num_kv_heads, int head_dim, bool hnd,
                           bool f8 = false) {
    const CacheMapKey key{base, (int)dtype, num_blocks, block_size, num_kv_heads, head_dim, hnd, f8};
    {
        std::lock_guard<std::mutex> lock(g_map_mutex);
        for (int i = 0; i < g_map_count; ++i)
            if (g_map_keys[i] == key) {
                *map = g_maps[i];
                return true;
            }
    }
    if (!encode_cache_map(map, base, dtype, num_blocks, block_size, num_kv_heads, head_dim, hnd,
                          f8))
        return false;
    std::lock_guard<std::mutex> lock(g_map_mutex);
    const int i = g_map_count < kCacheMapEntries ? g_map_count++ : g_map_next;
    g_map_next = (i + 1) % kCacheMapEntries;
    g_map_keys[i] = key;
    g_maps[i] = *map;
    return true;
}

static bool encode_cache_map(CUtensorMap* map, const void* base, pkv_dtype dtype, int num_blocks,
                             int block_size, int num_kv_heads, int head_dim, bool hnd, bool f8) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t e = f8 ? 1 : 2;
    const cuuint64_t inner = hnd ? (cuuint64_t)block_size : (cuuint64_t)num_kv_heads;
    const cuuint64_t outer = hnd ? (cuuint64_t)num_kv_heads : (cuuint64_t)block_size;
    cuuint64_t dims[4] = {(cuuint64_t)head_dim, inner, outer, (cuuint64_t)num_blocks};
    cuuint64_t strides[3] = {(cuuint64_t)head_dim * e, inner * head_dim * e,
                             outer * inner * head_dim * e};
    cuuint32_t box[4] = {(cuuint32_t)(128 / e), hnd ? (cuuint32_t)kStageTokens : 1u,
                         hnd ? 1u : (cuuint32_t)kStageTokens, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                       : dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                           : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    4, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <typename T, int D, int NT, bool F8, bool MQ = false>
static cudaError_t launch_decode_t(const CUtensorMap& mk, const CUtensorMap& mv,
                                   const DecodeParams& p, dim3 grid, cudaStream_t stream) {
    auto kern = decode_kernel<T, D, NT, F8, MQ>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        Tile<D, F8>::kSmemBytes + q_tile_bytes<D, NT, F8>());
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Tile<D, F8>::kSmemBytes + q_tile_bytes<D, NT, F8>();
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, mk, mv, p);
}

// f8: an E4M3 cache (head_dim 128 only).
template <typename T>
static cudaError_t launch_decode(const CUtensorMap& mk, const CUtensorMap& mv,
                                 const DecodeParams& p, int head_dim, dim3 grid,
                                 cudaStream_t stream, bool f8 = false) {
    const bool wide = p.group > 8;
    if (f8)
        return wide ? launch_decode_t<T, 128, 2, true>(mk, mv, p, grid, stream)
                    : launch_decode_t<T, 128, 1, true>(mk, mv, p, grid, stream);
    if (head_dim == 64)
        return wide ? launch_decode_t<T, 64, 2, false>(mk, mv, p, grid, stream)
                    : launch_decode_t<T, 64, 1, false>(mk, mv, p, grid, stream);
    return wide ? launch_decode_t<T, 128, 2, false>(mk, mv, p, grid, stream)
                : launch_decode_t<T, 128, 1, false>(mk, mv, p, grid, stream);
}

// Multi-query rows on the decode kernel: up to 16 columns per CTA (two
// 8-column groups whenever the rows need more than one CTA).
template <typename T>
static cudaError_t launch_decode_mq(const CUtensorMap& mk, const CUtensorMap& mv,
                                    const DecodeParams& p, int head_dim, dim3 grid,
                                    cudaStream_t stream) {
    const bool wide = p.q_len * p.group > 8;
    if (head_dim == 64)
        return wide ? launch_decode_t<T, 64, 2, false, true>(mk, mv, p, grid, stream)
                    : launch_decode_t<T, 64, 1, false, true>(mk, mv, p, grid, stream);
    return wide ? launch_decode_t<T, 128, 2, false, true>(mk, mv, p, grid, stream)
                : launch_decode_t<T, 128, 1, false, true>(mk, mv, p, grid, stream);
}

template <typename T>
static cudaError_t launch_merge(const MergeParams& p, int groups, int seqs, cudaStream_t stream) {
    MergeParams q = p;
    q.rows = (int64_t)groups * seqs;
    const int64_t ctas = (q.rows + kMergeRowsPerCta - 1) / kMergeRowsPerCta;
    if (ctas > INT_MAX) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::max<int64_t>(1, ctas));
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, merge_kernel<T>, q);
}

template <typename T, int D, int MODE = 0>
static cudaError_t launch_prefix_t(const CUtensorMap& mk, const CUtensorMap& mv,
                                   const PrefixParams& p, dim3 grid, cudaStream_t stream) {
    auto kern = prefix_kernel<T, D, MODE>;
    using Cfg = PrefixTile<D, MODE != 0 ? mq_stages<D>() : kPrefixStages, MODE != 0>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        Cfg::kSmemBytes);
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(((MODE != 0 ? 4 : kPrefixSoftmaxWarps) + 2) * 32);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, mk, mv, p);
}

// Modes of the tcgen05 kernel per path: multi-query with at most 64 query
// rows per (sequence, KV head) MODE 1, with more MODE 2 (one CTA per 128 rows,
// two CTAs an SM: C4 q_len 16 42.7 -> 45.2 % against MODE 0); shared prefixes
// MODE 0 (MODE 2 ran C5 at 80.2 % against 81.7 %).
constexpr int kMqDupMode = 1;
constexpr int kMqFullMode = 2;
constexpr int kPrefixMode = 0;
constexpr int ctas_per_sm_of_mode(int mode) { return mode != 0 ? 2 : 1; }
constexpr int kMqDupCtasPerSm = ctas_per_sm_of_mode(kMqDupMode);

// Plan of a shared-prefix call: the suffixes planned like a plain decode; the
// prefix in partitions of whole 64-token tiles, as many as give about one
// prefix CTA (128 query rows) per kPrefixSmShare SMs, at most kMaxChunkPages
// pages each; per (sequence, query head) the prefix partials first, then the
// suffix partials.  The prefix kernel runs beside the suffix decode, so it
// takes only part of the GPU and the decode keeps the rest.
constexpr int kPrefixSmShare = 2;
struct PrefixPlan {
    Plan suffix;
    int prefix_chunk;
    int prefix_parts;
    int total_splits;
    int row_tiles;
    size_t workspace_bytes;
};

static pkv_status make_prefix_plan(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, int max_context_len, int num_groups,
                                   int max_group_size, int max_prefix_len, PrefixPlan* pp) {
    if (num_groups < 0 || max_group_size < 0 || max_prefix_len < 0) return PKV_ERR_INVALID_ARG;
    pkv_status st = make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                              max_context_len, 0, &pp->suffix);
    if (st != PKV_OK) return st;
    const int group = num_q_heads / num_kv_heads;
    const int64_t rows = (int64_t)max_group_size * group;
    pp->row_tiles = (int)std::max<int64_t>(1, (rows + kPrefixTileRows - 1) / kPrefixTileRows);
    if ((int64_t)num_groups * num_kv_heads > 65535 || pp->row_tiles > 65535)
        return PKV_ERR_UNSUPPORTED;
    const int sms = current_sm_count();
    if (sms <= 0) return PKV_ERR_CUDA;
    const int64_t units = std::max<int64_t>(1, (int64_t)num_groups * num_kv_heads * pp->row_tiles);
    const int64_t want = std::max<int64_t>(
        1, (int64_t)sms * ctas_per_sm_of_mode(kPrefixMode) / (kPrefixSmShare * units));
    const int tiles = (max_prefix_len + kPrefixTileTokens - 1) / kPrefixTileTokens;
    const int max_tiles = kMaxChunkPages * block_size / kPrefixTileTokens;
    const int chunk_tiles =
        std::min<int64_t>(max_tiles, std::max<int64_t>(1, (tiles + want - 1) / want));
    pp->prefix_chunk = chunk_tiles * kPrefixTileTokens;
    pp->prefix_parts = max_prefix_len > 0 ? (max_prefix_len + pp->prefix_chunk - 1) / pp->prefix_chunk
                                          : 0;
    pp->total_splits = pp->prefix_parts + pp->suffix.num_splits;
    if (pp->total_splits > PKV_MAX_SPLITS) return PKV_ERR_UNSUPPORTED;
    const size_t partial_floats = (size_t)num_seqs * num_q_heads * pp->total_splits * (head_dim + 1);
    const size_t items = (size_t)num_seqs * num_kv_heads * pp->suffix.num_splits;
    // partials | per-sequence records | work list | its length | per-unit counts
    pp->workspace_bytes = ((partial_floats * sizeof(float) + 15) & ~size_t(15)) +
                          (size_t)num_seqs * sizeof(int2) + items * sizeof(int2) + 16 +
                          (size_t)num_seqs * num_kv_heads * sizeof(int) + 256;
    return PKV_OK;
}

// Plan of a multi-query call.  At most 2 * kMaxGroup (query token, query
// head) rows per (sequence, KV head) (speculative verification of a few
// tokens, a small GQA group or MHA): the decode kernel with those rows as its
// columns, in one CTA of up to kMaxGroup rows or two adjacent ones that read
// the same context together, planned like a decode.  More rows: 128-row
// tiles per (sequence, KV head) on the tensor-core kernel; the context in
// partitions of whole 64-token tiles, as many as give about one CTA per SM,
// at most kPrefixMaxChunkPages pages each.
constexpr int kMqDecodeRowBlocks = 2;
struct MultiQueryPlan {
    bool on_decode;  // the decode kernel's multi-query form
    int row_blocks;  // on the decode kernel: CTAs per (sequence, KV head)
    int chunk;
    int parts;
    int row_tiles;
    bool dup;      // at most 64 query rows per (sequence, KV head): two partials per partition
    int slots;     // partial slots per row: parts, or 2 * parts with dup
    size_t workspace_bytes;
};

static pkv_status make_mq_plan(int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                               int head_dim, int block_size, int max_context_len,
                               MultiQueryPlan* mp) {
    pkv_status st = check_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                 max_context_len, 0);
    if (st != PKV_OK) return st;
    if (q_len <= 0) return PKV_ERR_INVALID_ARG;
    const int group = num_q_heads / num_kv_heads;
    const int64_t rows = (int64_t)q_len * group;
    mp->row_tiles = (int)((rows + kPrefixTileRows - 1) / kPrefixTileRows);
    if ((int64_t)num_seqs * num_kv_heads > 65535 || mp->row_tiles > 65535 ||
        (int64_t)num_seqs * q_len > 65535)
        return PKV_ERR_UNSUPPORTED;
    mp->on_decode = rows <= kMqDecodeRowBlocks * kMaxGroup;
    mp->row_blocks = (int)((rows + kMaxGroup - 1) / kMaxGroup);
    if ((int64_t)num_kv_heads * mp->row_blocks > INT_MAX) return PKV_ERR_UNSUPPORTED;
    if (mp->on_decode) {
        Plan dp;
        st = make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                       max_context_len, 0, &dp, 3, mp->row_blocks);
        if (st != PKV_OK) return st;
        mp->dup = false;
        mp->chunk = dp.chunk_tokens;
        mp->parts = dp.num_splits;
        mp->slots = dp.num_splits;
        mp->workspace_bytes =
            (mp->parts > 1
                 ? (size_t)num_seqs * q_len * num_q_heads * mp->slots * (head_dim + 1) * sizeof(float)
                 : 0) +
            256;
        return PKV_OK;
    }
    const int sms = current_sm_count();
    if (sms <= 0) return PKV_ERR_CUDA;
    mp->dup = rows <= kPrefixTileRows / 2;
    const int64_t units = std::max<int64_t>(1, (int64_t)num_seqs * num_kv_heads * mp->row_tiles);
    const int64_t want = std::max<int64_t>(
        1, (int64_t)sms * (mp->dup ? kMqDupCtasPerSm : ctas_per_sm_of_mode(kMqFullMode)) / units);
    const int tiles = std::max(1, (max_context_len + kPrefixTileTokens - 1) / kPrefixTileTokens);
    const int max_tiles = kPrefixMaxChunkPages * block_size / kPrefixTileTokens;
    const int chunk_tiles =
        (int)std::min<int64_t>(max_tiles, std::max<int64_t>(1, (tiles + want - 1) / want));
    mp->chunk = chunk_tiles * kPrefixTileTokens;
    mp->parts = std::max(1, (max_context_len + mp->chunk - 1) / mp->chunk);
    if (mp->parts > PKV_MAX_SPLITS || mp->parts > 65535) return PKV_ERR_UNSUPPORTED;
    mp->slots = mp->parts * (mp->dup ? 2 : 1);
    if (mp->slots > 65535) return PKV_ERR_UNSUPPORTED;
    mp->workspace_bytes =
        (size_t)num_seqs * q_len * num_q_heads * mp->slots * (head_dim + 1) * sizeof(float) + 256;
    return PKV_OK;
}

pkv_status decode_workspace_16bit(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                  int block_size, int max_context_len, int num_splits,
                                  size_t* bytes) {
    Plan plan;
    const pkv_status st = make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                    max_context_len, num_splits, &plan);
    if (st == PKV_OK) *bytes = plan.workspace_bytes;
    return st;
}

}  // namespace pkv

using namespace pkv;

extern "C" size_t pkv_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                            int head_dim, int block_size, int max_context_len,
                                            int num_splits) {
    // Enough for the 16-bit kernel's plan and the E4M3 kernel's (whose
    // automatic plan counts four resident CTAs an SM).
    Plan plan, plan4;
    if (make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                  num_splits, &plan) != PKV_OK ||
        make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                  num_splits, &plan4, 4) != PKV_OK)
        return SIZE_MAX;
    return std::max(plan.workspace_bytes, plan4.workspace_bytes);
}

extern "C" int pkv_decode_num_splits(int num_seqs, int num_q_heads, int num_kv_heads,
                                     int head_dim, int block_size, int max_context_len,
                                     int num_splits) {
    Plan plan;
    if (make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                  num_splits, &plan) != PKV_OK)
        return -1;
    return plan.num_splits;
}

extern "C" int pkv_decode_num_splits_fp8(int num_seqs, int num_q_heads, int num_kv_heads,
                                         int head_dim, int block_size, int max_context_len,
                                         int num_splits) {
    Plan plan;
    if (make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                  num_splits, &plan, num_q_heads > 0 && num_kv_heads > 0 &&
                                         num_q_heads / num_kv_heads <= 8 ? 4 : 3) != PKV_OK)
        return -1;
    return plan.num_splits;
}

// The plain decode, with the new tokens' K/V appended by the decode kernel
// itself when k_new / v_new are given.
static pkv_status decode_impl(void* out, const void* q, const void* k_new, const void* v_new,
                              void* k_cache, void* v_cache, const int32_t* block_tables,
                              int max_blocks_per_seq, const int32_t* context_lens,
                              int max_context_len, int num_seqs, int num_blocks, int block_size,
                              int num_q_heads, int num_kv_heads, int head_dim, float scale,
                              int num_splits, void* workspace, size_t workspace_bytes,
                              pkv_dtype dtype, int32_t* err_flag, void* stream, bool f8 = false,
                              float k_scale = 1.f, float v_scale = 1.f) {
    const bool hnd = take_layout(dtype);
    pkv_status st = check_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                 max_context_len, num_splits);
    if (st != PKV_OK) return st;
    if ((dtype != PKV_FP16 && dtype != PKV_BF16) || max_blocks_per_seq <= 0 || num_blocks <= 0 ||
        !std::isfinite(scale))
        return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return PKV_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
        (reinterpret_cast<uintptr_t>(context_lens) & 3u))
        return PKV_ERR_INVALID_ARG;
    if ((k_new == nullptr) != (v_new == nullptr) ||
        (k_new != nullptr && (!aligned16(k_new) || !aligned16(v_new))))
        return PKV_ERR_INVALID_ARG;
    if (f8 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (f8 && (!std::isfinite(k_scale) || !std::isfinite(v_scale) || k_scale <= 0.f ||
               v_scale <= 0.f))
        return PKV_ERR_INVALID_ARG;
    if ((int64_t)max_blocks_per_seq * block_size > INT_MAX) return PKV_ERR_UNSUPPORTED;
    Plan plan;
    st = make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                   num_splits, &plan, f8 && num_q_heads / num_kv_heads <= 8 ? 4 : 3);
    if (st != PKV_OK) return st;
    if (plan.workspace_bytes > 0 && (workspace == nullptr || workspace_bytes < plan.workspace_bytes))
        return PKV_ERR_WORKSPACE;
    if (workspace != nullptr && !aligned16(workspace)) return PKV_ERR_INVALID_ARG;

    CUtensorMap mk, mv;
    if (!make_cache_map(&mk, k_cache, dtype, num_blocks, block_size, num_kv_heads, head_dim, hnd,
                        f8) ||
        !make_cache_map(&mv, v_cache, dtype, num_blocks, block_size, num_kv_heads, head_dim, hnd,
                        f8))
        return PKV_ERR_CUDA;

    DecodeParams p = {};
    p.out = out;
    p.q = q;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.err_flag = err_flag;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.block_size = block_size;
    p.num_q_heads = num_q_heads;
    p.group = num_q_heads / num_kv_heads;
    p.num_splits = plan.num_splits;
    p.chunk_tokens = plan.chunk_tokens;
    p.num_kv_heads = num_kv_heads;
    p.max_context_len = max_context_len;
    p.scale_log2 = scale * k_scale * kLog2e;
    p.v_scale = v_scale;
    p.partial_o = nullptr;
    p.partial_lse = nullptr;
    p.seq_info = nullptr;
    p.items = nullptr;
    p.item_count = nullptr;
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_scale = k_scale;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.hnd = hnd;
    if (plan.num_splits > 1) {
        p.partial_o = static_cast<float*>(workspace);
        p.partial_lse = p.partial_o + (size_t)num_seqs * num_q_heads * plan.num_splits * head_dim;
    }
    cudaStream_t s = (cudaStream_t)stream;
    dim3 grid(num_kv_heads, num_seqs, plan.num_splits);
    cudaError_t e = dtype == PKV_FP16
                        ? launch_decode<__half>(mk, mv, p, head_dim, grid, s, f8)
                        : launch_decode<__nv_bfloat16>(mk, mv, p, head_dim, grid, s, f8);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    if (plan.num_splits > 1) {
        MergeParams mp = {};
        mp.out = out;
        mp.partial_o = p.partial_o;
        mp.partial_lse = p.partial_lse;
        mp.context_lens = context_lens;
        mp.seq_info = nullptr;
        mp.num_q_heads = num_q_heads;
        mp.num_kv_heads = num_kv_heads;
        mp.group = num_q_heads / num_kv_heads;
        mp.num_splits = plan.num_splits;
        mp.head_dim = head_dim;
        mp.chunk_tokens = plan.chunk_tokens;
        mp.cap = std::min(max_blocks_per_seq * block_size, max_context_len);
        e = dtype == PKV_FP16 ? launch_merge<__half>(mp, num_q_heads, num_seqs, s)
                              : launch_merge<__nv_bfloat16>(mp, num_q_heads, num_seqs, s);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return PKV_ERR_CUDA;
        }
    }
    return PKV_OK;
}

extern "C" pkv_status pkv_decode_attention(void* out, const void* q, const void* k_cache,
                                           const void* v_cache, const int32_t* block_tables,
                                           int max_blocks_per_seq, const int32_t* context_lens,
                                           int max_context_len, int num_seqs, int num_blocks,
                                           int block_size, int num_q_heads, int num_kv_heads,
                                           int head_dim, float scale, int num_splits,
                                           void* workspace, size_t workspace_bytes,
                                           pkv_dtype dtype, int32_t* err_flag, void* stream) {
    return decode_impl(out, q, nullptr, nullptr, const_cast<void*>(k_cache),
                       const_cast<void*>(v_cache), block_tables, max_blocks_per_seq, context_lens,
                       max_context_len, num_seqs, num_blocks, block_size, num_q_heads,
                       num_kv_heads, head_dim, scale, num_splits, workspace, workspace_bytes,
                       dtype, err_flag, stream);
}

extern "C" pkv_status pkv_decode_attention_fp8(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int max_context_len, int num_seqs, int num_blocks, int block_size, int num_q_heads,
    int num_kv_heads, int head_dim, float scale, float k_scale, float v_scale, int num_splits,
    void* workspace, size_t workspace_bytes, pkv_dtype dtype, int32_t* err_flag, void* stream) {
    return decode_impl(out, q, nullptr, nullptr, const_cast<void*>(k_cache),
                       const_cast<void*>(v_cache), block_tables, max_blocks_per_seq, context_lens,
                       max_context_len, num_seqs, num_blocks, block_size, num_q_heads,
                       num_kv_heads, head_dim, scale, num_splits, workspace, workspace_bytes,
                       dtype, err_flag, stream, true, k_scale, v_scale);
}

extern "C" pkv_status pkv_append_decode_attention(
    void* out, const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int max_context_len, int num_seqs, int num_blocks, int block_size, int num_q_heads,
    int num_kv_heads, int head_dim, float scale, int num_splits, void* workspace,
    size_t workspace_bytes, pkv_dtype dtype, int32_t* err_flag, void* stream) {
    const pkv_status st = check_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                       max_context_len, num_splits);
    if (st != PKV_OK) return st;
    if (num_seqs > 0 && (k_new == nullptr || v_new == nullptr)) return PKV_ERR_INVALID_ARG;
    return decode_impl(out, q, k_new, v_new, k_cache, v_cache, block_tables, max_blocks_per_seq,
                       context_lens, max_context_len, num_seqs, num_blocks, block_size,
                       num_q_heads, num_kv_heads, head_dim, scale, num_splits, workspace,
                       workspace_bytes, dtype, err_flag, stream);
}

extern "C" pkv_status pkv_append_decode_attention_fp8(
    void* out, const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int max_context_len, int num_seqs, int num_blocks, int block_size, int num_q_heads,
    int num_kv_heads, int head_dim, float scale, float k_scale, float v_scale, int num_splits,
    void* workspace, size_t workspace_bytes, pkv_dtype dtype, int32_t* err_flag, void* stream) {
    const pkv_status st = check_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                       max_context_len, num_splits);
    if (st != PKV_OK) return st;
    if (num_seqs > 0 && (k_new == nullptr || v_new == nullptr)) return PKV_ERR_INVALID_ARG;
    return decode_impl(out, q, k_new, v_new, k_cache, v_cache, block_tables, max_blocks_per_seq,
                       context_lens, max_context_len, num_seqs, num_blocks, block_size,
                       num_q_heads, num_kv_heads, head_dim, scale, num_splits, workspace,
                       workspace_bytes, dtype, err_flag, stream, true, k_scale, v_scale);
}

extern "C" pkv_status pkv_merge(void* out, const float* partial_o, const float* partial_lse,
                                int num_seqs, int num_q_heads, int num_splits, int head_dim,
                                pkv_dtype dtype, void* stream) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_splits <= 0 || num_splits > PKV_MAX_SPLITS ||
        head_dim <= 0 || (dtype != PKV_FP16 && dtype != PKV_BF16))
        return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !partial_o || !partial_lse) return PKV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(out) & 7u) || (reinterpret_cast<uintptr_t>(partial_o) & 15u) ||
        (reinterpret_cast<uintptr_t>(partial_lse) & 3u))
        return PKV_ERR_INVALID_ARG;
    if (head_dim % 4 != 0 || head_dim > kMergeMaxHeadDim) return PKV_ERR_UNSUPPORTED;
    if (num_seqs > 65535) return PKV_ERR_UNSUPPORTED;
    MergeParams mp = {};
    mp.out = out;
    mp.partial_o = partial_o;
    mp.partial_lse = partial_lse;
    mp.context_lens = nullptr;
    mp.seq_info = nullptr;
    mp.num_q_heads = num_q_heads;
    mp.num_kv_heads = num_q_heads;
    mp.group = 1;  // partition geometry is not used without context_lens
    mp.num_splits = num_splits;
    mp.head_dim = head_dim;
    mp.chunk_tokens = 1;
    mp.cap = 0;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = dtype == PKV_FP16 ? launch_merge<__half>(mp, num_q_heads, num_seqs, s)
                                      : launch_merge<__nv_bfloat16>(mp, num_q_heads, num_seqs, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

extern "C" pkv_status pkv_selftest_wait_timeout(int32_t* err_flag, unsigned long long limit_ns,
                                                void* stream) {
    if (err_flag == nullptr || limit_ns == 0 || limit_ns > 1000000000ull)
        return PKV_ERR_INVALID_ARG;
    wait_timeout_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(err_flag, limit_ns);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" size_t pkv_prefix_shared_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                                   int head_dim, int block_size,
                                                   int max_context_len, int num_groups,
                                                   int max_group_size, int max_prefix_len) {
    PrefixPlan pp;
    if (make_prefix_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                         max_context_len, num_groups, max_group_size, max_prefix_len,
                         &pp) != PKV_OK)
        return SIZE_MAX;
    return pp.workspace_bytes;
}

extern "C" pkv_status pkv_decode_attention_prefix_shared(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int max_context_len, int num_seqs, int num_blocks, int block_size, int num_q_heads,
    int num_kv_heads, int head_dim, float scale, int num_groups, const int32_t* group_start,
    const int32_t* group_prefix_len, int max_group_size, int max_prefix_len, void* workspace,
    size_t workspace_bytes, pkv_dtype dtype, int32_t* err_flag, void* stream) {
    const bool hnd = take_layout(dtype);
    pkv_status st = check_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                 max_context_len, 0);
    if (st != PKV_OK) return st;
    if ((dtype != PKV_FP16 && dtype != PKV_BF16) || max_blocks_per_seq <= 0 || num_blocks <= 0 ||
        !std::isfinite(scale) || num_groups < 0 || max_group_size < 0 || max_prefix_len < 0)
        return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !workspace ||
        (num_groups > 0 && (!group_start || !group_prefix_len)))
        return PKV_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned16(workspace) || (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
        (reinterpret_cast<uintptr_t>(context_lens) & 3u) ||
        (reinterpret_cast<uintptr_t>(group_start) & 3u) ||
        (reinterpret_cast<uintptr_t>(group_prefix_len) & 3u))
        return PKV_ERR_INVALID_ARG;
    if ((int64_t)max_blocks_per_seq * block_size > INT_MAX) return PKV_ERR_UNSUPPORTED;
    PrefixPlan pp;
    st = make_prefix_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                          max_context_len, num_groups, max_group_size, max_prefix_len, &pp);
    if (st != PKV_OK) return st;
    if (workspace_bytes < pp.workspace_bytes) return PKV_ERR_WORKSPACE;

    CUtensorMap mk, mv;
    if (!make_cache_map(&mk, k_cache, dtype, num_blocks, block_size, num_kv_heads, head_dim, hnd) ||
        !make_cache_map(&mv, v_cache, dtype, num_blocks, block_size, num_kv_heads, head_dim, hnd))
        return PKV_ERR_CUDA;

    float* partial_o = static_cast<float*>(workspace);
    float* partial_lse = partial_o + (size_t)num_seqs * num_q_heads * pp.total_splits * head_dim;
    const size_t partial_floats = (size_t)num_seqs * num_q_heads * pp.total_splits * (head_dim + 1);
    int2* seq_info = reinterpret_cast<int2*>(static_cast<char*>(workspace) +
                                             ((partial_floats * sizeof(float) + 15) & ~size_t(15)));
    const int64_t num_items = (int64_t)num_seqs * num_kv_heads * pp.suffix.num_splits;
    int2* items = seq_info + num_seqs;
    int* item_count = reinterpret_cast<int*>(items + num_items);
    int* unit_left = item_count + 4;
    const int cap = std::min(max_blocks_per_seq * block_size, max_context_len);
    cudaStream_t s = (cudaStream_t)stream;

    // every sequence's prefix record and the list of suffix partitions with
    // tokens: the plan
    PlanParams pl = {};
    pl.context_lens = context_lens;
    pl.group_start = group_start;
    pl.group_prefix_len = group_prefix_len;
    pl.seq_info = seq_info;
    pl.items = items;
    pl.item_count = item_count;
    pl.err_flag = err_flag;
    pl.num_seqs = num_seqs;
    pl.num_kv_heads = num_kv_heads;
    pl.num_groups = num_groups;
    pl.max_group_size = max_group_size;
    pl.max_prefix_len = max_prefix_len;
    pl.block_size = block_size;
    pl.max_blocks_per_seq = max_blocks_per_seq;
    pl.prefix_chunk = pp.prefix_chunk;
    pl.chunk_tokens = pp.suffix.chunk_tokens;
    pl.cap = cap;
    pl.unit_left = unit_left;
    pl.group = num_q_heads / num_kv_heads;

    // the prefix partials of every group (tcgen05); the last contribution to
    // a unit merges it
    PrefixParams pr = {};
    pr.q = q;
    pr.block_tables = block_tables;
    pr.context_lens = context_lens;
    pr.group_start = group_start;
    pr.group_prefix_len = group_prefix_len;
    pr.partial_o = partial_o;
    pr.partial_lse = partial_lse;
    pr.err_flag = err_flag;
    pr.max_blocks_per_seq = max_blocks_per_seq;
    pr.num_blocks = num_blocks;
    pr.block_size = block_size;
    pr.num_seqs = num_seqs;
    pr.num_q_heads = num_q_heads;
    pr.num_kv_heads = num_kv_heads;
    pr.group = num_q_heads / num_kv_heads;
    pr.num_splits = pp.total_splits;
    pr.num_groups = num_groups;
    pr.max_group_size = max_group_size;
    pr.max_prefix_len = max_prefix_len;
    pr.prefix_chunk = pp.prefix_chunk;
    pr.cap = cap;
    pr.hnd = hnd;
    pr.scale_log2 = scale * kLog2e;
    pr.unit_left = unit_left;
    pr.out = out;
    pr.seq_info = seq_info;
    pr.suffix_chunk = pp.suffix.chunk_tokens;

    // suffix partials (or the whole answer for sequences without a prefix),
    // CTA x taking the plan's item x
    DecodeParams p = {};
    p.out = out;
    p.q = q;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.partial_o = partial_o;
    p.partial_lse = partial_lse;
    p.seq_info = seq_info;
    p.items = items;
    p.item_count = item_count;
    p.err_flag = err_flag;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.block_size = block_size;
    p.num_q_heads = num_q_heads;
    p.group = num_q_heads / num_kv_heads;
    p.num_splits = pp.total_splits;
    p.chunk_tokens = pp.suffix.chunk_tokens;
    p.num_kv_heads = num_kv_heads;
    p.max_context_len = max_context_len;
    p.hnd = hnd;
    p.scale_log2 = scale * kLog2e;
    p.v_scale = 1.f;
    p.unit_left = unit_left;

    auto launch_prefix = [&](cudaStream_t st) {
        const dim3 pgrid(pp.row_tiles, std::max(1, num_groups * num_kv_heads),
                         std::max(1, pp.prefix_parts));
        if (head_dim == 64)
            return dtype == PKV_FP16 ? launch_prefix_t<__half, 64, kPrefixMode>(mk, mv, pr, pgrid, st)
                                     : launch_prefix_t<__nv_bfloat16, 64, kPrefixMode>(mk, mv, pr, pgrid, st);
        return dtype == PKV_FP16 ? launch_prefix_t<__half, 128, kPrefixMode>(mk, mv, pr, pgrid, st)
                                 : launch_prefix_t<__nv_bfloat16, 128, kPrefixMode>(mk, mv, pr, pgrid, st);
    };
    auto launch_plan = [&](cudaStream_t st) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1);
        cfg.blockDim = dim3(kPlanThreads);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, plan_kernel, pl);
    };
    auto launch_suffix = [&](cudaStream_t st) {
        const dim3 grid((unsigned)num_items);
        return dtype == PKV_FP16 ? launch_decode<__half>(mk, mv, p, head_dim, grid, st)
                                 : launch_decode<__nv_bfloat16>(mk, mv, p, head_dim, grid, st);
    };

    // 1. the plan; 2. the prefix kernel on the side stream, forked from the
    // caller's stream after the plan, and the suffix decode on the caller's
    // stream at the same time; the caller's stream then waits for the prefix.
    // Whichever kernel writes a unit's last partial merges it, so no merge
    // launch follows.  Without a side stream, the prefix runs after the plan
    // on the caller's stream, then the decode.
    cudaError_t e = launch_plan(s);
    if (e == cudaSuccess) {
        std::lock_guard<std::mutex> lock(g_side_mutex);
        const SideStream* side = pp.prefix_parts > 0 ? side_stream_locked() : nullptr;
        if (side != nullptr) {
            e = cudaEventRecord(side->fork, s);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(side->stream, side->fork, 0);
            if (e == cudaSuccess) e = launch_prefix(side->stream);
            // the join is queued even if a launch failed, so the side stream
            // never runs ahead of the caller's later work
            const cudaError_t r = cudaEventRecord(side->join, side->stream);
            if (e == cudaSuccess) e = r;
            if (e == cudaSuccess) e = launch_suffix(s);
            const cudaError_t w = cudaStreamWaitEvent(s, side->join, 0);
            if (e == cudaSuccess) e = w;
        } else {
            if (pp.prefix_parts > 0) e = launch_prefix(s);
            if (e == cudaSuccess) e = launch_suffix(s);
        }
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

extern "C" size_t pkv_multi_query_workspace_size(int num_seqs, int q_len, int num_q_heads,
                                                 int num_kv_heads, int head_dim, int block_size,
                                                 int max_context_len) {
    MultiQueryPlan mp;
    if (make_mq_plan(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size,
                     max_context_len, &mp) != PKV_OK)
        return SIZE_MAX;
    return mp.workspace_bytes;
}

extern "C" int pkv_multi_query_plan(int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                                    int head_dim, int block_size, int max_context_len,
                                    int* num_partitions) {
    MultiQueryPlan mp;
    if (make_mq_plan(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size,
                     max_context_len, &mp) != PKV_OK)
        return -1;
    if (num_partitions != nullptr) *num_partitions = mp.parts;
    return mp.on_decode ? 1 : 0;
}

extern "C" pkv_status pkv_multi_query_attention(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int max_context_len, int num_seqs, int q_len, int num_blocks, int block_size,
    int num_q_heads, int num_kv_heads, int head_dim, float scale, void* workspace,
    size_t workspace_bytes, pkv_dtype dtype, int32_t* err_flag, void* stream) {
    const bool hnd = take_layout(dtype);
    if ((dtype != PKV_FP16 && dtype != PKV_BF16) || max_blocks_per_seq <= 0 || num_blocks <= 0 ||
        !std::isfinite(scale) || q_len <= 0)
        return PKV_ERR_INVALID_ARG;
    pkv_status st = check_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                 max_context_len, 0);
    if (st != PKV_OK) return st;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !workspace)
        return PKV_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned16(workspace) || (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
        (reinterpret_cast<uintptr_t>(context_lens) & 3u))
        return PKV_ERR_INVALID_ARG;
    if ((int64_t)max_blocks_per_seq * block_size > INT_MAX) return PKV_ERR_UNSUPPORTED;
    MultiQueryPlan mq;
    st = make_mq_plan(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size,
                      max_context_len, &mq);
    if (st != PKV_OK) return st;
    if (workspace_bytes < mq.workspace_bytes) return PKV_ERR_WORKSPACE;

    CUtensorMap mk, mv;
    if (!make_cache_map(&mk, k_cache, dtype, num_blocks, block_size, num_kv_heads, head_dim, hnd) ||
        !make_cache_map(&mv, v_cache, dtype, num_blocks, block_size, num_kv_heads, head_dim, hnd))
        return PKV_ERR_CUDA;
    float* partial_o = static_cast<float*>(workspace);
    float* partial_lse = partial_o + (size_t)num_seqs * q_len * num_q_heads * mq.slots * head_dim;
    const int cap = std::min(max_blocks_per_seq * block_size, max_context_len);
    const int group = num_q_heads / num_kv_heads;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e;

    if (mq.on_decode) {
        // 1. every row's attention (contexts of one partition) or its partials
        DecodeParams p = {};
        p.out = out;
        p.q = q;
        p.block_tables = block_tables;
        p.context_lens = context_lens;
        p.err_flag = err_flag;
        p.max_blocks_per_seq = max_blocks_per_seq;
        p.num_blocks = num_blocks;
        p.block_size = block_size;
        p.num_q_heads = num_q_heads;
        p.group = group;
        p.num_splits = mq.parts;
        p.chunk_tokens = mq.chunk;
        p.num_kv_heads = num_kv_heads;
        p.max_context_len = max_context_len;
        p.q_len = q_len;
        p.row_blocks = mq.row_blocks;
        p.hnd = hnd;
        p.scale_log2 = scale * kLog2e;
        p.v_scale = 1.f;
        if (mq.parts > 1) {
            p.partial_o = partial_o;
            p.partial_lse = partial_lse;
        }
        // a (sequence, KV head)'s row blocks are adjacent CTAs
        const dim3 grid(num_kv_heads * mq.row_blocks, num_seqs, mq.parts);
        e = dtype == PKV_FP16 ? launch_decode_mq<__half>(mk, mv, p, head_dim, grid, s)
                              : launch_decode_mq<__nv_bfloat16>(mk, mv, p, head_dim, grid, s);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return PKV_ERR_CUDA;
        }
        if (mq.parts == 1) return PKV_OK;
        // 2. merge the rows of contexts longer than one partition
        MergeParams mp = {};
        mp.out = out;
        mp.partial_o = partial_o;
        mp.partial_lse = partial_lse;
        mp.context_lens = context_lens;
        mp.num_q_heads = num_q_heads;
        mp.num_kv_heads = num_kv_heads;
        mp.group = group;
        mp.num_splits = mq.parts;
        mp.head_dim = head_dim;
        mp.chunk_tokens = mq.chunk;
        mp.cap = cap;
        mp.q_len = q_len;
        mp.mq_slots = 1;
        mp.mq_direct = true;
        e = dtype == PKV_FP16 ? launch_merge<__half>(mp, num_q_heads, num_seqs * q_len, s)
                              : launch_merge<__nv_bfloat16>(mp, num_q_heads, num_seqs * q_len, s);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return PKV_ERR_CUDA;
        }
        return PKV_OK;
    }

    // 1. partials of every (query token, query head) row per context partition (tcgen05)
    PrefixParams pr = {};
    pr.q = q;
    pr.block_tables = block_tables;
    pr.context_lens = context_lens;
    pr.partial_o = partial_o;
    pr.partial_lse = partial_lse;
    pr.err_flag = err_flag;
    pr.max_blocks_per_seq = max_blocks_per_seq;
    pr.num_blocks = num_blocks;
    pr.block_size = block_size;
    pr.num_seqs = num_seqs;
    pr.num_q_heads = num_q_heads;
    pr.num_kv_heads = num_kv_heads;
    pr.group = group;
    pr.num_splits = mq.slots;
    pr.prefix_chunk = mq.chunk;
    pr.cap = cap;
    pr.q_len = q_len;
    pr.hnd = hnd;
    pr.scale_log2 = scale * kLog2e;
    const dim3 pgrid(mq.row_tiles, num_seqs * num_kv_heads, mq.parts);
    if (mq.dup) {
        if (head_dim == 64)
            e = dtype == PKV_FP16 ? launch_prefix_t<__half, 64, kMqDupMode>(mk, mv, pr, pgrid, s)
                                  : launch_prefix_t<__nv_bfloat16, 64, kMqDupMode>(mk, mv, pr, pgrid, s);
        else
            e = dtype == PKV_FP16 ? launch_prefix_t<__half, 128, kMqDupMode>(mk, mv, pr, pgrid, s)
                                  : launch_prefix_t<__nv_bfloat16, 128, kMqDupMode>(mk, mv, pr, pgrid, s);
    } else if (head_dim == 64) {
        e = dtype == PKV_FP16 ? launch_prefix_t<__half, 64, kMqFullMode>(mk, mv, pr, pgrid, s)
                              : launch_prefix_t<__nv_bfloat16, 64, kMqFullMode>(mk, mv, pr, pgrid, s);
    } else {
        e = dtype == PKV_FP16 ? launch_prefix_t<__half, 128, kMqFullMode>(mk, mv, pr, pgrid, s)
                              : launch_prefix_t<__nv_bfloat16, 128, kMqFullMode>(mk, mv, pr, pgrid, s);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }

    // 2. merge every row
    MergeParams mp = {};
    mp.out = out;
    mp.partial_o = partial_o;
    mp.partial_lse = partial_lse;
    mp.context_lens = context_lens;
    mp.num_q_heads = num_q_heads;
    mp.num_kv_heads = num_kv_heads;
    mp.group = group;
    mp.num_splits = mq.slots;
    mp.head_dim = head_dim;
    mp.chunk_tokens = mq.chunk;
    mp.cap = cap;
    mp.q_len = q_len;
    mp.mq_slots = mq.dup ? 2 : 1;
    e = dtype == PKV_FP16 ? launch_merge<__half>(mp, num_q_heads, num_seqs * q_len, s)
                          : launch_merge<__nv_bfloat16>(mp, num_q_heads, num_seqs * q_len, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}
