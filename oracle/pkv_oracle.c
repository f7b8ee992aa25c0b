/*
 * Oracle for paged-KV decode attention — TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct fp64 CPU implementation of what the GPU
 * library computes.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load this file's shared object.  It shares no code,
 * header, table or helper with the CUDA library and includes none of it.
 *
 * What it follows (page "推理优化 / inference" and its companions):
 *  - Cache layout: K and V are stored page by page as
 *    [num_pages][page_size][num_heads][head_dim]
 *    (inference.html, "PagedAttention 内核实现").
 *  - Addressing: token t of a request lives in physical block
 *    block_table[t / block_size] at offset t % block_size
 *    (gsyq.cn essay, §三.2 PagedAttentionManager.get_kv_cache; tutorial
 *    chapter 12, PagedKVCache.update).
 *  - Attention with a cache: out = softmax(q K^T * scale) V over the t cached
 *    tokens, scale = 1/sqrt(head_dim) (inference.html, chunked-prefill
 *    attention and NPUAttention; tutorial chapter 12, Attention(Q_t, K_1:t,
 *    V_1:t)).
 *  - GQA: query heads are split into contiguous groups that share one KV head
 *    (gsyq.cn essay, §三.6 GQA).
 *
 * Readings where the pages are silent:
 *  - tokens at positions >= context_len are never read (masked, not zeroed);
 *  - context_len == 0 gives an all-zero output row;
 *  - the maximum score is subtracted before exp, as in every softmax on the
 *    pages.
 *
 * Inputs are the raw 16-bit patterns of fp16 (dtype 0) or bf16 (dtype 1)
 * values; this file decodes them itself, exactly, into double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE-754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_fp16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);               /* subnormal: frac * 2^-14 * 2^-10 */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), expo - 25); /* (1 + frac/1024) * 2^(expo-15) */
    }
    return sign ? -v : v;
}

/* bfloat16: the upper half of an IEEE-754 binary32. */
static double decode_bf16(uint16_t b) {
    uint32_t bits = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double decode(uint16_t x, int dtype) {
    return dtype == 0 ? decode_fp16(x) : decode_bf16(x);
}

/* Decodes n 16-bit values into doubles (used by the tests to check the two
 * decoders against an independent library conversion). */
void oracle_decode_values(double* out, const uint16_t* in, int64_t n, int dtype) {
    for (int64_t i = 0; i < n; ++i) out[i] = decode(in[i], dtype);
}

/*
 * Decode attention over a paged cache, one query token per sequence.
 *
 *   q            [num_seqs][num_q_heads][head_dim]            (16-bit)
 *   k_cache      [num_blocks][block_size][num_kv_heads][head_dim]
 *   v_cache      same layout as k_cache
 *   block_tables [num_seqs][max_blocks_per_seq]   int32, physical block ids
 *   context_lens [num_seqs]                       int32, tokens to attend to
 *   out          [num_seqs][num_q_heads][head_dim] double
 *
 * Returns 0, or -1 if an argument is inconsistent, or -2 if a block id that
 * would be read lies outside [0, num_blocks) (nothing is read then; the
 * affected row is left as NaN).
 */
int oracle_decode_attention(double* out, const uint16_t* q, const uint16_t* k_cache,
                            const uint16_t* v_cache, const int32_t* block_tables,
                            int max_blocks_per_seq, const int32_t* context_lens,
                            int num_seqs, int num_blocks, int block_size, int num_q_heads,
                            int num_kv_heads, int head_dim, double scale, int dtype) {
    if (num_seqs < 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        num_q_heads <= 0 || num_q_heads % num_kv_heads != 0 || (dtype != 0 && dtype != 1))
        return -1;
    const int group = num_q_heads / num_kv_heads; /* query heads per KV head */
    int status = 0;

#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < num_seqs; ++b) {
        for (int h = 0; h < num_q_heads; ++h) {
            double* o = out + ((int64_t)b * num_q_heads + h) * head_dim;
            const uint16_t* qv = q + ((int64_t)b * num_q_heads + h) * head_dim;
            const int g = h / group; /* the KV head this query head reads */
            const int n = context_lens[b];
            for (int j = 0; j < head_dim; ++j) o[j] = 0.0;
            if (n <= 0) continue;
            if (n > max_blocks_per_seq * block_size) {
                for (int j = 0; j < head_dim; ++j) o[j] = NAN;
#pragma omp atomic write
                status = -2;
                continue;
            }

            double* qd = (double*)malloc(sizeof(double) * (size_t)head_dim);
            double* s = (double*)malloc(sizeof(double) * (size_t)n);
            for (int j = 0; j < head_dim; ++j) qd[j] = decode(qv[j], dtype);

            /* scores s_t = scale * <q, K_t> over the gathered tokens */
            int bad = 0;
            for (int t = 0; t < n && !bad; ++t) {
                int32_t blk = block_tables[(int64_t)b * max_blocks_per_seq + t / block_size];
                int off = t % block_size;
                if (blk < 0 || blk >= num_blocks) { bad = 1; break; }
                const uint16_t* kt =
                    k_cache + (((int64_t)blk * block_size + off) * num_kv_heads + g) * head_dim;
                double dot = 0.0;
                for (int j = 0; j < head_dim; ++j) dot += qd[j] * decode(kt[j], dtype);
                s[t] = scale * dot;
            }
            if (bad) {
                for (int j = 0; j < head_dim; ++j) o[j] = NAN;
#pragma omp atomic write
                status = -2;
                free(qd);
                free(s);
                continue;
            }

            /* softmax with the maximum subtracted, then the weighted sum of V */
            double m = -INFINITY;
            for (int t = 0; t < n; ++t) if (s[t] > m) m = s[t];
            double z = 0.0;
            for (int t = 0; t < n; ++t) {
                s[t] = exp(s[t] - m);
                z += s[t];
            }
            for (int t = 0; t < n; ++t) {
                int32_t blk = block_tables[(int64_t)b * max_blocks_per_seq + t / block_size];
                int off = t % block_size;
                const uint16_t* vt =
                    v_cache + (((int64_t)blk * block_size + off) * num_kv_heads + g) * head_dim;
                double w = s[t] / z;
                for (int j = 0; j < head_dim; ++j) o[j] += w * decode(vt[j], dtype);
            }
            free(qd);
            free(s);
        }
    }
    return status;
}

/*
 * Append: for each new token i with slot_mapping[i] = s >= 0, copy its K and V
 * rows ([num_kv_heads][head_dim] 16-bit values) into block s / block_size at
 * offset s % block_size.  A negative slot is padding and is skipped.
 * (inference.html, KVCachePool.write_tokens; tutorial chapter 12,
 * PagedKVCache.update; gsyq.cn essay, kv_cache.append.)
 *
 * Returns 0, or -2 if a slot lies at or beyond num_blocks * block_size (that
 * token is skipped).
 */
int oracle_append(uint16_t* k_cache, uint16_t* v_cache, const uint16_t* k_new,
                  const uint16_t* v_new, const int64_t* slot_mapping, int num_tokens,
                  int num_blocks, int block_size, int num_kv_heads, int head_dim) {
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    int status = 0;
    for (int i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_blocks * block_size) {
            status = -2;
            continue;
        }
        int64_t blk = slot / block_size;
        int64_t off = slot % block_size;
        int64_t dst = (blk * block_size + off) * row;
        memcpy(k_cache + dst, k_new + (int64_t)i * row, sizeof(uint16_t) * (size_t)row);
        memcpy(v_cache + dst, v_new + (int64_t)i * row, sizeof(uint16_t) * (size_t)row);
    }
    return status;
}

/* ------------------------------------------------------------------------
 * FP8 KV cache (E4M3).  The vLLM deep dive (GPU execution, kernels and
 * graphs, 3.3 FP8 inference) gives E4M3 as the inference format, with the
 * value range held by a scale (per tensor or per token); its fusion list
 * (2.2) pairs the KV-cache write with quantisation.  Here: one fp32 scale
 * for K and one for V; a stored code is E4M3(x / scale), the fp32 quotient
 * rounded to nearest-even and saturated at +-448, and the value it stands for
 * is code * scale.
 *
 * E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits, no
 * infinities; S.1111.111 is NaN; the largest finite value is 448.
 * ------------------------------------------------------------------------ */
static double decode_e4m3(uint8_t x) {
    int sign = (x >> 7) & 1;
    int expo = (x >> 3) & 0xf;
    int frac = x & 7;
    double v;
    if (expo == 15 && frac == 7) {
        v = NAN;
    } else if (expo == 0) {
        v = ldexp((double)frac, -9);               /* subnormal: frac/8 * 2^-6 */
    } else {
        v = ldexp((double)(8 + frac), expo - 10);  /* (1 + frac/8) * 2^(expo-7) */
    }
    return sign ? -v : v;
}

void oracle_decode_e4m3(double* out, const uint8_t* in, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = decode_e4m3(in[i]);
}

/* Round half to even of a non-negative double that is an exact multiple of 1/2. */
static double round_half_even(double n) {
    double f = floor(n);
    double r = n - f;
    if (r > 0.5) return f + 1.0;
    if (r < 0.5) return f;
    return fmod(f, 2.0) == 0.0 ? f : f + 1.0;
}

/* Nearest E4M3 code to x (ties to the even code), saturating to +-448; NaN
 * gives the NaN code 0x7F. */
static uint8_t encode_e4m3(float x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;        /* saturate (also +-inf) */
    if (a == 0.0) return sign;
    int ex;
    frexp(a, &ex);                             /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;                            /* a in [2^e, 2^(e+1)) */
    if (e < -6) e = -6;                        /* subnormals: the spacing of binade -6 */
    double q = ldexp(1.0, e - 3);              /* spacing of E4M3 values there */
    double v = round_half_even(a / q) * q;     /* a / q is exact: q is a power of 2 */
    if (v >= 448.0) return sign | 0x7E;
    if (v == 0.0) return sign;
    if (v < ldexp(1.0, -6)) return sign | (uint8_t)(v / ldexp(1.0, -9));
    frexp(v, &ex);
    e = ex - 1;
    int frac = (int)(v / ldexp(1.0, e - 3)) - 8;
    return sign | (uint8_t)((e + 7) << 3) | (uint8_t)frac;
}

void oracle_encode_e4m3(uint8_t* out, const float* in, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = encode_e4m3(in[i]);
}

/* Quantising append: as oracle_append, with each element of the new K (V)
 * row stored as E4M3(x / k_scale) (E4M3(x / v_scale)), the quotient taken in
 * fp32.  new rows are 16-bit values of new_dtype (0 fp16, 1 bf16). */
int oracle_append_fp8(uint8_t* k_cache, uint8_t* v_cache, const uint16_t* k_new,
                      const uint16_t* v_new, const int64_t* slot_mapping, int num_tokens,
                      int num_blocks, int block_size, int num_kv_heads, int head_dim,
                      float k_scale, float v_scale, int new_dtype) {
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    int status = 0;
    for (int i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_blocks * block_size) {
            status = -2;
            continue;
        }
        int64_t dst = slot * row;  /* [num_blocks][block_size] rows, row = [heads][dim] */
        for (int64_t j = 0; j < row; ++j) {
            float kx = (float)decode(k_new[(int64_t)i * row + j], new_dtype);
            float vx = (float)decode(v_new[(int64_t)i * row + j], new_dtype);
            k_cache[dst + j] = encode_e4m3(kx / k_scale);
            v_cache[dst + j] = encode_e4m3(vx / v_scale);
        }
    }
    return status;
}

/*
 * Decode attention over an E4M3 cache: K_t = code * k_scale, V_t = code *
 * v_scale; q is 16-bit (q_dtype 0 fp16, 1 bf16); otherwise as
 * oracle_decode_attention (same layouts, masking and return codes).
 */
int oracle_decode_attention_fp8(double* out, const uint16_t* q, const uint8_t* k_cache,
                                const uint8_t* v_cache, const int32_t* block_tables,
                                int max_blocks_per_seq, const int32_t* context_lens,
                                int num_seqs, int num_blocks, int block_size, int num_q_heads,
                                int num_kv_heads, int head_dim, double scale, double k_scale,
                                double v_scale, int q_dtype) {
    if (num_seqs < 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        num_q_heads <= 0 || num_q_heads % num_kv_heads != 0 || (q_dtype != 0 && q_dtype != 1))
        return -1;
    const int group = num_q_heads / num_kv_heads;
    int status = 0;

#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < num_seqs; ++b) {
        for (int h = 0; h < num_q_heads; ++h) {
            double* o = out + ((int64_t)b * num_q_heads + h) * head_dim;
            const uint16_t* qv = q + ((int64_t)b * num_q_heads + h) * head_dim;
            const int kvh = h / group;
            const int n = context_lens[b];
            for (int j = 0; j < head_dim; ++j) o[j] = 0.0;
            if (n <= 0) continue;
            int bad = n > max_blocks_per_seq * block_size;
            for (int t = 0; t < n && !bad; ++t) {
                int32_t blk = block_tables[(int64_t)b * max_blocks_per_seq + t / block_size];
                if (blk < 0 || blk >= num_blocks) bad = 1;
            }
            if (bad) {
                for (int j = 0; j < head_dim; ++j) o[j] = NAN;
#pragma omp atomic write
                status = -2;
                continue;
            }
            double* qd = (double*)malloc(sizeof(double) * (size_t)head_dim);
            double* sc = (double*)malloc(sizeof(double) * (size_t)n);
            for (int j = 0; j < head_dim; ++j) qd[j] = decode(qv[j], q_dtype);
            double m = -INFINITY;
            for (int t = 0; t < n; ++t) {
                int32_t blk = block_tables[(int64_t)b * max_blocks_per_seq + t / block_size];
                const uint8_t* kt = k_cache +
                    (((int64_t)blk * block_size + t % block_size) * num_kv_heads + kvh) * head_dim;
                double dot = 0.0;
                for (int j = 0; j < head_dim; ++j) dot += qd[j] * (decode_e4m3(kt[j]) * k_scale);
                sc[t] = scale * dot;
                if (sc[t] > m) m = sc[t];
            }
            double z = 0.0;
            for (int t = 0; t < n; ++t) {
                sc[t] = exp(sc[t] - m);
                z += sc[t];
            }
            for (int t = 0; t < n; ++t) {
                int32_t blk = block_tables[(int64_t)b * max_blocks_per_seq + t / block_size];
                const uint8_t* vt = v_cache +
                    (((int64_t)blk * block_size + t % block_size) * num_kv_heads + kvh) * head_dim;
                double w = sc[t] / z;
                for (int j = 0; j < head_dim; ++j) o[j] += w * (decode_e4m3(vt[j]) * v_scale);
            }
            free(qd);
            free(sc);
        }
    }
    return status;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
