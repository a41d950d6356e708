/*
 * kvc_oracle.c -- plain, slow CPU oracle for the single-token KV-cache decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call this file:
 * only the tests, the package's smoke check and the benchmark's CPU-baseline arm use it.
 * It shares no code, header, table or constant with the CUDA library; it includes only
 * the C standard library.
 *
 * Every floating-point reduction is done in double precision, in the order the
 * definition is written, with no blocking, fusion or reordering.
 *
 * Sources (web pages on the KV cache; page title, then section):
 *   [KVG]  "KV 缓存" (llm-glossary, terms/kv-cache): "两条数学等价的 decode 路径",
 *          "可直接运行的对照实验", "容量公式：先算逻辑 payload，再谈 allocator".
 *   [W1D4] "第 1 周 · Day 4：KV Cache 与 MQA / GQA" (CME295 notes): §1.2, §1.3, §1.4,
 *          §2.3, §3.1, §3.3, §3.4.
 *   [M11]  "11.7 KV Cache：形状、显存与带宽" (Linear-Algebra-to-LLM): §2.2, §2.3, §4.2-§5.4.
 *
 * Readings taken where the pages are silent or garbled (listed in the design notes too):
 *   - score scale is 1/sqrt(D): [M11] §2.2 prints "/d_k" (the square root was lost in
 *     extraction); the teaching code in [KVG] divides by math.sqrt(head_dim).
 *   - the new token attends to itself: append first, then attend over all L slots
 *     ([W1D4] §1.3: after the append the new query attends to all t+1 cached keys).
 *   - lens[b] is the valid length AFTER the call's write; append writes slot lens[b]-1.
 *   - query head j reads KV head floor(j / (H_q/H_kv))  ([W1D4] §3.4, repeat_interleave).
 *   - a row with lens[b] < 1 or lens[b] > T_max is invalid: its output is zero and it is
 *     counted in the return value.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_BF16 0
#define OR_F32 1

/* Planted mistakes, for the tests that show the pins have teeth.  They exist only in a second
 * build of this file (-DORACLE_PLANTED, libkvc_oracle_planted.so) that the tests switch to while
 * a mistake is planted; in the oracle itself PLANTED(n) is the constant 0 and no branch is left. */
#ifdef ORACLE_PLANTED
static int g_fault = 0;
void oracle_set_fault(int which) { g_fault = which; }
int oracle_get_fault(void) { return g_fault; }
#define PLANTED(n) (g_fault == (n))
#else
#define PLANTED(n) 0
#endif

static int g_threads = 1;
/* Number of host threads the decode routine may use (1 = plain single-threaded loop). */
int oracle_set_threads(int n) {
    g_threads = n < 1 ? 1 : n;
#ifdef _OPENMP
    return g_threads;
#else
    g_threads = 1;
    return 1;
#endif
}

/* One stored element as a double.  bf16 is the top half of an IEEE binary32, so widening
 * it is exact; fp32 widens exactly too. */
static double load_elem(const void* base, int dtype, size_t idx) {
    if (dtype == OR_F32) return (double)((const float*)base)[idx];
    uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static int elem_bytes_of(int dtype) { return dtype == OR_F32 ? 4 : 2; }

/* ---------------------------------------------------------------------------------------
 * Capacity: [KVG] 容量公式 and [W1D4] §1.4: bytes = 2 * L * H_kv * D * (B * T) * s, the 2
 * counting K and V.  The ragged form ([KVG], same section) replaces B*T by sum_i T_i.
 * ------------------------------------------------------------------------------------- */
uint64_t oracle_kv_bytes(int64_t L, int64_t B, int64_t H_kv, int64_t D, int64_t T, int64_t s) {
    return (uint64_t)2 * (uint64_t)L * (uint64_t)H_kv * (uint64_t)D * ((uint64_t)B * (uint64_t)T) *
           (uint64_t)s;
}

uint64_t oracle_kv_bytes_ragged(int64_t L, int64_t H_kv, int64_t D, int64_t s, const int32_t* T_i,
                                int n) {
    uint64_t sum = 0;
    for (int i = 0; i < n; ++i) sum += (uint64_t)T_i[i];
    return (uint64_t)2 * (uint64_t)L * (uint64_t)H_kv * (uint64_t)D * (uint64_t)s * sum;
}

/* ---------------------------------------------------------------------------------------
 * Cache writes.  [W1D4] §3.1: the cache is preallocated to max_len and the new rows are
 * written in place at [pos, pos+T); [KVG] "从教学代码到生产实现还差什么" item 1.
 * Layout [B, H_kv, T_max, D], row = one token's D-vector.
 * ------------------------------------------------------------------------------------- */

/* Writes k_new[b,h,:] / v_new[b,h,:] (layout [B,H_kv,D]) into slot lens[b]-1.
 * Returns the number of batch rows skipped because lens[b] is out of [1, T_max]. */
int oracle_append(void* Kc, void* Vc, const void* k_new, const void* v_new, const int32_t* lens,
                  int B, int H_kv, int T_max, int D, int dtype) {
    const size_t row = (size_t)D * elem_bytes_of(dtype);
    int bad = 0;
    for (int b = 0; b < B; ++b) {
        int L = lens[b];
        if (L < 1 || L > T_max) {
            ++bad;
            continue;
        }
        int slot = L - 1;
        if (PLANTED(3)) slot = L; /* planted: off-by-one slot */
        if (slot >= T_max) continue;
        for (int h = 0; h < H_kv; ++h) {
            size_t dst = (((size_t)b * H_kv + h) * T_max + slot) * row;
            size_t src = ((size_t)b * H_kv + h) * row;
            memcpy((char*)Kc + dst, (const char*)k_new + src, row);
            memcpy((char*)Vc + dst, (const char*)v_new + src, row);
        }
    }
    return bad;
}

/* Writes K[b,h,0:lens[b],:] (layout [B,H_kv,T_in,D]) into cache slots [0, lens[b]).
 * Returns the number of rows skipped because lens[b] is out of [0, min(T_in, T_max)]. */
int oracle_prefill_write(void* Kc, void* Vc, const void* K, const void* V, int T_in,
                         const int32_t* lens, int B, int H_kv, int T_max, int D, int dtype) {
    const size_t row = (size_t)D * elem_bytes_of(dtype);
    int bad = 0;
    for (int b = 0; b < B; ++b) {
        int L = lens[b];
        if (L < 0 || L > T_in || L > T_max) {
            ++bad;
            continue;
        }
        for (int h = 0; h < H_kv; ++h)
            for (int t = 0; t < L; ++t) {
                size_t dst = (((size_t)b * H_kv + h) * T_max + t) * row;
                size_t src = (((size_t)b * H_kv + h) * T_in + t) * row;
                memcpy((char*)Kc + dst, (const char*)K + src, row);
                memcpy((char*)Vc + dst, (const char*)V + src, row);
            }
    }
    return bad;
}

/* ---------------------------------------------------------------------------------------
 * Decode attention for one query row, in double.  [M11] §2.2:
 *   s_t = q . k_t / sqrt(D),   o = softmax(s) V
 * over t in [0, L).  The softmax subtracts the row maximum before exponentiating (the same
 * value mathematically; it keeps exp finite).
 * q: D doubles; K, V: L rows of D doubles at stride `ld`; o: D doubles.
 * ------------------------------------------------------------------------------------- */
static void decode_row_f64(const double* q, const double* K, const double* V, int L, int D,
                           size_t ld, double* o, double* s /* scratch, L doubles */) {
    double scale = 1.0 / sqrt((double)D);
    if (PLANTED(2)) scale = 1.0 / (double)D; /* planted: the garbled "/d_k" reading */
    int Lr = (PLANTED(4)) ? L - 1 : L;       /* planted: new token left out */
    if (Lr < 1) Lr = 1;
    for (int t = 0; t < Lr; ++t) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += q[d] * K[(size_t)t * ld + d];
        s[t] = acc * scale;
    }
    double m = s[0];
    for (int t = 1; t < Lr; ++t)
        if (s[t] > m) m = s[t];
    double Z = 0.0;
    for (int t = 0; t < Lr; ++t) {
        s[t] = exp(s[t] - m);
        Z += s[t];
    }
    for (int d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int t = 0; t < Lr; ++t) acc += s[t] * V[(size_t)t * ld + d];
        o[d] = acc / Z;
    }
}

/* KV head read by query head j: [W1D4] §3.4, floor(j / (H_q / H_kv)). */
static int kv_head_of(int j, int H_q, int H_kv) {
    int g = H_q / H_kv;
    if (PLANTED(1)) return j % H_kv; /* planted: interleaved ("repeat") grouping */
    return j / g;
}

/* Decode attention over the cache.
 *   q     [B, H_q, D]           (dtype)
 *   Kc,Vc [B, H_kv, T_max, D]   (dtype)
 *   lens  [B]                   valid length of each sequence (the new token included)
 *   out   [B, H_q, D]           double
 * Returns the number of invalid rows (lens out of [1, T_max]); their output is zero. */
int oracle_decode_attn(const void* q, const void* Kc, const void* Vc, const int32_t* lens, int B,
                       int H_q, int H_kv, int T_max, int D, int dtype, double* out) {
    int bad = 0;
    for (int b = 0; b < B; ++b)
        if (lens[b] < 1 || lens[b] > T_max) ++bad;
    const int rows = B * H_q;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(g_threads) if (g_threads > 1)
#endif
    for (int r = 0; r < rows; ++r) {
        int b = r / H_q, j = r % H_q;
        int L = lens[b];
        double* o = out + (size_t)r * D;
        if (L < 1 || L > T_max) {
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            continue;
        }
        int h = kv_head_of(j, H_q, H_kv);
        double* qd = (double*)malloc(sizeof(double) * D);
        double* Kd = (double*)malloc(sizeof(double) * (size_t)L * D);
        double* Vd = (double*)malloc(sizeof(double) * (size_t)L * D);
        double* s = (double*)malloc(sizeof(double) * (size_t)L);
        for (int d = 0; d < D; ++d) qd[d] = load_elem(q, dtype, (size_t)r * D + d);
        size_t base = ((size_t)b * H_kv + h) * (size_t)T_max * D;
        for (size_t i = 0; i < (size_t)L * D; ++i) {
            Kd[i] = load_elem(Kc, dtype, base + i);
            Vd[i] = load_elem(Vc, dtype, base + i);
        }
        decode_row_f64(qd, Kd, Vd, L, D, (size_t)D, o, s);
        free(qd);
        free(Kd);
        free(Vd);
        free(s);
    }
    return bad;
}

/* ---------------------------------------------------------------------------------------
 * Paged cache.  The pages describe storage cut into fixed-size blocks handed out on demand,
 * found through a table, with the attention arithmetic unchanged ([W1D4] §1.6; [KVG]
 * "先把它放回推理链路" and "成本转移、失败场景与常见误解"; [M11] §8).  They fix no layout; the
 * reading taken here:
 *   pool  [num_blocks, H_kv, bs, D]   (dtype), one per layer for K and one for V
 *   table [B, max_blocks]             int32, physical block of logical block j of sequence b
 *   token t of sequence b, head h  ->  pool[table[b, t / bs], h, t % bs, :]
 * A row is invalid when lens[b] is out of [1, max_blocks * bs] (appends and attention) or
 * when a table entry it needs is out of [0, num_blocks).
 * ------------------------------------------------------------------------------------- */

static int paged_row_ok(const int32_t* table, int b, int L, int L_min, int bs, int max_blocks,
                        int num_blocks) {
    if (L < L_min || L > max_blocks * bs) return 0;
    int nb = (L + bs - 1) / bs;
    for (int j = 0; j < nb; ++j) {
        int e = table[(size_t)b * max_blocks + j];
        if (e < 0 || e >= num_blocks) return 0;
    }
    return 1;
}

static size_t paged_row_offset(const int32_t* table, int b, int h, int t, int H_kv, int bs,
                               int max_blocks) {
    int e = table[(size_t)b * max_blocks + t / bs];
    if (PLANTED(5)) /* planted: token-major block ([bs, H_kv] instead of [H_kv, bs]) */
        return ((size_t)e * bs + (size_t)(t % bs)) * H_kv + h;
    return (((size_t)e * H_kv + h) * bs + (size_t)(t % bs));
}

/* Writes k_new[b,h,:] (layout [B,H_kv,D]) into token lens[b]-1 of sequence b.  Returns the
 * number of invalid rows (skipped). */
int oracle_paged_append(void* Kp, void* Vp, const void* k_new, const void* v_new,
                        const int32_t* table, const int32_t* lens, int B, int H_kv, int D,
                        int bs, int max_blocks, int num_blocks, int dtype) {
    const size_t row = (size_t)D * elem_bytes_of(dtype);
    int bad = 0;
    for (int b = 0; b < B; ++b) {
        int L = lens[b];
        if (!paged_row_ok(table, b, L, 1, bs, max_blocks, num_blocks)) {
            ++bad;
            continue;
        }
        for (int h = 0; h < H_kv; ++h) {
            size_t dst = paged_row_offset(table, b, h, L - 1, H_kv, bs, max_blocks) * row;
            size_t src = ((size_t)b * H_kv + h) * row;
            memcpy((char*)Kp + dst, (const char*)k_new + src, row);
            memcpy((char*)Vp + dst, (const char*)v_new + src, row);
        }
    }
    return bad;
}

/* Writes K[b,h,0:lens[b],:] (layout [B,H_kv,T_in,D]) into tokens [0, lens[b]) of sequence b.
 * Returns the number of invalid rows (lens[b] > T_in counts as invalid; lens[b] = 0 writes
 * nothing and is valid). */
int oracle_paged_prefill_write(void* Kp, void* Vp, const void* K, const void* V, int T_in,
                               const int32_t* table, const int32_t* lens, int B, int H_kv, int D,
                               int bs, int max_blocks, int num_blocks, int dtype) {
    const size_t row = (size_t)D * elem_bytes_of(dtype);
    int bad = 0;
    for (int b = 0; b < B; ++b) {
        int L = lens[b];
        if (L > T_in || !paged_row_ok(table, b, L, 0, bs, max_blocks, num_blocks)) {
            ++bad;
            continue;
        }
        for (int h = 0; h < H_kv; ++h)
            for (int t = 0; t < L; ++t) {
                size_t dst = paged_row_offset(table, b, h, t, H_kv, bs, max_blocks) * row;
                size_t src = (((size_t)b * H_kv + h) * T_in + t) * row;
                memcpy((char*)Kp + dst, (const char*)K + src, row);
                memcpy((char*)Vp + dst, (const char*)V + src, row);
            }
    }
    return bad;
}

/* Decode attention over a paged cache: for every query row, the history rows are read
 * through the table in token order, then the same arithmetic as oracle_decode_attn.
 * out [B, H_q, D] double; invalid rows are zero.  Returns the number of invalid rows. */
int oracle_paged_decode_attn(const void* q, const void* Kp, const void* Vp, const int32_t* table,
                             const int32_t* lens, int B, int H_q, int H_kv, int D, int bs,
                             int max_blocks, int num_blocks, int dtype, double* out) {
    int bad = 0;
    for (int b = 0; b < B; ++b)
        if (!paged_row_ok(table, b, lens[b], 1, bs, max_blocks, num_blocks)) ++bad;
    const int rows = B * H_q;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(g_threads) if (g_threads > 1)
#endif
    for (int r = 0; r < rows; ++r) {
        int b = r / H_q, j = r % H_q;
        int L = lens[b];
        double* o = out + (size_t)r * D;
        if (!paged_row_ok(table, b, L, 1, bs, max_blocks, num_blocks)) {
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            continue;
        }
        int h = kv_head_of(j, H_q, H_kv);
        double* qd = (double*)malloc(sizeof(double) * D);
        double* Kd = (double*)malloc(sizeof(double) * (size_t)L * D);
        double* Vd = (double*)malloc(sizeof(double) * (size_t)L * D);
        double* s = (double*)malloc(sizeof(double) * (size_t)L);
        for (int d = 0; d < D; ++d) qd[d] = load_elem(q, dtype, (size_t)r * D + d);
        for (int t = 0; t < L; ++t) {
            size_t base = paged_row_offset(table, b, h, t, H_kv, bs, max_blocks) * D;
            for (int d = 0; d < D; ++d) {
                Kd[(size_t)t * D + d] = load_elem(Kp, dtype, base + d);
                Vd[(size_t)t * D + d] = load_elem(Vp, dtype, base + d);
            }
        }
        decode_row_f64(qd, Kd, Vd, L, D, (size_t)D, o, s);
        free(qd);
        free(Kd);
        free(Vd);
        free(s);
    }
    return bad;
}

/* ---------------------------------------------------------------------------------------
 * Quantized cache.  The pages list int8 / fp8 caches as a way to read fewer bytes, with the
 * softmax accumulated in higher precision, and name per-token / per-head scales among the
 * formats ([KVG] "MHA、GQA、MLA 与量化如何改变容量"; [M11] §3.1 and §8; [W1D4] §1.5).  Reading
 * taken: symmetric int8, one fp32 scale per (sequence, KV head, token) row, no zero point:
 *   scale = max_d |x_d| / 127           (fp32)
 *   code_d = round_half_even(x_d / scale), clamped to [-127, 127]   (fp32 division)
 *   x_d ~ code_d * scale                 (the attention reads these values)
 * A row of zeros has scale 0 and codes 0.  Layout per layer: codes [B, H_kv, T_max, D] int8,
 * scales [B, H_kv, T_max] fp32, for K and for V.
 * ------------------------------------------------------------------------------------- */

static float load_f32(const void* base, int dtype, size_t idx) {
    if (dtype == OR_F32) return ((const float*)base)[idx];
    return (float)load_elem(base, dtype, idx); /* bf16 -> float is exact */
}

static void quant_row(const void* x, int dtype, size_t off, int D, int8_t* codes, float* scale) {
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) {
        float a = fabsf(load_f32(x, dtype, off + d));
        if (a > amax) amax = a;
    }
    float s = amax / 127.0f;
    if (PLANTED(8)) s = amax / 128.0f; /* planted: scale off by one level */
    *scale = s;
    for (int d = 0; d < D; ++d) {
        float c = 0.0f;
        if (s > 0.0f) c = rintf(load_f32(x, dtype, off + d) / s);
        if (c > 127.0f) c = 127.0f;
        if (c < -127.0f) c = -127.0f;
        codes[d] = (int8_t)c;
    }
}

/* Quantizes rows of a [n_rows, D] array (dtype) into codes [n_rows, D] and scales [n_rows]. */
void oracle_quantize_rows(const void* x, int n_rows, int D, int dtype, int8_t* codes, float* scales) {
    for (int r = 0; r < n_rows; ++r)
        quant_row(x, dtype, (size_t)r * D, D, codes + (size_t)r * D, scales + r);
}

/* Appends k_new/v_new [B, H_kv, D] (dtype), quantized, at slot lens[b]-1.  Returns the number of
 * invalid rows (lens out of [1, T_max]; skipped). */
int oracle_quant_append(int8_t* Kq, float* Ks, int8_t* Vq, float* Vs, const void* k_new,
                        const void* v_new, const int32_t* lens, int B, int H_kv, int T_max, int D,
                        int dtype) {
    int bad = 0;
    for (int b = 0; b < B; ++b) {
        int L = lens[b];
        if (L < 1 || L > T_max) {
            ++bad;
            continue;
        }
        for (int h = 0; h < H_kv; ++h) {
            size_t row = ((size_t)b * H_kv + h) * T_max + (size_t)(L - 1);
            size_t src = ((size_t)b * H_kv + h) * D;
            quant_row(k_new, dtype, src, D, Kq + row * D, Ks + row);
            quant_row(v_new, dtype, src, D, Vq + row * D, Vs + row);
        }
    }
    return bad;
}

/* Writes K/V [B, H_kv, T_in, D] (dtype) rows [0, lens[b]), quantized.  Returns the number of
 * invalid rows (lens out of [0, min(T_in, T_max)]). */
int oracle_quant_prefill_write(int8_t* Kq, float* Ks, int8_t* Vq, float* Vs, const void* K,
                               const void* V, int T_in, const int32_t* lens, int B, int H_kv,
                               int T_max, int D, int dtype) {
    int bad = 0;
    for (int b = 0; b < B; ++b) {
        int L = lens[b];
        if (L < 0 || L > T_in || L > T_max) {
            ++bad;
            continue;
        }
        for (int h = 0; h < H_kv; ++h)
            for (int t = 0; t < L; ++t) {
                size_t row = ((size_t)b * H_kv + h) * T_max + (size_t)t;
                size_t src = (((size_t)b * H_kv + h) * T_in + t) * D;
                quant_row(K, dtype, src, D, Kq + row * D, Ks + row);
                quant_row(V, dtype, src, D, Vq + row * D, Vs + row);
            }
    }
    return bad;
}

/* Decode attention over a quantized cache: the same arithmetic as oracle_decode_attn on the
 * values code * scale (formed in double).  out [B, H_q, D] double. */
int oracle_quant_decode_attn(const void* q, const int8_t* Kq, const float* Ks, const int8_t* Vq,
                             const float* Vs, const int32_t* lens, int B, int H_q, int H_kv,
                             int T_max, int D, int dtype, double* out) {
    int bad = 0;
    for (int b = 0; b < B; ++b)
        if (lens[b] < 1 || lens[b] > T_max) ++bad;
    const int rows = B * H_q;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(g_threads) if (g_threads > 1)
#endif
    for (int r = 0; r < rows; ++r) {
        int b = r / H_q, j = r % H_q;
        int L = lens[b];
        double* o = out + (size_t)r * D;
        if (L < 1 || L > T_max) {
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            continue;
        }
        int h = kv_head_of(j, H_q, H_kv);
        double* qd = (double*)malloc(sizeof(double) * D);
        double* Kd = (double*)malloc(sizeof(double) * (size_t)L * D);
        double* Vd = (double*)malloc(sizeof(double) * (size_t)L * D);
        double* sc = (double*)malloc(sizeof(double) * (size_t)L);
        for (int d = 0; d < D; ++d) qd[d] = load_elem(q, dtype, (size_t)r * D + d);
        size_t row0 = ((size_t)b * H_kv + h) * (size_t)T_max;
        for (int t = 0; t < L; ++t) {
            double sk = (double)Ks[row0 + t], sv = (double)Vs[row0 + t];
            for (int d = 0; d < D; ++d) {
                Kd[(size_t)t * D + d] = (double)Kq[(row0 + t) * D + d] * sk;
                Vd[(size_t)t * D + d] = (double)Vq[(row0 + t) * D + d] * sv;
            }
        }
        decode_row_f64(qd, Kd, Vd, L, D, (size_t)D, o, sc);
        free(qd);
        free(Kd);
        free(Vd);
        free(sc);
    }
    return bad;
}

/* ---------------------------------------------------------------------------------------
 * fp8 cache.  The pages name fp8 beside int8 as a cache format read with higher-precision
 * softmax accumulation ([M11] §3.1 and §8; [KVG] "MHA、GQA、MLA 与量化如何改变容量").  Reading
 * taken: E4M3 codes as the OCP 8-bit floating-point format defines them -- 1 sign bit, 4
 * exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds the subnormals m * 2^-9;
 * there is no infinity and S.1111.111 is NaN, so the largest finite magnitude is
 * 1.75 * 2^8 = 448 -- with one fp32 scale per (sequence, KV head, token) row:
 *   scale = max_d |x_d| / 448                      (fp32)
 *   code_d = e4m3(x_d / scale)                     (fp32 division, then round to the nearest
 *                                                   code, ties to the even code; magnitudes
 *                                                   beyond 448 saturate to 448)
 *   x_d ~ value(code_d) * scale                    (the attention reads these values)
 * A row of zeros has scale 0 and codes 0.  Layout as for int8: codes [B, H_kv, T_max, D] (one
 * byte each), scales [B, H_kv, T_max] fp32, for K and for V.
 * ------------------------------------------------------------------------------------- */

/* The value a code stands for (NaN for the two NaN codes). */
double oracle_e4m3_value(uint8_t c) {
    int e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    double v = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return (c & 0x80) ? -v : v;
}

/* Nearest code to x (ties to the even code), saturating at +-448; the sign bit follows x's
 * (so -0 gives 0x80).  x is finite.  The non-negative finite codes 0x00 .. 0x7E are ordered by
 * value, so the code below x is found by bisection over them. */
uint8_t oracle_e4m3_encode(float x) {
    const uint8_t sign = signbit(x) ? 0x80 : 0;
    double v = fabs((double)x);
    if (v >= 448.0) return sign | 0x7E;
    int lo = 0, hi = 0x7E; /* value(lo) <= v < value(hi) */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (oracle_e4m3_value((uint8_t)mid) <= v) lo = mid; else hi = mid;
    }
    double a = oracle_e4m3_value((uint8_t)lo), b = oracle_e4m3_value((uint8_t)hi);
    int c;
    if (v - a < b - v) c = lo;
    else if (v - a > b - v) c = hi;
    else c = (lo & 1) ? hi : lo; /* a tie: the even code */
    if (PLANTED(9) && v - a == b - v) c = hi; /* planted: ties away from zero */
    return sign | (uint8_t)c;
}

static void fp8_row(const void* x, int dtype, size_t off, int D, uint8_t* codes, float* scale) {
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) {
        float a = fabsf(load_f32(x, dtype, off + d));
        if (a > amax) amax = a;
    }
    float s = amax / 448.0f;
    if (PLANTED(10)) s = amax / 240.0f; /* planted: the range of the other E4M3 variant */
    *scale = s;
    for (int d = 0; d < D; ++d) codes[d] = s > 0.0f ? oracle_e4m3_encode(load_f32(x, dtype, off + d) / s) : 0;
}

/* Quantizes rows of a [n_rows, D] array (dtype) into E4M3 codes [n_rows, D] and scales [n_rows]. */
void oracle_fp8_quantize_rows(const void* x, int n_rows, int D, int dtype, uint8_t* codes, float* scales) {
    for (int r = 0; r < n_rows; ++r) fp8_row(x, dtype, (size_t)r * D, D, codes + (size_t)r * D, scales + r);
}

/* Appends k_new/v_new [B, H_kv, D] (dtype), as fp8 rows, at slot lens[b]-1.  Returns the number
 * of invalid rows (lens out of [1, T_max]; skipped). */
int oracle_fp8_append(uint8_t* Kq, float* Ks, uint8_t* Vq, float* Vs, const void* k_new,
                      const void* v_new, const int32_t* lens, int B, int H_kv, int T_max, int D,
                      int dtype) {
    int bad = 0;
    for (int b = 0; b < B; ++b) {
        int L = lens[b];
        if (L < 1 || L > T_max) {
            ++bad;
            continue;
        }
        for (int h = 0; h < H_kv; ++h) {
            size_t row = ((size_t)b * H_kv + h) * T_max + (size_t)(L - 1);
            size_t src = ((size_t)b * H_kv + h) * D;
            fp8_row(k_new, dtype, src, D, Kq + row * D, Ks + row);
            fp8_row(v_new, dtype, src, D, Vq + row * D, Vs + row);
        }
    }
    return bad;
}

/* Writes K/V [B, H_kv, T_in, D] (dtype) rows [0, lens[b]) as fp8 rows.  Returns the number of
 * invalid rows (lens out of [0, min(T_in, T_max)]). */
int oracle_fp8_prefill_write(uint8_t* Kq, float* Ks, uint8_t* Vq, float* Vs, const void* K,
                             const void* V, int T_in, const int32_t* lens, int B, int H_kv,
                             int T_max, int D, int dtype) {
    int bad = 0;
    for (int b = 0; b < B; ++b) {
        int L = lens[b];
        if (L < 0 || L > T_in || L > T_max) {
            ++bad;
            continue;
        }
        for (int h = 0; h < H_kv; ++h)
            for (int t = 0; t < L; ++t) {
                size_t row = ((size_t)b * H_kv + h) * T_max + (size_t)t;
                size_t src = (((size_t)b * H_kv + h) * T_in + t) * D;
                fp8_row(K, dtype, src, D, Kq + row * D, Ks + row);
                fp8_row(V, dtype, src, D, Vq + row * D, Vs + row);
            }
    }
    return bad;
}

/* Decode attention over an fp8 cache: the same arithmetic as oracle_decode_attn on the values
 * value(code) * scale (formed in double).  out [B, H_q, D] double. */
int oracle_fp8_decode_attn(const void* q, const uint8_t* Kq, const float* Ks, const uint8_t* Vq,
                           const float* Vs, const int32_t* lens, int B, int H_q, int H_kv,
                           int T_max, int D, int dtype, double* out) {
    int bad = 0;
    for (int b = 0; b < B; ++b)
        if (lens[b] < 1 || lens[b] > T_max) ++bad;
    const int rows = B * H_q;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(g_threads) if (g_threads > 1)
#endif
    for (int r = 0; r < rows; ++r) {
        int b = r / H_q, j = r % H_q;
        int L = lens[b];
        double* o = out + (size_t)r * D;
        if (L < 1 || L > T_max) {
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            continue;
        }
        int h = kv_head_of(j, H_q, H_kv);
        double* qd = (double*)malloc(sizeof(double) * D);
        double* Kd = (double*)malloc(sizeof(double) * (size_t)L * D);
        double* Vd = (double*)malloc(sizeof(double) * (size_t)L * D);
        double* sc = (double*)malloc(sizeof(double) * (size_t)L);
        for (int d = 0; d < D; ++d) qd[d] = load_elem(q, dtype, (size_t)r * D + d);
        size_t row0 = ((size_t)b * H_kv + h) * (size_t)T_max;
        for (int t = 0; t < L; ++t) {
            double sk = (double)Ks[row0 + t], sv = (double)Vs[row0 + t];
            for (int d = 0; d < D; ++d) {
                Kd[(size_t)t * D + d] = oracle_e4m3_value(Kq[(row0 + t) * D + d]) * sk;
                Vd[(size_t)t * D + d] = oracle_e4m3_value(Vq[(row0 + t) * D + d]) * sv;
            }
        }
        decode_row_f64(qd, Kd, Vd, L, D, (size_t)D, o, sc);
        free(qd);
        free(Kd);
        free(Vd);
        free(sc);
    }
    return bad;
}

/* ---------------------------------------------------------------------------------------
 * Several new tokens per step (chunked prefill, speculative decoding).  With a cache holding
 * S keys after appending T new tokens, new query i (absolute position S - T + i) sees keys
 * 0 .. S - T + i: the causal mask aligned to the lower right of the T x S score matrix
 * ([W1D4] §3.3, third case; the upper-left alignment is the pitfall the same section names).
 *   q, out  [B, H_q, T_q, D]      k_new, v_new  [B, H_kv, T_q, D]
 * lens[b] is the post-append length S; a row is invalid unless T_q <= lens[b] <= T_max.
 * ------------------------------------------------------------------------------------- */

/* Writes the T_q new rows of every (b, h) into slots [lens[b] - T_q, lens[b]).  Returns the
 * number of invalid rows (skipped). */
int oracle_append_multi(void* Kc, void* Vc, const void* k_new, const void* v_new,
                        const int32_t* lens, int B, int H_kv, int T_max, int D, int T_q, int dtype) {
    const size_t row = (size_t)D * elem_bytes_of(dtype);
    int bad = 0;
    for (int b = 0; b < B; ++b) {
        int L = lens[b];
        if (T_q < 1 || L < T_q || L > T_max) {
            ++bad;
            continue;
        }
        for (int h = 0; h < H_kv; ++h)
            for (int i = 0; i < T_q; ++i) {
                size_t dst = (((size_t)b * H_kv + h) * T_max + (size_t)(L - T_q + i)) * row;
                size_t src = (((size_t)b * H_kv + h) * T_q + i) * row;
                memcpy((char*)Kc + dst, (const char*)k_new + src, row);
                memcpy((char*)Vc + dst, (const char*)v_new + src, row);
            }
    }
    return bad;
}

/* Decode attention of T_q new queries per head over the cache [B, H_kv, T_max, D].
 * out [B, H_q, T_q, D] double; invalid rows are zero.  Returns the number of invalid rows. */
int oracle_decode_multi(const void* q, const void* Kc, const void* Vc, const int32_t* lens, int B,
                        int H_q, int H_kv, int T_max, int D, int T_q, int dtype, double* out) {
    int bad = 0;
    for (int b = 0; b < B; ++b)
        if (T_q < 1 || lens[b] < T_q || lens[b] > T_max) ++bad;
    const int rows = B * H_q * T_q;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(g_threads) if (g_threads > 1)
#endif
    for (int r = 0; r < rows; ++r) {
        int b = r / (H_q * T_q), j = (r / T_q) % H_q, i = r % T_q;
        int L = lens[b];
        double* o = out + (size_t)r * D;
        if (T_q < 1 || L < T_q || L > T_max) {
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            continue;
        }
        int visible = L - T_q + i + 1; /* keys 0 .. L - T_q + i */
        if (PLANTED(7)) visible = i + 1; /* planted: upper-left aligned causal mask */
        int h = kv_head_of(j, H_q, H_kv);
        double* qd = (double*)malloc(sizeof(double) * D);
        double* Kd = (double*)malloc(sizeof(double) * (size_t)visible * D);
        double* Vd = (double*)malloc(sizeof(double) * (size_t)visible * D);
        double* sc = (double*)malloc(sizeof(double) * (size_t)visible);
        for (int d = 0; d < D; ++d) qd[d] = load_elem(q, dtype, (size_t)r * D + d);
        size_t base = ((size_t)b * H_kv + h) * (size_t)T_max * D;
        for (size_t e = 0; e < (size_t)visible * D; ++e) {
            Kd[e] = load_elem(Kc, dtype, base + e);
            Vd[e] = load_elem(Vc, dtype, base + e);
        }
        decode_row_f64(qd, Kd, Vd, visible, D, (size_t)D, o, sc);
        free(qd);
        free(Kd);
        free(Vd);
        free(sc);
    }
    return bad;
}

/* ---------------------------------------------------------------------------------------
 * Sliding window and rolling cache.  With a window of W tokens the query of the newest token
 * (position L-1) attends to the W most recent positions [max(0, L-W), L), and the cache only
 * needs W slots: position p lives in slot p mod W, the oldest entry being overwritten
 * ([W1D4] §2.7 and §1.6, the rolling cache of a sliding-window model; [M11] §8).
 * ------------------------------------------------------------------------------------- */

/* First position of the window of a sequence of length L. */
static int window_start(int L, int W) {
    int t0 = L - W;
    if (PLANTED(6)) t0 = L - W - 1; /* planted: one position too many */
    return t0 > 0 ? t0 : 0;
}

/* Sliding-window decode over a full-history cache [B, H_kv, T_max, D]: positions
 * [max(0, L-W), L).  out [B, H_q, D] double.  Returns the number of invalid rows. */
int oracle_window_decode_attn(const void* q, const void* Kc, const void* Vc, const int32_t* lens,
                              int B, int H_q, int H_kv, int T_max, int D, int W, int dtype,
                              double* out) {
    int bad = 0;
    for (int r = 0; r < B * H_q; ++r) {
        int b = r / H_q, j = r % H_q;
        int L = lens[b];
        double* o = out + (size_t)r * D;
        if (L < 1 || L > T_max || W < 1) {
            if (j == 0) ++bad;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            continue;
        }
        int h = kv_head_of(j, H_q, H_kv);
        int t0 = window_start(L, W), n = L - t0;
        double* qd = (double*)malloc(sizeof(double) * D);
        double* Kd = (double*)malloc(sizeof(double) * (size_t)n * D);
        double* Vd = (double*)malloc(sizeof(double) * (size_t)n * D);
        double* sc = (double*)malloc(sizeof(double) * (size_t)n);
        for (int d = 0; d < D; ++d) qd[d] = load_elem(q, dtype, (size_t)r * D + d);
        size_t base = (((size_t)b * H_kv + h) * (size_t)T_max + (size_t)t0) * D;
        for (size_t i = 0; i < (size_t)n * D; ++i) {
            Kd[i] = load_elem(Kc, dtype, base + i);
            Vd[i] = load_elem(Vc, dtype, base + i);
        }
        decode_row_f64(qd, Kd, Vd, n, D, (size_t)D, o, sc);
        free(qd);
        free(Kd);
        free(Vd);
        free(sc);
    }
    return bad;
}

/* Rolling cache [B, H_kv, W, D]: writes k_new/v_new of position lens[b]-1 into slot
 * (lens[b]-1) mod W.  Returns the number of rows with lens[b] < 1 (skipped). */
int oracle_rolling_append(void* Kr, void* Vr, const void* k_new, const void* v_new,
                          const int32_t* lens, int B, int H_kv, int W, int D, int dtype) {
    const size_t row = (size_t)D * elem_bytes_of(dtype);
    int bad = 0;
    for (int b = 0; b < B; ++b) {
        int L = lens[b];
        if (L < 1 || W < 1) {
            ++bad;
            continue;
        }
        int slot = (L - 1) % W;
        for (int h = 0; h < H_kv; ++h) {
            size_t dst = (((size_t)b * H_kv + h) * W + slot) * row;
            size_t src = ((size_t)b * H_kv + h) * row;
            memcpy((char*)Kr + dst, (const char*)k_new + src, row);
            memcpy((char*)Vr + dst, (const char*)v_new + src, row);
        }
    }
    return bad;
}

/* Decode over a rolling cache: positions [max(0, L-W), L) in position order, position p read
 * from slot p mod W.  Returns the number of rows with lens[b] < 1 (zero output). */
int oracle_rolling_decode_attn(const void* q, const void* Kr, const void* Vr, const int32_t* lens,
                               int B, int H_q, int H_kv, int W, int D, int dtype, double* out) {
    int bad = 0;
    for (int r = 0; r < B * H_q; ++r) {
        int b = r / H_q, j = r % H_q;
        int L = lens[b];
        double* o = out + (size_t)r * D;
        if (L < 1 || W < 1) {
            if (j == 0) ++bad;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            continue;
        }
        int h = kv_head_of(j, H_q, H_kv);
        int t0 = window_start(L, W), n = L - t0;
        double* qd = (double*)malloc(sizeof(double) * D);
        double* Kd = (double*)malloc(sizeof(double) * (size_t)n * D);
        double* Vd = (double*)malloc(sizeof(double) * (size_t)n * D);
        double* sc = (double*)malloc(sizeof(double) * (size_t)n);
        for (int d = 0; d < D; ++d) qd[d] = load_elem(q, dtype, (size_t)r * D + d);
        for (int i = 0; i < n; ++i) {
            size_t base = (((size_t)b * H_kv + h) * (size_t)W + (size_t)((t0 + i) % W)) * D;
            for (int d = 0; d < D; ++d) {
                Kd[(size_t)i * D + d] = load_elem(Kr, dtype, base + d);
                Vd[(size_t)i * D + d] = load_elem(Vr, dtype, base + d);
            }
        }
        decode_row_f64(qd, Kd, Vd, n, D, (size_t)D, o, sc);
        free(qd);
        free(Kd);
        free(Vd);
        free(sc);
    }
    return bad;
}

/* ---------------------------------------------------------------------------------------
 * One attention layer, two ways ([KVG] "两条数学等价的 decode 路径"; [W1D4] §1.3).
 * x: [B, T, hidden]; W_Q [hidden, H_q*D], W_K / W_V [hidden, H_kv*D], W_O [H_q*D, hidden],
 * all double, row-major.  No RoPE, no norm: the pages' single-layer teaching setting.
 * ------------------------------------------------------------------------------------- */

/* y[T, n] = x[T, k] @ W[k, n] */
static void matmul(const double* x, const double* W, double* y, int T, int k, int n) {
    for (int t = 0; t < T; ++t)
        for (int c = 0; c < n; ++c) {
            double acc = 0.0;
            for (int i = 0; i < k; ++i) acc += x[(size_t)t * k + i] * W[(size_t)i * n + c];
            y[(size_t)t * n + c] = acc;
        }
}

/* Path A: dense causal attention over all T positions (the prefill of the pages): every
 * query position i sees keys 0..i (the triu(-inf) mask).  Writes out[B,T,hidden] and, when
 * Kout/Vout are non-null, the projected K/V in cache layout [B, H_kv, T, D]. */
void oracle_layer_full(const double* x, int B, int T, int hidden, int H_q, int H_kv, int D,
                       const double* WQ, const double* WK, const double* WV, const double* WO,
                       double* out, double* Kout, double* Vout) {
    const int nq = H_q * D, nkv = H_kv * D;
    double* Q = (double*)malloc(sizeof(double) * (size_t)T * nq);
    double* K = (double*)malloc(sizeof(double) * (size_t)T * nkv);
    double* V = (double*)malloc(sizeof(double) * (size_t)T * nkv);
    double* ctx = (double*)malloc(sizeof(double) * (size_t)T * nq);
    double* s = (double*)malloc(sizeof(double) * (size_t)T);
    const double scale = 1.0 / sqrt((double)D);
    for (int b = 0; b < B; ++b) {
        const double* xb = x + (size_t)b * T * hidden;
        matmul(xb, WQ, Q, T, hidden, nq);
        matmul(xb, WK, K, T, hidden, nkv);
        matmul(xb, WV, V, T, hidden, nkv);
        for (int j = 0; j < H_q; ++j) {
            int h = j / (H_q / H_kv);
            for (int i = 0; i < T; ++i) {
                /* full score row with the causal mask: positions > i get -inf */
                for (int t = 0; t < T; ++t) {
                    if (t > i) {
                        s[t] = -INFINITY;
                        continue;
                    }
                    double acc = 0.0;
                    for (int d = 0; d < D; ++d)
                        acc += Q[(size_t)i * nq + j * D + d] * K[(size_t)t * nkv + h * D + d];
                    s[t] = acc * scale;
                }
                double m = -INFINITY;
                for (int t = 0; t < T; ++t)
                    if (s[t] > m) m = s[t];
                double Z = 0.0;
                for (int t = 0; t < T; ++t) {
                    s[t] = exp(s[t] - m); /* exp(-inf) = 0 for masked positions */
                    Z += s[t];
                }
                for (int d = 0; d < D; ++d) {
                    double acc = 0.0;
                    for (int t = 0; t < T; ++t) acc += s[t] * V[(size_t)t * nkv + h * D + d];
                    ctx[(size_t)i * nq + j * D + d] = acc / Z;
                }
            }
        }
        matmul(ctx, WO, out + (size_t)b * T * hidden, T, nq, hidden);
        if (Kout && Vout)
            for (int h = 0; h < H_kv; ++h)
                for (int t = 0; t < T; ++t)
                    for (int d = 0; d < D; ++d) {
                        size_t c = (((size_t)b * H_kv + h) * T + t) * D + d;
                        Kout[c] = K[(size_t)t * nkv + h * D + d];
                        Vout[c] = V[(size_t)t * nkv + h * D + d];
                    }
    }
    free(Q);
    free(K);
    free(V);
    free(ctx);
    free(s);
}

/* Path B: prefill the first T_p positions once (path A on the prompt, keeping its K/V in a
 * preallocated cache of T_total slots), then for each later position project only that
 * token, write its k/v at the next slot, and attend with the decode routine over all slots
 * written so far.  out[B, T_total - T_p, hidden] holds the decode outputs; Kc/Vc
 * [B, H_kv, T_total, D] hold the final cache. */
void oracle_layer_incremental(const double* x, int B, int T_p, int T_total, int hidden, int H_q,
                              int H_kv, int D, const double* WQ, const double* WK,
                              const double* WV, const double* WO, double* out, double* Kc,
                              double* Vc) {
    const int nq = H_q * D, nkv = H_kv * D;
    double* pre_out = (double*)malloc(sizeof(double) * (size_t)T_p * hidden);
    double* Kp = (double*)malloc(sizeof(double) * (size_t)H_kv * T_p * D);
    double* Vp = (double*)malloc(sizeof(double) * (size_t)H_kv * T_p * D);
    double* q = (double*)malloc(sizeof(double) * nq);
    double* k = (double*)malloc(sizeof(double) * nkv);
    double* v = (double*)malloc(sizeof(double) * nkv);
    double* ctx = (double*)malloc(sizeof(double) * nq);
    double* s = (double*)malloc(sizeof(double) * (size_t)T_total);
    for (int b = 0; b < B; ++b) {
        const double* xb = x + (size_t)b * T_total * hidden;
        double* Kb = Kc + (size_t)b * H_kv * T_total * D;
        double* Vb = Vc + (size_t)b * H_kv * T_total * D;
        memset(Kb, 0, sizeof(double) * (size_t)H_kv * T_total * D);
        memset(Vb, 0, sizeof(double) * (size_t)H_kv * T_total * D);
        oracle_layer_full(xb, 1, T_p, hidden, H_q, H_kv, D, WQ, WK, WV, WO, pre_out, Kp, Vp);
        for (int h = 0; h < H_kv; ++h)
            for (int t = 0; t < T_p; ++t)
                for (int d = 0; d < D; ++d) {
                    Kb[((size_t)h * T_total + t) * D + d] = Kp[((size_t)h * T_p + t) * D + d];
                    Vb[((size_t)h * T_total + t) * D + d] = Vp[((size_t)h * T_p + t) * D + d];
                }
        for (int pos = T_p; pos < T_total; ++pos) {
            const double* xt = xb + (size_t)pos * hidden;
            matmul(xt, WQ, q, 1, hidden, nq);
            matmul(xt, WK, k, 1, hidden, nkv);
            matmul(xt, WV, v, 1, hidden, nkv);
            for (int h = 0; h < H_kv; ++h)
                for (int d = 0; d < D; ++d) {
                    Kb[((size_t)h * T_total + pos) * D + d] = k[h * D + d];
                    Vb[((size_t)h * T_total + pos) * D + d] = v[h * D + d];
                }
            const int L = pos + 1;
            for (int j = 0; j < H_q; ++j) {
                int h = kv_head_of(j, H_q, H_kv);
                decode_row_f64(q + j * D, Kb + (size_t)h * T_total * D,
                               Vb + (size_t)h * T_total * D, L, D, (size_t)D, ctx + j * D, s);
            }
            matmul(ctx, WO, out + ((size_t)b * (T_total - T_p) + (pos - T_p)) * hidden, 1, nq,
                   hidden);
        }
    }
    free(pre_out);
    free(Kp);
    free(Vp);
    free(q);
    free(k);
    free(v);
    free(ctx);
    free(s);
}
