/*
 * kvc.h -- C ABI of the GB300 (sm_103a) single-token KV-cache decode step.
 *
 * What it computes (sources are web pages on the KV cache, cited by title and section):
 *   - a per-layer cache K, V in layout [B, H_kv, T_max, D], preallocated once and written
 *     in place ("第 1 周 · Day 4：KV Cache 与 MQA / GQA" §3.1; "KV 缓存" glossary page,
 *     "从教学代码到生产实现还差什么" item 1);
 *   - append: the new token's k_t, v_t go to slot lens[b]-1 of every KV head
 *     ("KV 缓存", "两条数学等价的 decode 路径", path B);
 *   - decode attention: for every query head j of sequence b,
 *         o[b,j,:] = softmax_t( q[b,j,:] . K[b,h,t,:] / sqrt(D) ) V[b,h,t,:],  t in [0, lens[b]),
 *     with h = floor(j / (H_q/H_kv))  ("11.7 KV Cache：形状、显存与带宽" §2.2 single-step
 *     decode; "第 1 周 · Day 4" §3.4 for the grouped-query head map);
 *   - capacity: bytes = 2 * L * H_kv * D * B * T * s  ("第 1 周 · Day 4" §1.4; "KV 缓存",
 *     容量公式, whose ragged form replaces B*T by sum_i T_i).
 *
 * Conventions used by every call:
 *   - lens (int32 [B], DEVICE memory) is the valid length of each sequence AFTER the call's
 *     own write.  One decode step is: lens += 1; kvc_append(...lens); kvc_decode_attn(...lens),
 *     or the fused kvc_decode_step(...lens).  The new token attends to itself.
 *   - All tensor pointers are DEVICE pointers, dense row-major, in the cache dtype
 *     (bf16 bit patterns or fp32), 16-byte aligned.  The caller owns them.
 *   - stream is a cudaStream_t passed as void* (NULL = legacy default stream).  Every call
 *     that launches work is asynchronous on that stream and never synchronises, except
 *     kvc_last_error and kvc_destroy.  All calls on one handle must come from one host thread
 *     at a time.
 *   - Errors: a problem visible on the host (null pointer, bad layer index, unsupported
 *     shape, CUDA launch failure) returns a nonzero status and launches nothing.  lens lives
 *     on the device, so an out-of-range lens[b] is found by the kernels: they skip that row
 *     (append writes nothing, attention writes a zero output row), never read or write out of
 *     bounds, and set the handle's device error word, which kvc_last_error reports.
 */
#ifndef KVC_H
#define KVC_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct kvc_cache* kvc_t;

/* Cache element types. */
#define KVC_BF16 0
#define KVC_F32 1

/* Status codes. */
#define KVC_OK 0
#define KVC_EINVAL 1       /* bad argument (null pointer, negative size, layer out of range) */
#define KVC_ENOMEM 2       /* device allocation failed or would exceed free memory */
#define KVC_ECUDA 3        /* a CUDA runtime call or kernel launch failed */
#define KVC_ERANGE 4       /* a size is out of the supported range (T_in > T_max, B > 1024) */
#define KVC_EDEVICE 5      /* a kernel found bad input on the device (see kvc_last_error) */
#define KVC_EUNSUPPORTED 6 /* shape or device not supported (D, group size, not sm_103) */

/* Bits of the device error word returned through kvc_last_error's `detail`. */
#define KVC_DEV_BAD_LENS 1u     /* some lens[b] < 1 (or < 0 for prefill) or > T_max */
#define KVC_DEV_WAIT_TIMEOUT 2u /* an in-kernel wait gave up (internal error; output invalid) */
#define KVC_DEV_BAD_BLOCK 4u    /* a paged call met a block-table entry outside [0, num_blocks) */

/* Create a cache of `layers` layers, each holding K and V of shape [B, H_kv, T_max, D].
 * Supported: dtype KVC_BF16 with D in {64, 128, 256}; KVC_F32 with D in {4, 64, 128, 256};
 * H_q % H_kv == 0 with H_q/H_kv in {1, 2, 4, 8, 16, 32}; 1 <= B <= 1024; T_max >= 1.
 * The cache (kvc_bytes(h) bytes, one device allocation) is zero-filled, like a preallocated
 * torch.zeros cache.  Workspace for split sequences and a device error word are allocated
 * here too, so no later call allocates.  Uses the current CUDA device.
 * Returns KVC_OK and *out, or an error status and *out = NULL. */
int kvc_create(kvc_t* out, int layers, int B, int H_q, int H_kv, int D, int T_max, int dtype);

/* Synchronise the device, free everything the handle owns.  NULL is a no-op. */
int kvc_destroy(kvc_t h);

/* Prefill write: copy K, V ([B, H_kv, T_in, D], device) slots [0, lens[b]) into the cache of
 * `layer`.  Requires 1 <= T_in <= T_max; a lens[b] outside [0, T_in] skips row b and sets
 * KVC_DEV_BAD_LENS.  Slots >= lens[b] are not touched. */
int kvc_prefill_write(kvc_t h, int layer, const void* K, const void* V, int T_in,
                      const int32_t* lens, void* stream);

/* Append: write k_new[b,h,:], v_new[b,h,:] ([B, H_kv, D], device) into slot lens[b]-1 of every
 * KV head h of `layer`.  Every other slot keeps its exact bytes.  A lens[b] outside
 * [1, T_max] skips row b and sets KVC_DEV_BAD_LENS. */
int kvc_append(kvc_t h, int layer, const void* k_new, const void* v_new, const int32_t* lens,
               void* stream);

/* Decode attention over the cache of `layer`: q, out are [B, H_q, D] (device, cache dtype);
 * out[b,j,:] as in the header comment, fp32 softmax and accumulation, rounded to the cache
 * dtype (nearest-even for bf16).  Reads slots [0, lens[b]).  A lens[b] outside [1, T_max]
 * gives a zero row and sets KVC_DEV_BAD_LENS.  Long sequences are split across CTAs
 * (split-T) and their partial softmax states merged on the device. */
int kvc_decode_attn(kvc_t h, int layer, const void* q, void* out, const int32_t* lens,
                    void* stream);

/* Fused decode step = kvc_append followed by kvc_decode_attn, in one launch: the new token's
 * k/v are read from k_new/v_new for the attention and written to slot lens[b]-1 of the cache.
 * Same results as the two calls in sequence. */
int kvc_decode_step(kvc_t h, int layer, const void* q, const void* k_new, const void* v_new,
                    void* out, const int32_t* lens, void* stream);

/* Allocated payload of the handle: 2 * layers * H_kv * D * B * T_max * elem_bytes. */
uint64_t kvc_bytes(kvc_t h);

/* The closed form 2 * L * H_kv * D * (B * T) * elem_bytes (no allocation, host only).
 * Returns 0 if any argument is negative or the product overflows 64 bits. */
uint64_t kvc_bytes_formula(int64_t L, int64_t B, int64_t H_kv, int64_t D, int64_t T,
                           int64_t elem_bytes);

/* Ragged payload 2 * layers * H_kv * D * elem_bytes * sum_b lens_host[b] (lens in HOST memory,
 * B entries). */
uint64_t kvc_payload_bytes(kvc_t h, const int32_t* lens_host);

/* Device pointers of layer `layer`'s K and V caches ([B, H_kv, T_max, D], owned by h). */
int kvc_layer_ptrs(kvc_t h, int layer, void** K, void** V);

/* Synchronise `stream`, read and clear the device error word.  Returns KVC_OK if it was zero,
 * else KVC_EDEVICE with the KVC_DEV_* bits in *detail (detail may be NULL). */
int kvc_last_error(kvc_t h, void* stream, uint32_t* detail);

/* Number of CTAs the attention kernel splits the work over (0 restores the default: one per
 * SM, or four fifths of the SMs when the combine kernel merges the streams, see
 * kvc_set_combine_mode).  1 <= ctas <= 4 * SMs.  Changes only the split, never the result beyond
 * rounding.  kvc_get_ctas returns the setting (the SM count while it is 0). */
int kvc_set_ctas(kvc_t h, int ctas);
int kvc_get_ctas(kvc_t h);

/* How streams cut across CTAs are merged: -1 automatic (default), 0 by the last CTA to finish
 * the stream (arrival counter; no CTA ever waits on another), 1 by a separate combine kernel
 * launched right after on the same stream.  Changes nothing beyond rounding. */
int kvc_set_combine_mode(kvc_t h, int mode);

/* Which units compute the two small contractions of the attention (q.K and p.V):
 *   0 automatic: tcgen05 tensor cores for bf16 caches with D = 128, CUDA cores otherwise;
 *   1 CUDA cores (fp32 arithmetic; the only path for fp32 caches);
 *   2 warp-level mma.sync tensor instructions (bf16 caches);
 *   3 tcgen05 tensor cores with tensor-memory accumulators (bf16 caches, D = 128).
 * Paths 2 and 3 need B*H_kv*T_max < 2^31 (tensor-map coordinates), else KVC_EUNSUPPORTED.
 * All paths agree within the bf16 tolerance.  kvc_get_math returns the path the next call
 * takes (1, 2 or 3). */
int kvc_set_math(kvc_t h, int mode);
int kvc_get_math(kvc_t h);

/* Launch overlap (default 0).  The tcgen05 attention kernel is launched with programmatic
 * dependent launch: its CTAs may become resident while the preceding kernel on the stream is
 * still finishing.  With 0 they read nothing before that kernel has completed.  With 1 they
 * read lens[] and start loading the history rows [0, lens[b] - 1) of each stream before it has
 * completed, and wait for it before touching anything else (q, k_new, v_new, the new row
 * lens[b] - 1, outputs, workspace).  Set 1 only when the kernel launched just before on the
 * stream writes neither lens nor those rows: e.g. a decode loop over layers where the
 * preceding kernel is another layer's kvc_decode_step or a projection writing q / k_new /
 * v_new.  Results are identical either way; only the start of each launch moves earlier.
 * Not part of the pages' method (a scheduling choice of this implementation).  Other math
 * paths ignore it.  Returns KVC_EINVAL for a value other than 0 or 1. */
int kvc_set_launch_overlap(kvc_t h, int on);
int kvc_get_launch_overlap(kvc_t h);

/* ---------------------------------------------------------------------------------------
 * Quantized cache.  The pages list int8 / fp8 caches with per-token or per-head scales as a
 * way to read fewer bytes, with the softmax accumulated in higher precision ("KV 缓存",
 * "MHA、GQA、MLA 与量化如何改变容量"; "11.7 KV Cache" §3.1 and §8).  kvc_create_quantized makes a
 * contiguous handle whose cache is symmetric int8 with one fp32 scale per (sequence, KV head,
 * token) row, for K and for V:
 *     scale = max_d |x_d| / 127,   code_d = round-half-even(x_d / scale) in [-127, 127]
 * (IEEE fp32 division; a zero row has scale 0), and the attention reads code * scale.  q, out,
 * k_new, v_new and the prefill source stay bf16 (dtype must be KVC_BF16); the ordinary calls
 * (kvc_prefill_write, kvc_append, kvc_decode_attn, kvc_decode_step) quantize on write.
 * Per layer: codes [B, H_kv, T_max, D] int8 (kvc_layer_ptrs) and scales [B, H_kv, T_max] fp32
 * (kvc_layer_scales).  Supported: D = 128, H_q / H_kv <= 8, one new token per step, the
 * tcgen05 path (math 0 or 3); else KVC_EUNSUPPORTED. */
int kvc_create_quantized(kvc_t* out, int layers, int B, int H_q, int H_kv, int D, int T_max,
                         int dtype);
int kvc_layer_scales(kvc_t h, int layer, float** Ks, float** Vs);

/* fp8 cache: as kvc_create_quantized, with E4M3 codes (the OCP 8-bit float: 1 sign, 4 exponent
 * bits with bias 7, 3 mantissa bits, subnormals m * 2^-9, no infinity, largest finite 448) and
 * one fp32 scale per (sequence, KV head, token) row for K and for V:
 *     scale = max_d |x_d| / 448,   code_d = E4M3(x_d / scale)
 * (IEEE fp32 division; round to the nearest code, ties to even, saturating at +-448; a zero row
 * has scale 0), and the attention reads value(code) * scale.  The same names as for int8 ("KV 缓存",
 * "MHA、GQA、MLA 与量化如何改变容量"; "11.7 KV Cache" §3.1 and §8 list int8 and fp8 caches).
 * The tcgen05 kernel multiplies the K codes by q directly (q split exactly into three E4M3 terms),
 * so only V is widened (to f16) on chip.  Per layer: codes [B, H_kv, T_max, D] (one byte each,
 * kvc_layer_ptrs) and scales (kvc_layer_scales).  Supported: dtype KVC_BF16, D = 128,
 * H_q / H_kv <= 8, one new token per step, math 0 or 3; else KVC_EUNSUPPORTED. */
int kvc_create_fp8(kvc_t* out, int layers, int B, int H_q, int H_kv, int D, int T_max, int dtype);

/* The handle's cache format: KVC_CACHE_PLAIN (bf16 / fp32 values), KVC_CACHE_INT8, KVC_CACHE_FP8;
 * -1 for NULL. */
#define KVC_CACHE_PLAIN 0
#define KVC_CACHE_INT8 1
#define KVC_CACHE_FP8 2
int kvc_get_cache_format(kvc_t h);

/* ---------------------------------------------------------------------------------------
 * Several new tokens per step (chunked prefill, speculative decoding).  After T_q new tokens
 * are appended to a sequence of S = lens[b] positions, new query i sits at position S - T_q + i
 * and attends to positions 0 .. S - T_q + i: the causal mask aligned to the lower right of the
 * T_q x S score matrix ("第 1 周 · Day 4" §3.3, third case).  Layouts:
 *   q, out        [B, H_q, T_q, D]   (per head, the T_q new tokens in order)
 *   k_new, v_new  [B, H_kv, T_q, D]  written to slots [S - T_q, S)
 * lens[b] < T_q or > T_max is invalid (KVC_DEV_BAD_LENS, zero output rows).  Supported when T_q
 * is a power of two with (H_q / H_kv) * T_q <= 32, on contiguous handles, math paths 0, 1, 3;
 * else KVC_EUNSUPPORTED.  T_q = 1 is kvc_append / kvc_decode_attn / kvc_decode_step. */
int kvc_append_multi(kvc_t h, int layer, const void* k_new, const void* v_new, const int32_t* lens,
                     int T_q, void* stream);
int kvc_decode_attn_multi(kvc_t h, int layer, const void* q, void* out, const int32_t* lens, int T_q,
                          void* stream);
int kvc_decode_step_multi(kvc_t h, int layer, const void* q, const void* k_new, const void* v_new,
                          void* out, const int32_t* lens, int T_q, void* stream);

/* ---------------------------------------------------------------------------------------
 * Rolling cache for sliding-window attention.  With a window of W tokens the newest query
 * attends to the W most recent positions, and the cache needs only W slots: position p lives
 * in slot p mod W, overwriting position p - W ("第 1 周 · Day 4" §2.7 and §1.6, the rolling
 * cache of a sliding-window model; "11.7 KV Cache" §8).  kvc_create_rolling makes a contiguous
 * handle [B, H_kv, W, D] per layer (T_max = W) whose calls read lens as positions, unbounded:
 *   - kvc_append / kvc_decode_step write position lens[b] - 1 into slot (lens[b] - 1) mod W;
 *   - kvc_decode_attn / kvc_decode_step attend over positions [max(0, lens[b] - W), lens[b]),
 *     i.e. slots [0, min(lens[b], W)) (softmax over a set: the slot order does not matter);
 *   - kvc_prefill_write takes T_in >= lens[b] positions and keeps the last W of them.
 * lens[b] < 1 is invalid (KVC_DEV_BAD_LENS).  Math paths 0, 1, 3 (2 is KVC_EUNSUPPORTED).
 * kvc_get_window returns W (0 for a handle that does not roll). */
int kvc_create_rolling(kvc_t* out, int layers, int B, int H_q, int H_kv, int D, int window,
                       int dtype);
int kvc_get_window(kvc_t h);

/* ---------------------------------------------------------------------------------------
 * Paged cache.  The pages describe storage cut into fixed-size blocks that are handed out on
 * demand and found through a table, with the attention arithmetic unchanged ("第 1 周 · Day 4"
 * §1.6; "KV 缓存", "先把它放回推理链路" and "成本转移、失败场景与常见误解"; "11.7 KV Cache" §8).
 * They fix no layout; this one:
 *   - per layer, K and V are pools [num_blocks, H_kv, block_size, D] owned by the handle
 *     (zero at create), block_size in {16, 32, 64, 128, 256};
 *   - block_table (int32 [B, max_blocks], DEVICE memory, owned by the caller, who also
 *     decides which blocks a sequence gets) maps logical block j of sequence b to a pool block;
 *     the same table serves every layer;
 *   - token t of sequence b, KV head h is row (block_table[b][t / block_size], h,
 *     t % block_size) of the layer's pools; a sequence holds up to T_max = max_blocks *
 *     block_size tokens (lens[b] <= T_max, else KVC_DEV_BAD_LENS as for contiguous caches).
 * Only table entries of blocks [0, ceil(lens[b] / block_size)) are read.  An entry outside
 * [0, num_blocks) sets KVC_DEV_BAD_BLOCK: writes to that row are skipped and attention reads
 * pool block 0 in its place (no out-of-bounds access; the outputs of that sequence are then
 * unspecified).  A paged handle accepts only the kvc_paged_* writes and attention calls
 * below (the contiguous ones return KVC_EINVAL, and vice versa); kvc_layer_ptrs returns the
 * pools, kvc_bytes the pools' size, kvc_get_shape T_max = max_blocks * block_size.  Math
 * paths: 0, 1, 3 (warp MMA, 2, is KVC_EUNSUPPORTED).  With launch overlap on, block-table
 * entries of history blocks are read early as well. */
int kvc_create_paged(kvc_t* out, int layers, int num_blocks, int block_size, int B, int max_blocks,
                     int H_q, int H_kv, int D, int dtype);
/* K, V: [B, H_kv, T_in, D]; writes tokens [0, lens[b]) of each sequence (lens[b] <= T_in). */
int kvc_paged_prefill_write(kvc_t h, int layer, const void* K, const void* V, int T_in,
                            const int32_t* block_table, const int32_t* lens, void* stream);
/* k_new, v_new: [B, H_kv, D]; writes token lens[b] - 1 of each sequence. */
int kvc_paged_append(kvc_t h, int layer, const void* k_new, const void* v_new,
                     const int32_t* block_table, const int32_t* lens, void* stream);
/* Decode attention over tokens [0, lens[b]) read through the table; q, out [B, H_q, D]. */
int kvc_paged_decode_attn(kvc_t h, int layer, const void* q, void* out, const int32_t* block_table,
                          const int32_t* lens, void* stream);
/* kvc_paged_append + kvc_paged_decode_attn in one launch (same results). */
int kvc_paged_decode_step(kvc_t h, int layer, const void* q, const void* k_new, const void* v_new,
                          void* out, const int32_t* block_table, const int32_t* lens, void* stream);
/* Paged geometry (any pointer may be NULL); KVC_EINVAL for a contiguous handle. */
int kvc_get_paged_shape(kvc_t h, int* num_blocks, int* block_size, int* max_blocks);

/* Shape query: writes layers, B, H_q, H_kv, D, T_max, dtype (any pointer may be NULL). */
int kvc_get_shape(kvc_t h, int* layers, int* B, int* H_q, int* H_kv, int* D, int* T_max,
                  int* dtype);

/* Split-T partition used by the attention kernels (host copy of the device arithmetic, for
 * tests).  The B*H_kv (sequence, KV head) streams are laid end to end, stream u = b*H_kv + h
 * holding lens[b] tokens, and each stream is cut into units of `grain` tokens (its last unit
 * may be partial); with U units in total, CTA i of P takes units [floor(i*U/P), floor((i+1)*U/P)).
 * So every CTA holds floor(U/P) or ceil(U/P) units and every cut falls on a unit boundary of its
 * stream.  The kernels use grain 128 (one tcgen05 tile: no tile is shared by two CTAs), except
 * that query groups of 16 or 32 heads whose split streams are merged inside the kernel
 * (combine_mode 0) use the plain token split: grain 1, or a paged cache's block size.
 * kvc_plan_grain(G, combine_mode, block_size) returns it (block_size 1 for a contiguous cache;
 * -1 for bad arguments).  kvc_plan_cta_of returns the CTA that owns unit x (0 <= x < U), -1 for
 * bad arguments. */
int kvc_plan_grain(int G, int combine_mode, int block_size);
int kvc_plan_cta_of(int64_t x, int64_t U, int P);

/* The partition the attention kernels use, on the host (for tests).  lens_host [B] holds
 * post-append lengths (invalid ones count as 0).  The kernels use
 * Pu = min(P, ceil(W / min_tokens), U) CTAs for W tokens in U units; CTA i takes stream
 * positions [cuts[i], cuts[i+1]).  Writes cuts[0..Pu] (Pu + 1 values; cuts must hold P + 1) and
 * returns Pu (0 when W = 0, -1 for bad arguments, including B * T_max >= 2^31). */
int kvc_plan_cuts(const int32_t* lens_host, int B, int H_kv, int T_max, int grain, int P,
                  int min_tokens, int64_t* cuts);
/* First and last CTA holding stream (b, h) under that partition (KVC_EINVAL if it is empty,
 * KVC_ERANGE if B * T_max >= 2^31). */
int kvc_plan_stream_ctas(const int32_t* lens_host, int B, int H_kv, int T_max, int grain, int P,
                         int min_tokens, int b, int h, int* first, int* last);

/* Decode attention for callers that cannot allocate device memory.  The pages have no
 * counterpart: this is an interface variant of kvc_decode_attn.  It runs the kernel that
 * kvc_decode_attn picks by default for the same cache (tcgen05 for a bf16 cache with D = 128,
 * the CUDA-core kernel otherwise), with the same split over one CTA per SM and the same merge
 * rule, so its results agree with kvc_decode_attn's within rounding (not bit for bit: the order
 * in which a split sequence's partial states are folded may differ from run to run).
 * Who needs it: code that must not call cudaMalloc (a plugin whose host engine owns all device
 * memory, a latency-critical loop where the allocator's device synchronisation is forbidden, a
 * runtime with a fixed memory plan) and that keeps its K/V cache in memory it owns.
 * Arguments: K, V are one layer's cache [B, H_kv, T_max, D] (device, dtype KVC_BF16 or
 * KVC_F32, the same layout and limits as kvc_create); q, out [B, H_q, D] and lens [B] as in
 * kvc_decode_attn; err is an optional device uint32 that receives the KVC_DEV_* bits (NULL:
 * not reported); stream as elsewhere.  K, V, q and out must be 16-byte aligned, lens and err
 * 4-byte aligned, else KVC_EINVAL before any launch.  err accumulates: bits are ORed in and
 * never cleared by the library, so zero it before the calls you want to check.
 * Scratch: a fixed 8 MiB __device__ array inside the library (held by every device that loads
 * it, until exit).  Shapes whose split-T scratch would exceed it return KVC_ERANGE before any
 * launch.  Nothing is allocated: no cudaMalloc, no cudaFree, no allocating library call.
 * The first call on a device looks the array's address up (cudaGetSymbolAddress) with that
 * device current, so make it before any stream capture.  All calls share the array: calls
 * that may overlap on the GPU (unordered streams) race and must not be made. */
int kvc_decode_attn_noalloc(const void* K, const void* V, int B, int H_q, int H_kv, int D,
                            int T_max, int dtype, const void* q, void* out, const int32_t* lens,
                            uint32_t* err, void* stream);

/* Self-test of the bounded in-kernel wait.  The pages have no counterpart: every attention
 * kernel waits on shared-memory barriers, and each wait gives up after a time limit (2 s),
 * sets KVC_DEV_WAIT_TIMEOUT in the device error word and lets the kernel finish instead of
 * hanging the GPU.  A correct launch never reaches that limit, so this call makes a wait reach
 * it on purpose, with no fault: one CTA of 64 threads waits on a barrier phase that nothing
 * completes, for limit_ns nanoseconds (limit_ns <= 0: the kernels' own 2 s limit; more than
 * that: KVC_ERANGE).  It ORs KVC_DEV_WAIT_TIMEOUT into *err (device uint32, 4-byte aligned)
 * and writes info[0] = threads whose wait reported completion (0 when the wait works),
 * info[1] = nanoseconds thread 0 waited (device int64[2], 8-byte aligned).  Asynchronous on
 * stream; the context stays usable afterwards. */
int kvc_selftest_wait_timeout(uint32_t* err, long long* info, long long limit_ns, void* stream);

/* Human-readable name of a status code. */
const char* kvc_status_str(int status);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H */
