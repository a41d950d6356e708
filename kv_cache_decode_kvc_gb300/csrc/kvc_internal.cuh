// kvc_internal.cuh -- device helpers and launch plumbing shared by the CUDA translation units
// of libkvc (never by the CPU oracle).
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the encoder is fetched at run time)
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace kvc {

constexpr uint32_t DEV_BAD_LENS = 1u;      // mirrors KVC_DEV_BAD_LENS
constexpr uint32_t DEV_WAIT_TIMEOUT = 2u;  // mirrors KVC_DEV_WAIT_TIMEOUT
constexpr uint32_t DEV_BAD_BLOCK = 4u;     // mirrors KVC_DEV_BAD_BLOCK
constexpr int MAX_B = 1024;
// An in-kernel wait that has not completed after this long gives up, flags
// DEV_WAIT_TIMEOUT and lets the kernel run to its end (no hang, output marked invalid).
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

// ------------------------------------------------------------------ split-T partition
// The B*H_kv (sequence b, KV head h) streams are laid end to end, stream u = b*H_kv + h
// holding L_b tokens; W = H_kv * sum_b L_b.  Each stream is cut into units of g tokens (the
// stream's last unit may be partial): n_b = ceil(L_b / g) units, U = H_kv * sum_b n_b in all.
// CTA i of P owns units [cta_begin(i), cta_begin(i+1)), so every CTA holds floor(U / P) or
// ceil(U / P) units and every cut falls on a unit boundary of its stream.  With g = GRAIN = 128
// (one tcgen05 tile) a tile never straddles two CTAs and the split adds no partial tiles (a
// CTA's tile count is its unit count); paged blocks of 16..128 tokens divide a unit, a 256-token
// block may be cut at its 128-token boundary.  g = 1 is the plain token split (every CTA holds
// W / P tokens; a paged cache takes g = its block size), used where groups of 16+ query heads
// merge their split streams inside the kernel: measured faster there (MQA, B = 64 streams of
// 4097 tokens: 38.2 against 42.3 us per layer), the merges of their large partial states falling
// better behind the streaming of other CTAs; with the separate combine kernel (one long stream)
// the tile-aligned split is the faster one (29.1 against 31.0 us).
// prefix[b] = sum_{b' < b} L_b' and uprefix[b] = sum_{b' < b} n_b' (B + 1 entries each,
// 32-bit: creation keeps B * T_max below 2^31).  U and P <= 2^12 keep products below 2^63.
constexpr int GRAIN = 128;
__host__ __device__ inline int64_t units_of(int64_t L, int g) {
    return (L + g - 1) / g;
}
// With g = GRAIN each stream is charged one more unit for its start (stream_cost): a segment
// start costs its CTA a q switch, a segment epilogue and the stream's partial last tile, measured
// at about 1.4 units' time on the 8B GQA layers (CTAs holding three segments streamed 1.8 %
// longer than two-segment ones with equal units).  The extra unit sits before the stream's first
// real unit; a cut inside it falls on the stream's start.  Stream u then costs n_u + 1 units, U
// counts them, and a CTA holding only such a unit holds no tokens (its range is empty).
__host__ __device__ inline int stream_cost(int g) {
    return g == GRAIN ? 1 : 0;
}
// Partition units of a stream of L valid tokens (none for an empty stream).
__host__ __device__ inline int64_t stream_units(int64_t L, int g) {
    return L > 0 ? units_of(L, g) + stream_cost(g) : 0;
}
// Partition unit for a query group of G heads, the merge mode (0: in the kernel, 1: combine
// kernel) and the block size of a paged cache (1: contiguous).
__host__ __device__ inline int partition_grain(int G, int combine_mode, int bs) {
    if (G >= 16 && combine_mode == 0) return bs > 1 ? bs : 1;
    return GRAIN;
}
__host__ __device__ inline int64_t cta_begin(int64_t i, int64_t U, int64_t P) {
    return (i * U) / P;
}
// CTA owning unit x: the largest i with cta_begin(i) <= x.
__host__ __device__ inline int64_t cta_of(int64_t x, int64_t U, int64_t P) {
    return ((x + 1) * P - 1) / U;
}
// Token position of CTA i's first unit (i = P: the end, W).
__host__ __device__ inline int64_t cta_cut(int64_t i, const int32_t* prefix, const int32_t* uprefix,
                                           int B, int H_kv, int64_t U, int64_t P, int g) {
    if (i >= P) return (int64_t)H_kv * prefix[B];
    const int64_t x = cta_begin(i, U, P);
    int lo = 0, hi = B - 1;  // largest b with H_kv * uprefix[b] <= x (a sequence with units)
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)H_kv * uprefix[mid] <= x) lo = mid; else hi = mid - 1;
    }
    const int64_t nb = uprefix[lo + 1] - uprefix[lo];  // one stream's units
    const int64_t r = x - (int64_t)H_kv * uprefix[lo];
    const int64_t h = r / nb, j = r - h * nb, c = stream_cost(g);
    return (int64_t)H_kv * prefix[lo] + h * (int64_t)(prefix[lo + 1] - prefix[lo]) + (j > c ? j - c : 0) * g;
}
// CTAs actually used: at most P, at least min_tokens positions each, at least one unit each
// (with stream costs a CTA may still hold no tokens).
__host__ __device__ inline int64_t plan_ctas(int64_t W, int64_t U, int64_t P, int min_tokens) {
    int64_t want = (W + min_tokens - 1) / min_tokens;
    if (U < want) want = U;
    return want < P ? want : P;
}

// ------------------------------------------------------------------ launch parameters
struct DecodeParams {
    const void* K;        // layer base, [B, H_kv, T_max, D]
    const void* V;
    const void* q;        // [B, H_q, D]
    void* out;            // [B, H_q, D]
    const void* k_new;    // [B, H_kv, D] for the fused append, else nullptr
    const void* v_new;
    const int32_t* lens;  // [B], valid length after this step's append
    float* part_o;        // [slots][G][D] unnormalised partial outputs of split streams
    float* part_ml;       // [slots][G][2] (running max in log2 units, denominator)
    int* counters;        // [B*H_kv] arrivals per split stream (all zero between calls)
    uint32_t* err;        // device error word
    int B, H_kv, T_max;
    int P;                // CTAs of the partition (grid size)
    int min_tokens;       // fewer CTAs when W / P would drop below this (1 = never)
    int grain;            // partition unit in tokens (partition_grain of the query group)
    int combine_mode;     // 0: the last CTA of a split stream merges it; 1: combine kernel
    float qscale;         // log2(e) / sqrt(D), folded into q
    int overlap;          // 1: lens and history rows may be read before the preceding grid ends
    // paged cache (table == nullptr: contiguous [B, H_kv, T_max, D] layer)
    const int32_t* table; // [B, max_blocks] physical block of each logical block
    int bs;               // tokens per block (1 for a contiguous cache)
    int max_blocks;
    int num_blocks;       // K / V are pools [num_blocks, H_kv, bs, D]; T_max = max_blocks * bs
    int box_rows;         // tcgen05 path: rows per tensor-copy box of a paged tile (min(bs, 128))
    int rolling;          // 1: rolling cache, T_max = window slots, position p in slot p mod T_max
    int m2p;              // tcgen05, paged pool: MMA2 issued by the producer warp (else the MMA warp)
    int T_q;              // new tokens per sequence (>= 1); the group's G query rows are
                          // [head][token], token i seeing positions up to lens[b] - T_q + i
    const float* Ksc;     // int8 cache: K / V are codes [B, H_kv, T_max, D] and these the row
    const float* Vsc;     // scales [B, H_kv, T_max] (value = code * scale); else nullptr
};

struct CopyParams {
    void* Kc;             // layer base of the cache
    void* Vc;
    const void* K;        // source: [B, H_kv, T_in, D] (prefill) or [B, H_kv, D] (append)
    const void* V;
    const int32_t* lens;
    uint32_t* err;
    int B, H_kv, T_max, T_in;
    int row_bytes;        // D * element bytes (a multiple of 16)
    const int32_t* table; // paged cache: [B, max_blocks] block table, else nullptr
    int bs, max_blocks, num_blocks;
    int rolling;          // rolling cache: position p in slot p mod T_max (lens may exceed T_max)
    float* Ksc;           // int8 / fp8 cache: row scales of K / V; the rows are quantized on write
    float* Vsc;
    int fp8;              // 1: the codes are E4M3 (fp8 cache), 0: int8
};

// One launcher per (dtype, D) translation unit; G selects the instantiation.  Each returns
// a cudaError_t (0 = launched) and writes the kernel's dynamic shared memory to *smem_out.
#define KVC_DECLARE_LAUNCHER(NAME) \
    int NAME(int G, const DecodeParams& p, cudaStream_t s, int* smem_out);
KVC_DECLARE_LAUNCHER(launch_decode_bf16_d64)
KVC_DECLARE_LAUNCHER(launch_decode_bf16_d128)
KVC_DECLARE_LAUNCHER(launch_decode_bf16_d256)
KVC_DECLARE_LAUNCHER(launch_decode_f32_d4)
KVC_DECLARE_LAUNCHER(launch_decode_f32_d64)
KVC_DECLARE_LAUNCHER(launch_decode_f32_d128)
KVC_DECLARE_LAUNCHER(launch_decode_f32_d256)
// Tensor-core decode (bf16 cache), one launcher per head dimension; tmK / tmV are the layer's
// 2-D tensor maps (rows = B*H_kv*T_max, columns = D; boxes of 64 columns x 32 rows, 128-byte
// swizzle), built by make_kv_tensor_map.
int launch_decode_tc_d64(int G, const DecodeParams& p, const CUtensorMap& tmK,
                         const CUtensorMap& tmV, cudaStream_t s, int* smem_out);
int launch_decode_tc_d128(int G, const DecodeParams& p, const CUtensorMap& tmK,
                          const CUtensorMap& tmV, cudaStream_t s, int* smem_out);
int launch_decode_tc_d256(int G, const DecodeParams& p, const CUtensorMap& tmK,
                          const CUtensorMap& tmV, cudaStream_t s, int* smem_out);
// tcgen05 decode (bf16 cache, D = 128): maps[0..3] = K and V with TC_BOX_ROWS-row boxes, then
// K and V with TC_FULL_ROWS-row boxes (whole 128-token tiles).
int launch_decode_tc5_d128(int G, const DecodeParams& p, const CUtensorMap* maps, cudaStream_t s,
                           int* smem_out);
// the same kernel for a paged pool (p.table set; maps with min(bs, 128)-row boxes) and for a
// rolling cache (p.rolling set)
int launch_decode_tc5p_d128(int G, const DecodeParams& p, const CUtensorMap* maps, cudaStream_t s,
                            int* smem_out);
int launch_decode_tc5r_d128(int G, const DecodeParams& p, const CUtensorMap* maps, cudaStream_t s,
                            int* smem_out);
// ... and for an int8 cache (p.Ksc / p.Vsc set; maps over the int8 rows, no swizzle)
int launch_decode_tc5q_d128(int G, const DecodeParams& p, const CUtensorMap* maps, cudaStream_t s,
                            int* smem_out);
// ... and for an fp8 cache (E4M3 codes and row scales; maps over the code rows, 128-byte swizzle)
int launch_decode_tc5f_d128(int G, const DecodeParams& p, const CUtensorMap* maps, cudaStream_t s,
                            int* smem_out);
constexpr int TC_BOX_ROWS = 32;
constexpr int TC_FULL_ROWS = 128;
// Tensor maps of a bf16 cache (host; encoded by the driver, no allocation).  2-D: columns D,
// rows B*H_kv*T_max, boxes of 64 columns x box_rows, 128-byte swizzle.  3-D (D = 128): a whole
// box_rows-row tile of both 64-column blocks in one copy.  False if the encoder is unavailable
// or base is not 16-byte aligned.
bool make_kv_tensor_map(CUtensorMap* map, void* base, uint64_t rows, int D, int box_rows);
bool make_kv3_tensor_map(CUtensorMap* map, void* base, uint64_t rows, int box_rows);
int launch_combine(int dtype, int D, int G, const DecodeParams& p, cudaStream_t s);

// cudaFuncSetAttribute applies to the current device only: a launcher sets a kernel's
// attributes once per device (devices 0..63; beyond that, on every launch).  Setting them twice
// from racing threads is harmless.
struct PerDeviceOnce {
    std::atomic<uint64_t> done{0};
    template <class F>
    int run(F&& set) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return (int)cudaErrorInvalidDevice;
        if (dev < 0 || dev >= 64) return set();
        const uint64_t bit = 1ull << dev;
        if (done.load(std::memory_order_acquire) & bit) return 0;
        const int e = set();
        if (e == 0) done.fetch_or(bit, std::memory_order_acq_rel);
        return e;
    }
};
int launch_append(const CopyParams& p, cudaStream_t s);
int launch_prefill(const CopyParams& p, cudaStream_t s);

// ------------------------------------------------------------------ device primitives
#ifdef __CUDACC__
// Attended length of a sequence with post-append length L: 0 if invalid (L < T_q, i.e. fewer
// positions than the step's new tokens, or L > T_max for a cache that does not roll),
// min(L, T_max) for a rolling cache, else L.
__host__ __device__ __forceinline__ int eff_len(int L, int T_max, int rolling, int T_q = 1) {
    if (L < (T_q > 1 ? T_q : 1) || (!rolling && L > T_max)) return 0;
    return rolling && L > T_max ? T_max : L;
}

// Slot of a sequence's new row in the fused step (the row an append writes): L_eff - 1, or for a
// rolling cache (lens[b] - 1) mod T_max.
__device__ __forceinline__ int new_row_slot(const DecodeParams& p, int b, int L_eff) {
    return p.rolling ? (__ldg(p.lens + b) - 1) % p.T_max : L_eff - 1;
}

// Cache row of token t of stream (b, h): contiguous [B, H_kv, T_max] rows, or through the block
// table of a paged pool [num_blocks, H_kv, bs].  A table entry outside [0, num_blocks) flags
// DEV_BAD_BLOCK and gives -1: readers then load row 0 instead (in bounds; that sequence's
// output is unspecified), writers skip the row.
__device__ __forceinline__ int64_t cache_row(const int32_t* table, int bs, int max_blocks,
                                             int num_blocks, int H_kv, int T_max, int b, int h, int t,
                                             uint32_t* err) {
    if (table == nullptr) return ((int64_t)b * H_kv + h) * T_max + t;
    const int e = __ldg(table + (size_t)b * max_blocks + t / bs);
    if ((unsigned)e >= (unsigned)num_blocks) {
        atomicOr(err, DEV_BAD_BLOCK);
        return -1;
    }
    return ((int64_t)e * H_kv + h) * bs + (t % bs);
}
__device__ __forceinline__ int64_t cache_row_rd(const int32_t* table, int bs, int max_blocks,
                                                int num_blocks, int H_kv, int T_max, int b, int h,
                                                int t, uint32_t* err) {
    const int64_t r = cache_row(table, bs, max_blocks, num_blocks, H_kv, T_max, b, h, t, err);
    return r < 0 ? 0 : r;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}


__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity to complete, for at most limit_ns (the kernels use
// WAIT_LIMIT_NS).  On timeout (or once another thread of the CTA has timed out) it returns
// false, having set the CTA's abort flag and the device error word; callers then skip work but
// keep the protocol.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* err, uint64_t limit_ns = WAIT_LIMIT_NS) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (*abort_flag) return false;
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            atomicOr(err, DEV_WAIT_TIMEOUT);
            return false;
        }
    }
}

// One bulk (TMA engine) copy global -> shared, completing `bytes` on the mbarrier.
// dst, src 16-byte aligned; bytes a multiple of 16.  The L2 policy marks the stream as
// evict-first: every KV byte is read once per step.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
        "%2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// 2^x with the SFU's approximate exp2 (relative error about 2^-22; results below the
// smallest normal flush to zero, which the softmax weights tolerate: they are < 2^-126).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// bf16 pair (one 32-bit word) -> two floats, exact.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <typename T>
struct Elem;
template <>
struct Elem<__nv_bfloat16> {
    static constexpr int BYTES = 2;
    static constexpr int VEC = 8;  // elements per 16-byte vector
    __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[8]) {
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
        f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
        f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    }
    __device__ __forceinline__ static void unpack2(const uint4& v, float2 (&f)[4]) {
        f[0] = make_float2(bf16_lo(v.x), bf16_hi(v.x));
        f[1] = make_float2(bf16_lo(v.y), bf16_hi(v.y));
        f[2] = make_float2(bf16_lo(v.z), bf16_hi(v.z));
        f[3] = make_float2(bf16_lo(v.w), bf16_hi(v.w));
    }
    __device__ __forceinline__ static void store(void* base, size_t idx, float x) {
        reinterpret_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(x);
    }
};
template <>
struct Elem<float> {
    static constexpr int BYTES = 4;
    static constexpr int VEC = 4;
    __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[4]) {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static void unpack2(const uint4& v, float2 (&f)[2]) {
        f[0] = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
        f[1] = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
    }
    __device__ __forceinline__ static void store(void* base, size_t idx, float x) {
        reinterpret_cast<float*>(base)[idx] = x;
    }
};
// Symmetric int8 quantization of one bf16 row of D = 128 values, as the cache stores it:
// scale = max |x| / 127, code = round-half-even(x / scale) clamped to [-127, 127] (IEEE fp32
// division; a zero row gets scale 0 and codes 0).
__device__ __forceinline__ float q8_row_scale(const __nv_bfloat16* x) {
    float amax = 0.f;
    const uint4* v = reinterpret_cast<const uint4*>(x);
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
        const uint4 w = __ldg(v + i);
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(u[j])), fabsf(bf16_hi(u[j]))));
    }
    return __fdiv_rn(amax, 127.f);
}
// Warp-cooperative: lane l quantizes elements 4l .. 4l+3 of the row and stores their codes;
// lane 0 stores the scale.
__device__ __forceinline__ void q8_store_row(const __nv_bfloat16* x, int8_t* codes, float* scale,
                                             int lane) {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(x) + lane);
    const float f[4] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y)};
    float amax = fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3])));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    const float s = __fdiv_rn(amax, 127.f);
    uint32_t packed = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        int c = s > 0.f ? __float2int_rn(__fdiv_rn(f[j], s)) : 0;
        c = c > 127 ? 127 : (c < -127 ? -127 : c);
        packed |= (uint32_t)(c & 0xFF) << (8 * j);
    }
    reinterpret_cast<uint32_t*>(codes)[lane] = packed;
    if (lane == 0) *scale = s;
}

// ---- fp8 (E4M3) cache: one fp32 scale per row, scale = max |x| / 448, code = E4M3 of x / scale
// (IEEE fp32 division; round to nearest even, saturating at +-448; a zero row gets scale 0).
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {  // a in the low byte
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float2 e4m3x2_value(uint32_t c2) {    // the two codes of the low 16 bits
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(c2 & 0xFFFFu), __NV_E4M3);
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
}
__device__ __forceinline__ float f8_row_scale(const __nv_bfloat16* x) {
    float amax = 0.f;
    const uint4* v = reinterpret_cast<const uint4*>(x);
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
        const uint4 w = __ldg(v + i);
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(u[j])), fabsf(bf16_hi(u[j]))));
    }
    return __fdiv_rn(amax, 448.f);
}
// The K and V row scales of a fused step's new row, computed from k_new / v_new as its append
// computes them (fp8 != 0: E4M3 scales, else int8).  Out of line: it runs once per stream, and
// inlined at each call site of the tile loops it would crowd their instruction cache.
static __device__ __noinline__ float2 new_row_scales(const __nv_bfloat16* kr, const __nv_bfloat16* vr, int fp8);
static __device__ __noinline__ float2 new_row_scales(const __nv_bfloat16* kr, const __nv_bfloat16* vr, int fp8) {
    return fp8 ? make_float2(f8_row_scale(kr), f8_row_scale(vr)) : make_float2(q8_row_scale(kr), q8_row_scale(vr));
}
// Warp-cooperative: lane l encodes elements 4l .. 4l+3 of a D = 128 row; lane 0 stores the scale.
__device__ __forceinline__ void f8_store_row(const __nv_bfloat16* x, uint8_t* codes, float* scale, int lane) {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(x) + lane);
    const float f[4] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y)};
    float amax = fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3])));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    const float s = __fdiv_rn(amax, 448.f);
    uint32_t packed = 0;
    if (s > 0.f)
        packed = e4m3x2(__fdiv_rn(f[0], s), __fdiv_rn(f[1], s)) |
                 (e4m3x2(__fdiv_rn(f[2], s), __fdiv_rn(f[3], s)) << 16);
    reinterpret_cast<uint32_t*>(codes)[lane] = packed;
    if (lane == 0) *scale = s;
}
// q of one head as three E4M3 terms: q = 2^e (t0 + t1 + t2).  e puts the head's largest |q| in
// [128, 256) (the exponent of amax minus 7, clamped so 2^-e stays a normal fp32); the scaled
// value v = q 2^-e is exact, t0 is its nearest code and t1, t2 those of the (exact) residues, so a
// bf16 value within the codes' normal range is represented exactly.
__device__ __forceinline__ int f8_head_exp(float amax) {
    const int E = (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127;
    const int e = amax > 0.f ? E - 7 : 0;
    return e < -100 ? -100 : (e > 100 ? 100 : e);
}
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }
// Eight scaled values -> their three E4M3 terms, 8 bytes each (value i in byte i).
__device__ __forceinline__ void e4m3_split3(const float (&v)[8], uint2& t0, uint2& t1, uint2& t2) {
    uint32_t c[3][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float a = v[2 * i], b = v[2 * i + 1];
#pragma unroll
        for (int t = 0; t < 3; ++t) {
            c[t][i] = e4m3x2(a, b);
            const float2 r = e4m3x2_value(c[t][i]);
            a -= r.x;
            b -= r.y;
        }
    }
    t0 = make_uint2(c[0][0] | (c[0][1] << 16), c[0][2] | (c[0][3] << 16));
    t1 = make_uint2(c[1][0] | (c[1][1] << 16), c[1][2] | (c[1][3] << 16));
    t2 = make_uint2(c[2][0] | (c[2][1] << 16), c[2][2] | (c[2][3] << 16));
}

#endif  // __CUDACC__

}  // namespace kvc
