// kvc_host.cu -- the C ABI of include/kvc.h: handle, allocation, argument checks, dispatch.
//
// Capacity: bytes = 2 * L * H_kv * D * (B * T) * s ("第 1 周 · Day 4：KV Cache 与 MQA / GQA"
// §1.4; "KV 缓存" glossary page, 容量公式, ragged form with sum_i T_i).  The cache is one
// preallocated, zero-filled device slab, written in place (same notes, §3.1).
#include <math.h>
#include <string.h>

#include <new>
#include <vector>

#include "../../include/kvc.h"
#include "kvc_internal.cuh"

struct kvc_cache {
    int layers, B, H_q, H_kv, D, T_max, dtype, es, G;
    int device, sms;
    int ctas;          // 0 = one per SM
    int combine_mode;  // -1 = automatic
    int max_ctas;
    char* slab;        // layer l: K at (2l) * layer_bytes, V at (2l+1) * layer_bytes
    size_t layer_bytes;
    float* part_o;
    float* part_ml;
    int* counters;
    uint32_t* err;
    int math;                        // 0 automatic, 1 CUDA cores, 2 warp MMA, 3 tcgen05
    int overlap;                     // 1: early history reads before the preceding grid ends
    bool tc_ok;                      // tensor maps built (bf16 cache, rows < 2^31)
    std::vector<CUtensorMap> tmaps;  // per layer: K, V (32-row boxes), K, V (128-row boxes; 3-D
                                     // maps of whole tiles for a contiguous D = 128 cache);
                                     // paged: K, V, K, V with min(bs, 128)-row boxes
    bool paged;                      // K / V of a layer are pools [num_blocks, H_kv, bs, D]
    bool rolling;                    // T_max = window slots, position p in slot p mod T_max
    bool quant;                      // 8-bit codes + fp32 row scales (q, out, new rows in dtype)
    bool fp8;                        // the codes are E4M3 (else int8)
    float* scales;                   // int8 cache: K / V row scales of layer l at 2l, 2l + 1
    size_t scale_stride;             // floats between consecutive scale arrays (256-byte aligned)
    int bs, max_blocks, num_blocks;  // paged geometry (T_max = max_blocks * bs)
};

namespace {

bool d_supported(int dtype, int D) {
    if (dtype == KVC_BF16) return D == 64 || D == 128 || D == 256;
    if (dtype == KVC_F32) return D == 4 || D == 64 || D == 128 || D == 256;
    return false;
}

bool g_supported(int G) { return G == 1 || G == 2 || G == 4 || G == 8 || G == 16 || G == 32; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, fetched through the runtime (no link-time libcuda); looked up
// once per process (thread-safe static initialisation).
EncodeTiledFn encode_fn() {
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(f);
        return nullptr;
    }();
    return fn;
}

}  // namespace

namespace kvc {

// 2-D map over one layer's K or V cache: columns D (contiguous), rows B*H_kv*T_max; boxes of 64
// columns (128 bytes) x box_rows rows, 128-byte swizzle, zero fill past the last row.
bool make_kv_tensor_map(CUtensorMap* map, void* base, uint64_t rows, int D, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over a contiguous cache with D = 128 (rows of 256 bytes): dimensions (64 columns, rows,
// 2 column blocks) with byte strides (256, 128) for dimensions 1..2, so one box of box_rows rows
// lands in shared memory as [column block][row][128 B] (128-byte swizzle): a whole tile of K or
// V in one copy.
bool make_kv3_tensor_map(CUtensorMap* map, void* base, uint64_t rows, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
    const cuuint64_t dims[3] = {64, (cuuint64_t)rows, 2};
    const cuuint64_t strides[2] = {256, 128};
    const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace kvc

namespace {

// 4-D map over a paged pool with D = 128 (rows of 256 bytes): dimensions (64 columns, 8 rows,
// 2 column blocks, rows / 8 groups) with byte strides (256, 128, 2048) for dimensions 1..3, so
// one box of box_rows / 8 groups lands in shared memory as [group][column block][8 rows][128 B]
// (128-byte swizzle); both column blocks of a block's rows come in one copy.
bool make_paged_tensor_map(CUtensorMap* map, void* base, uint64_t rows, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || (reinterpret_cast<uintptr_t>(base) & 15) || rows % 8 != 0) return false;
    const cuuint64_t dims[4] = {64, 8, 2, (cuuint64_t)(rows / 8)};
    const cuuint64_t strides[3] = {256, 128, 2048};
    const cuuint32_t box[4] = {64, 8, 2, (cuuint32_t)(box_rows / 8)};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over an int8 cache with D = 128 (rows of 128 bytes): boxes of 128 bytes x box_rows rows,
// no swizzle (the kernel widens them to bf16 itself).
bool make_q8_tensor_map(CUtensorMap* map, void* base, uint64_t rows, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
    const cuuint64_t dims[2] = {128, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over an 8-bit cache with D = 128 (rows of 128 codes): boxes of 128 bytes x box_rows
// rows, 128-byte swizzle (an fp8 K tile is MMA1's operand as it lands; an int8 K tile is read a
// row per thread).
bool make_f8_tensor_map(CUtensorMap* map, void* base, uint64_t rows, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
    const cuuint64_t dims[2] = {128, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// a * b with overflow detection (all operands >= 0)
bool mul_ok(uint64_t a, uint64_t b, uint64_t* r) {
    if (a != 0 && b > UINT64_MAX / a) return false;
    *r = a * b;
    return true;
}

// Which kernel computes the attention: 1 CUDA cores, 2 warp-level MMA, 3 tcgen05.
int kvc_math_path(const kvc_cache* h) {
    if (!h->tc_ok || h->math == 1) return 1;
    if (h->math == 2) return 2;
    if (h->math == 3) return 3;
    return h->D == 128 ? 3 : 1;  // automatic
}

int launch_decode(const kvc_cache* h, int layer, const kvc::DecodeParams& p, cudaStream_t s) {
    int smem = 0;
    int e;
    const int Gq = h->G * p.T_q;  // query rows per KV head: G heads x T_q new tokens
    const int path = kvc_math_path(h);
    if (path == 3) {
        const CUtensorMap* maps = &h->tmaps[4 * (size_t)layer];
        e = h->paged     ? kvc::launch_decode_tc5p_d128(Gq, p, maps, s, &smem)
            : h->rolling ? kvc::launch_decode_tc5r_d128(Gq, p, maps, s, &smem)
            : h->quant   ? (h->fp8 ? kvc::launch_decode_tc5f_d128(Gq, p, maps, s, &smem)
                                   : kvc::launch_decode_tc5q_d128(Gq, p, maps, s, &smem))
                         : kvc::launch_decode_tc5_d128(Gq, p, maps, s, &smem);
    } else if (path == 2) {
        const CUtensorMap& tk = h->tmaps[4 * (size_t)layer];
        const CUtensorMap& tv = h->tmaps[4 * (size_t)layer + 1];
        switch (h->D) {
            case 64: e = kvc::launch_decode_tc_d64(Gq, p, tk, tv, s, &smem); break;
            case 128: e = kvc::launch_decode_tc_d128(Gq, p, tk, tv, s, &smem); break;
            case 256: e = kvc::launch_decode_tc_d256(Gq, p, tk, tv, s, &smem); break;
            default: return KVC_EUNSUPPORTED;
        }
    } else if (h->dtype == KVC_BF16) {
        switch (h->D) {
            case 64: e = kvc::launch_decode_bf16_d64(Gq, p, s, &smem); break;
            case 128: e = kvc::launch_decode_bf16_d128(Gq, p, s, &smem); break;
            case 256: e = kvc::launch_decode_bf16_d256(Gq, p, s, &smem); break;
            default: return KVC_EUNSUPPORTED;
        }
    } else {
        switch (h->D) {
            case 4: e = kvc::launch_decode_f32_d4(Gq, p, s, &smem); break;
            case 64: e = kvc::launch_decode_f32_d64(Gq, p, s, &smem); break;
            case 128: e = kvc::launch_decode_f32_d128(Gq, p, s, &smem); break;
            case 256: e = kvc::launch_decode_f32_d256(Gq, p, s, &smem); break;
            default: return KVC_EUNSUPPORTED;
        }
    }
    if (e != 0) return KVC_ECUDA;
    if (p.combine_mode == 1) {
        if (kvc::launch_combine(h->dtype, h->D, Gq, p, s) != 0) return KVC_ECUDA;
    }
    return KVC_OK;
}

int attn_common(kvc_t h, int layer, const void* q, const void* k_new, const void* v_new, void* out,
                const int32_t* table, const int32_t* lens, void* stream, int T_q = 1) {
    if (!h || !q || !out || !lens) return KVC_EINVAL;
    if (T_q < 1) return KVC_EINVAL;
    if (T_q > 1) {
        // several new tokens: the group's G * T_q query rows must be a supported row count, on a
        // plain contiguous cache, with a kernel that masks per query row
        if ((T_q & (T_q - 1)) != 0 || h->G * T_q > 32) return KVC_EUNSUPPORTED;
        if (h->paged || h->rolling || h->quant || kvc_math_path(h) == 2) return KVC_EUNSUPPORTED;
    }
    if (h->quant && kvc_math_path(h) != 3) return KVC_EUNSUPPORTED;  // only tcgen05 reads int8
    if (layer < 0 || layer >= h->layers) return KVC_EINVAL;
    if ((k_new == nullptr) != (v_new == nullptr)) return KVC_EINVAL;
    if (h->paged != (table != nullptr)) return KVC_EINVAL;  // paged calls on paged handles only
    kvc::DecodeParams p{};
    p.K = h->slab + (size_t)(2 * layer) * h->layer_bytes;
    p.V = h->slab + (size_t)(2 * layer + 1) * h->layer_bytes;
    p.q = q;
    p.out = out;
    p.k_new = k_new;
    p.v_new = v_new;
    p.lens = lens;
    p.part_o = h->part_o;
    p.part_ml = h->part_ml;
    p.counters = h->counters;
    p.err = h->err;
    p.B = h->B;
    p.H_kv = h->H_kv;
    p.T_max = h->T_max;
    p.P = h->ctas > 0 ? h->ctas : h->sms;
    p.min_tokens = h->ctas > 0 ? 1 : 256;
    p.table = table;
    p.bs = h->paged ? h->bs : 1;
    p.max_blocks = h->max_blocks;
    p.num_blocks = h->num_blocks;
    p.box_rows = h->paged ? (h->bs < kvc::TC_FULL_ROWS ? h->bs : kvc::TC_FULL_ROWS) : 0;
    p.rolling = h->rolling ? 1 : 0;
    // tcgen05 kernel on a paged pool: which warp issues MMA2.  Measured (8B GQA, per layer): the
    // producer warp for 32- and 64-token blocks (2-4 copies per tile), the MMA warp for 16-token
    // blocks (8 copies per tile keep the producer busy) and for blocks of 128 tokens or more.
    p.m2p = (h->paged && h->bs >= 32 && h->bs < 128) ? 1 : 0;
    p.T_q = T_q;
    if (h->quant) {
        p.Ksc = h->scales + (size_t)(2 * layer) * h->scale_stride;
        p.Vsc = h->scales + (size_t)(2 * layer + 1) * h->scale_stride;
    }
    const int U = h->B * h->H_kv;
    int mode = h->combine_mode;
    if (mode < 0) {
        // Merge cost of the last-arriving CTA grows with the segments per stream times the
        // group's outputs; when streams are few and long, hand the merge to a wide kernel.
        const long long nseg = (p.P + U - 1) / U + 1;
        mode = (nseg * h->G * T_q * h->D * 4 > 65536) ? 1 : 0;
    }
    p.combine_mode = mode;
    // Few long streams merged by the combine kernel (a segment per CTA): a decode grid of four
    // fifths of the SMs measured faster on MQA B = 1, T = 131072, G = 32 (us per layer with
    // 104 / 120 / 136 / 152 CTAs: 26.8 / 26.5 / 29.8 / 29.2; this rule's 121 on one box: 28.2-28.5
    // against 26.2-26.4 with 120 and 29.2 with 152, a step not understood).  Grids merged in-kernel
    // keep one CTA per SM (MQA B = 64 with 120 CTAs: 44.7 against 37.5).
    if (mode == 1 && h->ctas <= 0) p.P = h->sms * 4 / 5;
    p.grain = kvc::partition_grain(h->G, mode, p.bs);
    p.qscale = (float)(1.4426950408889634 / sqrt((double)h->D));
    p.overlap = h->overlap;
    return launch_decode(h, layer, p, static_cast<cudaStream_t>(stream));
}

// int8 cache: the layer's row-scale arrays for the quantizing writes
void set_quant_scales(const kvc_cache* h, int layer, kvc::CopyParams& p) {
    if (!h->quant) return;
    p.fp8 = h->fp8 ? 1 : 0;
    p.Ksc = h->scales + (size_t)(2 * layer) * h->scale_stride;
    p.Vsc = h->scales + (size_t)(2 * layer + 1) * h->scale_stride;
}

}  // namespace

extern "C" {

const char* kvc_status_str(int status) {
    switch (status) {
        case KVC_OK: return "ok";
        case KVC_EINVAL: return "invalid argument";
        case KVC_ENOMEM: return "out of device memory";
        case KVC_ECUDA: return "CUDA error";
        case KVC_ERANGE: return "size out of range";
        case KVC_EDEVICE: return "device-side check failed";
        case KVC_EUNSUPPORTED: return "unsupported shape or device";
        default: return "unknown status";
    }
}

uint64_t kvc_bytes_formula(int64_t L, int64_t B, int64_t H_kv, int64_t D, int64_t T,
                           int64_t elem_bytes) {
    if (L < 0 || B < 0 || H_kv < 0 || D < 0 || T < 0 || elem_bytes < 0) return 0;
    uint64_t r = 2;
    const int64_t f[6] = {L, H_kv, D, B, T, elem_bytes};
    for (int i = 0; i < 6; ++i)
        if (!mul_ok(r, (uint64_t)f[i], &r)) return 0;
    return r;
}

int kvc_plan_grain(int G, int combine_mode, int block_size) {
    if (G < 1 || (combine_mode != 0 && combine_mode != 1) || block_size < 1) return -1;
    return kvc::partition_grain(G, combine_mode, block_size);
}

int kvc_plan_cta_of(int64_t x, int64_t U, int P) {
    if (U <= 0 || P <= 0 || x < 0 || x >= U) return -1;
    return (int)kvc::cta_of(x, U, P);
}

namespace {
// prefix[b] / uprefix[b] = valid lengths / partition units before b (host copy of the kernels'
// first step; B * T_max < 2^31 keeps both in 32 bits)
bool plan_prefix(const int32_t* lens, int B, int T_max, int grain, std::vector<int32_t>& prefix,
                 std::vector<int32_t>& uprefix) {
    if ((int64_t)B * T_max >= (int64_t(1) << 31)) return false;
    prefix.assign((size_t)B + 1, 0);
    uprefix.assign((size_t)B + 1, 0);
    for (int b = 0; b < B; ++b) {
        const int L = (lens[b] >= 1 && lens[b] <= T_max) ? lens[b] : 0;
        prefix[b + 1] = prefix[b] + L;
        uprefix[b + 1] = uprefix[b] + (int32_t)kvc::stream_units(L, grain);
    }
    return true;
}
}  // namespace

int kvc_plan_cuts(const int32_t* lens_host, int B, int H_kv, int T_max, int grain, int P,
                  int min_tokens, int64_t* cuts) {
    if (!lens_host || !cuts || B < 1 || B > kvc::MAX_B || H_kv < 1 || T_max < 1 || grain < 1 ||
        P < 1 || min_tokens < 1)
        return -1;
    std::vector<int32_t> prefix, uprefix;
    if (!plan_prefix(lens_host, B, T_max, grain, prefix, uprefix)) return -1;
    const int64_t W = (int64_t)H_kv * prefix[B], U = (int64_t)H_kv * uprefix[B];
    if (W == 0) return 0;
    const int64_t Pu = kvc::plan_ctas(W, U, P, min_tokens);
    for (int64_t i = 0; i <= Pu; ++i)
        cuts[i] = kvc::cta_cut(i, prefix.data(), uprefix.data(), B, H_kv, U, Pu, grain);
    return (int)Pu;
}

int kvc_plan_stream_ctas(const int32_t* lens_host, int B, int H_kv, int T_max, int grain, int P,
                         int min_tokens, int b, int h, int* first, int* last) {
    if (!lens_host || !first || !last || B < 1 || B > kvc::MAX_B || T_max < 1 || grain < 1 || b < 0 ||
        b >= B || h < 0 || h >= H_kv || P < 1 || min_tokens < 1)
        return KVC_EINVAL;
    std::vector<int32_t> prefix, uprefix;
    if (!plan_prefix(lens_host, B, T_max, grain, prefix, uprefix)) return KVC_ERANGE;
    const int64_t W = (int64_t)H_kv * prefix[B], U = (int64_t)H_kv * uprefix[B];
    const int64_t nu = uprefix[b + 1] - uprefix[b];
    if (W == 0 || nu == 0) return KVC_EINVAL;
    const int64_t Pu = kvc::plan_ctas(W, U, P, min_tokens);
    const int64_t u0 = (int64_t)H_kv * uprefix[b] + (int64_t)h * nu;
    *first = (int)kvc::cta_of(u0 + kvc::stream_cost(grain), U, Pu);
    *last = (int)kvc::cta_of(u0 + nu - 1, U, Pu);
    return KVC_OK;
}

static int create_common(kvc_t* out, int layers, int B, int H_q, int H_kv, int D, int T_max,
                         int dtype, int bs, int max_blocks, int num_blocks, bool quant = false,
                         bool fp8 = false) {
    const bool paged = bs > 0;
    if (!out) return KVC_EINVAL;
    *out = nullptr;
    if (layers < 1 || B < 1 || H_q < 1 || H_kv < 1 || D < 1 || T_max < 1) return KVC_EINVAL;
    if (dtype != KVC_BF16 && dtype != KVC_F32) return KVC_EINVAL;
    if (H_q % H_kv != 0) return KVC_EINVAL;
    if (B > kvc::MAX_B) return KVC_ERANGE;
    const int G = H_q / H_kv;
    if (!g_supported(G) || !d_supported(dtype, D)) return KVC_EUNSUPPORTED;
    const int es = dtype == KVC_BF16 ? 2 : 4;
    // the kernels keep prefix sums of the sequence lengths in 32 bits: B * T_max < 2^31
    if ((int64_t)B * T_max >= (int64_t(1) << 31)) return KVC_ERANGE;
    // rows of one layer's K (or V): streams x T_max, or the pool's blocks x heads x bs
    uint64_t rows = 0;
    if (!mul_ok(paged ? (uint64_t)num_blocks : (uint64_t)B, (uint64_t)H_kv, &rows) ||
        !mul_ok(rows, paged ? (uint64_t)bs : (uint64_t)T_max, &rows))
        return KVC_ERANGE;
    // cache element bytes: the dtype, or 1 for int8 codes (their fp32 row scales follow all codes)
    const int ces = quant ? 1 : es;
    uint64_t total = 0;
    if (!mul_ok(rows, 2ull * (uint64_t)layers * (uint64_t)D * (uint64_t)ces, &total)) return KVC_ERANGE;
    const size_t scale_stride = quant ? (size_t)((rows + 63) / 64 * 64) : 0;  // floats, 256-B aligned
    const size_t codes_total = (size_t)total;
    total += 2ull * (uint64_t)layers * scale_stride * 4;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVC_ECUDA;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return KVC_ECUDA;
    if (!(prop.major == 10 && prop.minor == 3)) return KVC_EUNSUPPORTED;  // built for sm_103a

    kvc_cache* h = new (std::nothrow) kvc_cache();
    if (!h) return KVC_ENOMEM;
    h->layers = layers; h->B = B; h->H_q = H_q; h->H_kv = H_kv; h->D = D; h->T_max = T_max;
    h->dtype = dtype; h->es = es; h->G = G; h->device = dev;
    h->sms = prop.multiProcessorCount;
    h->ctas = 0;
    h->combine_mode = -1;
    h->overlap = 0;
    h->math = 0;
    h->tc_ok = false;
    h->paged = paged;
    h->rolling = false;
    h->quant = quant;
    h->fp8 = quant && fp8;
    h->scale_stride = scale_stride;
    h->bs = paged ? bs : 1;
    h->max_blocks = paged ? max_blocks : 0;
    h->num_blocks = paged ? num_blocks : 0;
    h->max_ctas = 4 * h->sms;
    h->layer_bytes = (size_t)rows * D * ces;

    const size_t U = (size_t)B * H_kv;
    const size_t slots = (size_t)h->max_ctas + U;
    // partial states for up to 32 query rows per KV head (G heads x T_q new tokens)
    const size_t GW = G > 32 ? (size_t)G : 32;
    const size_t ws_bytes = slots * GW * (size_t)D * 4 + slots * GW * 2 * 4 + U * 4 + 256;
    size_t free_b = 0, total_b = 0;
    if (cudaMemGetInfo(&free_b, &total_b) != cudaSuccess) { delete h; return KVC_ECUDA; }
    if (total + ws_bytes > free_b) { delete h; return KVC_ENOMEM; }

    if (cudaMalloc(&h->slab, total) != cudaSuccess) { cudaGetLastError(); delete h; return KVC_ENOMEM; }
    h->scales = quant ? reinterpret_cast<float*>(h->slab + codes_total) : nullptr;
    char* ws = nullptr;
    if (cudaMalloc(&ws, ws_bytes) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(h->slab);
        delete h;
        return KVC_ENOMEM;
    }
    h->part_o = reinterpret_cast<float*>(ws);
    h->part_ml = h->part_o + slots * GW * D;
    h->counters = reinterpret_cast<int*>(h->part_ml + slots * GW * 2);
    h->err = reinterpret_cast<uint32_t*>(h->counters + U);
    if (cudaMemset(h->slab, 0, total) != cudaSuccess || cudaMemset(ws, 0, ws_bytes) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        cudaFree(ws);
        cudaFree(h->slab);
        delete h;
        return KVC_ECUDA;
    }
    // tensor maps for the tensor-core kernels (bf16 caches whose rows fit the map's coordinates);
    // a paged pool is copied one block (at most 128 rows) per box
    const int box_small = paged ? (bs < kvc::TC_FULL_ROWS ? bs : kvc::TC_FULL_ROWS) : kvc::TC_BOX_ROWS;
    const int box_full = paged ? box_small : kvc::TC_FULL_ROWS;
    if (dtype == KVC_BF16 && rows < (1ull << 31) && ((!paged && !quant) || D == 128)) {
        h->tmaps.resize(4 * (size_t)layers);
        bool ok = true;
        for (int l = 0; l < layers && ok; ++l) {
            void* kb = h->slab + (size_t)(2 * l) * h->layer_bytes;
            void* vb = h->slab + (size_t)(2 * l + 1) * h->layer_bytes;
            CUtensorMap* m4 = &h->tmaps[4 * (size_t)l];
            if (quant && fp8)  // E4M3 rows of 128 bytes, 128-byte swizzled
                ok = make_f8_tensor_map(&m4[0], kb, rows, box_small) &&
                     make_f8_tensor_map(&m4[1], vb, rows, box_small) &&
                     make_f8_tensor_map(&m4[2], kb, rows, box_full) &&
                     make_f8_tensor_map(&m4[3], vb, rows, box_full);
            else if (quant)  // int8 rows of 128 bytes: K 128-byte swizzled (each converter thread
                             // widens a whole row), V unswizzled (widened in place)
                ok = make_f8_tensor_map(&m4[0], kb, rows, box_small) &&
                     make_q8_tensor_map(&m4[1], vb, rows, box_small) &&
                     make_f8_tensor_map(&m4[2], kb, rows, box_full) &&
                     make_q8_tensor_map(&m4[3], vb, rows, box_full);
            else if (paged)  // the tcgen05 kernel's paged variant (D = 128) reads 4-D boxes
                ok = make_paged_tensor_map(&m4[0], kb, rows, box_small) &&
                     make_paged_tensor_map(&m4[1], vb, rows, box_small) &&
                     make_paged_tensor_map(&m4[2], kb, rows, box_full) &&
                     make_paged_tensor_map(&m4[3], vb, rows, box_full);
            else if (D == 128)  // whole tiles (tcgen05 kernel only) in one 3-D copy per tensor
                ok = kvc::make_kv_tensor_map(&m4[0], kb, rows, D, box_small) &&
                     kvc::make_kv_tensor_map(&m4[1], vb, rows, D, box_small) &&
                     kvc::make_kv3_tensor_map(&m4[2], kb, rows, box_full) &&
                     kvc::make_kv3_tensor_map(&m4[3], vb, rows, box_full);
            else
                ok = kvc::make_kv_tensor_map(&m4[0], kb, rows, D, box_small) &&
                     kvc::make_kv_tensor_map(&m4[1], vb, rows, D, box_small) &&
                     kvc::make_kv_tensor_map(&m4[2], kb, rows, D, box_full) &&
                     kvc::make_kv_tensor_map(&m4[3], vb, rows, D, box_full);
        }
        h->tc_ok = ok;
        if (!ok) h->tmaps.clear();
    }
    *out = h;
    return KVC_OK;
}

int kvc_create(kvc_t* out, int layers, int B, int H_q, int H_kv, int D, int T_max, int dtype) {
    return create_common(out, layers, B, H_q, H_kv, D, T_max, dtype, 0, 0, 0);
}

int kvc_create_quantized(kvc_t* out, int layers, int B, int H_q, int H_kv, int D, int T_max,
                         int dtype) {
    if (!out) return KVC_EINVAL;
    *out = nullptr;
    // the tcgen05 kernel reads int8 tiles: bf16 queries, D = 128, up to 8 query heads per KV head
    if (dtype != KVC_BF16 || D != 128 || H_kv < 1 || H_q % H_kv != 0 || H_q / H_kv > 8)
        return KVC_EUNSUPPORTED;
    const int rc = create_common(out, layers, B, H_q, H_kv, D, T_max, dtype, 0, 0, 0, true);
    if (rc == KVC_OK && !(*out)->tc_ok) {  // no tensor maps: nothing can read this cache
        kvc_destroy(*out);
        *out = nullptr;
        return KVC_EUNSUPPORTED;
    }
    return rc;
}

int kvc_create_fp8(kvc_t* out, int layers, int B, int H_q, int H_kv, int D, int T_max, int dtype) {
    if (!out) return KVC_EINVAL;
    *out = nullptr;
    // the tcgen05 kernel reads E4M3 tiles: bf16 queries, D = 128, up to 8 query heads per KV head
    if (dtype != KVC_BF16 || D != 128 || H_kv < 1 || H_q % H_kv != 0 || H_q / H_kv > 8)
        return KVC_EUNSUPPORTED;
    const int rc = create_common(out, layers, B, H_q, H_kv, D, T_max, dtype, 0, 0, 0, true, true);
    if (rc == KVC_OK && !(*out)->tc_ok) {  // no tensor maps: nothing can read this cache
        kvc_destroy(*out);
        *out = nullptr;
        return KVC_EUNSUPPORTED;
    }
    return rc;
}

int kvc_get_cache_format(kvc_t h) {
    if (!h) return -1;
    return h->quant ? (h->fp8 ? KVC_CACHE_FP8 : KVC_CACHE_INT8) : KVC_CACHE_PLAIN;
}

int kvc_layer_scales(kvc_t h, int layer, float** Ks, float** Vs) {
    if (!h || !h->quant || layer < 0 || layer >= h->layers) return KVC_EINVAL;
    if (Ks) *Ks = h->scales + (size_t)(2 * layer) * h->scale_stride;
    if (Vs) *Vs = h->scales + (size_t)(2 * layer + 1) * h->scale_stride;
    return KVC_OK;
}

int kvc_create_rolling(kvc_t* out, int layers, int B, int H_q, int H_kv, int D, int window,
                       int dtype) {
    const int rc = create_common(out, layers, B, H_q, H_kv, D, window, dtype, 0, 0, 0);
    if (rc == KVC_OK) (*out)->rolling = true;
    return rc;
}

int kvc_get_window(kvc_t h) {
    if (!h) return -1;
    return h->rolling ? h->T_max : 0;
}

int kvc_create_paged(kvc_t* out, int layers, int num_blocks, int block_size, int B, int max_blocks,
                     int H_q, int H_kv, int D, int dtype) {
    if (!out) return KVC_EINVAL;
    *out = nullptr;
    if (num_blocks < 1 || max_blocks < 1) return KVC_EINVAL;
    if (block_size != 16 && block_size != 32 && block_size != 64 && block_size != 128 &&
        block_size != 256)
        return KVC_EUNSUPPORTED;
    if ((int64_t)max_blocks * block_size >= (1ll << 31)) return KVC_ERANGE;
    return create_common(out, layers, B, H_q, H_kv, D, max_blocks * block_size, dtype, block_size,
                         max_blocks, num_blocks);
}

int kvc_destroy(kvc_t h) {
    if (!h) return KVC_OK;
    int rc = KVC_OK;
    if (cudaDeviceSynchronize() != cudaSuccess) rc = KVC_ECUDA;
    cudaFree(h->part_o);  // workspace base
    cudaFree(h->slab);
    delete h;
    return rc;
}

uint64_t kvc_bytes(kvc_t h) {
    if (!h) return 0;
    // paged: the whole block pool; int8: codes plus the fp32 row scales
    return 2ull * (uint64_t)h->layers * (h->layer_bytes + h->scale_stride * 4);
}

uint64_t kvc_payload_bytes(kvc_t h, const int32_t* lens_host) {
    if (!h || !lens_host) return 0;
    uint64_t sum = 0;
    for (int b = 0; b < h->B; ++b) sum += (uint64_t)(lens_host[b] > 0 ? lens_host[b] : 0);
    const uint64_t row = h->quant ? (uint64_t)h->D + 4 : (uint64_t)h->D * h->es;  // int8: + scale
    return 2ull * h->layers * h->H_kv * row * sum;
}

int kvc_layer_ptrs(kvc_t h, int layer, void** K, void** V) {
    if (!h || layer < 0 || layer >= h->layers) return KVC_EINVAL;
    if (K) *K = h->slab + (size_t)(2 * layer) * h->layer_bytes;
    if (V) *V = h->slab + (size_t)(2 * layer + 1) * h->layer_bytes;
    return KVC_OK;
}

int kvc_get_shape(kvc_t h, int* layers, int* B, int* H_q, int* H_kv, int* D, int* T_max,
                  int* dtype) {
    if (!h) return KVC_EINVAL;
    if (layers) *layers = h->layers;
    if (B) *B = h->B;
    if (H_q) *H_q = h->H_q;
    if (H_kv) *H_kv = h->H_kv;
    if (D) *D = h->D;
    if (T_max) *T_max = h->T_max;
    if (dtype) *dtype = h->dtype;
    return KVC_OK;
}

int kvc_set_ctas(kvc_t h, int ctas) {
    if (!h || ctas < 0 || ctas > h->max_ctas) return KVC_EINVAL;
    h->ctas = ctas;
    return KVC_OK;
}

int kvc_get_ctas(kvc_t h) {
    if (!h) return -1;
    return h->ctas > 0 ? h->ctas : h->sms;
}

int kvc_set_math(kvc_t h, int mode) {
    if (!h || mode < 0 || mode > 3) return KVC_EINVAL;
    if (mode >= 2 && !h->tc_ok) return KVC_EUNSUPPORTED;
    if (mode == 3 && h->D != 128) return KVC_EUNSUPPORTED;
    if (mode == 2 && (h->paged || h->rolling)) return KVC_EUNSUPPORTED;  // warp MMA: plain caches only
    if (h->quant && mode != 0 && mode != 3) return KVC_EUNSUPPORTED;     // int8: tcgen05 only
    h->math = mode;
    return KVC_OK;
}

int kvc_get_math(kvc_t h) {
    if (!h) return -1;
    return kvc_math_path(h);
}

int kvc_set_launch_overlap(kvc_t h, int on) {
    if (!h || on < 0 || on > 1) return KVC_EINVAL;
    h->overlap = on;
    return KVC_OK;
}

int kvc_get_launch_overlap(kvc_t h) {
    if (!h) return -1;
    return h->overlap;
}

int kvc_set_combine_mode(kvc_t h, int mode) {
    if (!h || mode < -1 || mode > 1) return KVC_EINVAL;
    h->combine_mode = mode;
    return KVC_OK;
}

int kvc_prefill_write(kvc_t h, int layer, const void* K, const void* V, int T_in,
                      const int32_t* lens, void* stream) {
    if (!h || !K || !V || !lens) return KVC_EINVAL;
    if (layer < 0 || layer >= h->layers) return KVC_EINVAL;
    if (T_in < 1 || (!h->rolling && T_in > h->T_max)) return KVC_ERANGE;
    if (h->paged) return KVC_EINVAL;
    kvc::CopyParams p{};
    p.Kc = h->slab + (size_t)(2 * layer) * h->layer_bytes;
    p.Vc = h->slab + (size_t)(2 * layer + 1) * h->layer_bytes;
    p.K = K;
    p.V = V;
    p.lens = lens;
    p.err = h->err;
    p.B = h->B; p.H_kv = h->H_kv; p.T_max = h->T_max; p.T_in = T_in;
    p.row_bytes = h->D * h->es;
    p.rolling = h->rolling ? 1 : 0;
    set_quant_scales(h, layer, p);
    return kvc::launch_prefill(p, static_cast<cudaStream_t>(stream)) == 0 ? KVC_OK : KVC_ECUDA;
}

int kvc_append(kvc_t h, int layer, const void* k_new, const void* v_new, const int32_t* lens,
               void* stream) {
    if (!h || !k_new || !v_new || !lens) return KVC_EINVAL;
    if (layer < 0 || layer >= h->layers) return KVC_EINVAL;
    if (h->paged) return KVC_EINVAL;
    kvc::CopyParams p{};
    p.Kc = h->slab + (size_t)(2 * layer) * h->layer_bytes;
    p.Vc = h->slab + (size_t)(2 * layer + 1) * h->layer_bytes;
    p.K = k_new;
    p.V = v_new;
    p.lens = lens;
    p.err = h->err;
    p.B = h->B; p.H_kv = h->H_kv; p.T_max = h->T_max; p.T_in = 1;
    p.row_bytes = h->D * h->es;
    p.rolling = h->rolling ? 1 : 0;
    set_quant_scales(h, layer, p);
    return kvc::launch_append(p, static_cast<cudaStream_t>(stream)) == 0 ? KVC_OK : KVC_ECUDA;
}

int kvc_decode_attn(kvc_t h, int layer, const void* q, void* out, const int32_t* lens,
                    void* stream) {
    return attn_common(h, layer, q, nullptr, nullptr, out, nullptr, lens, stream);
}

int kvc_decode_step(kvc_t h, int layer, const void* q, const void* k_new, const void* v_new,
                    void* out, const int32_t* lens, void* stream) {
    if (!k_new || !v_new) return KVC_EINVAL;
    return attn_common(h, layer, q, k_new, v_new, out, nullptr, lens, stream);
}

int kvc_append_multi(kvc_t h, int layer, const void* k_new, const void* v_new, const int32_t* lens,
                     int T_q, void* stream) {
    if (!h || !k_new || !v_new || !lens || T_q < 1) return KVC_EINVAL;
    if (layer < 0 || layer >= h->layers || h->paged) return KVC_EINVAL;
    if (T_q > 1 && (h->rolling || h->quant)) return KVC_EUNSUPPORTED;
    if (T_q > h->T_max) return KVC_ERANGE;
    kvc::CopyParams p{};
    p.Kc = h->slab + (size_t)(2 * layer) * h->layer_bytes;
    p.Vc = h->slab + (size_t)(2 * layer + 1) * h->layer_bytes;
    p.K = k_new;
    p.V = v_new;
    p.lens = lens;
    p.err = h->err;
    p.B = h->B; p.H_kv = h->H_kv; p.T_max = h->T_max; p.T_in = T_q;
    p.row_bytes = h->D * h->es;
    p.rolling = h->rolling ? 1 : 0;
    return kvc::launch_append(p, static_cast<cudaStream_t>(stream)) == 0 ? KVC_OK : KVC_ECUDA;
}

int kvc_decode_attn_multi(kvc_t h, int layer, const void* q, void* out, const int32_t* lens, int T_q,
                          void* stream) {
    return attn_common(h, layer, q, nullptr, nullptr, out, nullptr, lens, stream, T_q);
}

int kvc_decode_step_multi(kvc_t h, int layer, const void* q, const void* k_new, const void* v_new,
                          void* out, const int32_t* lens, int T_q, void* stream) {
    if (!k_new || !v_new) return KVC_EINVAL;
    return attn_common(h, layer, q, k_new, v_new, out, nullptr, lens, stream, T_q);
}

int kvc_paged_prefill_write(kvc_t h, int layer, const void* K, const void* V, int T_in,
                            const int32_t* block_table, const int32_t* lens, void* stream) {
    if (!h || !K || !V || !lens || !block_table) return KVC_EINVAL;
    if (!h->paged || layer < 0 || layer >= h->layers) return KVC_EINVAL;
    if (T_in < 1 || T_in > h->T_max) return KVC_ERANGE;
    kvc::CopyParams p{};
    p.Kc = h->slab + (size_t)(2 * layer) * h->layer_bytes;
    p.Vc = h->slab + (size_t)(2 * layer + 1) * h->layer_bytes;
    p.K = K;
    p.V = V;
    p.lens = lens;
    p.err = h->err;
    p.B = h->B; p.H_kv = h->H_kv; p.T_max = h->T_max; p.T_in = T_in;
    p.row_bytes = h->D * h->es;
    p.table = block_table; p.bs = h->bs; p.max_blocks = h->max_blocks; p.num_blocks = h->num_blocks;
    return kvc::launch_prefill(p, static_cast<cudaStream_t>(stream)) == 0 ? KVC_OK : KVC_ECUDA;
}

int kvc_paged_append(kvc_t h, int layer, const void* k_new, const void* v_new,
                     const int32_t* block_table, const int32_t* lens, void* stream) {
    if (!h || !k_new || !v_new || !lens || !block_table) return KVC_EINVAL;
    if (!h->paged || layer < 0 || layer >= h->layers) return KVC_EINVAL;
    kvc::CopyParams p{};
    p.Kc = h->slab + (size_t)(2 * layer) * h->layer_bytes;
    p.Vc = h->slab + (size_t)(2 * layer + 1) * h->layer_bytes;
    p.K = k_new;
    p.V = v_new;
    p.lens = lens;
    p.err = h->err;
    p.B = h->B; p.H_kv = h->H_kv; p.T_max = h->T_max; p.T_in = 1;
    p.row_bytes = h->D * h->es;
    p.table = block_table; p.bs = h->bs; p.max_blocks = h->max_blocks; p.num_blocks = h->num_blocks;
    return kvc::launch_append(p, static_cast<cudaStream_t>(stream)) == 0 ? KVC_OK : KVC_ECUDA;
}

int kvc_paged_decode_attn(kvc_t h, int layer, const void* q, void* out, const int32_t* block_table,
                          const int32_t* lens, void* stream) {
    if (!block_table) return KVC_EINVAL;
    return attn_common(h, layer, q, nullptr, nullptr, out, block_table, lens, stream);
}

int kvc_paged_decode_step(kvc_t h, int layer, const void* q, const void* k_new, const void* v_new,
                          void* out, const int32_t* block_table, const int32_t* lens, void* stream) {
    if (!k_new || !v_new || !block_table) return KVC_EINVAL;
    return attn_common(h, layer, q, k_new, v_new, out, block_table, lens, stream);
}

int kvc_get_paged_shape(kvc_t h, int* num_blocks, int* block_size, int* max_blocks) {
    if (!h || !h->paged) return KVC_EINVAL;
    if (num_blocks) *num_blocks = h->num_blocks;
    if (block_size) *block_size = h->bs;
    if (max_blocks) *max_blocks = h->max_blocks;
    return KVC_OK;
}

int kvc_last_error(kvc_t h, void* stream, uint32_t* detail) {
    if (!h) return KVC_EINVAL;
    if (detail) *detail = 0;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVC_ECUDA;
    uint32_t v = 0;
    if (cudaMemcpy(&v, h->err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return KVC_ECUDA;
    if (v == 0) return KVC_OK;
    if (cudaMemset(h->err, 0, sizeof v) != cudaSuccess) return KVC_ECUDA;
    if (detail) *detail = v;
    return KVC_EDEVICE;
}

}  // extern "C"
