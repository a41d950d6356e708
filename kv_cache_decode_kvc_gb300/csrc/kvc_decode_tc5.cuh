// kvc_decode_tc5.cuh -- decode attention over a bf16 cache with the two contractions on the
// 5th-generation tensor cores (tcgen05: single-thread MMA issue, operands in shared memory,
// accumulators in tensor memory).
//
// Same computation, split-T partition and merging as decode_kernel (kvc_decode.cuh): for every
// query head j of sequence b, o = softmax_t(q . K_t / sqrt(D)) V over t < lens[b]
// ("11.7 KV Cache：形状、显存与带宽" §2.2; head map of "第 1 周 · Day 4：KV Cache 与 MQA /
// GQA" §3.4).  A CTA (producer warp, MMA warp, 4 or 8 softmax warps, 2 epilogue warps)
// consumes 128-token tiles:
//   MMA1  S^T[128 tok x N]  = K[128 x D] . Q^T[D x N]   A = K tile (K-major), B = q (K-major)
//   softmax: a thread owns one token (one tensor-memory lane) and all N head columns
//   MMA2  O^T[D x N]        = V^T[D x 128] . P^T[128 x N]  A = V tile read MN-major, B = P
//   O^T is read back per tile (a thread owns output element d = its lane) and accumulated in
//   registers with the online-softmax rescale.  S^T, O^T and P are double-buffered so MMA1 of
//   tile k+1 overlaps the softmax of tile k.
// N = the query-head group padded to at least 16 (tcgen05 needs N % 16 == 0 at M = 128); the
// padded q rows are zero.  P is stored as P_hi + P_lo (two bf16 terms, stacked as 2N operand
// columns of one MMA2) so the weights keep fp32-level accuracy while V is read once.
// Everything the tensor cores read is in the 128-byte-swizzled K-major or MN-major canonical
// layout: K/V tiles arrive that way from TMA tensor copies, q and P are written that way by the
// threads.
// HBM traffic is unchanged: every K/V byte once per step, shared by the whole group.
#pragma once

#include "kvc_decode_tc.cuh"

namespace kvc {

template <int G_, int MODE_ = 0>
struct Tc5Cfg {
    static constexpr int D = 128;
    static constexpr int G = G_;
    // fp8 cache (MODE 4): MMA1 reads the E4M3 K tile as it lands and q as three E4M3 terms per
    // head (rows [t G, (t + 1) G) hold term t); only V is widened (to f16) for MMA2
    static constexpr bool FP8 = MODE_ == 4;
    static constexpr int NP = G < 16 ? 16 : G;          // heads, padded (P rows and O^T columns)
    static constexpr int N = FP8 ? (3 * G + 15) / 16 * 16 : NP;  // MMA1 N (q rows, padded)
    static constexpr int ROWB = D * 2;
    static constexpr int HALVES = D / 64;               // 128-byte column blocks of a 16-bit row
    // softmax warps (+ producer + MMA warp): HSPLIT per tensor-memory lane quadrant, each with
    // GH = G / HSPLIT of the group's head columns (large groups: more warps, fewer registers each)
    static constexpr int HSPLIT = G >= 16 ? 2 : 1;
    static constexpr int GH = G / HSPLIT;
    static constexpr int NW = 4 * HSPLIT;
    // segment-epilogue warps (int8 cache with groups of up to 4 heads: one, which leaves room
    // for the MMA2 warp within 16 warps)
    static constexpr int NEPI = MODE_ == 3 && G_ <= 4 ? 1 : 2;
    static constexpr int NTHREADS = (2 + NW + NEPI) * 32;
    static constexpr int NCONV = MODE_ == 3 && G_ <= 4 ? 8 : 4;  // converter warps (int8 and fp8 caches)
    static constexpr int TT = 128;                      // tokens per tile = MMA M
    static constexpr int BOX_ROWS = TC_BOX_ROWS;
    static constexpr int HALF_BYTES = TT * 128;         // one column block of a 16-bit K or V tile
    static constexpr int TILE_BYTES = TT * ROWB;        // a 16-bit tile
    // a ring stage holds one tile of K and one of V as they land: 16-bit tiles; for an fp8
    // cache 8-bit ones (TT rows of D bytes, 128-byte swizzled), whose V is widened into one of
    // two f16 working tiles (VW); for an int8 cache the K codes (128-byte swizzled, widened into
    // tensor memory) and a 16-bit V tile area whose back column block the V codes land in
    static constexpr bool Q8 = MODE_ == 3;
    static constexpr int KLAND = (FP8 || Q8) ? TT * D : TILE_BYTES;  // K area of a stage
    static constexpr int VAREA = FP8 ? TT * D : TILE_BYTES;          // V area of a stage
    static constexpr int STAGE_BYTES = KLAND + VAREA;
    static constexpr int VW_BYTES = FP8 ? 2 * TILE_BYTES : 0;
    static constexpr int OPB_BLOCK = N * 128;           // one column block of a K-major [N][128 B] operand
    static constexpr int OPB_BYTES = (FP8 ? 1 : HALVES) * OPB_BLOCK;
    // P operand of MMA2, P_hi and P_lo side by side as the N2 columns of one MMA:
    //  K-major (G <= 8): rows [0, NP) = P_hi, rows [NP, 2NP) = P_lo, in 64-token column blocks of
    //    PBLOCK bytes (a thread stores its token's weights one 16-bit value at a time);
    //  MN-major (G >= 16): one 128-byte row per token, P_hi at columns [0, NP) and P_lo at
    //    [32, 32 + NP) (a thread stores its token's weights in 16-byte vectors).
    // PBUF = one whole 128-token buffer.  (fp8 cache: P and the widened V are f16, else bf16.)
    static constexpr bool PMN = G >= 16;
    static constexpr int N2 = PMN ? 64 : 2 * NP;
    static constexpr int LOOFF = PMN ? 32 : NP;         // column of P_lo, and of O^T_lo
    static constexpr int PBLOCK = N2 * 128;
    static constexpr int PBUF = PMN ? TT * 128 : (TT / 64) * PBLOCK;
    static constexpr int HS = G < 8 ? G : 8;            // head slices for finish_segment
    static constexpr int MERGE_FLOATS = G * (D + 2);
    static constexpr int PREFIX_BYTES = 2 * (MAX_B + 1) * 4;  // prefix and uprefix (int32)
    static constexpr int RED_BYTES = 6 * N * 4;         // reductions [quadrant][N], rescale factors [2][N]
    // 4 tensor maps: K and V with 128-row boxes (full tiles) and 32-row boxes (partial tiles)
    static constexpr int MISC_BYTES = 512;              // mbarriers and flags
    static constexpr int ALIGN_PAD = 1024;
    static constexpr int BUDGET = 232448;               // opt-in maximum per CTA (227 KB)
    static constexpr int FIXED = OPB_BYTES + 2 * PBUF + VW_BYTES + MERGE_FLOATS * 4 + PREFIX_BYTES +
                                 RED_BYTES + MISC_BYTES + ALIGN_PAD;
    // Groups of 16+ heads on a contiguous or rolling cache keep K and V in separate rings of
    // 16-bit tiles: a K slot is refilled as soon as MMA1 has read it, a V slot once MMA2 has, so
    // the V loads get two tiles of lead where one joint ring (two stages fit) gives them one.
    static constexpr bool SPLIT = PMN && (MODE_ == 0 || MODE_ == 2);
    static constexpr int NSLOT = (BUDGET - FIXED) / TILE_BYTES;
    static constexpr int NV = SPLIT ? 2 : 0;                         // V slots
    static constexpr int NST_A = SPLIT ? NSLOT - NV : (BUDGET - FIXED) / STAGE_BYTES;
    static constexpr int NST = NST_A > 4 ? 4 : NST_A;                // stages (SPLIT: K slots)
    static constexpr int RING_BYTES = SPLIT ? (NST + NV) * TILE_BYTES : NST * STAGE_BYTES;
    static constexpr int SMEM = RING_BYTES + FIXED;
    // S^T buffers [0, N) and [N, 2N); O^T buffers (hi and lo columns) [2N, 2N + N2), [2N + N2, 2N + 2 N2)
    // int8 cache: two bf16 K tiles, MMA1's A operand (lane = token, 64 columns of 2 dims each),
    // at columns [KA_COL, KA_COL + 128)
    static constexpr int KA_COL = 128;
    static constexpr int TMEM_NEED = Q8 ? KA_COL + 128 : 2 * N + 2 * N2;
    static constexpr int TMEM_COLS = TMEM_NEED <= 32 ? 32 : (TMEM_NEED <= 64 ? 64 : (TMEM_NEED <= 128 ? 128 : 256));
    static_assert(NST >= 2, "ring too shallow");
    static_assert(!SPLIT || NST >= 3, "split rings: at least 3 K slots");
    static_assert(N % 16 == 0 && N <= 256, "MMA N");
    static_assert(HSPLIT == 1 || GH % 8 == 0, "head slices start on a swizzle row group");
    static_assert(!PMN || NP <= 32, "P_hi and P_lo share one 64-column row");
    static_assert(!FP8 || G <= 8, "fp8 cache: up to 8 query heads per KV head");
    static_assert(!Q8 || 2 * N + 2 * N2 <= KA_COL, "int8 cache: S^T and O^T below the K tiles");
    static_assert(OPB_BLOCK % 1024 == 0 && STAGE_BYTES % 1024 == 0, "swizzle atoms aligned");
};

// ---- tcgen05 descriptors
// Shared-memory matrix descriptor: start address, leading / stride byte offsets (>> 4), the
// descriptor version of this tensor-core generation (1), 128-byte swizzle layout (2).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}
// 8-bit caches with groups of up to 4 heads: one more warp, which issues MMA2 alone (the MMA warp
// then issues only MMA1; each tcgen05.mma holds its issuing thread ~90-110 cycles, and the two
// contractions plus their waits exceeded an 8-bit tile's time on one thread; from the producer
// thread, MMA2 delayed the next tile's copies)
template <int G, int MODE>
__host__ __device__ constexpr bool tc5_mma2_warp() {
    return (MODE == 3 || MODE == 4) && G <= 4;
}
// Threads of the kernel instantiation: a quantized cache adds the converter warps.
template <int G, int MODE>
__host__ __device__ constexpr int tc5_threads() {
    return Tc5Cfg<G, MODE>::NTHREADS + ((MODE == 3 || MODE == 4) ? Tc5Cfg<G, MODE>::NCONV * 32 : 0) +
           (tc5_mma2_warp<G, MODE>() ? 32 : 0);
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A/B major-ness (0 = K-major,
// 1 = MN-major), N >> 3, M >> 4.
__host__ __device__ constexpr uint32_t instr_desc_bf16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor with f16 A and B (format code 0; fp32 accumulator), and for kind::f8f6f4
// with E4M3 A and B (format code 0 there too; both K-major).
__host__ __device__ constexpr uint32_t instr_desc_f16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t instr_desc_e4m3(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void tc5_mma_f8(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc5_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
// A (M = 128 rows, K-major 16-bit) from tensor memory: row m in lane m, two K elements per column.
__device__ __forceinline__ void tc5_mma_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
// 16 consecutive 32-bit columns of this thread's tensor-memory lane (completion: tc5_wait_st).
__device__ __forceinline__ void tc5_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
        "%12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tc5_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void named_bar_arrive(int id, int n) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void tc5_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}
__device__ __forceinline__ void tc5_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc5_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 16 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tc5_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 8 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tc5_ld8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
// NC (8 or 16) consecutive columns.
template <int NC>
__device__ __forceinline__ void tc5_ld(uint32_t taddr, float (&v)[NC]) {
    if constexpr (NC == 8) tc5_ld8(taddr, v);
    else tc5_ld16(taddr, v);
}

// Issues one tile: a whole tile of a contiguous cache is one 3-D copy per tensor (maps tmKf /
// tmVf), a paged block one 4-D copy, a partial contiguous tile 32-row boxes per column block
// (tmK / tmV), rows past the stream's end being loaded and masked.
// 4-D tensor copy for a paged pool: the map views the pool's rows as (64 columns, 8 rows, 2
// column blocks, row groups of 8) with strides (2, 256, 128, 2048) bytes, so one box of `groups`
// row groups arrives as [group][column block][8 rows x 128 B]: 8-row swizzle atoms of the two
// column blocks interleaved (column-block stride 1024 B, group stride 2048 B).  `group` is the
// first row / 8 (block rows start at multiples of 16).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int group, int groups,
                                            uint64_t* bar, uint64_t policy) {
    (void)groups;  // fixed by the map's box
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::"
        "cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(0), "r"(0), "r"(group), "r"(smem_addr(bar)),
        "l"(policy)
        : "memory");
}
// 3-D tensor copy of a whole contiguous tile: the map views the cache as (64 columns, rows, 2
// column blocks) with byte strides (256, 128), so the box lands as [column block][row][128 B].
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int row, uint64_t* bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::"
        "cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(0), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}
// Shared-memory layout of a K / V tile: contiguous caches [column block][128 rows][128 B]
// (2-D copies); paged pools [8-row group][column block][8 rows][128 B] (4-D copies above).
template <class C, bool PAGED>
struct Tc5Layout {
    static constexpr uint32_t HSTR = PAGED ? 1024u : (uint32_t)C::HALF_BYTES;  // column-block stride
    static constexpr uint32_t GSTR = PAGED ? 2048u : 1024u;                    // 8-row group stride
};
// Paged cache: the tile's blocks are table[b][t / bs + i] for i < ceil(n / bs) (one block when
// bs >= 128).  The whole producer warp runs a paged tile: lane i looks up block i (ahead, so the
// lookup latency hides behind a stage wait) and issues its copies.
template <int TT>
__device__ __forceinline__ int tile_block(const DecodeParams& p, const TileCursor<TT>& c, int lane) {
    const int nb = p.bs >= TT ? 1 : (c.n() + p.bs - 1) / p.bs;
    return lane < nb ? __ldg(p.table + (size_t)c.it.b * p.max_blocks + c.t / p.bs + lane) : 0;
}
// Run by lane 0 of the producer warp (contiguous) or by the whole warp (paged, lane = block).
template <class C, int TT, int MODE>
__device__ __forceinline__ void issue_tile_tc5(const DecodeParams& p, const TileCursor<TT>& c,
                                               uint32_t ring, uint64_t* full_bar, int stage,
                                               uint64_t pol, const CUtensorMap* tmK,
                                               const CUtensorMap* tmV, const CUtensorMap* tmKf,
                                               const CUtensorMap* tmVf, int ent, int lane) {
    const int n = c.n();
    const size_t unit = (size_t)c.it.b * p.H_kv + c.it.h;
    const uint32_t ks = ring + stage * C::STAGE_BYTES;
    const uint32_t vs = ks + C::KLAND;
    constexpr bool PAGED = MODE == 1, QUANT = MODE == 3, FP8 = MODE == 4;
    constexpr bool paged = PAGED;
    const bool full = n == TT && !paged;
    const int rows = paged ? p.box_rows : (full ? TT : C::BOX_ROWS);
    const int nbox = full ? 1 : (n + rows - 1) / rows;
    // bf16 tiles: 2 x 128-byte column blocks per row; int8 and fp8 tiles: one row of D bytes
    const uint32_t kv_bytes = (uint32_t)(2 * nbox * rows * ((QUANT || FP8) ? C::D : C::HALVES * 128));
    if (lane == 0) mbar_arrive_expect_tx(&full_bar[stage], kv_bytes);
    if constexpr (PAGED) {
        {
            __syncwarp();  // the stage's expected bytes are registered before any copy lands
            // lane bx: box bx = block bx (or the 128-row piece of a larger block)
            if (lane < nbox) {
                int e = ent;
                if ((unsigned)e >= (unsigned)p.num_blocks) {
                    atomicOr(p.err, DEV_BAD_BLOCK);
                    e = 0;
                }
                const int tt = c.t + lane * rows;
                const int row = (int)(((int64_t)e * p.H_kv + c.it.h) * p.bs + tt % p.bs);
                // both column blocks in one copy: the 4-D map lands [8-row group][half][8 rows][128 B]
                const uint32_t off = (uint32_t)(lane * rows * C::ROWB);
                tma_load_4d(ks + off, tmK, row >> 3, rows >> 3, &full_bar[stage], pol);
                tma_load_4d(vs + off, tmV, row >> 3, rows >> 3, &full_bar[stage], pol);
            }
        }
    } else if (FP8) {
        // E4M3 rows (128 bytes, 128-byte swizzled) as they are: K is MMA1's operand, V is widened
        // by the converter warps
        const int row0 = (int)(unit * p.T_max + c.t);
        const CUtensorMap* mk = full ? tmKf : tmK;
        const CUtensorMap* mv = full ? tmVf : tmV;
        for (int bx = 0; bx < nbox; ++bx) {
            const uint32_t off = bx * C::BOX_ROWS * C::D;
            tma_load_2d(ks + off, mk, 0, row0 + bx * C::BOX_ROWS, &full_bar[stage], pol);
            tma_load_2d(vs + off, mv, 0, row0 + bx * C::BOX_ROWS, &full_bar[stage], pol);
        }
    } else if (QUANT) {
        // int8 rows (128 bytes): K's 128-byte swizzled into the K area (widened into tensor
        // memory later), V's unswizzled into the back column block of the V tile area (widened
        // in place later)
        const int row0 = (int)(unit * p.T_max + c.t);
        const CUtensorMap* mk = full ? tmKf : tmK;
        const CUtensorMap* mv = full ? tmVf : tmV;
        for (int bx = 0; bx < nbox; ++bx) {
            const uint32_t off = bx * C::BOX_ROWS * C::D;
            tma_load_2d(ks + off, mk, 0, row0 + bx * C::BOX_ROWS, &full_bar[stage], pol);
            tma_load_2d(vs + C::HALF_BYTES + off, mv, 0, row0 + bx * C::BOX_ROWS, &full_bar[stage], pol);
        }
    } else {
        const int row0 = (int)(unit * p.T_max + c.t);
        if (full) {
            // a whole tile: both column blocks in one 3-D copy per tensor
            tma_load_3d(ks, tmKf, row0, &full_bar[stage], pol);
            tma_load_3d(vs, tmVf, row0, &full_bar[stage], pol);
        } else {
#pragma unroll
            for (int hf = 0; hf < C::HALVES; ++hf)
                for (int bx = 0; bx < nbox; ++bx) {
                    const uint32_t off = hf * C::HALF_BYTES + bx * C::BOX_ROWS * 128;
                    tma_load_2d(ks + off, tmK, hf * 64, row0 + bx * C::BOX_ROWS, &full_bar[stage], pol);
                    tma_load_2d(vs + off, tmV, hf * 64, row0 + bx * C::BOX_ROWS, &full_bar[stage], pol);
                }
        }
    }
}

// Split rings: one tensor's tile (K or V, 16-bit, contiguous or rolling cache) into a 32 KB slot:
// a whole tile in one 3-D copy, a partial tile in 32-row 2-D boxes per column block.
template <class C, int TT>
__device__ __forceinline__ void issue_one_tc5(const DecodeParams& p, const TileCursor<TT>& c, uint32_t dst,
                                              uint64_t* bar, uint64_t pol, const CUtensorMap* tm,
                                              const CUtensorMap* tmf) {
    const int n = c.n();
    const bool full = n == TT;
    const int nbox = full ? 1 : (n + C::BOX_ROWS - 1) / C::BOX_ROWS;
    const int row0 = (int)(((size_t)c.it.b * p.H_kv + c.it.h) * p.T_max + c.t);
    mbar_arrive_expect_tx(bar, (uint32_t)(full ? C::TILE_BYTES : nbox * C::BOX_ROWS * C::ROWB));
    if (full) {
        tma_load_3d(dst, tmf, row0, bar, pol);
    } else {
#pragma unroll
        for (int hf = 0; hf < C::HALVES; ++hf)
            for (int bx = 0; bx < nbox; ++bx)
                tma_load_2d(dst + hf * C::HALF_BYTES + bx * C::BOX_ROWS * 128, tm, hf * 64, row0 + bx * C::BOX_ROWS,
                            bar, pol);
    }
}

// 16 int8 values -> 16 bf16, exactly, with full-rate integer and bf16x2 operations: for the
// byte x = l - 128 s (l its low 7 bits, s its sign bit), the bf16 with bits 0x43:l is 128 + l and
// the one with bits 0x43:(s << 7) is 128 + 128 s; their difference is x, exactly representable.
__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ void widen_i8x16(const uint4& v, uint4& o0, uint4& o1) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t r[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t lo = w[j] & 0x7F7F7F7Fu, hi = w[j] & 0x80808080u;
        r[2 * j] = bf16x2_sub(__byte_perm(lo, 0x43434343u, 0x4140), __byte_perm(hi, 0x43434343u, 0x4140));
        r[2 * j + 1] = bf16x2_sub(__byte_perm(lo, 0x43434343u, 0x4342), __byte_perm(hi, 0x43434343u, 0x4342));
    }
    o0 = make_uint4(r[0], r[1], r[2], r[3]);
    o1 = make_uint4(r[4], r[5], r[6], r[7]);
}

// Named barrier BAR of NT threads with an OR reduction of a predicate.
template <int BAR, int NT>
__device__ __forceinline__ bool group_any(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "n"(BAR), "n"(NT)
        : "memory");
    return r != 0;
}

// Warp roles: warp 0 issues the tensor copies (producer) and MMA2 (for a paged pool with
// m2p = 0, warp 1 does; for an 8-bit cache with G <= 4, a warp of its own), warp 1 issues MMA1
// and loads q, warps 2 .. 2+NW-1 run the softmax, write P and accumulate O (thread <->
// tensor-memory lane 32*(warp%4) + lane), the next NEPI warps finish segments (output or
// partial state, and the merge of a stream whose last segment this CTA completes) while the
// next segment streams; the CTA's last segment is finished by the epilogue and softmax warps
// together.  8-bit caches add NCONV converter warps after those, then the MMA2 warp if any.
// Double buffers: S^T and O^T in tensor memory, P in shared memory; MMA1 of tile k+1 runs while
// the softmax warps work on tile k, and O^T(k-1) is folded in after the softmax of tile k.
// Slot of a stream's new row in the fused step (the row a preceding append may just have
// written): the last row, or for a rolling cache of W = T_max slots, (lens[b] - 1) mod W.  The
// rolling slot comes from lens[b] (one load per stream, kept while the cursor stays on it).
template <bool ROLL>
struct NewRow {
    int b = -1, slot = 0;
    // does tile [t, t + n) hold a new row (one of the last T_q rows, or the rolling slot)?
    __device__ __forceinline__ bool in_tile(const DecodeParams& p, int sb, int L, int t, int n) {
        if constexpr (!ROLL) {
            (void)sb;
            return t + n > L - p.T_q;
        } else {
            if (sb != b) {
                b = sb;
                slot = (__ldg(p.lens + sb) - 1) % p.T_max;
            }
            return t <= slot && slot < t + n;
        }
    }
};

// MODE: 0 contiguous cache, 1 paged pool (block table), 2 rolling cache (T_max = window slots,
// position p in slot p mod T_max; lens may exceed T_max and the attention covers
// min(lens, T_max) slots), 3 int8 cache with per-row scales (tiles arrive as int8 in the back
// half of the stage's tile area and are widened in place to bf16 by the converter warps; the
// row scales multiply the scores and the weights).  Each mode is its own instantiation.
template <int G, int MODE>
__global__ void __launch_bounds__(tc5_threads<G, MODE>(), 1)
    decode_tc5_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmKf,
                      const __grid_constant__ CUtensorMap tmVf) {
    using C = Tc5Cfg<G, MODE>;
    using T = __nv_bfloat16;
    constexpr bool PAGED = MODE == 1, ROLL = MODE == 2, QUANT = MODE == 3, FP8 = MODE == 4;
    constexpr bool SCALED = QUANT || FP8;  // rows carry fp32 scales (K: scores, V: weights)
    constexpr bool DED2 = tc5_mma2_warp<G, MODE>();  // a warp of its own issues MMA2
    constexpr int D = C::D, N = C::N, NP = C::NP, TT = C::TT, NST = C::NST, TS = TT / 16;
    constexpr int KS = FP8 ? D / 32 : D / 16;  // MMA1 k-steps of 32 bytes
    using Cur = TileCursor<TT>;

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* ring = smem;
    unsigned char* vw = ring + C::RING_BYTES;                 // fp8 cache: f16 V working tiles [2]
    unsigned char* qsw = ring + C::RING_BYTES + C::VW_BYTES;  // q, [N][D] K-major swizzled
    // split rings (groups of 16+): K slots [0, NST), then V slots [NST, NST + NV), one tile each
    unsigned char* vring = ring + NST * C::TILE_BYTES;
    unsigned char* pbuf = qsw + C::OPB_BYTES;                 // [2 buffers][2 blocks][2N rows][128 B]
    float* merge = reinterpret_cast<float*>(pbuf + 2 * C::PBUF);
    int32_t* prefix = reinterpret_cast<int32_t*>(merge + C::MERGE_FLOATS);
    int32_t* uprefix = prefix + MAX_B + 1;
    float* red = reinterpret_cast<float*>(uprefix + MAX_B + 1);  // [4][N]
    float* alpha_s = red + 4 * N;                                  // [2][N]: rescale factor of a tile
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(red + 6 * N);
    uint64_t* empty_bar = full_bar + NST;
    uint64_t* s_full = empty_bar + NST;   // [2]
    uint64_t* s_empty = s_full + 2;
    uint64_t* p_full = s_empty + 2;
    uint64_t* o_full = p_full + 2;
    uint64_t* o_empty = o_full + 2;
    uint64_t* m_full = o_empty + 2;       // merge buffer written (softmax warps -> epilogue warps)
    uint64_t* m_empty = m_full + 1;       // merge buffer consumed
    int* issued = reinterpret_cast<int*>(m_empty + 1);       // [NST]
    volatile int* abort_flag = issued + NST;
    int* last_flag = issued + NST + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(issued + NST + 2);
    int* mma_issued = issued + NST + 3;                      // MMA2 commits issued (abort drain)
    int* mma1_issued = issued + NST + 4;                     // MMA1 commits issued (abort drain)
    // (append_bar follows at the next 8-byte boundary)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = p.B, H_kv = p.H_kv;
    const size_t row_elems_q = (size_t)H_kv * G * D;
    uint64_t* append_bar = reinterpret_cast<uint64_t*>(
        (reinterpret_cast<uintptr_t>(mma1_issued + 1) + 7) & ~uintptr_t(7));
    uint64_t* conv_full = append_bar + 1;  // [NST] int8 cache: the stage's tiles are bf16 now
    uint64_t* vw_full = conv_full + NST;   // [2] fp8 cache: V working tile written (converters)
    uint64_t* vw_empty = vw_full + 2;      // [2] fp8 cache: V working tile read (MMA2 commit)
    uint64_t* sv_full = vw_empty + 2;      // [NV] split rings: V slot landed
    uint64_t* sv_empty = sv_full + 2;      // [NV] split rings: V slot read by MMA2
    int* vissued = reinterpret_cast<int*>(sv_empty + 2);  // [NV] V copies issued per slot (abort drain)
    uint64_t* ka_empty = reinterpret_cast<uint64_t*>(vissued + 2);  // [2] int8: K tile read (MMA1 commit)

    // Programmatic dependent launch: the next kernel on the stream may be scheduled now (its
    // CTAs take SMs as ours exit) but waits in griddepcontrol.wait until this grid is complete.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (tid == 32) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full_bar[s], 1);
            // a stage is free once MMA2 has read it; fp8: once MMA1 has read K and the converters V
            mbar_init(&empty_bar[s], FP8 ? 2 : 1);
            issued[s] = 0;
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], C::NW);
            mbar_init(&p_full[i], C::NW);
            mbar_init(&o_full[i], 1);
            mbar_init(&o_empty[i], C::NW);
        }
        mbar_init(m_full, C::NW * 32);
        mbar_init(m_empty, C::NEPI * 32);
        mbar_init(append_bar, 1);
        if constexpr (QUANT) {
            for (int s = 0; s < NST; ++s) mbar_init(&conv_full[s], C::NCONV * 32);
            for (int i = 0; i < 2; ++i) mbar_init(&ka_empty[i], 1);
        }
        if constexpr (FP8)
            for (int i = 0; i < 2; ++i) {
                mbar_init(&vw_full[i], C::NCONV * 32);
                mbar_init(&vw_empty[i], 1);
            }
        if constexpr (C::SPLIT)
            for (int i = 0; i < C::NV; ++i) {
                mbar_init(&sv_full[i], 1);
                mbar_init(&sv_empty[i], 1);
                vissued[i] = 0;
            }
        *abort_flag = 0;
        *last_flag = 0;
        *mma_issued = 0;
        *mma1_issued = 0;
        fence_mbar_init();
    }
    if (tid == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmK)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmV)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmKf)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmVf)) : "memory");
    }
    // With overlap, lens and the history rows below each stream's last row are read before the
    // preceding grid on the stream has finished (the caller guarantees it does not write them);
    // everything else waits for it.
    const bool early = p.overlap != 0;
    if (!early) asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == 0) scan_lengths(p, ROLL ? 1 : 0, prefix, uprefix, lane);
    __syncthreads();

    const int64_t W = (int64_t)H_kv * prefix[B], U = (int64_t)H_kv * uprefix[B];
    const int64_t P = W > 0 ? plan_ctas(W, U, p.P, p.min_tokens) : 0;
    const int64_t r0 = W > 0 ? cta_cut(blockIdx.x, prefix, uprefix, B, H_kv, U, P, p.grain) : 0;
    const int64_t r1 = W > 0 ? cta_cut(blockIdx.x + 1, prefix, uprefix, B, H_kv, U, P, p.grain) : 0;
    const bool work = W > 0 && (int64_t)blockIdx.x < P && r0 < r1;
    const uint32_t ring_s = smem_addr(ring);
    const uint64_t pol = policy_evict_first();
    constexpr bool paged = PAGED;  // paged pool through the block table (separate instantiation)
    Cur pref;  // producer's cursor (thread 0; the whole warp 0 when paged)
    NewRow<ROLL> nrow;    // producer: where the stream's new row is
    int ent = 0;          // paged: this lane's block of the tile at pref
    int npre = 0;         // tiles whose K/V copies started before the grid dependency wait
    // How many: copies in flight at the grid wait delay its release (measured with a plain
    // kernel chain: 0.9 us with none, 2.2 us with 192 KB per CTA in flight), while the early
    // tiles save their load latency.  Small layers gain from one (Llama-2-7B MHA, ~7 tiles per
    // CTA: 17.0 against 17.7 us per layer with a full ring), long ones from a full ring (8B GQA,
    // ~48 tiles per CTA: 71.4 against 72.6 with one): a quarter of the CTA's tiles, 1 to NST.
    const int64_t tiles_per_cta = P > 0 ? (U / P) * p.grain / TT : 0;
    const int emax = tiles_per_cta / 4 < 1 ? 1 : (tiles_per_cta / 4 > NST ? NST : (int)(tiles_per_cta / 4));
    if (work && (PAGED ? warp == 0 : tid == 0)) {
        pref.init(prefix, B, H_kv, r0, r1);
        if (early)
            while (pref.valid && npre < emax && !nrow.in_tile(p, pref.it.b, pref.it.L, pref.t, pref.n())) {
                if constexpr (PAGED) ent = tile_block<TT>(p, pref, lane);
                if constexpr (C::SPLIT) {
                    issued[npre] += 1;
                    issue_one_tc5<C, TT>(p, pref, ring_s + npre * C::TILE_BYTES, &full_bar[npre], pol, &tmK, &tmKf);
                    if (npre < C::NV) {
                        vissued[npre] += 1;
                        issue_one_tc5<C, TT>(p, pref, smem_addr(vring) + npre * C::TILE_BYTES, &sv_full[npre], pol,
                                             &tmV, &tmVf);
                    }
                } else {
                    if (lane == 0) issued[npre] += 1;
                    issue_tile_tc5<C, TT, MODE>(p, pref, ring_s, full_bar, npre, pol, &tmK, &tmV, &tmKf, &tmVf, ent,
                                                 lane);
                }
                pref.advance();
                ++npre;
            }
    }
    if (early) asm volatile("griddepcontrol.wait;" ::: "memory");

    for (int b = blockIdx.x; b < B; b += gridDim.x) {
        if (prefix[b + 1] == prefix[b]) {
            if (tid == 0) atomicOr(p.err, DEV_BAD_LENS);
            for (size_t i = tid; i < row_elems_q; i += blockDim.x)
                Elem<T>::store(p.out, (size_t)b * row_elems_q + i, 0.f);
        }
    }
    if (!work) return;
    const bool fused = p.k_new != nullptr;
    uint32_t tmem = 0;
    // The CTA's last segment is finished (output, partial state, and the stream's merge when
    // this CTA is the last of it) by the epilogue and the softmax warps together (named
    // barrier 5): nothing else is left to overlap it with.  Both groups always arrive; the
    // work is skipped by all of them if any member gave up on a wait.
    constexpr int NJ = C::NEPI + C::NW;
    auto final_segment = [&](bool ok, const SegIter& it, int jt) {
        const bool skip = group_any<5, NJ * 32>(!ok || *abort_flag != 0);
        if (!skip)
            finish_segment<T, G, D, C::HS, 1, NJ, 5>(p, merge, it, (size_t)it.b * H_kv + it.h, U, P,
                                                     last_flag, jt);
    };

    // MMA2(k): O^T[k&1] = V(stage st)^T . (P_hi + P_lo)^T, then its commits (run by one thread:
    // the producer's, or for a paged pool with m2p = 0 the MMA warp's: a producer warp that
    // issues one copy per block can be the slower of the two)
    // (fp8: the MMA warp issues MMA2 as well, one tile behind MMA1; a stage is free once MMA1
    // has read K and the converters V, and the producer thread only refills the ring: a tensor
    // copy can hold its issuing thread for hundreds of cycles, so no MMA waits behind one)
    const bool m2p = !FP8 && !DED2 && (!PAGED || p.m2p != 0);
    // V read MN-major x P; an fp8 cache's widened V and its weights are f16
    constexpr uint32_t IDESC2 = FP8 ? instr_desc_f16(128, C::N2, 1, C::PMN ? 1 : 0)
                                    : instr_desc_bf16(128, C::N2, 1, C::PMN ? 1 : 0);
    using LY = Tc5Layout<C, PAGED>;
    const uint32_t vw_s = smem_addr(vw);
    auto issue_mma2 = [&](int k, int st, uint32_t tm) {
        // V: the stage's tile, or (fp8) the f16 working tile k & 1
        const uint64_t dV0 = smem_desc_sw128(FP8 ? vw_s : (C::SPLIT ? smem_addr(vring) : ring_s + C::KLAND),
                                             LY::HSTR, LY::GSTR);
        // P: K-major rows of 64 tokens, or MN-major token rows (one 64-column pattern; the
        // leading offset is never stepped over)
        const uint32_t pbuf_s = smem_addr(pbuf);
        const uint64_t dP0 = C::PMN ? smem_desc_sw128(pbuf_s, (uint32_t)C::PBUF, 1024u)
                                    : smem_desc_sw128(pbuf_s, 16u, 1024u);
        const uint32_t tO = tm + (uint32_t)(2 * N + (k & 1) * C::N2);
        const uint32_t pb = (uint32_t)((k & 1) * C::PBUF);
#pragma unroll
        for (int kk = 0; kk < TS; ++kk) {
            const uint32_t voff = (uint32_t)((FP8 ? (k & 1) * C::TILE_BYTES
                                                  : C::SPLIT ? (k % C::NV) * C::TILE_BYTES : st * C::STAGE_BYTES) +
                                             kk * 2 * LY::GSTR);
            const uint32_t poff = C::PMN ? pb + (uint32_t)(kk * 2048)
                                         : pb + (uint32_t)((kk >> 2) * C::PBLOCK + (kk & 3) * 32);
            tc5_mma(tO, dV0 + (voff >> 4), dP0 + (poff >> 4), IDESC2, kk > 0 ? 1u : 0u);
        }
        tc5_commit(&o_full[k & 1]);
        if constexpr (FP8)
            tc5_commit(&vw_empty[k & 1]);  // the working tile is free (the stage was freed earlier)
        else if constexpr (C::SPLIT)
            tc5_commit(&sv_empty[k % C::NV]);  // the V slot is consumed (MMA1 freed the K slot)
        else
            tc5_commit(&empty_bar[st]);  // K/V of the stage are consumed
        *mma_issued += 1;
    };

    if (warp == 0) {
        // ======================================================= producer
        if (PAGED || lane == 0) {
            if constexpr (PAGED) if (pref.valid) ent = tile_block<TT>(p, pref, lane);
            // a tile that holds a stream's new token waits for the fused append's writes (lane 0
            // waits; the warp follows its verdict: paged, every lane issues a block)
            auto append_ready = [&]() {
                bool ok = true;
                if (lane == 0 && fused && nrow.in_tile(p, pref.it.b, pref.it.L, pref.t, pref.n()))
                    ok = mbar_wait(append_bar, 0u, abort_flag, p.err);
                if constexpr (PAGED) ok = __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;
                return ok;
            };
            auto issue_next = [&](int st) {
                if (lane == 0) issued[st] += 1;
                issue_tile_tc5<C, TT, MODE>(p, pref, ring_s, full_bar, st, pol, &tmK, &tmV, &tmKf, &tmVf, ent,
                                             lane);
                pref.advance();
                // the next tile's blocks load while lane 0 waits
                if constexpr (PAGED) if (pref.valid) ent = tile_block<TT>(p, pref, lane);
            };
            bool ok = true;
            if constexpr (C::SPLIT) {
                // K slots: tile k in slot k % NST, refilled with tile k + NST once MMA1(k) has read
                // it; V slots: tile k in slot k % NV, refilled with tile k + NV once MMA2(k) has.
                // This thread issues MMA2 (its V wait included) between the two refills.
                auto ready = [&](const Cur& c) {
                    return !(fused && nrow.in_tile(p, c.it.b, c.it.L, c.t, c.n())) ||
                           mbar_wait(append_bar, 0u, abort_flag, p.err);
                };
                Cur vp;  // V cursor
                vp.init(prefix, B, H_kv, r0, r1);
                const int nvpre = npre < C::NV ? npre : C::NV;
                for (int i = 0; i < nvpre && vp.valid; ++i) vp.advance();
                for (int st = npre; st < NST && pref.valid && ok; ++st) {
                    ok = ready(pref);
                    if (!ok) break;
                    issued[st] += 1;
                    issue_one_tc5<C, TT>(p, pref, ring_s + st * C::TILE_BYTES, &full_bar[st], pol, &tmK, &tmKf);
                    pref.advance();
                }
                for (int sv = nvpre; sv < C::NV && vp.valid && ok; ++sv) {
                    ok = ready(vp);
                    if (!ok) break;
                    vissued[sv] += 1;
                    issue_one_tc5<C, TT>(p, vp, smem_addr(vring) + sv * C::TILE_BYTES, &sv_full[sv], pol, &tmV, &tmVf);
                    vp.advance();
                }
                Cur mc;
                mc.init(prefix, B, H_kv, r0, r1);
                for (int k = 0; ok && mc.valid; ++k) {
                    const int sk = k % NST, sv = k % C::NV;
                    if (pref.valid) {
                        ok = mbar_wait(&empty_bar[sk], (uint32_t)((k / NST) & 1), abort_flag, p.err) && ready(pref);
                        if (ok) {
                            issued[sk] += 1;
                            issue_one_tc5<C, TT>(p, pref, ring_s + sk * C::TILE_BYTES, &full_bar[sk], pol, &tmK, &tmKf);
                            pref.advance();
                        }
                    }
                    ok = ok && mbar_wait(&p_full[k & 1], (k >> 1) & 1, abort_flag, p.err) &&
                         mbar_wait(&o_empty[k & 1], ((k >> 1) & 1) ^ 1u, abort_flag, p.err) &&
                         mbar_wait(&sv_full[sv], (uint32_t)((k / C::NV) & 1), abort_flag, p.err);
                    if (ok) {
                        tc5_fence_after();
                        if (k == 0) tmem = *tmem_slot;
                        issue_mma2(k, sk, tmem);
                    }
                    if (ok && vp.valid) {
                        ok = mbar_wait(&sv_empty[sv], (uint32_t)((k / C::NV) & 1), abort_flag, p.err) && ready(vp);
                        if (ok) {
                            vissued[sv] += 1;
                            issue_one_tc5<C, TT>(p, vp, smem_addr(vring) + sv * C::TILE_BYTES, &sv_full[sv], pol,
                                                 &tmV, &tmVf);
                            vp.advance();
                        }
                    }
                    mc.advance();
                }
            } else {
            // the rest of the ring's first pass: those stages are free
            for (int st = npre; st < NST && pref.valid; ++st) {
                ok = append_ready();
                if (!ok) break;
                issue_next(st);
            }
            if (m2p) {
                // MMA2 of each tile (this thread issues it: MMA1 is warp 1's), then the tile NST
                // ahead into the stage that MMA2 frees.  Issued here so that MMA1 of the next tile
                // never queues behind it in one thread (each tcgen05.mma takes ~90 cycles to issue).
                Cur mc;
                mc.init(prefix, B, H_kv, r0, r1);
                int s2 = 0;
                for (int k = 0; ok && mc.valid; ++k) {
                    if (lane == 0) {
                        ok = mbar_wait(&p_full[k & 1], (k >> 1) & 1, abort_flag, p.err) &&
                             mbar_wait(&o_empty[k & 1], ((k >> 1) & 1) ^ 1u, abort_flag, p.err);
                        if (FP8 && ok) ok = mbar_wait(&vw_full[k & 1], (k >> 1) & 1, abort_flag, p.err);
                        if (ok) {
                            tc5_fence_after();
                            // written by warp 1's allocation before the weights of tile 0 existed
                            if (k == 0) tmem = *tmem_slot;
                            issue_mma2(k, s2, tmem);
                        }
                    }
                    if constexpr (PAGED) ok = __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;
                    if (!FP8 && ok && pref.valid) {
                        // tile k + NST goes into stage s2 once MMA2(k) has read it
                        if (lane == 0) ok = mbar_wait(&empty_bar[s2], (uint32_t)((k / NST) & 1), abort_flag, p.err);
                        if constexpr (PAGED) ok = __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;
                        if (ok) ok = append_ready();
                        if (ok) issue_next(s2);
                    }
                    mc.advance();
                    if (++s2 == NST) s2 = 0;
                }
            } else {
                // each further tile into the next stage once it is free (MMA2 has read it; fp8: MMA1
                // has read K and the converters V)
                int s = 0;
                uint32_t ph = 1u;
                while (ok && pref.valid) {
                    if (lane == 0) ok = mbar_wait(&empty_bar[s], ph ^ 1u, abort_flag, p.err);
                    if constexpr (PAGED) ok = __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;  // (else lane 0 alone)
                    if (ok) ok = append_ready();
                    if (ok) issue_next(s);
                    if (++s == NST) { s = 0; ph ^= 1u; }
                }
            }
            }
        }
    } else if (warp == 1) {
        // ======================================================= MMA1 issue
        // Allocates tensor memory: S^T buffers at columns [0, N) and [N, 2N); O^T at
        // [2N, 2N + N2) and [2N + N2, 2N + 2 N2).  MMA1 of each tile is issued as soon as its K
        // tile and an S^T buffer are free; MMA2 is issued by the producer thread.  Each commits
        // its own MMAs (a commit tracks the issuing thread's operations); MMA1 of a tile has
        // completed before its MMA2 is issued (S^T -> softmax -> P), so MMA2's commit of the
        // stage's empty barrier covers both reads of the stage.
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "r"(C::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        if constexpr (QUANT) {
            // the converter warps write K tiles into tensor memory: the allocation is theirs to read
            tc5_fence_before();
            named_bar_arrive(6, 32 + C::NCONV * 32);
        }
        // Each segment's q rows (G rows of D bf16 at row unit * G of q) go into the swizzled
        // operand from registers, loaded one segment ahead and stored once the previous
        // segment's last MMA1 has read the operand.
        Cur cur;
        cur.init(prefix, B, H_kv, r0, r1);
        constexpr int QV = G * (D / 8), QPL = (QV + 31) / 32;
        uint4 qv[QPL];
        auto q_load = [&](const SegIter& it) {
            const uint4* src = reinterpret_cast<const uint4*>(p.q) + ((size_t)it.b * H_kv + it.h) * QV;
#pragma unroll
            for (int i = 0; i < QPL; ++i)
                if (lane + 32 * i < QV) qv[i] = __ldcg(src + lane + 32 * i);
        };
        auto q_store = [&]() {
#pragma unroll
            for (int i = 0; i < QPL; ++i) {
                const int c = lane + 32 * i;
                if constexpr (FP8) {
                    // a head's 16 chunks sit on 16 consecutive lanes of one slot: its largest |q| by a
                    // half-warp reduction, then 2^-e q as three E4M3 terms in rows t G + h (one
                    // 128-byte row per head and term, 8 bytes per chunk)
                    const uint4 w = c < QV ? qv[i] : make_uint4(0u, 0u, 0u, 0u);
                    float f[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                                  bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
                    float amax = 0.f;
#pragma unroll
                    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
#pragma unroll
                    for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, off));
                    const float sc = exp2i(-f8_head_exp(amax));
#pragma unroll
                    for (int j = 0; j < 8; ++j) f[j] *= sc;
                    uint2 t[3];
                    e4m3_split3(f, t[0], t[1], t[2]);
                    if (c < QV) {
                        const int h = c / (D / 8), cc = c % (D / 8);
#pragma unroll
                        for (int tt = 0; tt < 3; ++tt) {
                            const int r = tt * G + h;
                            *reinterpret_cast<uint2*>(qsw + r * 128 + (((cc >> 1) ^ (r & 7)) << 4) + (cc & 1) * 8) = t[tt];
                        }
                    }
                } else if (c < QV) {
                    const int h = c / (D / 8), cc = c % (D / 8);
                    *reinterpret_cast<uint4*>(qsw + (cc >> 3) * C::OPB_BLOCK + h * 128 + (((cc & 7) ^ (h & 7)) << 4)) =
                        qv[i];
                }
            }
        };
        if (cur.valid) q_load(cur.it);
        tc5_fence_before();
        named_bar_sync(2, 32 + C::NW * 32);
        tc5_fence_after();
        tmem = *tmem_slot;
        // K (K-major) x q (K-major): bf16, or E4M3 codes and terms (kind::f8f6f4)
        constexpr uint32_t IDESC1 = FP8 ? instr_desc_e4m3(128, N) : instr_desc_bf16(128, N, 0, 0);
        const uint32_t qsw_s = smem_addr(qsw);
        using LY = Tc5Layout<C, PAGED>;
        int s = 0;
        uint32_t ph = 0;
        bool alive = true;
        const uint64_t dK0 = smem_desc_sw128(ring_s, 16u, LY::GSTR);  // + stage, block, k-step
        const uint64_t dQ0 = smem_desc_sw128(qsw_s, 16u, 1024u);
        int s_prev = 0;
        // MMA2 of tile j from this warp (the m2p = 0 orders below)
        auto mma2_here = [&](int j) {
            alive = mbar_wait(&p_full[j & 1], (j >> 1) & 1, abort_flag, p.err) &&
                    mbar_wait(&o_empty[j & 1], ((j >> 1) & 1) ^ 1u, abort_flag, p.err);
            if (FP8 && alive) alive = mbar_wait(&vw_full[j & 1], (j >> 1) & 1, abort_flag, p.err);
            if (alive && lane == 0) {
                tc5_fence_after();
                issue_mma2(j, s_prev, tmem);
            }
            __syncwarp();
        };
        for (int k = 0;; ++k) {
            if (!m2p && !FP8 && !DED2) {
                // MMA2 of the previous tile here, first (it frees a ring stage as soon as the
                // weights are written)
                if (k > 0 && alive) mma2_here(k - 1);
            }
            if (FP8 && !cur.valid) {
                // the last tile's MMA2 (MMA1 runs one tile ahead of MMA2 here)
                if (!DED2 && k > 0 && alive) mma2_here(k - 1);
                break;
            }
            if (!cur.valid || !alive) break;
            // ---- MMA1(k): S^T[k&1] = K(stage s) . Q^T
            // int8 cache: wait until the converter warps have widened K into tensor memory and V
            // in place
            alive = mbar_wait(QUANT ? &conv_full[s] : &full_bar[s], ph, abort_flag, p.err);
            // (fp8: the K codes are read as they landed)
            if (alive && cur.first()) {
                // the previous MMA1 read q_sw: let it finish before q is replaced
                if (k > 0) alive = mbar_wait(&s_full[(k - 1) & 1], ((k - 1) >> 1) & 1, abort_flag, p.err);
                q_store();
                fence_async_smem();
                __syncwarp();
                SegIter nx = cur.it;
                nx.next();
                if (nx.valid) q_load(nx);
            }
            if (alive) alive = mbar_wait(&s_empty[k & 1], ((k >> 1) & 1) ^ 1u, abort_flag, p.err);
            if (alive && lane == 0) {
                tc5_fence_after();
                const uint32_t tS = tmem + (uint32_t)((k & 1) * N);
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    if constexpr (FP8) {
                        // one 128-byte column block: k-steps of 32 codes
                        const uint32_t off = (uint32_t)(s * C::STAGE_BYTES + kk * 32);
                        tc5_mma_f8(tS, dK0 + (off >> 4), dQ0 + ((uint32_t)(kk * 32) >> 4), IDESC1, kk > 0 ? 1u : 0u);
                    } else if constexpr (QUANT) {
                        // K tile k & 1 in tensor memory: k-step kk is columns 8 kk .. 8 kk + 7
                        const uint32_t qoff = (uint32_t)((kk >> 2) * C::OPB_BLOCK + (kk & 3) * 32);
                        tc5_mma_ta(tS, tmem + (uint32_t)(C::KA_COL + (k & 1) * 64 + kk * 8), dQ0 + (qoff >> 4),
                                   IDESC1, kk > 0 ? 1u : 0u);
                    } else {
                        // (split rings: K slots of one tile each)
                        const uint32_t off = (uint32_t)(s * (C::SPLIT ? C::TILE_BYTES : C::STAGE_BYTES) +
                                                        (kk >> 2) * LY::HSTR + (kk & 3) * 32);
                        const uint32_t qoff = (uint32_t)((kk >> 2) * C::OPB_BLOCK + (kk & 3) * 32);
                        tc5_mma(tS, dK0 + (off >> 4), dQ0 + (qoff >> 4), IDESC1, kk > 0 ? 1u : 0u);
                    }
                }
                tc5_commit(&s_full[k & 1]);
                if constexpr (FP8) tc5_commit(&empty_bar[s]);  // K read (the converters arrive for V)
                if constexpr (QUANT) tc5_commit(&ka_empty[k & 1]);  // the K tile in tensor memory is read
                if constexpr (C::SPLIT) tc5_commit(&empty_bar[s]);  // split rings: the K slot is free
                *mma1_issued += 1;
            }
            __syncwarp();
            // fp8: MMA2 of the previous tile after MMA1 of this one, so the scores run a tile ahead
            // of the weights (MMA1 of a tile is four instructions; the stage does not wait for MMA2)
            if (FP8 && !DED2 && k > 0 && alive) mma2_here(k - 1);
            s_prev = s;
            cur.advance();
            if (++s == NST) { s = 0; ph ^= 1u; }
        }
    } else if (DED2 && warp == 2 + C::NW + C::NEPI + C::NCONV) {
        // ======================================================= MMA2 issue (8-bit caches, groups <= 4)
        // MMA2 of each tile once its weights and its O^T buffer are ready, and for fp8 its f16 V
        // working tile (int8: the stage's V was widened before MMA1 of the tile; lane 0 issues,
        // the warp follows its verdict)
        Cur mc;
        mc.init(prefix, B, H_kv, r0, r1);
        bool ok = true;
        int s2 = 0;
        for (int k = 0; ok && mc.valid; ++k) {
            if (lane == 0) {
                ok = mbar_wait(&p_full[k & 1], (k >> 1) & 1, abort_flag, p.err) &&
                     mbar_wait(&o_empty[k & 1], ((k >> 1) & 1) ^ 1u, abort_flag, p.err) &&
                     (!FP8 || mbar_wait(&vw_full[k & 1], (k >> 1) & 1, abort_flag, p.err));
                if (ok) {
                    tc5_fence_after();
                    // written by warp 1's allocation before the weights of tile 0 existed
                    if (k == 0) tmem = *tmem_slot;
                    issue_mma2(k, s2, tmem);
                }
            }
            ok = __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;
            mc.advance();
            if (++s2 == NST) s2 = 0;
        }
    } else if (FP8 && warp >= 2 + C::NW + C::NEPI) {
        // ======================================================= E4M3 V -> f16 converters
        // Per tile, in order: wait for the copies and for working tile k & 1 to be free (MMA2 of
        // tile k - 2 has read it); widen the V codes (128-byte swizzled rows) into it, in the
        // 128-byte-swizzled MN-major layout MMA2 reads ([column block][row][128 B]); rows past
        // the loaded boxes become zeros (they meet weight 0, and stale bytes could be NaN codes).
        // Then publish the working tile to the tensor cores and hand the stage's V back (MMA1's
        // commit hands back K).
        const int ct = tid - (2 + C::NW + C::NEPI) * 32;  // 0 .. NCONV * 32 - 1
        Cur cc;
        cc.init(prefix, B, H_kv, r0, r1);
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int k = 0; cc.valid; ++k) {
            const int w = k & 1;
            ok = ok && mbar_wait(&full_bar[s], ph, abort_flag, p.err);
            ok = ok && mbar_wait(&vw_empty[w], ((k >> 1) & 1) ^ 1u, abort_flag, p.err);
            if (ok) {
                const int n = cc.n();
                const int loaded = n == TT ? TT : ((n + C::BOX_ROWS - 1) / C::BOX_ROWS) * C::BOX_ROWS;
                const unsigned char* vl = ring + s * C::STAGE_BYTES + C::KLAND;
                unsigned char* vt = vw + w * C::TILE_BYTES;
                // unit = (row r, 16-code column group c) -> 32 bytes of f16 (two 16-byte chunks).
                // The 8 lanes of a quarter warp take one c and 8 consecutive rows, so their loads
                // and stores hit 8 different swizzled chunks (no bank conflicts); each thread loads
                // all of its units before converting any.
                constexpr int PER = TT * 8 / (C::NCONV * 32);  // units per thread (8)
                uint4 v[PER];
#pragma unroll
                for (int i = 0; i < PER; ++i) {
                    const int u = ct + i * C::NCONV * 32;
                    const int r = ((u >> 6) << 3) | (u & 7), c = (u >> 3) & 7;
                    v[i] = r < loaded ? *reinterpret_cast<const uint4*>(vl + r * 128 + ((c ^ (r & 7)) << 4))
                                      : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int i = 0; i < PER; ++i) {
                    const int u = ct + i * C::NCONV * 32;
                    const int r = ((u >> 6) << 3) | (u & 7), c = (u >> 3) & 7;
                    // two codes per conversion (E4M3 -> f16 is exact; a zero code gives +0)
                    const uint32_t x[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
                    uint32_t h[8];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
                            "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
                            : "=r"(h[2 * j]), "=r"(h[2 * j + 1])
                            : "r"(x[j]));
                    }
                    // f16 columns [16c, 16c + 16): column block c / 4, chunks 2 (c % 4) and + 1
                    unsigned char* row = vt + (c >> 2) * C::HALF_BYTES + r * 128;
                    const int cb = 2 * (c & 3);
                    *reinterpret_cast<uint4*>(row + ((cb ^ (r & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
                    *reinterpret_cast<uint4*>(row + (((cb + 1) ^ (r & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
                }
            }
            fence_async_smem();  // generic-proxy writes before the tensor cores read them
            mbar_arrive(&vw_full[w]);
            named_bar_sync(4, C::NCONV * 32);  // every converter is done with the landed V
            if (ct == 0) mbar_arrive(&empty_bar[s]);
            cc.advance();
            if (++s == NST) { s = 0; ph ^= 1u; }
        }
    } else if (QUANT && warp >= 2 + C::NW + C::NEPI) {
        // ======================================================= int8 -> bf16 converters
        // Per stage, in tile order: wait for the copies, widen the K codes into tensor memory and
        // the V codes in place, publish to the tensor cores, arrive.
        //  K: MMA1's A operand in tensor memory (buffer k & 1, free once MMA1 of tile k - 2 has
        //   read it): a thread widens its own row (lane 32 (warp % 4) + lane, the quadrant this
        //   warp may access; the warps of a quadrant split the row) 32 codes at a time; the codes
        //   landed 128-byte swizzled, so the 8 rows of a quarter warp read 8 different bank groups.
        //  V: int8 rows at column block 1 -> bf16 rows in the 128-byte-swizzled layout of column
        //   blocks 0 and 1.  Every thread loads all its units before any thread writes (the bf16
        //   rows of column block 1 overwrite the int8 rows), then widens them.  A unit is 16 codes
        //   (group g) of one row; a quarter warp takes rows 2p and 2p + 1, groups 0-3 of one and
        //   4-7 of the other, so its 16-byte loads cover the 8 bank groups once, and so do its
        //   stores (row 2p + 1's chunks are row 2p's XOR 1 under the swizzle).
        const int ct = tid - (2 + C::NW + C::NEPI) * 32;  // 0 .. NCONV * 32 - 1
        const int cw = ct >> 5;                           // converter warp
        constexpr int PER = TT * 8 / (C::NCONV * 32);     // V units per thread (4 or 8)
        const int kr = 32 * (warp & 3) + lane;            // K row = tensor-memory lane
        constexpr int KP = 16 / C::NCONV;                 // 32-code pieces of that row per warp
        Cur cc;
        cc.init(prefix, B, H_kv, r0, r1);
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        named_bar_sync(6, 32 + C::NCONV * 32);  // the MMA warp has allocated tensor memory
        tc5_fence_after();
        const uint32_t tka = *tmem_slot + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)C::KA_COL;
        for (int k = 0; cc.valid; ++k) {
            ok = ok && mbar_wait(&full_bar[s], ph, abort_flag, p.err);
            ok = ok && mbar_wait(&ka_empty[k & 1], ((k >> 1) & 1) ^ 1u, abort_flag, p.err);
            ok = __all_sync(FULL, ok);  // the tensor-memory store below is warp-wide
            tc5_fence_after();
            unsigned char* st = ring + s * C::STAGE_BYTES;
            if (ok)
#pragma unroll 1
                for (int q = (cw >> 2) * KP; q < (cw >> 2) * KP + KP; ++q) {  // 32 codes (16 columns) a pass
                    uint4 c2[2];
#pragma unroll
                    for (int j = 0; j < 2; ++j)
                        c2[j] = *reinterpret_cast<const uint4*>(st + kr * 128 + (((2 * q + j) ^ (kr & 7)) << 4));
                    uint32_t w[16];
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        uint4 o0, o1;
                        widen_i8x16(c2[j], o0, o1);
                        w[8 * j + 0] = o0.x; w[8 * j + 1] = o0.y; w[8 * j + 2] = o0.z; w[8 * j + 3] = o0.w;
                        w[8 * j + 4] = o1.x; w[8 * j + 5] = o1.y; w[8 * j + 6] = o1.z; w[8 * j + 7] = o1.w;
                    }
                    tc5_st16(tka + (uint32_t)((k & 1) * 64 + q * 16), w);
                }
            unsigned char* tb = st + C::KLAND;
            uint4 v[PER];
            if (ok)
#pragma unroll
                for (int i = 0; i < PER; ++i) {
                    const int u = ct + i * C::NCONV * 32;
                    const int rs = (u >> 2) & 1;
                    const int r = ((u >> 4) << 1) | rs, g = ((rs ^ (u >> 3)) & 1) << 2 | (u & 3);
                    v[i] = *reinterpret_cast<const uint4*>(tb + C::HALF_BYTES + r * C::D + g * 16);
                }
            // (the barrier runs whatever ok is: a thread that gave up must not strand the others)
            named_bar_sync(4, C::NCONV * 32);
            if (ok)
#pragma unroll
                for (int i = 0; i < PER; ++i) {
                    const int u = ct + i * C::NCONV * 32;
                    const int rs = (u >> 2) & 1;
                    const int r = ((u >> 4) << 1) | rs, g = ((rs ^ (u >> 3)) & 1) << 2 | (u & 3);
                    uint4 o0, o1;
                    widen_i8x16(v[i], o0, o1);
                    unsigned char* row = tb + (g >> 2) * C::HALF_BYTES + r * 128;
                    const int c0 = 2 * (g & 3);
                    *reinterpret_cast<uint4*>(row + ((c0 ^ (r & 7)) << 4)) = o0;
                    *reinterpret_cast<uint4*>(row + (((c0 + 1) ^ (r & 7)) << 4)) = o1;
                }
            tc5_wait_st();
            tc5_fence_before();  // tensor-memory stores before the MMA warp's wait
            fence_async_smem();  // generic-proxy writes before the tensor cores read them
            mbar_arrive(&conv_full[s]);
            cc.advance();
            if (++s == NST) { s = 0; ph ^= 1u; }
        }
    } else if (warp >= 2 + C::NW) {
        // ======================================================= segment epilogues
        // For each segment of this CTA, in order: wait for the softmax warps' final state in
        // `merge`, write the output or the partial state, merge the stream if this CTA is the
        // last to finish it, release `merge`.  Runs beside the next segment's tiles.
        // The fused append's new rows, written by the first epilogue warp, idle until the first
        // segment ends: the producer waits for them only at the tile that holds them, and no warp
        // on the way to the first tile waits for their k_new / v_new loads.
        if (warp == 2 + C::NW && fused) {
            SegIter it;
            it.init(prefix, B, H_kv, r0, r1);
            while (it.valid) {
                // the new rows inside this segment: slots [r0, r1), k_new rows from i0
                int r0 = 0, r1 = 0, i0 = 0;
                if constexpr (ROLL) {
                    const int slot = (__ldg(p.lens + it.b) - 1) % p.T_max;
                    if (it.t0 <= slot && slot < it.t1) { r0 = slot; r1 = slot + 1; }
                } else {
                    const int first = it.L - p.T_q;  // the step's first new position
                    r0 = first > it.t0 ? first : it.t0;
                    r1 = it.t1;
                    i0 = r0 - first;
                }
                const size_t unit = (size_t)it.b * H_kv + it.h;
                if constexpr (QUANT) {
                    // quantize the new row (one per stream: T_q = 1) into codes + scale
                    for (int r = r0; r < r1; ++r) {
                        const size_t crow = unit * p.T_max + r;
                        q8_store_row(static_cast<const __nv_bfloat16*>(p.k_new) + unit * D,
                                     static_cast<int8_t*>(const_cast<void*>(p.K)) + crow * D,
                                     const_cast<float*>(p.Ksc) + crow, lane);
                        q8_store_row(static_cast<const __nv_bfloat16*>(p.v_new) + unit * D,
                                     static_cast<int8_t*>(const_cast<void*>(p.V)) + crow * D,
                                     const_cast<float*>(p.Vsc) + crow, lane);
                    }
                    r1 = r0;  // nothing left for the plain copy below
                }
                if constexpr (FP8) {
                    for (int r = r0; r < r1; ++r) {
                        const size_t crow = unit * p.T_max + r;
                        f8_store_row(static_cast<const __nv_bfloat16*>(p.k_new) + unit * D,
                                     static_cast<uint8_t*>(const_cast<void*>(p.K)) + crow * D,
                                     const_cast<float*>(p.Ksc) + crow, lane);
                        f8_store_row(static_cast<const __nv_bfloat16*>(p.v_new) + unit * D,
                                     static_cast<uint8_t*>(const_cast<void*>(p.V)) + crow * D,
                                     const_cast<float*>(p.Vsc) + crow, lane);
                    }
                    r1 = r0;
                }
                for (int r = r0; r < r1; ++r) {
                    int64_t arow;
                    if constexpr (PAGED)
                        arow = cache_row(p.table, p.bs, p.max_blocks, p.num_blocks, H_kv, p.T_max, it.b,
                                         it.h, r, p.err);
                    else
                        arow = ((int64_t)it.b * H_kv + it.h) * p.T_max + r;
                    if (arow < 0) continue;
                    const size_t src = (unit * p.T_q + (size_t)(i0 + r - r0)) * C::ROWB;
                    const uint4* ksrc = reinterpret_cast<const uint4*>(static_cast<const char*>(p.k_new) + src);
                    const uint4* vsrc = reinterpret_cast<const uint4*>(static_cast<const char*>(p.v_new) + src);
                    uint4* kd = reinterpret_cast<uint4*>(static_cast<char*>(const_cast<void*>(p.K)) + (size_t)arow * C::ROWB);
                    uint4* vd = reinterpret_cast<uint4*>(static_cast<char*>(const_cast<void*>(p.V)) + (size_t)arow * C::ROWB);
                    for (int v = lane; v < C::ROWB / 16; v += 32) {
                        kd[v] = __ldg(ksrc + v);
                        vd[v] = __ldg(vsrc + v);
                    }
                }
                it.next();
            }
            // order these generic-proxy writes before the producer's tensor copies of the rows
            asm volatile("fence.proxy.async.global;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(append_bar);
        }
        const int et = tid - (2 + C::NW) * 32;
        SegIter it;
        it.init(prefix, B, H_kv, r0, r1);
        bool ok = true;
        for (int sg = 0; it.valid; ++sg) {
            ok = ok && mbar_wait(m_full, (uint32_t)(sg & 1), abort_flag, p.err);
            SegIter nx = it;
            nx.next();
            if (!nx.valid) {
                final_segment(ok, it, et);
                break;
            }
            // the merge buffer goes back to the softmax warps as soon as it has been read; the
            // partial state's fence, arrival count and any merge of the stream follow
            if (ok)
                finish_segment<T, G, D, C::HS, 1, C::NEPI, 3>(p, merge, it, (size_t)it.b * H_kv + it.h,
                                                              U, P, last_flag, et,
                                                              [&]() { mbar_arrive(m_empty); });
            else
                mbar_arrive(m_empty);
            it = nx;
        }
    } else {
        // ======================================================= softmax + accumulate
        // zero the padded q rows and the P rows of padded heads (they stay zero); then meet the
        // MMA warp (named barrier 2) for the TMEM base
        for (int i = tid - 64; i < (C::OPB_BYTES + 2 * C::PBUF) / 16; i += C::NW * 32)
            reinterpret_cast<uint4*>(qsw)[i] = make_uint4(0u, 0u, 0u, 0u);
        fence_async_smem();
        tc5_fence_before();
        named_bar_sync(2, 32 + C::NW * 32);
        tc5_fence_after();
        tmem = *tmem_slot;
        constexpr int GH = C::GH, NT = C::NW * 32;
        constexpr int CH = GH <= 8 ? 8 : 16;  // tensor-memory columns per load
        const int q4 = warp & 3;            // tensor-memory lane quadrant of this warp
        const int h0 = ((warp - 2) >> 2) * GH;  // this warp's head slice [h0, h0 + GH)
        const int row = q4 * 32 + lane;     // token of S^T rows / element d of O^T rows
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const float qscale = p.qscale;
        // o: this thread's output element for the slice's heads; m: the group's running maxima
        // (the same in every thread), mt = m + TAU; l: this thread's share of the denominators.
        // The rescale factors of a tile whose maxima moved scale o when that tile's O^T is
        // folded in: kept in registers (alpha, alpha_prev) for small groups, in shared memory
        // (alpha_s[tile & 1], the same for every thread) for groups of 16+ heads, whose threads
        // have no registers to spare.
        constexpr bool ASH = C::PMN;
        float o[GH], m[GH], mt[GH], l[GH], alpha[GH], alpha_prev[GH];
        Cur cur;
        cur.init(prefix, B, H_kv, r0, r1);
        int s = 0, sg = 0;
        uint32_t ph = 0;
        bool alive = true;
        auto absorb = [&](int j, bool resc, const float* areg) {
            // O^T(j) into the accumulator: o = o * alpha_j + (O^T_hi + O^T_lo)(j)[row, :]
            alive = alive && mbar_wait(&o_full[j & 1], (j >> 1) & 1, abort_flag, p.err);
            tc5_fence_after();
            const uint32_t ob = tmem + (uint32_t)(2 * N + (j & 1) * C::N2 + h0) + lane_off;
            const float* al = ASH ? alpha_s + (j & 1) * N + h0 : areg;
            float hi[CH], lo[CH];
#pragma unroll
            for (int c0 = 0; c0 < GH; c0 += CH) {
                tc5_ld<CH>(ob + c0, hi);
                tc5_ld<CH>(ob + C::LOOFF + c0, lo);
#pragma unroll
                for (int i = 0; i < CH; ++i)
                    if (c0 + i < GH)
                        o[c0 + i] = fmaf(o[c0 + i], (ASH && !resc) ? 1.f : al[c0 + i], hi[i] + lo[i]);
            }
            tc5_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_empty[j & 1]);
        };
        // int8 / fp8 cache: the K and V scales of this thread's row of a tile; the new row of a
        // fused step takes them from k_new / v_new, as its append computes them
        auto load_scales = [&](const Cur& c, float& a, float& b) {
            a = 1.f;
            b = 1.f;
            if (row < c.n()) {
                const int t = c.t + row;
                const size_t unit = (size_t)c.it.b * H_kv + c.it.h;
                if (fused && t == c.it.L - 1) {
                    const __nv_bfloat16* kr = static_cast<const __nv_bfloat16*>(p.k_new) + unit * D;
                    const __nv_bfloat16* vr = static_cast<const __nv_bfloat16*>(p.v_new) + unit * D;
                    const float2 sc = new_row_scales(kr, vr, FP8 ? 1 : 0);
                    a = sc.x;
                    b = sc.y;
                } else {
                    a = __ldcg(p.Ksc + unit * p.T_max + t);
                    b = __ldcg(p.Vsc + unit * p.T_max + t);
                }
            }
        };
        float sk_next = 1.f, sv_next = 1.f;
        if constexpr (SCALED)
            if (cur.valid) load_scales(cur, sk_next, sv_next);
        // fp8 cache: 2^e of each head's q terms (the MMA warp derives the same e from the same q)
        float qe[FP8 ? GH : 1];
        qe[0] = 1.f;
        SegIter last_it = cur.it;  // the segment of the latest `last` tile
        bool resc_prev = false;    // the previous tile moved the maxima
        for (int k = 0; cur.valid; ++k) {
            const int n = cur.n();
            const bool first = cur.first(), last = cur.last();
            if (first) {
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    o[h] = 0.f; m[h] = -INFINITY; mt[h] = -INFINITY; l[h] = 0.f; alpha_prev[h] = 1.f;
                }
            }
            // int8 / fp8 cache: this row's K and V scales, loaded one tile ahead
            const float sk = sk_next, sv = sv_next;
            if constexpr (SCALED) {
                Cur nxt = cur;
                nxt.advance();
                if (nxt.valid) load_scales(nxt, sk_next, sv_next);
            }
            const float qk = SCALED ? qscale * sk : qscale;
            // fp8 cache, a segment's first tile: each head's largest |q| (lane l reads elements
            // 4l .. 4l+3; loads issued before the score wait), then 2^e after it
            uint2 qraw[FP8 ? GH : 1];
            if constexpr (FP8)
                if (first) {
                    const uint2* qg = reinterpret_cast<const uint2*>(p.q) + ((size_t)cur.it.b * H_kv + cur.it.h) * G * (D / 4);
#pragma unroll
                    for (int h = 0; h < GH; ++h) qraw[h] = __ldcg(qg + (size_t)h * (D / 4) + lane);
                }
            // ---- scores of tile k
            alive = alive && mbar_wait(&s_full[k & 1], (k >> 1) & 1, abort_flag, p.err);
            tc5_fence_after();
            float x[GH];
            if constexpr (FP8) {
                if (first) {
#pragma unroll
                    for (int h = 0; h < GH; ++h) {
                        float a = fmaxf(fmaxf(fabsf(bf16_lo(qraw[h].x)), fabsf(bf16_hi(qraw[h].x))),
                                        fmaxf(fabsf(bf16_lo(qraw[h].y)), fabsf(bf16_hi(qraw[h].y))));
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(FULL, a, off));
                        qe[h] = exp2i(f8_head_exp(a));
                    }
                }
                // the three terms of head h are columns h, G + h, 2G + h
                float v[N];
#pragma unroll
                for (int c0 = 0; c0 < N; c0 += 16) {
                    float w[16];
                    tc5_ld<16>(tmem + (uint32_t)((k & 1) * N + c0) + lane_off, w);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[c0 + i] = w[i];
                }
#pragma unroll
                for (int h = 0; h < GH; ++h) x[h] = ((v[h] + v[G + h]) + v[2 * G + h]) * qe[h];
            } else {
                float v[CH];
#pragma unroll
                for (int c0 = 0; c0 < GH; c0 += CH) {
                    tc5_ld<CH>(tmem + (uint32_t)((k & 1) * N + h0 + c0) + lane_off, v);
#pragma unroll
                    for (int i = 0; i < CH; ++i)
                        if (c0 + i < GH) x[c0 + i] = v[i];
                }
            }
            tc5_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_empty[k & 1]);
            const bool valid = row < n;
            // query row h is new token h mod T_q (T_q a power of two), which sees positions up
            // to L - T_q + (h mod T_q): this row is visible to new token i iff i >= dmask
            const int dmask = row - (cur.it.L - p.T_q - cur.t);
            bool need = false;
            if (dmask <= 0) {  // visible to every query row (always with one new token)
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    x[h] = valid ? x[h] * qk : -INFINITY;
                    need |= x[h] > mt[h];
                }
            } else {
                const int tq1 = p.T_q - 1;
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    x[h] = (valid && ((h0 + h) & tq1) >= dmask) ? x[h] * qk : -INFINITY;
                    need |= x[h] > mt[h];
                }
            }
            if constexpr (!ASH)
#pragma unroll
                for (int h = 0; h < GH; ++h) alpha[h] = 1.f;
            const bool resc = group_any<1, NT>(need);
            if (resc) {
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    float mx = x[h];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, off));
                    if (lane == 0) red[q4 * N + h0 + h] = mx;
                }
                named_bar_sync(1, NT);
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    float mx = red[h0 + h];
#pragma unroll
                    for (int w = 1; w < 4; ++w) mx = fmaxf(mx, red[w * N + h0 + h]);
                    const float mn = fmaxf(m[h], mx);
                    const float a = (mn == -INFINITY) ? 1.f : fast_exp2(m[h] - mn);
                    m[h] = mn;
                    mt[h] = mn + TAU;
                    l[h] *= a;
                    if constexpr (ASH) {
                        if (row == 0) alpha_s[(k & 1) * N + h0 + h] = a;
                    } else {
                        alpha[h] = a;
                    }
                }
                named_bar_sync(1, NT);  // red is reused; alpha_s is written
            }
            // ---- P(k) = P_hi + P_lo for this thread's token; a score of -inf (masked, or no key
            // seen yet: -inf - -inf) gives weight 0
            float pw[GH];
#pragma unroll
            for (int h = 0; h < GH; ++h) {
                const float pv = fast_exp2(fmaxf(x[h] - m[h], -INFINITY));
                l[h] += pv;
                // int8 / fp8 cache: the V row scale folds into the weight (MMA2 reads the codes)
                pw[h] = SCALED ? pv * sv : pv;
            }
            if constexpr (C::PMN) {
                // MN-major: the token's row of 64 columns, 16-byte chunks swizzled by token & 7
                unsigned char* pr = pbuf + (k & 1) * C::PBUF + row * 128;
                const int sw = row & 7;
#pragma unroll
                for (int c = 0; c < GH / 8; ++c) {
                    uint32_t whi[4], wlo[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const __nv_bfloat162 h2 = __floats2bfloat162_rn(pw[8 * c + 2 * i], pw[8 * c + 2 * i + 1]);
                        const float2 hf = __bfloat1622float2(h2);
                        const __nv_bfloat162 l2 = __floats2bfloat162_rn(pw[8 * c + 2 * i] - hf.x,
                                                                        pw[8 * c + 2 * i + 1] - hf.y);
                        whi[i] = *reinterpret_cast<const uint32_t*>(&h2);
                        wlo[i] = *reinterpret_cast<const uint32_t*>(&l2);
                    }
                    const int chi = (h0 >> 3) + c, clo = (C::LOOFF >> 3) + (h0 >> 3) + c;
                    *reinterpret_cast<uint4*>(pr + ((chi ^ sw) << 4)) = make_uint4(whi[0], whi[1], whi[2], whi[3]);
                    *reinterpret_cast<uint4*>(pr + ((clo ^ sw) << 4)) = make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
                }
            } else {
                // K-major: rows h (hi) and N + h (lo), column = this thread's token (h0 is a
                // multiple of 8: the swizzle phase is h & 7)
                unsigned char* pb = pbuf + (k & 1) * C::PBUF + (row >> 6) * C::PBLOCK + h0 * 128;
                const int chunk = (row & 63) >> 3, e = row & 7;
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    const uint32_t off = (((chunk ^ (h & 7)) << 4) | (e << 1));  // NP % 8 == 0
                    if constexpr (FP8) {  // f16 terms (the widened V is f16)
                        const __half hi = __float2half_rn(pw[h]);
                        const __half lo = __float2half_rn(pw[h] - __half2float(hi));
                        *reinterpret_cast<__half*>(pb + h * 128 + off) = hi;
                        *reinterpret_cast<__half*>(pb + (NP + h) * 128 + off) = lo;
                    } else {
                        const __nv_bfloat16 hi = __float2bfloat16_rn(pw[h]);
                        const __nv_bfloat16 lo = __float2bfloat16_rn(pw[h] - __bfloat162float(hi));
                        *reinterpret_cast<__nv_bfloat16*>(pb + h * 128 + off) = hi;
                        *reinterpret_cast<__nv_bfloat16*>(pb + (NP + h) * 128 + off) = lo;
                    }
                }
            }
            // V rows past the loaded boxes hold stale bytes: zero them (they meet p = 0 in MMA2;
            // fp8: the converters write zeros there)
            const int br = paged ? p.box_rows : C::BOX_ROWS;
            const int loaded = ((n + br - 1) / br) * br;
            if (!FP8 && h0 == 0 && row >= loaded) {
                using LY = Tc5Layout<C, PAGED>;
                unsigned char* vt = (C::SPLIT ? vring + (k % C::NV) * C::TILE_BYTES : ring + s * C::STAGE_BYTES + C::KLAND) +
                                    (row >> 3) * LY::GSTR + (row & 7) * 128;
#pragma unroll
                for (int hf = 0; hf < C::HALVES; ++hf)
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4*>(vt + hf * LY::HSTR + c * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[k & 1]);
            // ---- fold in O^T of the previous tile of this segment
            if (!first) absorb(k - 1, resc_prev, alpha_prev);
            resc_prev = resc;
            if constexpr (!ASH)
#pragma unroll
                for (int h = 0; h < GH; ++h) alpha_prev[h] = alpha[h];
            if (last) {
                absorb(k, resc, alpha);
                // ---- segment epilogue: group-wide denominators, then the shared merge
#pragma unroll
                for (int h = 0; h < GH; ++h) {
                    float s_ = l[h];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) s_ += __shfl_xor_sync(FULL, s_, off);
                    if (lane == 0) red[q4 * N + h0 + h] = s_;
                }
                named_bar_sync(1, NT);
                // hand the segment's state to the epilogue warps (merge: [G][D + 2])
                alive = alive && mbar_wait(m_empty, (uint32_t)(sg & 1) ^ 1u, abort_flag, p.err);
#pragma unroll
                for (int h = 0; h < GH; ++h) merge[(h0 + h) * (D + 2) + row] = o[h];
                if (q4 == 0 && lane < GH) {
                    // lane i of a slice's quadrant-0 warp: maximum and denominator of head h0 + i
                    float mv = m[0];
#pragma unroll
                    for (int h = 1; h < GH; ++h) mv = lane == h ? m[h] : mv;
                    float s_ = 0.f;
#pragma unroll
                    for (int w = 0; w < 4; ++w) s_ += red[w * N + h0 + lane];
                    merge[(h0 + lane) * (D + 2) + D] = mv;
                    merge[(h0 + lane) * (D + 2) + D + 1] = s_;
                }
                mbar_arrive(m_full);
                last_it = cur.it;
                ++sg;
            }
            cur.advance();
            if (++s == NST) { s = 0; ph ^= 1u; }
        }
        // join the epilogue warps on the last segment, once every softmax warp's state is in
        if (sg > 0) alive = alive && mbar_wait(m_full, (uint32_t)((sg - 1) & 1), abort_flag, p.err);
        final_segment(alive && sg > 0, last_it, C::NEPI * 32 + (tid - 64));
    }
    __syncthreads();  // every role is out of its loop (all waits are bounded)
    if (*abort_flag) {
        // broken protocol (a wait timed out): let issued copies and MMAs land, bounded
        if (tid == 0) {
            for (int s = 0; s < NST; ++s) {
                if (issued[s] == 0) continue;
                const uint32_t par = (uint32_t)((issued[s] - 1) & 1);
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(&full_bar[s], par) && global_ns() - t0 < WAIT_LIMIT_NS) {
                }
            }
            if constexpr (C::SPLIT)
                for (int v = 0; v < C::NV; ++v) {
                    if (vissued[v] == 0) continue;
                    const uint32_t par = (uint32_t)((vissued[v] - 1) & 1);
                    const uint64_t t0 = global_ns();
                    while (!mbar_try_wait(&sv_full[v], par) && global_ns() - t0 < WAIT_LIMIT_NS) {
                    }
                }
        }
        if (tid == 32 && *mma_issued > 0) {
            const int j = *mma_issued - 1;
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(&o_full[j & 1], (j >> 1) & 1) && global_ns() - t0 < WAIT_LIMIT_NS) {
            }
        }
        if (tid == 33 && *mma1_issued > 0) {
            const int j = *mma1_issued - 1;
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(&s_full[j & 1], (j >> 1) & 1) && global_ns() - t0 < WAIT_LIMIT_NS) {
            }
        }
    }
    tc5_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc5_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(C::TMEM_COLS)
                     : "memory");
    }
}

}  // namespace kvc
