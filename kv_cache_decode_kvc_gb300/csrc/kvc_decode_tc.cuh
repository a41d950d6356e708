// kvc_decode_tc.cuh -- decode attention over a bf16 cache with the two small contractions on
// tensor cores.
//
// Same computation, split-T partition and merging as decode_kernel (kvc_decode.cuh): for every
// query head j of sequence b, o = softmax_t(q . K_t / sqrt(D)) V over t < lens[b]
// ("11.7 KV Cache：形状、显存与带宽" §2.2; the head map of "第 1 周 · Day 4：KV Cache 与
// MQA / GQA" §3.4).  What changes is how a CTA consumes a tile.  On CUDA cores a GQA group of
// g heads costs about 2g FMAs plus a share of shuffles and unpacking per cached element; at
// group 4 and above that issue work, not HBM, bounds the stream.  Here a warp takes a slab of
// 16 tokens and one slice of up to 8 query heads of the group:
//   S^T[16 tok x 8 heads] = K[16 x D] . Q^T[D x 8]          (D/16 mma.m16n8k16, bf16 -> fp32)
//   online softmax on the accumulator fragment (fp32; a lane holds 2 tokens x 2 heads)
//   O^T[D x 8 heads]     += V^T[D x 16] . P^T[16 x 8]        (2 D/16 mma: P = P_hi + P_lo)
// P^T's operand fragment is the score fragment transposed in registers (movmatrix).  K and V
// tiles arrive by TMA tensor copies (cp.async.bulk.tensor, 128-byte swizzle, boxes of 32 rows x
// 64 columns) so the ldmatrix reads of both operands are free of bank conflicts; the q rows come
// with a plain bulk copy.  Each K/V byte is still read from HBM once per step.
//
// The fused append (kvc_decode_step) writes the new token's rows into the cache in the
// prologue of the CTA that owns the stream's last position, and orders those writes before its
// own tensor copies with a proxy fence; the tile then reads the row from the cache.
#pragma once

#include <cuda.h>  // CUtensorMap

#include "kvc_decode.cuh"

namespace kvc {

template <int D_, int G_>
struct TcCfg {
    static constexpr int D = D_;
    static constexpr int G = G_;
    static constexpr int ROWB = D * 2;
    static constexpr int HALVES = D / 64;              // 128-byte column blocks of a row
    static constexpr int HS = G < 8 ? G : 8;           // heads per warp slice (mma N = 8)
    static constexpr int NS = G / HS;                  // slices
    static constexpr int NW = 4;                       // warps
    static constexpr int NWT = NW / NS > 0 ? NW / NS : 1;
    static constexpr int NTHREADS = NW * 32;
    static constexpr int TT = 64;                      // tokens per tile
    static constexpr int SLABS = TT / 16;
    static constexpr int BOX_ROWS = TC_BOX_ROWS;
    static constexpr int HALF_BYTES = TT * 128;        // one column block of a tile
    static constexpr int TILE_BYTES = TT * ROWB;
    static constexpr int Q_BYTES = (G * ROWB + 1023) / 1024 * 1024;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES + Q_BYTES;
    static constexpr int MERGE_FLOATS = NW * HS * (D + 2);
    static constexpr int PREFIX_BYTES = 2 * (MAX_B + 1) * 4;  // prefix and uprefix (int32)
    static constexpr int MISC_BYTES = 256;
    static constexpr int ALIGN_PAD = 1024;
    static constexpr int BUDGET = 230400;
    static constexpr int NST_A =
        (BUDGET - MERGE_FLOATS * 4 - PREFIX_BYTES - MISC_BYTES - ALIGN_PAD) / STAGE_BYTES;
    static constexpr int NST = NST_A > 8 ? 8 : NST_A;
    static constexpr int SMEM =
        NST * STAGE_BYTES + MERGE_FLOATS * 4 + PREFIX_BYTES + MISC_BYTES + ALIGN_PAD;
    static_assert(D % 64 == 0, "whole 128-byte column blocks");
    static_assert(NS * NWT == NW, "warps split evenly over head slices");
    static_assert(SLABS % NWT == 0 || NWT <= SLABS, "slabs per warp");
    static_assert(NST >= 2, "ring too shallow");
    static_assert(TILE_BYTES % 1024 == 0 && STAGE_BYTES % 1024 == 0, "swizzle atoms stay aligned");
};

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
// D += A(16x16, row) . B(16x8, col), bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
// TMA tensor copy of a box {64 columns, BOX_ROWS rows} at (col, row) into shared memory.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int col, int row,
                                            uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::"
        "cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(col), "r"(row), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Issues one tile: ceil(n/BOX_ROWS) boxes per column block of K and of V (rows past the stream's
// end are loaded and masked; rows past the tensor read as zero), plus q on a segment's first tile.
template <class C, int TT>
__device__ __forceinline__ void issue_tile_tc(const DecodeParams& p, const TileCursor<TT>& c,
                                              uint32_t ring, uint64_t* full_bar, int stage,
                                              uint64_t pol, const CUtensorMap* tmK,
                                              const CUtensorMap* tmV) {
    const int n = c.n();
    const size_t unit = (size_t)c.it.b * p.H_kv + c.it.h;
    const uint32_t ks = ring + stage * C::STAGE_BYTES;
    const uint32_t vs = ks + C::TILE_BYTES;
    const uint32_t qs = vs + C::TILE_BYTES;
    const int nbox = (n + C::BOX_ROWS - 1) / C::BOX_ROWS;
    const bool with_q = c.first();
    uint32_t bytes = (uint32_t)(2 * C::HALVES * nbox * C::BOX_ROWS * 128);
    if (with_q) bytes += C::G * C::ROWB;
    mbar_arrive_expect_tx(&full_bar[stage], bytes);
    const int row0 = (int)(unit * p.T_max + c.t);
#pragma unroll
    for (int hf = 0; hf < C::HALVES; ++hf)
        for (int bx = 0; bx < nbox; ++bx) {
            const uint32_t off = hf * C::HALF_BYTES + bx * C::BOX_ROWS * 128;
            tma_load_2d(ks + off, tmK, hf * 64, row0 + bx * C::BOX_ROWS, &full_bar[stage], pol);
            tma_load_2d(vs + off, tmV, hf * 64, row0 + bx * C::BOX_ROWS, &full_bar[stage], pol);
        }
    if (with_q) {
        asm volatile(
            "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
            "[%1], %2, [%3], %4;" ::"r"(qs),
            "l"(static_cast<const char*>(p.q) + unit * C::G * C::ROWB), "r"(C::G * C::ROWB),
            "r"(smem_addr(&full_bar[stage])), "l"(pol)
            : "memory");
    }
}

// Shared-memory address of 16-byte chunk `chunk` (0..7) of row `row` of one column block of a
// tile written by the 128-byte-swizzled tensor copy (chunk index XOR row mod 8).
__device__ __forceinline__ uint32_t swz(uint32_t block, int row, int chunk) {
    return block + row * 128 + ((chunk ^ (row & 7)) << 4);
}

template <int D, int G>
__global__ void __launch_bounds__(TcCfg<D, G>::NTHREADS, 1)
    decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV) {
    using C = TcCfg<D, G>;
    using T = __nv_bfloat16;
    constexpr int HS = C::HS, TT = C::TT, NW = C::NW, NWT = C::NWT, NST = C::NST;
    constexpr int KS = D / 16;  // k-steps of q.k, m-tiles of p.V

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* ring = smem;
    float* merge = reinterpret_cast<float*>(smem + NST * C::STAGE_BYTES);
    int32_t* prefix = reinterpret_cast<int32_t*>(merge + C::MERGE_FLOATS);
    int32_t* uprefix = prefix + MAX_B + 1;
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(uprefix + MAX_B + 1);
    int* release_cnt = reinterpret_cast<int*>(full_bar + NST);
    int* issued = release_cnt + NST;
    volatile int* abort_flag = issued + NST;
    int* last_flag = issued + NST + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = p.B, H_kv = p.H_kv;
    const size_t row_elems_q = (size_t)H_kv * G * D;

    if (warp == 0) scan_lengths(p, 0, prefix, uprefix, lane);
    if (tid == 32) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full_bar[s], 1);
            release_cnt[s] = 0;
            issued[s] = 0;
        }
        *abort_flag = 0;
        *last_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    for (int b = blockIdx.x; b < B; b += gridDim.x) {
        if (prefix[b + 1] == prefix[b]) {
            if (tid == 0) atomicOr(p.err, DEV_BAD_LENS);
            for (size_t i = tid; i < row_elems_q; i += blockDim.x)
                Elem<T>::store(p.out, (size_t)b * row_elems_q + i, 0.f);
        }
    }

    const int64_t W = (int64_t)H_kv * prefix[B], U = (int64_t)H_kv * uprefix[B];
    if (W == 0) return;
    const int64_t P = plan_ctas(W, U, p.P, p.min_tokens);
    if ((int64_t)blockIdx.x >= P) return;
    const int64_t r0 = cta_cut(blockIdx.x, prefix, uprefix, B, H_kv, U, P, p.grain);
    const int64_t r1 = cta_cut(blockIdx.x + 1, prefix, uprefix, B, H_kv, U, P, p.grain);
    if (r0 >= r1) return;

    // ---- fused append: write the new rows of the streams whose last token this CTA owns,
    // then order those generic-proxy writes before this CTA's tensor copies
    if (p.k_new != nullptr && warp == 0) {
        SegIter it;
        it.init(prefix, B, H_kv, r0, r1);
        while (it.valid) {
            if (it.t1 == it.L) {
                const size_t unit = (size_t)it.b * H_kv + it.h;
                const size_t dst = (unit * p.T_max + (size_t)(it.L - 1)) * C::ROWB;
                const uint4* ksrc = reinterpret_cast<const uint4*>(static_cast<const char*>(p.k_new) + unit * C::ROWB);
                const uint4* vsrc = reinterpret_cast<const uint4*>(static_cast<const char*>(p.v_new) + unit * C::ROWB);
                uint4* kd = reinterpret_cast<uint4*>(static_cast<char*>(const_cast<void*>(p.K)) + dst);
                uint4* vd = reinterpret_cast<uint4*>(static_cast<char*>(const_cast<void*>(p.V)) + dst);
                for (int v = lane; v < C::ROWB / 16; v += 32) {
                    kd[v] = __ldg(ksrc + v);
                    vd[v] = __ldg(vsrc + v);
                }
            }
            it.next();
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __syncwarp();
    }
    __syncthreads();

    const uint64_t pol = policy_evict_first();
    const uint32_t ring_s = smem_addr(ring);
    TileCursor<TT> pref;
    pref.init(prefix, B, H_kv, r0, r1);
    for (int k = 0; k < NST && pref.valid; ++k) {
        if (tid == 0) {
            issue_tile_tc<C, TT>(p, pref, ring_s, full_bar, k, pol, &tmK, &tmV);
            issued[k] += 1;
        }
        pref.advance();
    }

    const int wt = warp % NWT;   // token warp within the head slice
    const int sl = warp / NWT;   // head slice
    const int g = lane >> 2, t4 = lane & 3;
    const int lj = lane >> 3, lr = lane & 7;  // ldmatrix: which 8x8 matrix, which row of it
    const float qscale = p.qscale;

    uint32_t qb[KS][2];  // B fragments of Q^T for this slice (head g of the slice)
    float o[KS][4];      // O^T fragments: d = 16 mt + g (+8), heads 2 t4, 2 t4 + 1
    float m[2], l[2];    // reference max (log2 units) and denominator of heads 2 t4, 2 t4 + 1

    int stage = 0;
    uint32_t phase = 0;
    TileCursor<TT> cur;
    cur.init(prefix, B, H_kv, r0, r1);
    while (cur.valid) {
        const size_t unit = (size_t)cur.it.b * H_kv + cur.it.h;
        const int n = cur.n();
        const bool ok = mbar_wait(&full_bar[stage], phase, abort_flag, p.err);
        const uint32_t ks = ring_s + stage * C::STAGE_BYTES;
        const uint32_t vs = ks + C::TILE_BYTES;
        if (cur.first()) {
            const bool live = g < HS;  // heads past the group are zero columns
            const unsigned char* qrow = ring + stage * C::STAGE_BYTES + 2 * C::TILE_BYTES +
                                        (size_t)(sl * HS + (live ? g : 0)) * C::ROWB;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                qb[kk][0] = live ? *reinterpret_cast<const uint32_t*>(qrow + (16 * kk + 2 * t4) * 2) : 0u;
                qb[kk][1] = live ? *reinterpret_cast<const uint32_t*>(qrow + (16 * kk + 2 * t4 + 8) * 2) : 0u;
            }
#pragma unroll
            for (int mt = 0; mt < KS; ++mt)
#pragma unroll
                for (int r = 0; r < 4; ++r) o[mt][r] = 0.f;
            m[0] = m[1] = -INFINITY;
            l[0] = l[1] = 0.f;
        }
        if (ok) {
#pragma unroll 1
            for (int slab = wt; slab < C::SLABS; slab += NWT) {
                const int sb = slab * 16;
                if (sb >= n) break;
                // ---- S^T = K . Q^T (two accumulators to halve the dependency chain)
                float sa[4] = {0.f, 0.f, 0.f, 0.f}, sc[4] = {0.f, 0.f, 0.f, 0.f};
                const int krow = sb + lr + 8 * (lj & 1);
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    const int chunk = (kk & 3) * 2 + (lj >> 1);
                    uint32_t a[4];
                    ldsm_x4(a, swz(ks + (kk >> 2) * C::HALF_BYTES, krow, chunk));
                    if (kk & 1) mma_bf16(sc, a, qb[kk][0], qb[kk][1]);
                    else mma_bf16(sa, a, qb[kk][0], qb[kk][1]);
                }
                const bool v0 = sb + g < n, v1 = sb + g + 8 < n;
                float x[4];
                x[0] = v0 ? (sa[0] + sc[0]) * qscale : -INFINITY;  // token g,   head 2 t4
                x[1] = v0 ? (sa[1] + sc[1]) * qscale : -INFINITY;  // token g,   head 2 t4 + 1
                x[2] = v1 ? (sa[2] + sc[2]) * qscale : -INFINITY;  // token g+8, head 2 t4
                x[3] = v1 ? (sa[3] + sc[3]) * qscale : -INFINITY;  // token g+8, head 2 t4 + 1
                // ---- online softmax, reference max raised lazily
                float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
                if (__any_sync(FULL, mx0 > m[0] + TAU || mx1 > m[1] + TAU)) {
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(FULL, mx0, off));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(FULL, mx1, off));
                    }
                    const float n0 = fmaxf(m[0], mx0), n1 = fmaxf(m[1], mx1);
                    const float a0 = (n0 == -INFINITY) ? 1.f : fast_exp2(m[0] - n0);
                    const float a1 = (n1 == -INFINITY) ? 1.f : fast_exp2(m[1] - n1);
                    m[0] = n0; m[1] = n1;
                    l[0] *= a0; l[1] *= a1;
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt) {
                        o[mt][0] *= a0; o[mt][2] *= a0;
                        o[mt][1] *= a1; o[mt][3] *= a1;
                    }
                }
                const float p0 = x[0] == -INFINITY ? 0.f : fast_exp2(x[0] - m[0]);
                const float p1 = x[1] == -INFINITY ? 0.f : fast_exp2(x[1] - m[1]);
                const float p2 = x[2] == -INFINITY ? 0.f : fast_exp2(x[2] - m[0]);
                const float p3 = x[3] == -INFINITY ? 0.f : fast_exp2(x[3] - m[1]);
                l[0] += p0 + p2;
                l[1] += p1 + p3;
                // P^T operand: P = P_hi + P_lo, both bf16 (P_lo = the rounding residue), so the
                // product keeps fp32-level accuracy; each (token, head) fragment of the two
                // 8-token halves is transposed in registers.
                const uint32_t h01 = pack_bf16(p0, p1), h23 = pack_bf16(p2, p3);
                const uint32_t l01 = pack_bf16(p0 - bf16_lo(h01), p1 - bf16_hi(h01));
                const uint32_t l23 = pack_bf16(p2 - bf16_lo(h23), p3 - bf16_hi(h23));
                const uint32_t b0 = movmatrix_trans(h01), b1 = movmatrix_trans(h23);
                const uint32_t c0 = movmatrix_trans(l01), c1 = movmatrix_trans(l23);
                // ---- O^T += V^T . P^T; rows past n are zeroed in the operand (0 * stale = 0)
                const bool tail = sb + 16 > n;
                const int vrow = sb + lr + 8 * (lj >> 1);
                uint32_t mlo = 0xFFFFFFFFu, mhi = 0xFFFFFFFFu;
                if (tail) {
                    const int tA = sb + 2 * t4, tB = sb + 2 * t4 + 8;
                    mlo = (tA < n ? 0x0000FFFFu : 0u) | (tA + 1 < n ? 0xFFFF0000u : 0u);
                    mhi = (tB < n ? 0x0000FFFFu : 0u) | (tB + 1 < n ? 0xFFFF0000u : 0u);
                }
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    const int dcol = 16 * mt + 8 * (lj & 1);
                    uint32_t a[4];
                    ldsm_x4_trans(a, swz(vs + (dcol >> 6) * C::HALF_BYTES, vrow, (dcol & 63) >> 3));
                    a[0] &= mlo; a[1] &= mlo; a[2] &= mhi; a[3] &= mhi;
                    mma_bf16(o[mt], a, b0, b1);
                    mma_bf16(o[mt], a, c0, c1);
                }
            }
        }
        // ---- release the stage; the last warp out refills it with the tile NST ahead
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            if (atomicAdd(&release_cnt[stage], 1) == NW - 1) {
                release_cnt[stage] = 0;
                if (pref.valid && !*abort_flag) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    issue_tile_tc<C, TT>(p, pref, ring_s, full_bar, stage, pol, &tmK, &tmV);
                    issued[stage] += 1;
                }
            }
        }
        if (pref.valid) pref.advance();
        if (++stage == NST) { stage = 0; phase ^= 1u; }

        if (cur.last()) {
            // ---- segment epilogue: warp state -> merge[warp][head][D + 2]
            float lt0 = l[0], lt1 = l[1];
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                lt0 += __shfl_xor_sync(FULL, lt0, off);
                lt1 += __shfl_xor_sync(FULL, lt1, off);
            }
            float* mw = merge + warp * (HS * (D + 2));
            const int h0 = 2 * t4, h1 = 2 * t4 + 1;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                const int d0 = 16 * mt + g;
                if (h0 < HS) {
                    mw[h0 * (D + 2) + d0] = o[mt][0];
                    mw[h0 * (D + 2) + d0 + 8] = o[mt][2];
                }
                if (h1 < HS) {
                    mw[h1 * (D + 2) + d0] = o[mt][1];
                    mw[h1 * (D + 2) + d0 + 8] = o[mt][3];
                }
            }
            if (g == 0) {
                if (h0 < HS) { mw[h0 * (D + 2) + D] = m[0]; mw[h0 * (D + 2) + D + 1] = lt0; }
                if (h1 < HS) { mw[h1 * (D + 2) + D] = m[1]; mw[h1 * (D + 2) + D + 1] = lt1; }
            }
            __syncthreads();
            finish_segment<T, G, D, HS, NWT, NW>(p, merge, cur.it, unit, U, P, last_flag, tid);
        }
        cur.advance();
    }
    if (*abort_flag) {
        __syncthreads();
        if (tid == 0) {
            for (int s = 0; s < NST; ++s) {
                if (issued[s] == 0) continue;
                const uint32_t par = (uint32_t)((issued[s] - 1) & 1);
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(&full_bar[s], par) && global_ns() - t0 < WAIT_LIMIT_NS) {
                }
            }
        }
    }
}

}  // namespace kvc
