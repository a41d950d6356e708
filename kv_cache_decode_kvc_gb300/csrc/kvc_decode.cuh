// kvc_decode.cuh -- decode attention over a [B, H_kv, T_max, D] cache (CUDA cores, fp32 math).
//
// Computes, for every sequence b and query head j (KV head h = j / G):
//     o[b,j,:] = softmax_t(q[b,j,:] . K[b,h,t,:] / sqrt(D)) V[b,h,t,:],   t < lens[b]
// ("11.7 KV Cache：形状、显存与带宽" §2.2 single-step decode; head map from
// "第 1 周 · Day 4：KV Cache 与 MQA / GQA" §3.4).  Decode reads every cached byte once and does
// about G FLOP per byte, far below any tensor-core ridge (same pages, §1.5 / §1.1), so this
// kernel is built around the HBM stream:
//
// * Work split (split-T): the B*H_kv (b, h) streams are laid end to end and cut into P equal
//   contiguous ranges, one per CTA (cta_begin); a CTA may finish one stream and start the next.
//   A stream cut across several CTAs leaves per-CTA partial softmax states (running max m,
//   denominator l, unnormalised output) that are merged afterwards -- by the last CTA to finish
//   that stream (an arrival counter, no waiting) or by a separate combine kernel.
// * Data movement: K and V tiles of TT tokens are streamed by bulk (TMA engine) copies into an
//   NST-deep shared-memory ring guarded by mbarriers; every (b, h) row is a contiguous run of
//   lens[b]*D elements, so a tile is one copy per tensor.  There is no producer warp: the last
//   warp to finish with a stage (a shared-memory arrival counter) issues the copy of the tile
//   NST ahead into it.  The first tile of each stream segment also brings the group's q rows.
//   Each K/V byte comes from HBM once and serves all G query heads of its group.
// * Math: NW warps.  A token row is spread over LPT lanes (E elements each); the q.k partial
//   dots of TPI tokens x HS heads are reduced with a transposing butterfly so each lane ends
//   with one full score; the softmax is online with a lazily raised reference max (rescale only
//   when a score exceeds it by TAU in log2 units); p is gathered back to the LPT lanes for the
//   p.V accumulation.  Groups of more than 8 heads are split into slices served by separate
//   warps reading the same shared tile.
#pragma once

#include <math.h>

#include "kvc_internal.cuh"

namespace kvc {

template <typename T, int D_, int G_>
struct DecodeCfg {
    static constexpr int D = D_;
    static constexpr int G = G_;
    static constexpr int ES = Elem<T>::BYTES;
    static constexpr int VEC = Elem<T>::VEC;
    static constexpr int ROWB = D * ES;
    static constexpr int NVR = ROWB / 16;                   // 16-byte vectors per row
    static constexpr int HS = G < 8 ? G : 8;                // heads per slice
    static constexpr int NS = G / HS;                       // head slices
    static constexpr int LPT_A = 2 * HS > 4 ? 2 * HS : 4;
    static constexpr int LPT_B = (D * HS) / 64;             // keeps HS*E <= 64 registers
    static constexpr int LPT_T = LPT_A > LPT_B ? LPT_A : LPT_B;
    static constexpr int LPT_C = LPT_T > 32 ? 32 : LPT_T;
    static constexpr int LPT = NVR < LPT_C ? NVR : LPT_C;   // lanes per token
    static constexpr int NV = NVR / LPT;                    // vectors per lane per row
    static constexpr int E = NV * VEC;                      // elements per lane per row
    static constexpr int NGRP = 32 / LPT;                   // token groups per warp
    static constexpr int TPI = LPT >= HS ? LPT / HS : 1;    // tokens per group per iteration
    static constexpr int R = (TPI * HS) / LPT;              // scores per lane after reduction
    static constexpr int TPW = NGRP * TPI;                  // tokens per warp iteration
    static constexpr int NWT_MAX = 8 / NS;                  // token warps per slice (<= 8 warps)
    // Tile: 16 KB of each tensor, grown up to 32 KB when that is what 8 warps need, and never
    // smaller than one warp iteration.
    static constexpr int TT_16K = 16384 / ROWB > 0 ? 16384 / ROWB : 1;
    static constexpr int TT_32K = 32768 / ROWB > 0 ? 32768 / ROWB : 1;
    static constexpr int TT_WANT = NWT_MAX * TPW;
    static constexpr int TT_A = TT_WANT < TT_16K ? TT_16K : (TT_WANT < TT_32K ? TT_WANT : TT_32K);
    static constexpr int TT_B = TT_A > 512 ? 512 : TT_A;
    static constexpr int TT = TT_B < TPW ? TPW : TT_B;      // tokens per tile
    static constexpr int NWT = TT / TPW < NWT_MAX ? TT / TPW : NWT_MAX;
    static constexpr int NW = NS * NWT;                     // warps
    static constexpr int NTHREADS = NW * 32;
    static constexpr int ITERS = TT / (NWT * TPW);          // warp iterations per tile
    // Lanes of a quarter warp that read different rows at the same column would hit the
    // same banks (rows are multiples of 128 B); rotating the column order by group removes it.
    static constexpr int ROT = (LPT < 8 && NVR >= 8) ? 8 / LPT : 1;
    static constexpr int TILE_BYTES = TT * ROWB;
    static constexpr int Q_BYTES = (G * ROWB + 127) / 128 * 128;  // the group's q rows
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES + Q_BYTES;
    static constexpr int MERGE_FLOATS = NW * HS * (D + 2);
    static constexpr int PREFIX_BYTES = 2 * (MAX_B + 1) * 4;  // prefix and uprefix (int32)
    static constexpr int MISC_BYTES = 256;
    static constexpr int BUDGET = 230400;
    static constexpr int NST_A =
        (BUDGET - MERGE_FLOATS * 4 - PREFIX_BYTES - MISC_BYTES) / STAGE_BYTES;
    static constexpr int NST = NST_A > 8 ? 8 : NST_A;       // ring depth
    static constexpr int SMEM = NST * STAGE_BYTES + MERGE_FLOATS * 4 + PREFIX_BYTES + MISC_BYTES;
    static_assert(ROWB % 16 == 0, "rows must be whole 16-byte vectors");
    static_assert(R == 1 || LPT == 1, "lane mapping");
    static_assert(NST >= 2, "shared-memory ring too shallow");
    static_assert(TT % (NWT * TPW) == 0, "tile must split evenly over warps");
    static_assert(HS * E <= 64, "register budget");
};

constexpr float TAU = 8.0f;  // lazy-rescale threshold, log2 units (p <= 2^8 between rescales)
constexpr unsigned FULL = 0xFFFFFFFFu;

// Walks the (b, h) streams a CTA's range [r0, r1) touches, in order.
struct SegIter {
    // prefix[b] = sum_{b' < b} L_b' (invalid lengths count as 0); the partition-unit prefix
    // uprefix[b] = sum_{b' < b} ceil(L_b' / grain) follows it in shared memory at prefix + MAX_B + 1
    const int32_t* prefix;
    int B, H_kv;
    int64_t r1;
    int b, h, L;
    int64_t ustart;  // position of token 0 of stream (b, h)
    int t0, t1;      // this segment: tokens [t0, t1) of the stream
    bool valid;

    __device__ void init(const int32_t* pre, int B_, int H_kv_, int64_t r0, int64_t r1_) {
        prefix = pre; B = B_; H_kv = H_kv_; r1 = r1_;
        int lo = 0, hi = B - 1;  // largest b with H_kv * prefix[b] <= r0
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((int64_t)H_kv * prefix[mid] <= r0) lo = mid; else hi = mid - 1;
        }
        b = lo;
        L = prefix[b + 1] - prefix[b];
        h = (int)((r0 - (int64_t)H_kv * prefix[b]) / L);
        ustart = (int64_t)H_kv * prefix[b] + (int64_t)h * L;
        t0 = (int)(r0 - ustart);
        t1 = (int)((r1 < ustart + L ? r1 : ustart + L) - ustart);
        valid = true;
    }
    __device__ void next() {
        const int64_t pos = ustart + t1;
        if (pos >= r1) { valid = false; return; }
        if (++h == H_kv) {
            h = 0;
            do { ++b; } while (prefix[b + 1] == prefix[b]);  // skip empty sequences
            L = prefix[b + 1] - prefix[b];
        }
        ustart = (int64_t)H_kv * prefix[b] + (int64_t)h * L;
        t0 = 0;
        t1 = (int)((r1 < ustart + L ? r1 : ustart + L) - ustart);
    }
};

// Prefix sums of the sequences' valid lengths and of their partition units (one warp):
// prefix[b] = sum_{b' < b} L_b', uprefix[b] = sum_{b' < b} ceil(L_b' / p.grain), B + 1 entries.
__device__ __forceinline__ void scan_lengths(const DecodeParams& p, int rolling, int32_t* prefix,
                                             int32_t* uprefix, int lane) {
    int carry = 0, ucarry = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
        const int b = b0 + lane;
        int x = b < p.B ? eff_len(p.lens[b], p.T_max, rolling, p.T_q) : 0;
        int u = (int)stream_units(x, p.grain);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(FULL, x, o), v = __shfl_up_sync(FULL, u, o);
            if (lane >= o) {
                x += y;
                u += v;
            }
        }
        if (b < p.B) {
            prefix[b + 1] = carry + x;
            uprefix[b + 1] = ucarry + u;
        }
        carry += __shfl_sync(FULL, x, 31);
        ucarry += __shfl_sync(FULL, u, 31);
    }
    if (lane == 0) {
        prefix[0] = 0;
        uprefix[0] = 0;
    }
}

// Position in the CTA's tile sequence: segment + first token of the tile.
template <int TT>
struct TileCursor {
    SegIter it;
    int t;
    bool valid;
    __device__ void init(const int32_t* pre, int B, int H_kv, int64_t r0, int64_t r1) {
        it.init(pre, B, H_kv, r0, r1);
        t = it.t0;
        valid = it.valid;
    }
    __device__ int n() const { return (it.t1 - t) < TT ? (it.t1 - t) : TT; }
    __device__ bool first() const { return t == it.t0; }
    __device__ bool last() const { return t + TT >= it.t1; }
    __device__ void advance() {
        t += TT;
        if (t >= it.t1) {
            it.next();
            t = it.t0;
            valid = it.valid;
        }
    }
};

// Transposing butterfly: N == LPT partial sums per lane in, lane `lig` of the group ends with
// the full sum of value index `lig` in v[0].
template <int N, int LPT>
__device__ __forceinline__ void reduce_scatter(float (&v)[N], int lig) {
#pragma unroll
    for (int off = LPT / 2, n = N; off >= 1; off >>= 1, n >>= 1) {
        const bool up = (lig & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = up ? v[i] : v[i + n / 2];
            const float keep = up ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(FULL, send, off);
        }
    }
}

// Shared-memory vector index of register block i for a lane (see ROT).
template <class C>
__device__ __forceinline__ int vec_index(int i, int lig, int rot) {
    return lig + C::LPT * ((i + rot) % C::NV);
}

// Issues the bulk copies of one tile into `stage` (one thread).  The last token of a stream in
// the fused step comes from k_new / v_new instead of the cache; the first tile of a segment also
// brings the group's G query rows.
template <class C, int TT>
__device__ __forceinline__ void issue_tile(const DecodeParams& p, const TileCursor<TT>& c,
                                           unsigned char* ring, uint64_t* full_bar, int stage,
                                           uint64_t pol) {
    const int n = c.n();
    const size_t unit = (size_t)c.it.b * p.H_kv + c.it.h;
    unsigned char* ks = ring + stage * C::STAGE_BYTES;
    unsigned char* vs = ks + C::TILE_BYTES;
    unsigned char* qs = vs + C::TILE_BYTES;
    const bool with_q = c.first();
    // tile rows [ns, ne) hold the step's new tokens (k_new rows from i0) in the fused step
    int ns = -1, ne = -1, i0 = 0;
    if (p.k_new != nullptr) {
        if (p.rolling) {
            const int slot = new_row_slot(p, c.it.b, c.it.L);
            if (slot >= c.t && slot < c.t + n) { ns = slot - c.t; ne = ns + 1; }
        } else if (c.t + n > c.it.L - p.T_q) {  // the stream's last T_q rows
            const int first = c.it.L - p.T_q;
            ns = first > c.t ? first - c.t : 0;
            ne = n;
            i0 = c.t + ns - first;
        }
    }
    uint32_t bytes = (uint32_t)(2 * n * C::ROWB);
    if (with_q) bytes += C::G * C::ROWB;
    mbar_arrive_expect_tx(&full_bar[stage], bytes);
    // cache rows [r0, r1) of the tile
    auto copy_rows = [&](int r0, int r1) {
        if (r1 <= r0) return;
        if (p.table == nullptr) {
            const size_t off = (unit * p.T_max + c.t + r0) * C::ROWB;
            bulk_g2s(ks + r0 * C::ROWB, static_cast<const char*>(p.K) + off, (r1 - r0) * C::ROWB,
                     &full_bar[stage], pol);
            bulk_g2s(vs + r0 * C::ROWB, static_cast<const char*>(p.V) + off, (r1 - r0) * C::ROWB,
                     &full_bar[stage], pol);
            return;
        }
        // paged: one copy per block piece (the rows of one (block, head) are contiguous)
        for (int r = r0; r < r1;) {
            const int t = c.t + r;
            const int m = (p.bs - t % p.bs) < (r1 - r) ? (p.bs - t % p.bs) : (r1 - r);
            const int64_t row = cache_row_rd(p.table, p.bs, p.max_blocks, p.num_blocks, p.H_kv,
                                             p.T_max, c.it.b, c.it.h, t, p.err);
            bulk_g2s(ks + r * C::ROWB, static_cast<const char*>(p.K) + row * C::ROWB, m * C::ROWB,
                     &full_bar[stage], pol);
            bulk_g2s(vs + r * C::ROWB, static_cast<const char*>(p.V) + row * C::ROWB, m * C::ROWB,
                     &full_bar[stage], pol);
            r += m;
        }
    };
    if (ns < 0) {
        copy_rows(0, n);
    } else {
        // the new rows come straight from k_new / v_new [B, H_kv, T_q, D], the rest from the cache
        copy_rows(0, ns);
        const size_t src = (unit * p.T_q + i0) * C::ROWB;
        bulk_g2s(ks + ns * C::ROWB, static_cast<const char*>(p.k_new) + src, (ne - ns) * C::ROWB,
                 &full_bar[stage], pol);
        bulk_g2s(vs + ns * C::ROWB, static_cast<const char*>(p.v_new) + src, (ne - ns) * C::ROWB,
                 &full_bar[stage], pol);
        copy_rows(ne, n);
    }
    if (with_q)
        bulk_g2s(qs, static_cast<const char*>(p.q) + unit * C::G * C::ROWB, C::G * C::ROWB,
                 &full_bar[stage], pol);
}

// Second half of a segment epilogue, shared by the decode kernels.  On entry every warp's state
// (unnormalised output, max in log2 units, denominator) for its head slice is in `merge`
// ([NW][HS][D+2]) and the CTA has synchronised.  Merges the warps of each slice, then either
// writes the stream's output (the segment is the whole stream) or stores the partial state in
// slot (CTA + stream); with combine_mode 0 the last CTA to arrive merges all partial states.
// Synchronises the threads that run the epilogue: the whole CTA (BAR == 0) or the NT threads
// of named barrier BAR.
template <int BAR, int NT>
__device__ __forceinline__ void group_sync() {
    if constexpr (BAR == 0) __syncthreads();
    else named_bar_sync(BAR, NT);
}

// Merges the partial states (slots c + unit, c in [cfirst, clast]) of one stream into its
// output, o = sum_c w_c o_c / sum_c w_c l_c with w_c = 2^(m_c - M), M = max_c m_c.  A thread
// owns groups of 4 consecutive outputs (one head); for up to 4 segments at a time it issues
// every 16-byte partial-output load and 8-byte (max, denominator) load of its UNR groups before
// using any, and folds them in with a running maximum, so a stream split over at most 4 CTAs
// costs one round trip to L2 per UNR groups.  Run by NT threads.  Slots are 16-byte aligned
// (G * D is a multiple of 4).  With `loc`, the state of CTA `self` is taken from shared memory
// (layout [G][D + 2]: unnormalised output, max, denominator) instead of its slot.
template <typename T, int G, int D, int NT>
__device__ __forceinline__ void merge_partials(const DecodeParams& p, size_t unit, int64_t cfirst,
                                               int64_t clast, int tid, const float* loc = nullptr,
                                               int64_t self = -1) {
    const int nseg = (int)(clast - cfirst + 1);
    constexpr int V4 = G * D / 4;
    constexpr int PER = (V4 + NT - 1) / NT;
    constexpr int UMAX = NT >= 256 ? 2 : 4;  // fewer registers in the 8-warp CUDA-core kernel
    constexpr int UNR = PER < UMAX ? PER : UMAX;
    const size_t s0 = (size_t)(cfirst + (int64_t)unit);
    const float4* po4 = reinterpret_cast<const float4*>(p.part_o + s0 * G * D);
    const float2* pml = reinterpret_cast<const float2*>(p.part_ml + s0 * G * 2);
    for (int base = tid; base < V4; base += NT * UNR) {
        float4 acc[UNR];
        float M[UNR], den[UNR];
        int h[UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            M[u] = -INFINITY;
            den[u] = 0.f;
            const int hh = ((base + u * NT) * 4) / D;
            h[u] = hh < G ? hh : G - 1;
            if (loc != nullptr && base + u * NT < V4) {
                const float* lh = loc + h[u] * (D + 2);
                const int d0 = (base + u * NT) * 4 - h[u] * D;
                acc[u] = make_float4(lh[d0], lh[d0 + 1], lh[d0 + 2], lh[d0 + 3]);
                M[u] = lh[D];
                den[u] = lh[D + 1];
            }
        }
        for (int c0 = 0; c0 < nseg; c0 += 4) {
            float4 v[UNR][4];
            float2 ml[UNR][4];
#pragma unroll
            for (int u = 0; u < UNR; ++u)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const bool in = base + u * NT < V4 && c0 + j < nseg && cfirst + c0 + j != self;
                    v[u][j] = in ? __ldcg(po4 + (size_t)(c0 + j) * V4 + base + u * NT)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
                    ml[u][j] = in ? __ldcg(pml + (size_t)(c0 + j) * G + h[u]) : make_float2(-INFINITY, 0.f);
                }
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                float mn = M[u];
#pragma unroll
                for (int j = 0; j < 4; ++j) mn = fmaxf(mn, ml[u][j].x);
                if (mn == -INFINITY) continue;  // nothing valid yet
                const float sc = (M[u] == -INFINITY) ? 0.f : exp2f(M[u] - mn);
                acc[u].x *= sc; acc[u].y *= sc; acc[u].z *= sc; acc[u].w *= sc;
                den[u] *= sc;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float w = (ml[u][j].x == -INFINITY) ? 0.f : exp2f(ml[u][j].x - mn);
                    acc[u].x = fmaf(w, v[u][j].x, acc[u].x);
                    acc[u].y = fmaf(w, v[u][j].y, acc[u].y);
                    acc[u].z = fmaf(w, v[u][j].z, acc[u].z);
                    acc[u].w = fmaf(w, v[u][j].w, acc[u].w);
                    den[u] = fmaf(w, ml[u][j].y, den[u]);
                }
                M[u] = mn;
            }
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            const int i4 = base + u * NT;
            if (i4 < V4) {
                const float inv = 1.f / den[u];
                const size_t o = unit * G * D + (size_t)i4 * 4;
                Elem<T>::store(p.out, o, acc[u].x * inv);
                Elem<T>::store(p.out, o + 1, acc[u].y * inv);
                Elem<T>::store(p.out, o + 2, acc[u].z * inv);
                Elem<T>::store(p.out, o + 3, acc[u].w * inv);
            }
        }
    }
}

// `released` is called by every thread once, right after its last read of `merge` (a caller
// that overlaps the next segment may hand the buffer back there).
struct NoRelease {
    __device__ void operator()() const {}
};
template <typename T, int G, int D, int HS, int NWT, int NW, int BAR = 0, class Rel = NoRelease>
__device__ __forceinline__ void finish_segment(const DecodeParams& p, float* merge,
                                               const SegIter& it, size_t unit, int64_t U, int64_t P,
                                               int* last_flag, int tid, Rel released = Rel()) {
    const bool whole = (it.t0 == 0) && (it.t1 == it.L);
    const int64_t us = it.ustart;
    // the stream's partition units [u0, u0 + nu), its tokens in [u0 + stream_cost, u0 + nu)
    const int32_t* uprefix = it.prefix + MAX_B + 1;
    const int64_t nu = uprefix[it.b + 1] - uprefix[it.b];
    const int64_t u0 = (int64_t)it.H_kv * uprefix[it.b] + (int64_t)it.h * nu;
    const int64_t cfirst = cta_of(u0 + stream_cost(p.grain), U, P), clast = cta_of(u0 + nu - 1, U, P);
    const int64_t slot = (int64_t)blockIdx.x + (int64_t)unit;
    if constexpr (NWT == 1) {
        // `merge` holds this segment's final state.  If every other CTA of the stream has
        // already published its partial state (and counted itself), this CTA is the last: it
        // merges from shared memory without publishing its own.
        if (!whole && p.combine_mode == 0) {
            if (tid == 0) {
                int seen;
                asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(seen) : "l"(&p.counters[unit]) : "memory");
                *last_flag = (seen == (int)(clast - cfirst));
            }
            group_sync<BAR, NW * 32>();
            if (*last_flag) {
                merge_partials<T, G, D, NW * 32>(p, unit, cfirst, clast, tid, merge, (int64_t)blockIdx.x);
                released();
                if (tid == 0) p.counters[unit] = 0;  // every other arrival is in: ready for next call
                group_sync<BAR, NW * 32>();
                return;
            }
        }
    }
    if constexpr (NWT == 1) {
        // one state per head (merge row hg: D outputs, max, denominator): copied or normalised
        // two elements at a time
        static_assert(D % 2 == 0, "float2 rows");
        for (int i2 = tid; i2 < G * D / 2; i2 += NW * 32) {
            const int hg = (2 * i2) / D, d = 2 * i2 - hg * D;
            const float* bw = merge + hg * (D + 2);
            const float2 v = *reinterpret_cast<const float2*>(bw + d);
            if (whole) {
                const float den = bw[D + 1];
                Elem<T>::store(p.out, unit * G * D + 2 * i2, v.x / den);
                Elem<T>::store(p.out, unit * G * D + 2 * i2 + 1, v.y / den);
            } else {
                *reinterpret_cast<float2*>(p.part_o + (size_t)slot * G * D + 2 * i2) = v;
                if (d == 0)
                    *reinterpret_cast<float2*>(p.part_ml + ((size_t)slot * G + hg) * 2) = make_float2(bw[D], bw[D + 1]);
            }
        }
    } else
    for (int idx = tid; idx < G * D; idx += NW * 32) {
        const int hg = idx / D, d = idx - hg * D;
        const int s_ = hg / HS, hh = hg - s_ * HS;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NWT; ++w)
            M = fmaxf(M, merge[(s_ * NWT + w) * (HS * (D + 2)) + hh * (D + 2) + D]);
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int w = 0; w < NWT; ++w) {
            const float* bw = merge + (s_ * NWT + w) * (HS * (D + 2)) + hh * (D + 2);
            const float c = (bw[D] == -INFINITY) ? 0.f : exp2f(bw[D] - M);
            num = fmaf(c, bw[d], num);
            den = fmaf(c, bw[D + 1], den);
        }
        if (whole) {
            Elem<T>::store(p.out, unit * G * D + idx, num / den);
        } else {
            p.part_o[(size_t)slot * G * D + idx] = num;
            if (d == 0) {
                p.part_ml[((size_t)slot * G + hg) * 2] = M;
                p.part_ml[((size_t)slot * G + hg) * 2 + 1] = den;
            }
        }
    }
    released();
    if (!whole && p.combine_mode == 0) {
        __threadfence();
        group_sync<BAR, NW * 32>();  // also: every thread is done reading merge
        if (tid == 0) {
            const int prev = atomicAdd(&p.counters[unit], 1);
            *last_flag = (prev == (int)(clast - cfirst));
        }
        group_sync<BAR, NW * 32>();
        if (*last_flag) {
            __threadfence();
            merge_partials<T, G, D, NW * 32>(p, unit, cfirst, clast, tid);
            if (tid == 0) p.counters[unit] = 0;  // every arrival is in: ready for next call
        }
    }
    group_sync<BAR, NW * 32>();  // merge buffer and flags are reused by the next segment
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(DecodeCfg<T, D, G>::NTHREADS, 1)
    decode_kernel(const DecodeParams p) {
    using C = DecodeCfg<T, D, G>;
    constexpr int HS = C::HS, E = C::E, NV = C::NV, VEC = C::VEC, LPT = C::LPT, TPI = C::TPI;
    constexpr int R = C::R, TT = C::TT, NW = C::NW, NWT = C::NWT, NST = C::NST;

    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* ring = smem;
    float* merge = reinterpret_cast<float*>(smem + NST * C::STAGE_BYTES);
    int32_t* prefix = reinterpret_cast<int32_t*>(merge + C::MERGE_FLOATS);
    int32_t* uprefix = prefix + MAX_B + 1;
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(uprefix + MAX_B + 1);
    int* release_cnt = reinterpret_cast<int*>(full_bar + NST);   // [NST]
    int* issued = release_cnt + NST;                                // [NST] tiles issued per stage
    volatile int* abort_flag = issued + NST;
    int* last_flag = issued + NST + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = p.B, H_kv = p.H_kv;
    const size_t row_elems_q = (size_t)H_kv * G * D;  // one sequence of q / out

    // ---- lengths -> stream prefix sums (warp 0); barriers (thread 32)
    if (warp == 0) scan_lengths(p, p.rolling, prefix, uprefix, lane);
    if (tid == (NW > 1 ? 32 : 0)) {
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

    // ---- rows with an invalid length: zero output, flag (one CTA per row)
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
    const bool fused = p.k_new != nullptr;
    const uint64_t pol = policy_evict_first();

    // ---- prime the ring: tiles 0 .. NST-1 (thread 0); every warp keeps the same prefetch cursor
    TileCursor<TT> pref;
    pref.init(prefix, B, H_kv, r0, r1);
    for (int k = 0; k < NST && pref.valid; ++k) {
        if (tid == 0) {
            issue_tile<C, TT>(p, pref, ring, full_bar, k, pol);
            issued[k] += 1;
        }
        pref.advance();
    }

    const int wt = warp % NWT;   // token warp within the head slice
    const int sl = warp / NWT;   // head slice
    const int grp = lane / LPT, lig = lane % LPT;
    const int gbase = lane & ~(LPT - 1);
    const int rot = (C::ROT > 1) ? (grp % C::ROT) : 0;

    constexpr int PV = VEC / 2;  // fp32 pairs per 16-byte vector
    constexpr int E2 = E / 2;    // fp32 pairs per lane per row
    float2 q2[HS][E2];           // q, pre-scaled, as pairs of consecutive elements
    float2 o2[HS][E2];           // unnormalised output accumulators
    float m[R], l[R];

    int stage = 0;
    uint32_t phase = 0;
    TileCursor<TT> cur;
    cur.init(prefix, B, H_kv, r0, r1);
    while (cur.valid) {
        const size_t unit = (size_t)cur.it.b * H_kv + cur.it.h;
        const int n = cur.n();
        const bool ok = mbar_wait(&full_bar[stage], phase, abort_flag, p.err);
        const T* Ks = reinterpret_cast<const T*>(ring + stage * C::STAGE_BYTES);
        const T* Vs = Ks + TT * D;
        if (cur.first()) {
            // q rows of this slice from the stage, pre-scaled by log2(e)/sqrt(D)
            const T* qs = Vs + TT * D + (size_t)sl * HS * D;
            const float2 sc = make_float2(p.qscale, p.qscale);
#pragma unroll
            for (int hh = 0; hh < HS; ++hh)
#pragma unroll
                for (int i = 0; i < NV; ++i) {
                    const uint4 v = *reinterpret_cast<const uint4*>(
                        qs + (size_t)hh * D + vec_index<C>(i, lig, rot) * VEC);
                    float2 f[PV];
                    Elem<T>::unpack2(v, f);
#pragma unroll
                    for (int w = 0; w < PV; ++w) q2[hh][i * PV + w] = __fmul2_rn(f[w], sc);
                }
#pragma unroll
            for (int hh = 0; hh < HS; ++hh)
#pragma unroll
                for (int w = 0; w < E2; ++w) o2[hh][w] = make_float2(0.f, 0.f);
#pragma unroll
            for (int r = 0; r < R; ++r) { m[r] = -INFINITY; l[r] = 0.f; }
        }
        if (ok) {
#pragma unroll 1
            for (int itn = 0; itn < C::ITERS; ++itn) {
                if ((itn * NWT + wt) * C::TPW >= n) break;
                const int base = (itn * NWT + wt) * C::TPW + grp * TPI;
                // this lane's slices of the TPI token rows; masked rows read row 0 (p = 0 there).
                // When the slices are few, K and V are both loaded up front.
                constexpr bool PRE = TPI * NV <= 4;
                int roff[TPI];
#pragma unroll
                for (int k = 0; k < TPI; ++k) roff[k] = ((base + k < n) ? base + k : 0) * D;
                uint4 kv[TPI][NV], vv[PRE ? TPI : 1][PRE ? NV : 1];
#pragma unroll
                for (int k = 0; k < TPI; ++k)
#pragma unroll
                    for (int i = 0; i < NV; ++i) {
                        const int off = roff[k] + vec_index<C>(i, lig, rot) * VEC;
                        kv[k][i] = *reinterpret_cast<const uint4*>(Ks + off);
                        if constexpr (PRE) vv[k][i] = *reinterpret_cast<const uint4*>(Vs + off);
                    }
                // q . k partial dots: pairs of elements with packed fp32x2 FMAs
                float2 acc2[TPI * HS];
#pragma unroll
                for (int j = 0; j < TPI * HS; ++j) acc2[j] = make_float2(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < NV; ++i)
#pragma unroll
                    for (int k = 0; k < TPI; ++k) {
                        float2 f[PV];
                        Elem<T>::unpack2(kv[k][i], f);
#pragma unroll
                        for (int w = 0; w < PV; ++w)
#pragma unroll
                            for (int hh = 0; hh < HS; ++hh)
                                acc2[k * HS + hh] = __ffma2_rn(q2[hh][i * PV + w], f[w], acc2[k * HS + hh]);
                    }
                float acc[TPI * HS];
#pragma unroll
                for (int j = 0; j < TPI * HS; ++j) acc[j] = acc2[j].x + acc2[j].y;
                float s2[R];
                // query row c = sl * HS + hh of the group is new token c mod T_q (T_q a power of
                // two), which sees tile rows up to lim + (c mod T_q)
                const int lim = cur.it.L - p.T_q - cur.t, tq1 = p.T_q - 1;
                if constexpr (LPT == 1) {
                    const bool v0 = base < n;
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        s2[r] = (v0 && base <= lim + ((sl * HS + r) & tq1)) ? acc[r] : -INFINITY;
                } else {
                    reduce_scatter<LPT, LPT>(acc, lig);
                    const int tok = base + lig / HS;
                    s2[0] = (tok < n && tok <= lim + ((sl * HS + lig % HS) & tq1)) ? acc[0] : -INFINITY;
                }
                // online softmax with a lazily raised reference max
                bool need = false;
#pragma unroll
                for (int r = 0; r < R; ++r) need |= s2[r] > m[r] + TAU;
                if (__any_sync(FULL, need)) {
                    float alpha[R];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        float mx = s2[r];
#pragma unroll
                        for (int off = HS; off < LPT; off <<= 1)
                            mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, off));
                        const float mn = fmaxf(m[r], mx);
                        alpha[r] = (mn == -INFINITY) ? 1.f : fast_exp2(m[r] - mn);
                        m[r] = mn;
                        l[r] *= alpha[r];
                    }
#pragma unroll
                    for (int hh = 0; hh < HS; ++hh) {
                        float a;
                        if constexpr (LPT == 1) a = alpha[hh];
                        else a = __shfl_sync(FULL, alpha[0], gbase + hh);
                        const float2 a2 = make_float2(a, a);
#pragma unroll
                        for (int w = 0; w < E2; ++w) o2[hh][w] = __fmul2_rn(o2[hh][w], a2);
                    }
                }
                float pr[R];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    pr[r] = (s2[r] == -INFINITY) ? 0.f : fast_exp2(s2[r] - m[r]);
                    l[r] += pr[r];
                }
                // p . V
#pragma unroll
                for (int k = 0; k < TPI; ++k) {
                    float2 pp[HS];
#pragma unroll
                    for (int hh = 0; hh < HS; ++hh) {
                        float pv;
                        if constexpr (LPT == 1) pv = pr[hh];
                        else pv = __shfl_sync(FULL, pr[0], gbase + k * HS + hh);
                        pp[hh] = make_float2(pv, pv);
                    }
#pragma unroll
                    for (int i = 0; i < NV; ++i) {
                        float2 f[PV];
                        if constexpr (PRE) {
                            Elem<T>::unpack2(vv[k][i], f);
                        } else {
                            const uint4 v = *reinterpret_cast<const uint4*>(
                                Vs + roff[k] + vec_index<C>(i, lig, rot) * VEC);
                            Elem<T>::unpack2(v, f);
                        }
#pragma unroll
                        for (int w = 0; w < PV; ++w)
#pragma unroll
                            for (int hh = 0; hh < HS; ++hh)
                                o2[hh][i * PV + w] = __ffma2_rn(pp[hh], f[w], o2[hh][i * PV + w]);
                    }
                }
            }
            // fused append: warp 0 stores the new token's rows (now in the tile) into the cache
            // the tile rows [ns, ne) that hold the step's new tokens (now in shared memory)
            int ns = -1, ne = -1;
            if (fused && warp == 0) {
                if (p.rolling) {
                    const int slot = new_row_slot(p, cur.it.b, cur.it.L);
                    if (slot >= cur.t && slot < cur.t + n) { ns = slot - cur.t; ne = ns + 1; }
                } else if (cur.t + n > cur.it.L - p.T_q) {
                    const int first = cur.it.L - p.T_q;
                    ns = first > cur.t ? first - cur.t : 0;
                    ne = n;
                }
            }
            for (int tr = ns; tr >= 0 && tr < ne; ++tr) {
                const int64_t arow = cache_row(p.table, p.bs, p.max_blocks, p.num_blocks, H_kv, p.T_max,
                                               cur.it.b, cur.it.h, cur.t + tr, p.err);
                if (arow < 0) continue;
                const size_t dst = (size_t)arow * C::ROWB;
                const unsigned char* ksrc = reinterpret_cast<const unsigned char*>(Ks) + tr * C::ROWB;
                const unsigned char* vsrc = reinterpret_cast<const unsigned char*>(Vs) + tr * C::ROWB;
                unsigned char* kd = static_cast<unsigned char*>(const_cast<void*>(p.K)) + dst;
                unsigned char* vd = static_cast<unsigned char*>(const_cast<void*>(p.V)) + dst;
                for (int v = lane; v < C::NVR; v += 32) {
                    reinterpret_cast<uint4*>(kd)[v] = reinterpret_cast<const uint4*>(ksrc)[v];
                    reinterpret_cast<uint4*>(vd)[v] = reinterpret_cast<const uint4*>(vsrc)[v];
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
                    issue_tile<C, TT>(p, pref, ring, full_bar, stage, pol);
                    issued[stage] += 1;
                }
            }
        }
        if (pref.valid) pref.advance();
        if (++stage == NST) { stage = 0; phase ^= 1u; }

        if (cur.last()) {
            // ---- segment epilogue: merge groups (shuffles), then warps (shared memory)
            float o[HS][E];
#pragma unroll
            for (int hh = 0; hh < HS; ++hh)
#pragma unroll
                for (int w = 0; w < E2; ++w) { o[hh][2 * w] = o2[hh][w].x; o[hh][2 * w + 1] = o2[hh][w].y; }
            float mh[HS], lh[HS];
            if constexpr (LPT == 1) {
#pragma unroll
                for (int hh = 0; hh < HS; ++hh) { mh[hh] = m[hh]; lh[hh] = l[hh]; }
            } else {
                float lg = l[0];
#pragma unroll
                for (int off = HS; off < LPT; off <<= 1) lg += __shfl_xor_sync(FULL, lg, off);
#pragma unroll
                for (int hh = 0; hh < HS; ++hh) {
                    mh[hh] = __shfl_sync(FULL, m[0], gbase + hh);
                    lh[hh] = __shfl_sync(FULL, lg, gbase + hh);
                }
            }
            if constexpr (C::ROT > 1) {  // undo the per-group column rotation
#pragma unroll
                for (int rr = 1; rr < C::ROT; ++rr) {
                    if (rot == rr) {
#pragma unroll
                        for (int hh = 0; hh < HS; ++hh) {
                            float tmp[E];
#pragma unroll
                            for (int i = 0; i < NV; ++i)
#pragma unroll
                                for (int e = 0; e < VEC; ++e)
                                    tmp[((i + rr) % NV) * VEC + e] = o[hh][i * VEC + e];
#pragma unroll
                            for (int e = 0; e < E; ++e) o[hh][e] = tmp[e];
                        }
                    }
                }
            }
            if constexpr (C::NGRP > 1) {
#pragma unroll
                for (int hh = 0; hh < HS; ++hh) {
                    float M = mh[hh];
#pragma unroll
                    for (int off = LPT; off < 32; off <<= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, off));
                    const float c = (mh[hh] == -INFINITY) ? 0.f : fast_exp2(mh[hh] - M);
                    lh[hh] *= c;
#pragma unroll
                    for (int e = 0; e < E; ++e) o[hh][e] *= c;
#pragma unroll
                    for (int off = LPT; off < 32; off <<= 1) {
                        lh[hh] += __shfl_xor_sync(FULL, lh[hh], off);
#pragma unroll
                        for (int e = 0; e < E; ++e) o[hh][e] += __shfl_xor_sync(FULL, o[hh][e], off);
                    }
                    mh[hh] = M;
                }
            }
            float* mw = merge + warp * (HS * (D + 2));
            if (grp == 0) {
#pragma unroll
                for (int hh = 0; hh < HS; ++hh)
#pragma unroll
                    for (int i = 0; i < NV; ++i)
#pragma unroll
                        for (int e = 0; e < VEC; ++e)
                            mw[hh * (D + 2) + (lig + LPT * i) * VEC + e] = o[hh][i * VEC + e];
            }
            if (lane == 0) {
#pragma unroll
                for (int hh = 0; hh < HS; ++hh) {
                    mw[hh * (D + 2) + D] = mh[hh];
                    mw[hh * (D + 2) + D + 1] = lh[hh];
                }
            }
            __syncthreads();

            finish_segment<T, G, D, HS, NWT, NW>(p, merge, cur.it, unit, U, P, last_flag, tid);
        }
        cur.advance();
    }
    if (*abort_flag) {
        // A wait timed out (broken protocol): let every copy already issued land before the CTA
        // exits, each wait bounded on its own.
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

// Merges the partial states of streams cut across CTAs (combine_mode 1).  Block (u, hg, ds) of
// the U * G * DS grid merges columns [ds D / DS, (ds + 1) D / DS) of query head hg of stream u:
// DS > 1 spreads a few long streams (e.g. one sequence of 131k tokens, 153 segments) over many
// SMs.  The block recomputes the decode kernels' partition.  Its threads form SL segment lanes
// x C4 float4 column groups; lane j sums segments j, j + SL, j + 2 SL, ... with up to eight
// loads in flight, the first eight issued before the weights are known (the weights need the
// segments' maxima first), and the SL partial sums meet in shared memory.  Launched as a
// programmatic dependent of the decode kernel: lens is read before the grid dependency wait
// (the decode kernel does not write it) when launch overlap is on, the partials after it.
constexpr int COMBINE_MAX_SEG = 1024;
constexpr int COMBINE_THREADS = 256;
constexpr int COMBINE_CHUNK = 8;  // segment loads in flight per thread
template <typename T>
__global__ void __launch_bounds__(COMBINE_THREADS) combine_kernel(const DecodeParams p, int D, int G, int DS) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (!p.overlap) asm volatile("griddepcontrol.wait;" ::: "memory");
    constexpr int NWARP = COMBINE_THREADS / 32;
    const int ds = blockIdx.x % DS, ug = blockIdx.x / DS;
    const int u = ug / G, hg = ug % G;
    const int b = u / p.H_kv, h = u % p.H_kv;
    __shared__ int64_t sh_sum[4];
    __shared__ float sw[COMBINE_MAX_SEG];
    __shared__ float sred[NWARP];
    __shared__ float4 spart[COMBINE_THREADS];
    if (threadIdx.x < 4) sh_sum[threadIdx.x] = 0;
    __syncthreads();
    // tokens and partition units of the sequences before b, and of all
    int64_t before = 0, all = 0, ubefore = 0, uall = 0;
    for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
        const int L = p.lens[i];
        const int64_t v = eff_len(L, p.T_max, p.rolling, p.T_q), nv = stream_units(v, p.grain);
        all += v;
        uall += nv;
        if (i < b) {
            before += v;
            ubefore += nv;
        }
    }
    atomicAdd(reinterpret_cast<unsigned long long*>(&sh_sum[0]), (unsigned long long)before);
    atomicAdd(reinterpret_cast<unsigned long long*>(&sh_sum[1]), (unsigned long long)all);
    atomicAdd(reinterpret_cast<unsigned long long*>(&sh_sum[2]), (unsigned long long)ubefore);
    atomicAdd(reinterpret_cast<unsigned long long*>(&sh_sum[3]), (unsigned long long)uall);
    __syncthreads();
    if (p.overlap) asm volatile("griddepcontrol.wait;" ::: "memory");
    const int Lb = eff_len(p.lens[b], p.T_max, p.rolling, p.T_q);
    if (Lb == 0) return;
    const int64_t W = (int64_t)p.H_kv * sh_sum[1], U = (int64_t)p.H_kv * sh_sum[3];
    const int64_t P = plan_ctas(W, U, p.P, p.min_tokens);
    const int64_t nu = stream_units(Lb, p.grain), u0 = (int64_t)p.H_kv * sh_sum[2] + (int64_t)h * nu;
    const int64_t cfirst = cta_of(u0 + stream_cost(p.grain), U, P), clast = cta_of(u0 + nu - 1, U, P);
    if (cfirst == clast) return;  // written directly by its CTA
    const int nseg = (int)(clast - cfirst + 1);
    if (nseg > COMBINE_MAX_SEG) return;  // cannot happen: P <= 4 * SMs
    const size_t base = (size_t)(cfirst + u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this block's columns: C4 float4 groups (D / 4 divisible by DS, C4 divides the block)
    const int D4 = D >> 2, C4 = D4 / DS, SL = COMBINE_THREADS / C4;
    const int c4 = threadIdx.x % C4, j = threadIdx.x / C4;
    const size_t st4 = (size_t)G * D4;  // float4s between consecutive segments
    const float4* po = reinterpret_cast<const float4*>(p.part_o) + base * st4 + (size_t)hg * D4 + ds * C4 + c4;
    float4 v[COMBINE_CHUNK];
#pragma unroll
    for (int i = 0; i < COMBINE_CHUNK; ++i) {
        const int c = j + i * SL;
        v[i] = c < nseg ? __ldcg(po + (size_t)c * st4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // weights w_c = 2^(m_c - M), M = max_c m_c, and the denominator sum_c w_c l_c
    float mx = -INFINITY;
    for (int c = threadIdx.x; c < nseg; c += blockDim.x) {
        const float mc = p.part_ml[((base + c) * G + hg) * 2];
        sw[c] = mc;
        mx = fmaxf(mx, mc);
    }
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
    if (lane == 0) sred[warp] = mx;
    __syncthreads();
    float M = sred[0];
    for (int w = 1; w < NWARP; ++w) M = fmaxf(M, sred[w]);
    __syncthreads();
    float den = 0.f;
    for (int c = threadIdx.x; c < nseg; c += blockDim.x) {
        const float w = (sw[c] == -INFINITY) ? 0.f : exp2f(sw[c] - M);
        sw[c] = w;
        den = fmaf(w, p.part_ml[((base + c) * G + hg) * 2 + 1], den);
    }
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xFFFFFFFFu, den, off);
    if (lane == 0) sred[warp] = den;
    __syncthreads();  // also: every weight in sw is written
    float dsum = 0.f;
    for (int w = 0; w < NWARP; ++w) dsum += sred[w];
    const float inv = 1.f / dsum;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0;; c0 += COMBINE_CHUNK * SL) {
#pragma unroll
        for (int i = 0; i < COMBINE_CHUNK; ++i) {
            const int c = c0 + j + i * SL;
            const float w = c < nseg ? sw[c] : 0.f;
            acc.x = fmaf(w, v[i].x, acc.x);
            acc.y = fmaf(w, v[i].y, acc.y);
            acc.z = fmaf(w, v[i].z, acc.z);
            acc.w = fmaf(w, v[i].w, acc.w);
        }
        const int n0 = c0 + COMBINE_CHUNK * SL;
        if (n0 >= nseg) break;
#pragma unroll
        for (int i = 0; i < COMBINE_CHUNK; ++i) {
            const int c = n0 + j + i * SL;
            v[i] = c < nseg ? __ldcg(po + (size_t)c * st4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    spart[threadIdx.x] = acc;
    __syncthreads();
    if (j == 0) {
        for (int jj = 1; jj < SL; ++jj) {
            const float4 w4 = spart[jj * C4 + c4];
            acc.x += w4.x;
            acc.y += w4.y;
            acc.z += w4.z;
            acc.w += w4.w;
        }
        const size_t o = ((size_t)u * G + hg) * D + (size_t)(ds * C4 + c4) * 4;
        Elem<T>::store(p.out, o, acc.x * inv);
        Elem<T>::store(p.out, o + 1, acc.y * inv);
        Elem<T>::store(p.out, o + 2, acc.z * inv);
        Elem<T>::store(p.out, o + 3, acc.w * inv);
    }
}

}  // namespace kvc
