// kvc_copy.cu -- cache writes (bit-exact byte moves) and the split-T combine launcher.
//
// append: the new token's k_t, v_t go to slot lens[b]-1 of every KV head, in place in the
// preallocated cache ("第 1 周 · Day 4：KV Cache 与 MQA / GQA" §3.1; "KV 缓存" glossary page,
// "两条数学等价的 decode 路径", path B).  The write costs 2*B*H_kv*D*s bytes whatever the
// history length ("11.7 KV Cache：形状、显存与带宽" §1.1: constant-cost append).
// prefill write: the prompt's T_p rows per (b, h) go to slots [0, lens[b]).
// Paged caches reach token t of (b, h) through the block table (cache_row); a row whose table
// entry is out of range is not written (and DEV_BAD_BLOCK is flagged).
#include "kvc_decode.cuh"

namespace kvc {

// One warp per (b, h): the T_in new rows (T_in = T_q new tokens, source [B, H_kv, T_q, D])
// go to slots [L - T_q, L) (a rolling cache: T_q = 1, slot (L - 1) mod T_max); 16-byte vectors.
__global__ void append_kernel(const CopyParams p) {
    const int gw = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= p.B * p.H_kv) return;
    const int b = gw / p.H_kv, h = gw - b * p.H_kv;
    const int L = p.lens[b];
    const int T_q = p.T_in;
    if (L < T_q || L < 1 || (!p.rolling && L > p.T_max)) {
        if (h == 0 && lane == 0) atomicOr(p.err, DEV_BAD_LENS);
        return;
    }
    const int nvec = p.row_bytes >> 4;
    for (int i = 0; i < T_q; ++i) {
        // position L - T_q + i; a rolling cache stores it at slot position mod T_max
        const int pos = L - T_q + i;
        const int slot = p.rolling ? pos % p.T_max : pos;
        const int64_t drow = cache_row(p.table, p.bs, p.max_blocks, p.num_blocks, p.H_kv, p.T_max, b,
                                       h, slot, p.err);
        if (drow < 0) continue;
        const size_t dst = (size_t)drow * p.row_bytes;
        const size_t src = ((size_t)gw * T_q + i) * p.row_bytes;
        for (int v = lane; v < nvec; v += 32) {
            const uint4 kx = __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(p.K) + src) + v);
            const uint4 vx = __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(p.V) + src) + v);
            reinterpret_cast<uint4*>(static_cast<char*>(p.Kc) + dst)[v] = kx;
            reinterpret_cast<uint4*>(static_cast<char*>(p.Vc) + dst)[v] = vx;
        }
    }
}

// Grid-stride over the 16-byte vectors of all [B, H_kv, T_in] source rows.
__global__ void prefill_kernel(const CopyParams p) {
    const int nvec = p.row_bytes >> 4;
    const size_t rows = (size_t)p.B * p.H_kv * p.T_in;
    const size_t total = rows * nvec;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        const size_t row = i / nvec;
        const int v = (int)(i - row * nvec);
        const size_t bh = row / p.T_in;
        const int t = (int)(row - bh * p.T_in);
        const int b = (int)(bh / p.H_kv);
        const int L = p.lens[b];
        if (L < 0 || L > p.T_in) {
            if (t == 0 && v == 0 && bh % p.H_kv == 0) atomicOr(p.err, DEV_BAD_LENS);
            continue;
        }
        if (t >= L) continue;
        // a rolling cache keeps the last T_max positions, position t in slot t mod T_max
        if (p.rolling && t < L - p.T_max) continue;
        const uint4 kx = __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(p.K) + row * p.row_bytes) + v);
        const uint4 vx = __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(p.V) + row * p.row_bytes) + v);
        const int64_t drow = cache_row(p.table, p.bs, p.max_blocks, p.num_blocks, p.H_kv, p.T_max, b,
                                       (int)(bh - (size_t)b * p.H_kv), p.rolling ? t % p.T_max : t,
                                       p.err);
        if (drow < 0) continue;
        reinterpret_cast<uint4*>(static_cast<char*>(p.Kc) + drow * p.row_bytes)[v] = kx;
        reinterpret_cast<uint4*>(static_cast<char*>(p.Vc) + drow * p.row_bytes)[v] = vx;
    }
}

// int8 or fp8 cache (p.Ksc set; bf16 source rows, D = 128): one warp per (b, h, row) quantizes
// the source row into codes and a row scale (q8_store_row, or f8_store_row for E4M3 codes).  Append: rows [L - T_in, L) from the
// [B, H_kv, T_in, D] source; prefill: rows [0, L) from [B, H_kv, T_in, D].
__global__ void quant_write_kernel(const CopyParams p, int prefill) {
    const size_t gw = (blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const size_t rows = (size_t)p.B * p.H_kv * p.T_in;
    if (gw >= rows) return;
    const size_t bh = gw / p.T_in;
    const int i = (int)(gw - bh * p.T_in);
    const int b = (int)(bh / p.H_kv);
    const int L = p.lens[b];
    int t;
    if (prefill) {
        if (L < 0 || L > p.T_in || L > p.T_max) {
            if (i == 0 && lane == 0 && bh % p.H_kv == 0) atomicOr(p.err, DEV_BAD_LENS);
            return;
        }
        if (i >= L) return;
        t = i;
    } else {
        if (L < p.T_in || L > p.T_max) {
            if (i == 0 && lane == 0 && bh % p.H_kv == 0) atomicOr(p.err, DEV_BAD_LENS);
            return;
        }
        t = L - p.T_in + i;
    }
    const size_t crow = bh * p.T_max + t;
    const __nv_bfloat16* ks = static_cast<const __nv_bfloat16*>(p.K) + gw * 128;
    const __nv_bfloat16* vs = static_cast<const __nv_bfloat16*>(p.V) + gw * 128;
    if (p.fp8) {
        f8_store_row(ks, static_cast<uint8_t*>(p.Kc) + crow * 128, p.Ksc + crow, lane);
        f8_store_row(vs, static_cast<uint8_t*>(p.Vc) + crow * 128, p.Vsc + crow, lane);
    } else {
        q8_store_row(ks, static_cast<int8_t*>(p.Kc) + crow * 128, p.Ksc + crow, lane);
        q8_store_row(vs, static_cast<int8_t*>(p.Vc) + crow * 128, p.Vsc + crow, lane);
    }
}

static int launch_quant_write(const CopyParams& p, int prefill, cudaStream_t s) {
    const size_t warps = (size_t)p.B * p.H_kv * p.T_in;
    const int threads = 256;
    const size_t blocks = (warps * 32 + threads - 1) / threads;
    quant_write_kernel<<<(unsigned)blocks, threads, 0, s>>>(p, prefill);
    return (int)cudaGetLastError();
}

int launch_append(const CopyParams& p, cudaStream_t s) {
    if (p.Ksc != nullptr) return launch_quant_write(p, 0, s);
    const int warps = p.B * p.H_kv;
    const int threads = 256;
    const int blocks = (warps * 32 + threads - 1) / threads;
    append_kernel<<<blocks, threads, 0, s>>>(p);
    return (int)cudaGetLastError();
}

int launch_prefill(const CopyParams& p, cudaStream_t s) {
    if (p.Ksc != nullptr) return launch_quant_write(p, 1, s);
    const size_t total = (size_t)p.B * p.H_kv * p.T_in * (p.row_bytes >> 4);
    const int threads = 256;
    size_t blocks = (total + threads - 1) / threads;
    if (blocks > 65536) blocks = 65536;
    if (blocks == 0) blocks = 1;
    prefill_kernel<<<(unsigned)blocks, threads, 0, s>>>(p);
    return (int)cudaGetLastError();
}

// A programmatic dependent launch of the combine kernel behind the decode kernel.  Column
// slices per (stream, head): doubled while the grid is smaller than the decode grid (p.P, one
// CTA per SM by default), up to 8 and while each slice keeps at least one float4 column.
int launch_combine(int dtype, int D, int G, const DecodeParams& p, cudaStream_t s) {
    const long long ug = (long long)p.B * p.H_kv * G;
    int DS = 1;
    while (DS < 8 && 2 * DS <= D / 4 && ug * DS < p.P) DS *= 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(ug * DS));
    cfg.blockDim = dim3(COMBINE_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = dtype == 0 ? cudaLaunchKernelEx(&cfg, combine_kernel<__nv_bfloat16>, p, D, G, DS)
                                     : cudaLaunchKernelEx(&cfg, combine_kernel<float>, p, D, G, DS);
    if (e != cudaSuccess) return (int)e;
    return (int)cudaGetLastError();
}

}  // namespace kvc
