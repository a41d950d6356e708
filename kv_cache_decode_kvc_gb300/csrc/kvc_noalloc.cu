// kvc_noalloc.cu -- decode attention that allocates no device memory.
//
// kvc_decode_attn needs a handle, and kvc_create allocates the cache and the split-T
// workspace with cudaMalloc.  Some callers cannot do that: code whose device memory is owned
// by someone else (an engine that hands a plugin its buffers at enqueue time and forbids it to
// allocate, a real-time loop where cudaMalloc's implicit device synchronisation is not
// allowed, a runtime with a fixed memory budget planned ahead).  kvc_decode_attn_noalloc serves
// them: the caller passes the cache itself, and the scratch the kernel needs (partial softmax
// states of split sequences, their arrival counters and an error word) lives in a file-scope
// __device__ array of fixed size in this translation unit.
//
// The kernel is the one kvc_decode_attn picks by default for the same cache: the tcgen05 kernel
// for a bf16 cache with D = 128 (its tensor maps are host structures, encoded per call and
// passed by value), the CUDA-core kernel otherwise; same partition (one CTA per SM) and the same
// merge rule, so the results agree with kvc_decode_attn's within rounding (the order in which a
// split stream's partial states are folded can differ between runs).
//
// The array is SCRATCH_BYTES per device that loads the library, held until the process
// exits.  Its device address is looked up once per device (cudaGetSymbolAddress) on the first
// call made with that device current; that first call should therefore come before any stream
// capture.  Every call shares the one array: calls that overlap on the GPU (different streams,
// no ordering between them) race on it and must not be made.
#include <mutex>

#include "../../include/kvc.h"
#include "kvc_internal.cuh"

namespace {

constexpr size_t SCRATCH_BYTES = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_scratch[SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
void* g_scratch_ptr[MAX_DEVICES] = {};
int g_sms[MAX_DEVICES] = {};
std::mutex g_mu;

// Device address of g_scratch and the SM count for the current device (set up once).
int scratch_for(int dev, unsigned char** ptr, int* sms) {
    if (dev < 0 || dev >= MAX_DEVICES) return KVC_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        int major = 0, minor = 0, count = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return KVC_ECUDA;
        if (!(major == 10 && minor == 3)) return KVC_EUNSUPPORTED;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return KVC_ECUDA;
        g_scratch_ptr[dev] = p;
        g_sms[dev] = count;
    }
    *ptr = static_cast<unsigned char*>(g_scratch_ptr[dev]);
    *sms = g_sms[dev];
    return KVC_OK;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

extern "C" int kvc_decode_attn_noalloc(const void* K, const void* V, int B, int H_q, int H_kv,
                                       int D, int T_max, int dtype, const void* q, void* out,
                                       const int32_t* lens, uint32_t* err, void* stream) {
    if (!K || !V || !q || !out || !lens) return KVC_EINVAL;
    // 16-byte vectors and bulk copies read K, V, q and write out; lens and err are 32-bit words
    auto misaligned = [](const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) != 0; };
    if (misaligned(K, 16) || misaligned(V, 16) || misaligned(q, 16) || misaligned(out, 16) ||
        misaligned(lens, 4) || (err && misaligned(err, 4)))
        return KVC_EINVAL;
    if (B < 1 || H_q < 1 || H_kv < 1 || T_max < 1 || H_q % H_kv != 0) return KVC_EINVAL;
    if (dtype != KVC_BF16 && dtype != KVC_F32) return KVC_EINVAL;
    if (B > kvc::MAX_B) return KVC_ERANGE;
    const int G = H_q / H_kv;
    const bool g_ok = G == 1 || G == 2 || G == 4 || G == 8 || G == 16 || G == 32;
    const bool d_ok = dtype == KVC_BF16 ? (D == 64 || D == 128 || D == 256)
                                        : (D == 4 || D == 64 || D == 128 || D == 256);
    if (!g_ok || !d_ok) return KVC_EUNSUPPORTED;
    // the kernels keep prefix sums of the sequence lengths in 32 bits
    if ((int64_t)B * T_max >= (int64_t(1) << 31)) return KVC_ERANGE;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVC_ECUDA;
    unsigned char* base = nullptr;
    int sms = 0;
    const int rc = scratch_for(dev, &base, &sms);
    if (rc != KVC_OK) return rc;

    // scratch layout: [error word | counters (U ints) | part_ml | part_o], 256-byte aligned parts
    const size_t U = (size_t)B * H_kv;
    const size_t slots = (size_t)sms + U;
    const size_t off_cnt = 256;
    const size_t off_ml = round_up(off_cnt + U * 4, 256);
    const size_t off_o = round_up(off_ml + slots * G * 2 * 4, 256);
    const size_t need = off_o + slots * G * (size_t)D * 4;
    if (need > SCRATCH_BYTES) return KVC_ERANGE;

    // the tcgen05 kernel when kvc_decode_attn would take it: bf16, D = 128, rows addressable by
    // the tensor maps' 32-bit coordinates
    const uint64_t rows = (uint64_t)B * H_kv * (uint64_t)T_max;
    CUtensorMap maps[4];
    bool tc5 = dtype == KVC_BF16 && D == 128 && rows < (1ull << 31);
    if (tc5)
        tc5 = kvc::make_kv_tensor_map(&maps[0], const_cast<void*>(K), rows, D, kvc::TC_BOX_ROWS) &&
              kvc::make_kv_tensor_map(&maps[1], const_cast<void*>(V), rows, D, kvc::TC_BOX_ROWS) &&
              kvc::make_kv3_tensor_map(&maps[2], const_cast<void*>(K), rows, kvc::TC_FULL_ROWS) &&
              kvc::make_kv3_tensor_map(&maps[3], const_cast<void*>(V), rows, kvc::TC_FULL_ROWS);

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the counters must start at zero; the error word too when the kernel writes it here
    if (cudaMemsetAsync(base, 0, off_ml, s) != cudaSuccess) return KVC_ECUDA;

    kvc::DecodeParams p{};  // contiguous cache, no overlap
    p.K = K;
    p.V = V;
    p.q = q;
    p.out = out;
    p.k_new = nullptr;
    p.v_new = nullptr;
    p.lens = lens;
    p.part_o = reinterpret_cast<float*>(base + off_o);
    p.part_ml = reinterpret_cast<float*>(base + off_ml);
    p.counters = reinterpret_cast<int*>(base + off_cnt);
    p.err = err ? err : reinterpret_cast<uint32_t*>(base);
    p.B = B;
    p.H_kv = H_kv;
    p.T_max = T_max;
    p.P = sms;
    p.min_tokens = 256;
    p.bs = 1;
    p.T_q = 1;
    const long long nseg = ((long long)sms + (long long)U - 1) / (long long)U + 1;
    p.combine_mode = (nseg * G * D * 4 > 65536) ? 1 : 0;
    p.grain = kvc::partition_grain(G, p.combine_mode, 1);
    p.qscale = (float)(1.4426950408889634 / sqrt((double)D));

    int smem = 0, e;
    if (tc5) {
        e = kvc::launch_decode_tc5_d128(G, p, maps, s, &smem);
    } else if (dtype == KVC_BF16) {
        switch (D) {
            case 64: e = kvc::launch_decode_bf16_d64(G, p, s, &smem); break;
            case 128: e = kvc::launch_decode_bf16_d128(G, p, s, &smem); break;
            default: e = kvc::launch_decode_bf16_d256(G, p, s, &smem); break;
        }
    } else {
        switch (D) {
            case 4: e = kvc::launch_decode_f32_d4(G, p, s, &smem); break;
            case 64: e = kvc::launch_decode_f32_d64(G, p, s, &smem); break;
            case 128: e = kvc::launch_decode_f32_d128(G, p, s, &smem); break;
            default: e = kvc::launch_decode_f32_d256(G, p, s, &smem); break;
        }
    }
    if (e != 0) return KVC_ECUDA;
    if (p.combine_mode == 1 && kvc::launch_combine(dtype, D, G, p, s) != 0) return KVC_ECUDA;
    return KVC_OK;
}
