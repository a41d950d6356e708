// kvc_selftest.cu -- a self-test of the bounded in-kernel wait (kvc_selftest_wait_timeout).
//
// Every attention kernel waits on mbarriers (tile landed, scores ready, weights written, ...)
// through mbar_wait, which gives up after a time limit, flags KVC_DEV_WAIT_TIMEOUT in the error
// word and lets the kernel run to its end instead of hanging.  In a correct launch no wait ever
// runs out, so this kernel makes one run out on purpose, without any fault: its threads wait on
// a fresh mbarrier phase that nothing completes (no thread arrives on it and no copy targets it).
#include "../../include/kvc.h"
#include "kvc_internal.cuh"

namespace kvc {

constexpr int SELFTEST_THREADS = 64;

// info[0]: threads whose wait reported completion (0 expected); info[1]: nanoseconds thread 0
// spent in its wait.
__global__ void __launch_bounds__(SELFTEST_THREADS) wait_selftest_kernel(uint32_t* err, long long* info,
                                                                         uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    __shared__ int completed;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // one arrival would complete phase 0; none comes
        abort_flag = 0;
        completed = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const uint64_t t0 = global_ns();
    const bool ok = mbar_wait(&bar, 0u, &abort_flag, err, limit_ns);
    const uint64_t t1 = global_ns();
    if (ok) atomicAdd(&completed, 1);
    __syncthreads();
    if (threadIdx.x == 0) {
        info[0] = completed;
        info[1] = (long long)(t1 - t0);
    }
}

}  // namespace kvc

extern "C" int kvc_selftest_wait_timeout(uint32_t* err, long long* info, long long limit_ns, void* stream) {
    if (!err || !info) return KVC_EINVAL;
    if ((reinterpret_cast<uintptr_t>(err) & 3) || (reinterpret_cast<uintptr_t>(info) & 7)) return KVC_EINVAL;
    if (limit_ns > (long long)kvc::WAIT_LIMIT_NS) return KVC_ERANGE;
    const uint64_t lim = limit_ns <= 0 ? kvc::WAIT_LIMIT_NS : (uint64_t)limit_ns;
    kvc::wait_selftest_kernel<<<1, kvc::SELFTEST_THREADS, 0, static_cast<cudaStream_t>(stream)>>>(err, info, lim);
    return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ECUDA;
}
