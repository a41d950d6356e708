// kvc_decode_inst.cu -- instantiates the decode-attention kernel for one (dtype, D).
// Compiled once per pair with -DKVC_INST_BF16=0|1 -DKVC_INST_D=<D>, so the instantiations
// build in parallel; G (the query-head group) is dispatched here at run time.
#include "kvc_decode.cuh"

#if !defined(KVC_INST_BF16) || !defined(KVC_INST_D)
#error "compile with -DKVC_INST_BF16=0|1 -DKVC_INST_D=<head dim>"
#endif

#define KVC_CAT3(a, b, c) a##b##c
#define KVC_NAME(dt, d) KVC_CAT3(launch_decode_, dt, d)
#if KVC_INST_BF16
#define KVC_LAUNCHER KVC_NAME(bf16_d, KVC_INST_D)
#else
#define KVC_LAUNCHER KVC_NAME(f32_d, KVC_INST_D)
#endif

namespace kvc {

#if KVC_INST_BF16
using ElemT = __nv_bfloat16;
#else
using ElemT = float;
#endif

template <int G>
static int launch_g(const DecodeParams& p, cudaStream_t s, int* smem_out) {
    using C = DecodeCfg<ElemT, KVC_INST_D, G>;
    static PerDeviceOnce smem_attr;
    const int ea = smem_attr.run([] {
        return (int)cudaFuncSetAttribute(decode_kernel<ElemT, KVC_INST_D, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    });
    if (ea != 0) return ea;
    if (smem_out) *smem_out = C::SMEM;
    decode_kernel<ElemT, KVC_INST_D, G><<<p.P, C::NTHREADS, C::SMEM, s>>>(p);
    return (int)cudaGetLastError();
}

int KVC_LAUNCHER(int G, const DecodeParams& p, cudaStream_t s, int* smem_out) {
    switch (G) {
        case 1: return launch_g<1>(p, s, smem_out);
        case 2: return launch_g<2>(p, s, smem_out);
        case 4: return launch_g<4>(p, s, smem_out);
        case 8: return launch_g<8>(p, s, smem_out);
        case 16: return launch_g<16>(p, s, smem_out);
        case 32: return launch_g<32>(p, s, smem_out);
        default: return (int)cudaErrorInvalidValue;
    }
}

}  // namespace kvc
