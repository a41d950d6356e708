// kvc_decode_tc_inst.cu -- instantiates the tensor-core decode kernel (bf16 cache) for one head
// dimension (-DKVC_INST_D=<D>); the query-head group G is dispatched at run time.
#include "kvc_decode_tc.cuh"

#if !defined(KVC_INST_D)
#error "compile with -DKVC_INST_D=<head dim>"
#endif

#define KVC_CAT2(a, b) a##b
#define KVC_TC_NAME(d) KVC_CAT2(launch_decode_tc_d, d)

namespace kvc {

template <int G>
static int launch_tc_g(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                       cudaStream_t s, int* smem_out) {
    using C = TcCfg<KVC_INST_D, G>;
    static PerDeviceOnce smem_attr;
    const int ea = smem_attr.run([] {
        return (int)cudaFuncSetAttribute(decode_tc_kernel<KVC_INST_D, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    });
    if (ea != 0) return ea;
    if (smem_out) *smem_out = C::SMEM;
    decode_tc_kernel<KVC_INST_D, G><<<p.P, C::NTHREADS, C::SMEM, s>>>(p, tmK, tmV);
    return (int)cudaGetLastError();
}

int KVC_TC_NAME(KVC_INST_D)(int G, const DecodeParams& p, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, cudaStream_t s, int* smem_out) {
    switch (G) {
        case 1: return launch_tc_g<1>(p, tmK, tmV, s, smem_out);
        case 2: return launch_tc_g<2>(p, tmK, tmV, s, smem_out);
        case 4: return launch_tc_g<4>(p, tmK, tmV, s, smem_out);
        case 8: return launch_tc_g<8>(p, tmK, tmV, s, smem_out);
        case 16: return launch_tc_g<16>(p, tmK, tmV, s, smem_out);
        case 32: return launch_tc_g<32>(p, tmK, tmV, s, smem_out);
        default: return (int)cudaErrorInvalidValue;
    }
}

}  // namespace kvc
