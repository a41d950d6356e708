// kvc_decode_tc5_inst.cu -- instantiates the tcgen05 decode kernel (bf16 cache, D = 128); the
// query-head group G is dispatched at run time.  Compiled once per cache mode, so no kernel
// carries another mode's code: KVC_TC5_MODE = 0 contiguous (launch_decode_tc5_d128), 1 paged
// pool (launch_decode_tc5p_d128), 2 rolling cache (launch_decode_tc5r_d128), 3 int8 cache
// (launch_decode_tc5q_d128; group sizes up to 8, the converter warps leave fewer registers), 4 fp8
// cache (launch_decode_tc5f_d128; group sizes up to 8).
#include "kvc_decode_tc5.cuh"

#ifndef KVC_TC5_MODE
#define KVC_TC5_MODE 0
#endif
#if KVC_TC5_MODE == 1
#define KVC_TC5_LAUNCHER launch_decode_tc5p_d128
#elif KVC_TC5_MODE == 2
#define KVC_TC5_LAUNCHER launch_decode_tc5r_d128
#elif KVC_TC5_MODE == 3
#define KVC_TC5_LAUNCHER launch_decode_tc5q_d128
#elif KVC_TC5_MODE == 4
#define KVC_TC5_LAUNCHER launch_decode_tc5f_d128
#else
#define KVC_TC5_LAUNCHER launch_decode_tc5_d128
#endif

namespace kvc {

template <int G>
static int launch_tc5_g(const DecodeParams& p, const CUtensorMap* maps, cudaStream_t s,
                        int* smem_out) {
    using C = Tc5Cfg<G, KVC_TC5_MODE>;
    static PerDeviceOnce smem_attr;
    const int ea = smem_attr.run([] {
        return (int)cudaFuncSetAttribute(decode_tc5_kernel<G, KVC_TC5_MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    });
    if (ea != 0) return ea;
    if (smem_out) *smem_out = C::SMEM;
    // programmatic stream serialisation: this grid may be scheduled while the previous kernel on
    // the stream finishes; the kernel's griddepcontrol.wait holds every read of stream data
    // until that kernel is complete and its writes are visible
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.P);
    cfg.blockDim = dim3(tc5_threads<G, KVC_TC5_MODE>());
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, decode_tc5_kernel<G, KVC_TC5_MODE>, p, maps[0], maps[1], maps[2], maps[3]);
    if (e != cudaSuccess) return (int)e;
    return (int)cudaGetLastError();
}

int KVC_TC5_LAUNCHER(int G, const DecodeParams& p, const CUtensorMap* maps, cudaStream_t s,
                           int* smem_out) {
    switch (G) {
        case 1: return launch_tc5_g<1>(p, maps, s, smem_out);
        case 2: return launch_tc5_g<2>(p, maps, s, smem_out);
        case 4: return launch_tc5_g<4>(p, maps, s, smem_out);
        case 8: return launch_tc5_g<8>(p, maps, s, smem_out);
#if KVC_TC5_MODE != 3 && KVC_TC5_MODE != 4
        case 16: return launch_tc5_g<16>(p, maps, s, smem_out);
        case 32: return launch_tc5_g<32>(p, maps, s, smem_out);
#endif
        default: return (int)cudaErrorInvalidValue;
    }
}

}  // namespace kvc
