// The W8A8 instantiations of the GEMM kernels (W8 = true): the operands are
// INT8 codes held as BF16 integers, the accumulators exact integer sums (see
// compress_phase and w8_dequant_tile), and the epilogues dequantise.  Their
// own translation unit so that the BF16 kernels build in parallel with them.
#include "gemm_kernels.cuh"

namespace mlap {

cudaError_t gemm_w8a8_set_attributes() {
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(mla_compress_kernel<128, 6, false, true>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, CWide::BYTES)))
        return e;
    if ((e = cudaFuncSetAttribute(mla_compress_kernel<64, 4, false, true>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, CNarrow::BYTES)))
        return e;
    if ((e = cudaFuncSetAttribute(mla_compress_kernel<192, 5, false, true>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, C192::BYTES)))
        return e;
    if ((e = cudaFuncSetAttribute(mla_compress_kernel<256, 4, false, true>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, C256::BYTES)))
        return e;
    if ((e = cudaFuncSetAttribute(mla_expand_kernel<256, 4, true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  EWide::BYTES)))
        return e;
    if ((e = cudaFuncSetAttribute(mla_expand_kernel<192, 5, false, true>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, EMid::BYTES)))
        return e;
    if ((e = cudaFuncSetAttribute(mla_expand_kernel<64, 4, false, true>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, ENarrow::BYTES)))
        return e;
    if ((e = cudaFuncSetAttribute(mla_expand_kernel<64, 8, false, true>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, EDeep::BYTES)))
        return e;
    if ((e = cudaFuncSetAttribute(mla_expand_pair_kernel<256, 6, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  EPair::BYTES)))
        return e;
    if ((e = cudaFuncSetAttribute(mla_expand_kv_pair_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  KvResLayout::BYTES)))
        return e;
    return cudaSuccess;
}

cudaError_t launch_compress_w8(GemmShape s, int grid, const CUtensorMap& tm_x, const CUtensorMap& tm_wa,
                               const CompressParams& p, cudaStream_t st) {
    if (s == GemmShape::Wide)
        return launch_kernel(mla_compress_kernel<128, 6, false, true>, dim3(grid), dim3(kCompressThreads),
                             CWide::BYTES, st, false, tm_x, tm_wa, p);
    if (s == GemmShape::Wide192)
        return launch_kernel(mla_compress_kernel<192, 5, false, true>, dim3(grid), dim3(kCompressThreads),
                             C192::BYTES, st, false, tm_x, tm_wa, p);
    if (s == GemmShape::Wide256)
        return launch_kernel(mla_compress_kernel<256, 4, false, true>, dim3(grid), dim3(kCompressThreads),
                             C256::BYTES, st, false, tm_x, tm_wa, p);
    return launch_kernel(mla_compress_kernel<64, 4, false, true>, dim3(grid), dim3(kCompressThreads), CNarrow::BYTES,
                         st, false, tm_x, tm_wa, p);
}

cudaError_t launch_expand_w8(GemmShape s, int grid, const CUtensorMap& tm_aq, const CUtensorMap& tm_akv,
                             const CUtensorMap& tm_bq, const CUtensorMap& tm_bkv, const OutTensorMaps& om,
                             const ExpandParams& p, cudaStream_t st, const CUtensorMap* tm_bkvh) {
    const CUtensorMap& bkvh = tm_bkvh ? *tm_bkvh : tm_bkv;
    if (s == GemmShape::Wide)
        return launch_kernel(mla_expand_kernel<256, 4, true, true>, dim3(grid), dim3(kExpandThreads), EWide::BYTES,
                             st, true, tm_aq, tm_akv, tm_bq, tm_bkv, bkvh, om.q, om.k, om.v, p);
    if (s == GemmShape::Mid)
        return launch_kernel(mla_expand_kernel<192, 5, false, true>, dim3(grid), dim3(kExpandThreads), EMid::BYTES,
                             st, true, tm_aq, tm_akv, tm_bq, tm_bkv, bkvh, om.q, om.k, om.v, p);
    if (s == GemmShape::Deep)
        return launch_kernel(mla_expand_kernel<64, 8, false, true>, dim3(grid), dim3(kExpandThreads), EDeep::BYTES,
                             st, true, tm_aq, tm_akv, tm_bq, tm_bkv, bkvh, om.q, om.k, om.v, p);
    return launch_kernel(mla_expand_kernel<64, 4, false, true>, dim3(grid), dim3(kExpandThreads), ENarrow::BYTES, st,
                         true, tm_aq, tm_akv, tm_bq, tm_bkv, bkvh, om.q, om.k, om.v, p);
}

cudaError_t launch_expand_pair_w8(int pairs, const CUtensorMap& tm_aq, const CUtensorMap& tm_akv,
                                  const CUtensorMap& tm_bq, const CUtensorMap& tm_bkv, const OutTensorMaps& om,
                                  const ExpandParams& p, cudaStream_t st) {
    return launch_kernel(mla_expand_pair_kernel<256, 6, true>, dim3(2 * pairs), dim3(kExpandThreads), EPair::BYTES,
                         st, true, tm_aq, tm_akv, tm_bq, tm_bkv, om.q, om.k, om.v, p);
}

cudaError_t launch_expand_kv_pair_w8(int pairs, const CUtensorMap& tm_akv, const CUtensorMap& tm_bkv,
                                     const OutTensorMaps& om, const ExpandParams& p, int group, cudaStream_t st) {
    return launch_kernel(mla_expand_kv_pair_kernel<true>, dim3(2 * pairs), dim3(kExpandThreads), KvResLayout::BYTES,
                         st, true, tm_akv, tm_bkv, om.k, om.v, p, group);
}

}  // namespace mlap
