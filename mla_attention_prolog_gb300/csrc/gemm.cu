// Standalone tcgen05 GEMM kernels of the prolog (prefill, and decode
// shapes the cooperative kernel does not take): the compression projection
// (x . W_a^T, split-K partials) and the expansion projections (normed .
// W_b^T) with the split / RoPE / assemble epilogue.  Both are persistent: a
// grid of at most one CTA per SM walks a static job list (see engine.cuh).
#include "gemm_kernels.cuh"

namespace mlap {

// ------------------------------------------------------------ self-test

// One thread waits on a barrier phase that nothing completes; the bounded
// wait must give up and report it.
__global__ void mla_wait_selftest_kernel(int* status, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        const uint32_t b = smem_u32(&bar);
        mbar_init(b, 1);
        fence_barrier_init();
        if (!mbar_wait(b, 0, timeout_ns, nullptr)) atomicOr(status, kStatusWaitTimeout);
    }
}

// ------------------------------------------------------------ launchers

cudaError_t gemm_set_attributes() {
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(mla_compress_kernel<128, 6, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  CWide::BYTES)))
        return e;
    if ((e = cudaFuncSetAttribute(mla_compress_kernel<64, 4, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  CNarrow::BYTES)))
        return e;
    if ((e = cudaFuncSetAttribute(mla_compress_kernel<192, 5, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  C192::BYTES)))
        return e;
    if ((e = cudaFuncSetAttribute(mla_compress_kernel<256, 4, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  C256::BYTES)))
        return e;
    if ((e = cudaFuncSetAttribute(mla_expand_kernel<256, 4, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  EWide::BYTES)))
        return e;
    if ((e = cudaFuncSetAttribute(mla_expand_kernel<192, 5, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  EMid::BYTES)))
        return e;
    if ((e = cudaFuncSetAttribute(mla_expand_kernel<64, 4, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  ENarrow::BYTES)))
        return e;
    if ((e = cudaFuncSetAttribute(mla_expand_kernel<64, 8, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  EDeep::BYTES)))
        return e;
    if ((e = cudaFuncSetAttribute(mla_expand_pair_kernel<256, 6>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  EPair::BYTES)))
        return e;
    if ((e = cudaFuncSetAttribute(mla_expand_kv_pair_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  KvResLayout::BYTES)))
        return e;
    if ((e = cudaFuncSetAttribute(mla_compress_pair_kernel<256, 6>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  CPair::BYTES)))
        return e;
    return gemm_w8a8_set_attributes();
}

cudaError_t launch_compress(GemmShape s, int grid, const CUtensorMap& tm_x, const CUtensorMap& tm_wa,
                            const CompressParams& p, cudaStream_t st) {
    if (p.w8a8) return launch_compress_w8(s, grid, tm_x, tm_wa, p, st);
    if (s == GemmShape::Wide)
        return launch_kernel(mla_compress_kernel<128, 6, true>, dim3(grid), dim3(kCompressThreads), CWide::BYTES, st,
                             false, tm_x, tm_wa, p);
    if (s == GemmShape::Wide192)
        return launch_kernel(mla_compress_kernel<192, 5, false>, dim3(grid), dim3(kCompressThreads), C192::BYTES, st,
                             false, tm_x, tm_wa, p);
    if (s == GemmShape::Wide256)
        return launch_kernel(mla_compress_kernel<256, 4, false>, dim3(grid), dim3(kCompressThreads), C256::BYTES, st,
                             false, tm_x, tm_wa, p);
    return launch_kernel(mla_compress_kernel<64, 4, true>, dim3(grid), dim3(kCompressThreads), CNarrow::BYTES, st,
                         false, tm_x, tm_wa, p);
}

cudaError_t launch_expand(GemmShape s, int grid, const CUtensorMap& tm_aq, const CUtensorMap& tm_akv,
                          const CUtensorMap& tm_bq, const CUtensorMap& tm_bkv, const OutTensorMaps& om,
                          const ExpandParams& p, cudaStream_t st, const CUtensorMap* tm_bkvh) {
    if (p.w8a8) return launch_expand_w8(s, grid, tm_aq, tm_akv, tm_bq, tm_bkv, om, p, st, tm_bkvh);
    const CUtensorMap& bkvh = tm_bkvh ? *tm_bkvh : tm_bkv;
    if (s == GemmShape::Wide)
        return launch_kernel(mla_expand_kernel<256, 4, true>, dim3(grid), dim3(kExpandThreads), EWide::BYTES, st,
                             true, tm_aq, tm_akv, tm_bq, tm_bkv, bkvh, om.q, om.k, om.v, p);
    if (s == GemmShape::Mid)
        return launch_kernel(mla_expand_kernel<192, 5, false>, dim3(grid), dim3(kExpandThreads), EMid::BYTES, st,
                             true, tm_aq, tm_akv, tm_bq, tm_bkv, bkvh, om.q, om.k, om.v, p);
    if (s == GemmShape::Deep)
        return launch_kernel(mla_expand_kernel<64, 8, false>, dim3(grid), dim3(kExpandThreads), EDeep::BYTES, st,
                             true, tm_aq, tm_akv, tm_bq, tm_bkv, bkvh, om.q, om.k, om.v, p);
    return launch_kernel(mla_expand_kernel<64, 4, false>, dim3(grid), dim3(kExpandThreads), ENarrow::BYTES, st,
                         true, tm_aq, tm_akv, tm_bq, tm_bkv, bkvh, om.q, om.k, om.v, p);
}

cudaError_t expand_pair_max_active(int* clusters) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kExpandThreads);
    cfg.dynamicSmemBytes = EPair::BYTES;
    return cudaOccupancyMaxActiveClusters(clusters, mla_expand_pair_kernel<256, 6>, &cfg);
}

cudaError_t compress_pair_max_active(int* clusters) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kCompressThreads);
    cfg.dynamicSmemBytes = CPair::BYTES;
    return cudaOccupancyMaxActiveClusters(clusters, mla_compress_pair_kernel<256, 6>, &cfg);
}

cudaError_t launch_compress_pair(int pairs, const CUtensorMap& tm_x, const CUtensorMap& tm_wa,
                                 const CompressParams& p, cudaStream_t st) {
    return launch_kernel(mla_compress_pair_kernel<256, 6>, dim3(2 * pairs), dim3(kCompressThreads), CPair::BYTES, st,
                         false, tm_x, tm_wa, p);
}

cudaError_t launch_expand_pair(int pairs, const CUtensorMap& tm_aq, const CUtensorMap& tm_akv,
                               const CUtensorMap& tm_bq, const CUtensorMap& tm_bkv, const OutTensorMaps& om,
                               const ExpandParams& p, cudaStream_t st) {
    if (p.w8a8) return launch_expand_pair_w8(pairs, tm_aq, tm_akv, tm_bq, tm_bkv, om, p, st);
    return launch_kernel(mla_expand_pair_kernel<256, 6>, dim3(2 * pairs), dim3(kExpandThreads), EPair::BYTES, st,
                         true, tm_aq, tm_akv, tm_bq, tm_bkv, om.q, om.k, om.v, p);
}

cudaError_t expand_kv_pair_max_active(int* clusters) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kExpandThreads);
    cfg.dynamicSmemBytes = KvResLayout::BYTES;
    return cudaOccupancyMaxActiveClusters(clusters, mla_expand_kv_pair_kernel<false>, &cfg);
}

cudaError_t launch_expand_kv_pair(int pairs, const CUtensorMap& tm_akv, const CUtensorMap& tm_bkv,
                                  const OutTensorMaps& om, const ExpandParams& p, int group, cudaStream_t st) {
    if (p.w8a8) return launch_expand_kv_pair_w8(pairs, tm_akv, tm_bkv, om, p, group, st);
    return launch_kernel(mla_expand_kv_pair_kernel<false>, dim3(2 * pairs), dim3(kExpandThreads), KvResLayout::BYTES,
                         st, true, tm_akv, tm_bkv, om.k, om.v, p, group);
}

cudaError_t launch_wait_selftest(int* status, uint64_t timeout_ns, cudaStream_t st) {
    mla_wait_selftest_kernel<<<1, 32, 0, st>>>(status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace mlap
