// The persistent tcgen05 GEMM kernels of the prolog as templates (their
// shared-memory layouts below): the BF16 instantiations live in gemm.cu,
// the W8A8 ones (W8 = true: integer accumulators, dequantising epilogues)
// in gemm_w8a8.cu.
#pragma once

#include "engine.cuh"

namespace mlap {

// COMP: the drained chains may be summed with TwoSum (p.compensated); the
// wide tiles sum them with plain FP32 adds.
template <int BN_MAX, int STAGES, bool COMP, bool W8 = false>
__global__ void __launch_bounds__(kCompressThreads, 1)
    mla_compress_kernel(const __grid_constant__ CUtensorMap tm_x,
                        const __grid_constant__ CUtensorMap tm_wa, const CompressParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem sm = carve<BN_MAX, STAGES>(smem_raw);
    const uint32_t tmem = gemm_setup<BN_MAX, STAGES>(sm, kDrainEpiWarps);
    pdl_launch_dependents();
    RoleCounters rc;
    compress_phase<BN_MAX, STAGES, BN_MAX, 1, COMP, W8>(sm, tmem, &tm_x, &tm_wa, p, rc, blockIdx.x, gridDim.x);
    gemm_finish<BN_MAX, STAGES>(sm, tmem, rc, p.timeout_ns);
}

// TS: the kernel carries the epilogue's store staging area (the kv tiles and
// the per-token q tiles leave through bulk tensor stores when p.tma_store).
template <int BN_MAX, int STAGES, bool TS, bool W8 = false>
__global__ void __launch_bounds__(kExpandThreads, 1)
    mla_expand_kernel(const __grid_constant__ CUtensorMap tm_aq,
                      const __grid_constant__ CUtensorMap tm_akv,
                      const __grid_constant__ CUtensorMap tm_bq,
                      const __grid_constant__ CUtensorMap tm_bkv,
                      const __grid_constant__ CUtensorMap tm_bkvh,
                      const __grid_constant__ CUtensorMap tm_oq,
                      const __grid_constant__ CUtensorMap tm_ok,
                      const __grid_constant__ CUtensorMap tm_ov, const ExpandParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem sm = carve<BN_MAX, STAGES, 1, TS ? kStoreStageBytes : 0>(smem_raw);
    const uint32_t tmem = gemm_setup<BN_MAX, STAGES>(sm, kExpandEpiWarps);
    pdl_launch_dependents();
    RoleCounters rc;
    const CtaJobs jobs(p.job_table, expand_njobs(p));
    expand_phase<BN_MAX, STAGES, 1, TS, W8>(sm, tmem, &tm_aq, &tm_akv, &tm_bq, &tm_bkv, &tm_bkvh, p, rc, jobs, true,
                                        OutMaps{&tm_oq, &tm_ok, &tm_ov}, [] {
                                            pdl_wait();
                                            return true;
                                        });
    gemm_finish<BN_MAX, STAGES>(sm, tmem, rc, p.timeout_ns);
}

// Prefill compression on CTA pairs: each job is a 256-token x BN tile (M =
// 256); each CTA streams its 128 token rows and BN / 2 weight rows per K
// block and drains its own 128 rows' chains (plain FP32 sums, as the wide
// one-CTA tiles).
template <int BN_MAX, int STAGES, bool W8 = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kCompressThreads, 1)
    mla_compress_pair_kernel(const __grid_constant__ CUtensorMap tm_x,
                             const __grid_constant__ CUtensorMap tm_wa, const CompressParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem sm = carve<BN_MAX, STAGES, 2>(smem_raw);
    const uint32_t tmem = gemm_setup<BN_MAX, STAGES, 2>(sm, kDrainEpiWarps);
    pdl_launch_dependents();
    RoleCounters rc;
    compress_phase<BN_MAX, STAGES, BN_MAX, 2, false, W8>(sm, tmem, &tm_x, &tm_wa, p, rc, blockIdx.x, gridDim.x);
    gemm_finish<BN_MAX, STAGES, 2>(sm, tmem, rc, p.timeout_ns);
}

// Prefill expansion on CTA pairs (cta_group::2): each job is a 256-token x
// BN tile whose MMAs (M = 256) the even CTA issues; each CTA streams its own
// 128 token rows and half of the weight tile, so an SM receives 16 KB of
// activations + BN / 2 x 128 bytes of weights per K block instead of
// 16 KB + BN x 128 bytes for the same tensor-core work.
template <int BN_MAX, int STAGES, bool W8 = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kExpandThreads, 1)
    mla_expand_pair_kernel(const __grid_constant__ CUtensorMap tm_aq,
                           const __grid_constant__ CUtensorMap tm_akv,
                           const __grid_constant__ CUtensorMap tm_bq,
                           const __grid_constant__ CUtensorMap tm_bkv,
                           const __grid_constant__ CUtensorMap tm_oq,
                           const __grid_constant__ CUtensorMap tm_ok,
                           const __grid_constant__ CUtensorMap tm_ov, const ExpandParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem sm = carve<BN_MAX, STAGES, 2, kStoreStageBytes>(smem_raw);
    const uint32_t tmem = gemm_setup<BN_MAX, STAGES, 2>(sm, kExpandEpiWarps);
    pdl_launch_dependents();
    RoleCounters rc;
    const CtaJobs jobs(p.job_table, (p.nq_tiles + p.nkv_tiles) * p.m_tiles, 2);
    expand_phase<BN_MAX, STAGES, 2, true, W8>(sm, tmem, &tm_aq, &tm_akv, &tm_bq, &tm_bkv, &tm_bkv, p, rc, jobs, true,
                                          OutMaps{&tm_oq, &tm_ok, &tm_ov}, [] {
                                              pdl_wait();
                                              return true;
                                          });
    gemm_finish<BN_MAX, STAGES, 2>(sm, tmem, rc, p.timeout_ns);
}

// The kv tiles of the prefill expansion on CTA pairs with the activations
// resident in shared memory (see expand_kvres_phase): super-jobs of `group`
// kv tiles per pair token tile.
template <bool W8 = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kExpandThreads, 1)
    mla_expand_kv_pair_kernel(const __grid_constant__ CUtensorMap tm_akv,
                              const __grid_constant__ CUtensorMap tm_bkv,
                              const __grid_constant__ CUtensorMap tm_ok,
                              const __grid_constant__ CUtensorMap tm_ov, const ExpandParams p, int group) {
    extern __shared__ uint8_t smem_raw[];
    const KvResSmem k = kvres_carve(smem_raw);
    const uint32_t tmem = kvres_setup(k);
    pdl_launch_dependents();
    RoleCounters rc;
    OutMaps om;
    om.k = &tm_ok;
    om.v = &tm_ov;
    expand_kvres_phase<W8>(k, tmem, &tm_akv, &tm_bkv, p, om, group, rc);
    gemm_finish<256, kKvResStages, 2>(k.s, tmem, rc, p.timeout_ns);
}

// ------------------------------------------------------ shared-memory layouts

using EWide = Layout<256, 4, 1, kStoreStageBytes>;  // + the epilogue's store staging area
using EMid = Layout<192, 5>;
using ENarrow = Layout<64, 4>;
using EDeep = Layout<64, 8>;
using EPair = Layout<256, 6, 2, kStoreStageBytes>;  // per CTA: 16 KB activations + 16 KB weights per stage
using CPair = Layout<256, 6, 2>;  // per CTA: 16 KB activations + 16 KB weights per stage
using CWide = Layout<128, 6>;
using CNarrow = Layout<64, 4>;
using C192 = Layout<192, 5>;  // 16 KB activations + 24 KB weights per stage
using C256 = Layout<256, 4>;  // 16 KB activations + 32 KB weights per stage

}  // namespace mlap
