// Cooperative decode kernel: the whole prolog pass in one launch for batches
// of at most one 128-token tile.
//
// With so few tokens every step is latency bound, and the hand-offs between
// the four kernels (grid completion, the next kernel's CTAs waiting for an
// SM) cost as much as the work.  Here one CTA per SM runs the steps as
// phases and keeps its shared-memory ring, TMEM accumulators and barrier
// counters from one phase to the next:
//   A  compression projection (split-K partials, drained chains)
//   B  split-K reduction + BF16 cast + RMSNorm + k_pe RoPE, one token per CTA,
//      by the epilogue warps alone
//   C  expansion projections with the split / RoPE / assemble epilogues
//   D  per-token INT8 quantisation of q (q path only)
// The phases hand over through counters in global memory, not grid-wide
// barriers, so only the warps that need a result wait for it: the producer
// goes straight from the compression's loads to the expansion's weight tiles
// and waits for the norm only before its first activation tiles; the MMA
// warp waits on its ring as always; the epilogue warps wait for the
// compression before the norm and for every q tile before the quantisation.
// A grid-wide barrier costs about 2 us on GB300 (152 CTAs, two dies), so
// the weight stream must not stop at one.
//
// Counters (`DecodeParams::sync`): an epoch (runs completed) and four arrival
// counts that grow by a fixed amount per run, compared modulo 2^32 against
// (epoch + 1) x that amount.  Every CTA arrives on every counter in every run,
// also after a wait gave up, so the counts stay consistent; the last CTA to
// finish advances the epoch.  The launch is cooperative: all CTAs are
// resident, so no wait is on a CTA that has not started; every wait is
// bounded and reports MLA_STATUS_WAIT_TIMEOUT when it gives up.
#include "engine.cuh"
#include "rows.cuh"

namespace mlap {

constexpr int kDecodeThreads = kExpandThreads;  // 2 + 8 warps, as the standalone GEMM kernels
constexpr int kDecodeEpiFirst = kEpiFirst;      // the epilogue warps: threads [64, 320)
constexpr int kDecodeEpiThreads = kEpiThreads;
constexpr int kDecodeBN = 192;                  // smem ring / TMEM sized for a 192-wide q head
constexpr int kDecodeStages = 5;
constexpr int kDecodeCompressBN = 128;          // compression tile width (drain registers)
using DLayout = Layout<kDecodeBN, kDecodeStages>;
constexpr size_t kDecodeNormOff = (DLayout::BYTES + 127) & ~static_cast<size_t>(127);  // 16-byte aligned row
static_assert(kCompressThreads == kDecodeThreads, "compression and expansion roles share the CTA shape");
static_assert(kDecodeEpiThreads == 32 * kExpandEpiWarps, "the norm runs on the epilogue warps");

// Epilogue-group wait with the decode kernel's limit and status word.
__device__ __forceinline__ bool epi_wait(const unsigned* counter, unsigned target, const DecodeParams& p,
                                         const Smem& sm, int* ok_slot) {
    return epi_wait(counter, target, p.timeout_ns, p.status, sm.abort_flag, ok_slot);
}

__global__ void __launch_bounds__(kDecodeThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_wa,
                      const __grid_constant__ CUtensorMap tm_aq, const __grid_constant__ CUtensorMap tm_akv,
                      const __grid_constant__ CUtensorMap tm_bq, const __grid_constant__ CUtensorMap tm_bkv,
                      const DecodeParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ float red[2];
    __shared__ unsigned epoch_s;
    __shared__ int epi_ok;
    const Smem sm = carve<kDecodeBN, kDecodeStages>(smem_raw);
    // the norm phase's BF16 row lives after the ring (and its alignment slack)
    uint16_t* crow = reinterpret_cast<uint16_t*>(smem_raw + kDecodeNormOff);
    if (threadIdx.x == 0) epoch_s = *reinterpret_cast<volatile unsigned*>(p.sync + kSyncEpoch);
    const uint32_t tmem = gemm_setup<kDecodeBN, kDecodeStages>(sm, kExpandEpiWarps);  // includes __syncthreads
    const unsigned run = epoch_s + 1u;
    const unsigned grid = gridDim.x;
    const int warp = threadIdx.x >> 5;
    const bool epi = warp >= 2;
    RoleCounters rc;
    const CtaJobs jobs(p.b.job_table, (p.b.nq_tiles + p.b.nkv_tiles) * p.b.m_tiles);

    // A: compression projection (all roles)
    bool ok = compress_phase<kDecodeBN, kDecodeStages, kDecodeCompressBN>(sm, tmem, &tm_x, &tm_wa, p.a, rc,
                                                                          blockIdx.x, gridDim.x);
    if (epi) {
        // B: once every CTA's partials are out, the norm of this CTA's tokens
        // (`ok` is uniform over the epilogue group from here on)
        ok = epi_arrive(p.sync + kSyncCompressed, 1u, ok);
        ok = epi_wait(p.sync + kSyncCompressed, run * grid, p, sm, &epi_ok) && ok;
        for (int t = blockIdx.x; t < p.n.T; t += gridDim.x) {
            if (ok) norm_token<kDecodeEpiThreads, 8, kDecodeEpiFirst>(p.n, t, crow, red);
            epi_arrive(p.sync + kSyncNormed, 1u, true);
        }
        // The expansion epilogue's amax updates must follow every token's
        // amax clearing in the norm: acquire the norm count before them.
        ok = epi_wait(p.sync + kSyncNormed, run * static_cast<unsigned>(p.n.T), p, sm, &epi_ok) && ok;
    }

    // C: expansion projections; the producer's first activation tiles wait
    // for every token's normed row (its weight tiles do not)
    const unsigned normed_target = run * static_cast<unsigned>(p.n.T);
    const bool c_ok = expand_phase<kDecodeBN, kDecodeStages>(
        sm, tmem, &tm_aq, &tm_akv, &tm_bq, &tm_bkv, &tm_bkv, p.b, rc, jobs, false, OutMaps{}, [&] {
            const bool got = wait_counter(p.sync + kSyncNormed, normed_target, p.timeout_ns, sm.abort_flag);
            if (!got) atomicOr(p.status, kStatusWaitTimeout);
            fence_proxy_async_global();  // the normed rows were written with plain stores
            return got;
        });
    ok = ok && c_ok;

    // D: per-token INT8 quantisation of q, once every q tile is out
    if (epi && p.q.rows > 0) {
        ok = epi_arrive(p.sync + kSyncExpanded, 1u, ok);
        ok = epi_wait(p.sync + kSyncExpanded, run * grid, p, sm, &epi_ok) && ok;
        if (ok) {  // no barrier inside: a per-thread loop
            const int chunks = (p.q.row_len + p.q.chunk - 1) / p.q.chunk;
            for (int k = blockIdx.x; k < p.q.rows * chunks; k += gridDim.x) {
                const int row = k / chunks, c = k - row * chunks;
                const int c0 = c * p.q.chunk;
                const int c1 = c0 + p.q.chunk < p.q.row_len ? c0 + p.q.chunk : p.q.row_len;
                quant_span(p.q, row, c0, c1, __uint_as_float(p.q.amax[row]), threadIdx.x - kDecodeEpiFirst,
                           kDecodeEpiThreads);
            }
        }
    }
    gemm_finish<kDecodeBN, kDecodeStages>(sm, tmem, rc, p.timeout_ns);  // includes __syncthreads
    // the last CTA out advances the epoch for the next run
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned ticket = atomicAdd(p.sync + kSyncFinished, 1u);
        if (ticket + 1u == run * grid) atomicAdd(p.sync + kSyncEpoch, 1u);
    }
}

size_t decode_smem_bytes(int NA, int R, int Lq, int Lkv) {
    return kDecodeNormOff + norm_token_smem_bytes(NA, R, Lq, Lkv);
}

cudaError_t decode_set_attributes(size_t smem) {
    return cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem));
}

cudaError_t decode_occupancy(size_t smem, int* blocks_per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, mla_decode_kernel, kDecodeThreads, smem);
}

cudaError_t launch_decode(int grid, size_t smem, const CUtensorMap& tm_x, const CUtensorMap& tm_wa,
                          const CUtensorMap& tm_aq, const CUtensorMap& tm_akv, const CUtensorMap& tm_bq,
                          const CUtensorMap& tm_bkv, const DecodeParams& p, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kDecodeThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mla_decode_kernel, tm_x, tm_wa, tm_aq, tm_akv, tm_bq, tm_bkv, p);
}

}  // namespace mlap
