// Cooperative decode kernel: the whole prolog pass in one launch for batches
// of at most one 128-token tile.
//
// With so few tokens every step of the multi-kernel pipeline is latency
// bound, and the hand-offs between kernels (grid completion, the next
// kernel's CTAs waiting for shared memory and registers on each SM) cost as
// much as the work.  Here one CTA per SM runs the four steps as phases
// separated by grid-wide barriers, keeping its shared-memory ring, TMEM
// accumulators and barrier phase counters from one phase to the next:
//   A  compression projection (split-K partials, drained chains)
//   B  split-K reduction + BF16 cast + RMSNorm + k_pe RoPE, one token per CTA
//   C  expansion projections with the split / RoPE / assemble epilogues
//   D  per-token INT8 quantisation of q (q path only)
// During A, each CTA already prefetches (into L2) the first weights it will
// stream in C.  The launch is cooperative, so all CTAs are resident and the
// barriers cannot wait on a CTA that has not started; every barrier wait is
// bounded and reports MLA_STATUS_WAIT_TIMEOUT when it gives up.
//
// Measured on GB300 the kernel loses to the four-kernel path: one grid-wide
// barrier over 152 CTAs costs about 2 us even when every CTA arrives at once
// (atomic counter, acquire/release atomics, a two-level tree and a per-CTA
// flag array all land at 1.9-2.9 us), and each barrier here also drains the
// phase's outstanding stores, while the four kernels hand off with
// programmatic dependent launch and overlap each prologue with the previous
// kernel's tail.  It stays selectable (MLA_TUNE_DECODE_FUSED) and is held to
// bit-identical output with the four kernels.
#include "engine.cuh"
#include "rows.cuh"

namespace mlap {

constexpr int kDecodeThreads = kExpandThreads;  // 2 + 8 warps, as the standalone GEMM kernels
constexpr int kDecodeWarps = kDecodeThreads / 32;
constexpr int kDecodeBN = 192;                  // smem ring / TMEM sized for a 192-wide q head
constexpr int kDecodeStages = 5;
constexpr int kDecodeCompressBN = 128;          // compression tile width (drain registers)
using DLayout = Layout<kDecodeBN, kDecodeStages>;
constexpr size_t kDecodeNormOff = (DLayout::BYTES + 127) & ~static_cast<size_t>(127);  // 16-byte aligned row
static_assert(kCompressThreads == kDecodeThreads, "compression and expansion roles share the CTA shape");

// All-CTA barrier on a generation counter: bar[0] counts arrivals, bar[1] is
// the generation.  The last CTA to arrive resets the count and bumps the
// generation; the others wait (bounded) for the bump.  Writes before the
// barrier are visible to every CTA after it.  Returns, uniformly over the
// CTA, whether every thread of this CTA came in with `ok` and the wait did
// not give up.
__device__ __forceinline__ bool grid_barrier(bool ok_in, unsigned* bar, uint64_t timeout_ns, int* status,
                                             int* ok_slot) {
    const int all_ok = __syncthreads_and(ok_in ? 1 : 0);
    if (threadIdx.x == 0) {
        int ok = 1;
        volatile unsigned* vgen = bar + 1;
        const unsigned gen = *vgen;
        __threadfence();
        const unsigned arrived = atomicAdd(bar, 1u) + 1u;
        if (arrived == gridDim.x) {
            atomicExch(bar, 0u);
            __threadfence();
            atomicAdd(bar + 1, 1u);
        } else {
            const uint64_t t0 = global_timer_ns();
            while (*vgen == gen) {
                __nanosleep(64);
                if (global_timer_ns() - t0 > timeout_ns) {
                    ok = 0;
                    atomicOr(status, kStatusWaitTimeout);
                    break;
                }
            }
        }
        __threadfence();
        *ok_slot = ok && all_ok;
    }
    __syncthreads();
    // global data written by generic stores is read next by TMA (async proxy)
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return *ok_slot != 0;
}

__global__ void __launch_bounds__(kDecodeThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_wa,
                      const __grid_constant__ CUtensorMap tm_aq, const __grid_constant__ CUtensorMap tm_akv,
                      const __grid_constant__ CUtensorMap tm_bq, const __grid_constant__ CUtensorMap tm_bkv,
                      const DecodeParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ float red[2 * kDecodeWarps];
    __shared__ int bar_ok;
    const Smem sm = carve<kDecodeBN, kDecodeStages>(smem_raw);
    // the norm phase's BF16 row lives after the ring (and its alignment slack)
    uint16_t* crow = reinterpret_cast<uint16_t*>(smem_raw + kDecodeNormOff);
    const uint32_t tmem = gemm_setup<kDecodeBN, kDecodeStages>(sm, kExpandEpiWarps);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    RoleCounters rc;
    const CtaJobs jobs(p.b.job_table, (p.b.nq_tiles + p.b.nkv_tiles) * p.b.m_tiles);

    // Phase C's first weights, into L2 while A streams W_a (an idle lane of
    // the MMA warp; capped so that the partials of A stay resident).
    if (warp == 1 && lane == 1 && jobs.begin < jobs.end) {
        int tile, m;
        expand_job(p.b, jobs[jobs.begin], tile, m);
        const size_t cap = p.early_prefetch_bytes;
        if (tile < p.b.nq_tiles) {
            const size_t head = static_cast<size_t>(p.b.Dn + p.b.R) * p.b.Lq * 2;
            prefetch_slab(static_cast<const char*>(p.b.w_qb) + head * tile, head < cap ? head : cap);
        } else {
            const int n0 = (tile - p.b.nq_tiles) * p.b.bn_kv;
            const size_t bytes = static_cast<size_t>(p.b.bn_kv) * p.b.Lkv * 2;
            prefetch_slab(static_cast<const char*>(p.b.w_kvb) + static_cast<size_t>(n0) * p.b.Lkv * 2,
                          bytes < cap ? bytes : cap);
        }
    }

    // A: compression projection
    bool ok = compress_phase<kDecodeBN, kDecodeStages, kDecodeCompressBN>(sm, tmem, &tm_x, &tm_wa, p.a, rc,
                                                                          blockIdx.x, gridDim.x);
    ok = grid_barrier(ok, p.bar, p.timeout_ns, p.status, &bar_ok);

    // B: norm + k_pe RoPE, one token per CTA
    if (ok)
        for (int t = blockIdx.x; t < p.n.T; t += gridDim.x) norm_token<kDecodeThreads, 16>(p.n, t, crow, red);
    ok = grid_barrier(ok, p.bar, p.timeout_ns, p.status, &bar_ok);

    // C: expansion projections
    if (ok) ok = expand_phase<kDecodeBN, kDecodeStages>(sm, tmem, &tm_aq, &tm_akv, &tm_bq, &tm_bkv, p.b, rc, jobs,
                                                        false);

    // D: per-token INT8 quantisation of q
    if (p.q.rows > 0) {
        ok = grid_barrier(ok, p.bar, p.timeout_ns, p.status, &bar_ok);
        if (ok) {
            const int chunks = (p.q.row_len + p.q.chunk - 1) / p.q.chunk;
            for (int k = blockIdx.x; k < p.q.rows * chunks; k += gridDim.x) {
                const int row = k / chunks, c = k - row * chunks;
                const int c0 = c * p.q.chunk;
                const int c1 = c0 + p.q.chunk < p.q.row_len ? c0 + p.q.chunk : p.q.row_len;
                quant_span(p.q, row, c0, c1, __uint_as_float(p.q.amax[row]), threadIdx.x, kDecodeThreads);
            }
        }
    }
    gemm_finish<kDecodeBN, kDecodeStages>(sm, tmem, rc, p.timeout_ns);
}

size_t decode_smem_bytes(int norm_row_elems) {
    return kDecodeNormOff + ((static_cast<size_t>(norm_row_elems) * 2 + 15) & ~static_cast<size_t>(15));
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
