// tcgen05 GEMM kernels of the prolog: the compression projection (x . W_a^T,
// split-K partials) and the expansion projections (normed . W_b^T) with the
// split / RoPE / assemble epilogue.
//
// One CTA computes one 128 x BN tile with six warps:
//   warp 0     TMA producer: streams 128x64 A and BNx64 B tiles (128-byte
//              swizzle) into a STAGES-deep shared-memory ring;
//   warp 1     allocates the TMEM accumulator and issues tcgen05.mma
//              (M = 128, N = BN, K = 16 per instruction) from one thread;
//              each stage is released by tcgen05.commit on its "empty" barrier;
//   warps 2-5  epilogue: after the final commit, each warp reads its 32 TMEM
//              lanes (one token row per thread) with tcgen05.ld and stores.
// All waits are bounded (see ptx.cuh); a wait that gives up sets the status
// word and the CTA still drains its copies and frees TMEM before leaving.
#include "prolog.cuh"
#include "ptx.cuh"

namespace mlap {

template <int BN_MAX, int STAGES>
struct GemmLayout {
    static constexpr int A_BYTES = kBM * kBK * 2;
    static constexpr int B_BYTES = BN_MAX * kBK * 2;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int BARS = STAGES * STAGE;
    static constexpr int MISC = BARS + (2 * STAGES + 1) * 8;
    static constexpr int BYTES = MISC + 16 + 1024;  // + slack to align the ring to 1 KB
    static constexpr uint32_t TMEM_COLS = BN_MAX <= 32 ? 32 : BN_MAX <= 64 ? 64 : BN_MAX <= 128 ? 128 : 256;
    static_assert(STAGE % 1024 == 0, "stages must keep 1 KB alignment for the swizzle atoms");
};

struct TileJob {
    const CUtensorMap* tmA;  // activations, K-major [rows, K]
    const CUtensorMap* tmB;  // weights, K-major [N, K]
    int a_row, b_row;        // first row of the A and B tiles
    int kb0, nkb;            // first K block and number of K blocks (>= 1)
    int bn;                  // tile width, multiple of 16, <= BN_MAX
};

template <int BN_MAX, int STAGES, class Epilogue>
__device__ __forceinline__ void gemm_tile(uint8_t* smem_raw, const TileJob& job,
                                          uint64_t timeout_ns, int* status, const Epilogue& epi) {
    using L = GemmLayout<BN_MAX, STAGES>;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    const uint32_t base = raw + pad;
    uint8_t* base_ptr = smem_raw + pad;
    const uint32_t full0 = base + L::BARS;
    const uint32_t empty0 = full0 + 8 * STAGES;
    const uint32_t acc_full = empty0 + 8 * STAGES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + L::MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + L::MISC + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), L::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();
    if (warp != 0) pdl_wait();  // the producer waits after its early weight loads

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tensormap(job.tmA);
            prefetch_tensormap(job.tmB);
            const uint32_t tx = static_cast<uint32_t>(L::A_BYTES + job.bn * kBK * 2);
            // The weights (B) do not depend on the previous kernel: stream the
            // first ring of them before waiting for it, then the activations.
            const int pre = job.nkb < STAGES ? job.nkb : STAGES;
            for (int i = 0; i < pre; ++i) {
                const uint32_t sa = base + i * L::STAGE;
                mbar_arrive_expect_tx(full0 + 8 * i, tx);
                tma_load_2d(sa + L::A_BYTES, job.tmB, full0 + 8 * i, (job.kb0 + i) * kBK, job.b_row);
            }
            pdl_wait();
            for (int i = 0; i < pre; ++i)
                tma_load_2d(base + i * L::STAGE, job.tmA, full0 + 8 * i, (job.kb0 + i) * kBK, job.a_row);
            int issued = pre;
            bool ok = true;
            for (int i = pre; i < job.nkb; ++i) {
                const int s = i % STAGES;
                const uint32_t ph = (i / STAGES) & 1;
                if (!mbar_wait(empty0 + 8 * s, ph ^ 1, timeout_ns, abort_flag)) { ok = false; break; }
                const uint32_t sa = base + s * L::STAGE;
                mbar_arrive_expect_tx(full0 + 8 * s, tx);
                tma_load_2d(sa, job.tmA, full0 + 8 * s, (job.kb0 + i) * kBK, job.a_row);
                tma_load_2d(sa + L::A_BYTES, job.tmB, full0 + 8 * s, (job.kb0 + i) * kBK, job.b_row);
                ++issued;
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(status, kStatusWaitTimeout);
            }
            // No copy may still be landing in shared memory when the CTA leaves.
            for (int i = issued > STAGES ? issued - STAGES : 0; i < issued; ++i)
                mbar_wait(full0 + 8 * (i % STAGES), (i / STAGES) & 1, timeout_ns, nullptr);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kBM, job.bn);
            bool ok = true;
            for (int i = 0; i < job.nkb; ++i) {
                const int s = i % STAGES;
                const uint32_t ph = (i / STAGES) & 1;
                if (!mbar_wait(full0 + 8 * s, ph, timeout_ns, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sa = base + s * L::STAGE;
                const uint64_t ad = smem_desc_sw128(sa);
                const uint64_t bd = smem_desc_sw128(sa + L::A_BYTES);
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)  // +32 bytes of K per instruction
                    mma_bf16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (i | kk) != 0);
                mma_commit(empty0 + 8 * s);
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(status, kStatusWaitTimeout);
            }
            mma_commit(acc_full);
            // The accumulator must be complete before TMEM is released.
            mbar_wait(acc_full, 0, timeout_ns, nullptr);
        }
    } else {
        bool ok = mbar_wait(acc_full, 0, timeout_ns, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        tc_fence_after();
        if (ok) {
            epi(tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16), (warp & 3) * 32 + lane);
        } else if (lane == 0) {
            atomicOr(status, kStatusWaitTimeout);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

// ------------------------------------------------------- compression (x W_a^T)
//
// The tensor core adds each K=16 product group into its FP32 accumulator with
// a limited-precision aligned sum, and that error grows with the length of
// the accumulation chain (measured on GB300: one 448-instruction chain flips
// ~0.5% of the BF16-rounded outputs against the exact sum).  The compression
// output is rounded to BF16 and then feeds the RMSNorm, the q projection and
// the per-token INT8 codes, so this kernel keeps every tensor-core chain
// short: the MMA warp restarts a fresh TMEM accumulator every `group` K
// blocks (two TMEM buffers in turn), and the epilogue warps drain each chain
// into registers with error-free TwoSum accumulation while the next chain is
// being computed.

template <int BN_MAX, int STAGES>
struct DrainLayout {
    static constexpr int A_BYTES = kBM * kBK * 2;
    static constexpr int B_BYTES = BN_MAX * kBK * 2;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int BARS = STAGES * STAGE;
    // full[S], empty[S], acc_full[2], acc_empty[2], mma_done
    static constexpr int MISC = BARS + (2 * STAGES + 5) * 8;
    static constexpr int BYTES = MISC + 16 + 1024;
    static constexpr uint32_t TMEM_COLS = 2 * BN_MAX <= 64 ? 64 : 2 * BN_MAX <= 128 ? 128 : 2 * BN_MAX <= 256 ? 256 : 512;
    static_assert(STAGE % 1024 == 0, "stages must keep 1 KB alignment for the swizzle atoms");
};

constexpr int kDrainEpiWarps = 8;  // two warps per TMEM lane quarter, one per column half
constexpr int kCompressThreads = 64 + 32 * kDrainEpiWarps;

template <int BN_MAX, int STAGES>
__global__ void __launch_bounds__(kCompressThreads, 1)
    mla_compress_kernel(const __grid_constant__ CUtensorMap tm_x,
                        const __grid_constant__ CUtensorMap tm_wa, const CompressParams p) {
    using L = DrainLayout<BN_MAX, STAGES>;
    constexpr int HALF = BN_MAX / 2;  // columns per epilogue thread
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    const uint32_t base = raw + pad;
    uint8_t* base_ptr = smem_raw + pad;
    const uint32_t full0 = base + L::BARS;
    const uint32_t empty0 = full0 + 8 * STAGES;
    const uint32_t accf0 = empty0 + 8 * STAGES;  // acc_full[2]
    const uint32_t acce0 = accf0 + 16;           // acc_empty[2]
    const uint32_t mma_done = acce0 + 16;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + L::MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + L::MISC + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int n0 = blockIdx.x * p.bn;
    const int m0 = blockIdx.y * kBM;
    const int split = blockIdx.z;
    const int kb0 = split * p.kb_total / p.splits;
    const int nkb = (split + 1) * p.kb_total / p.splits - kb0;
    const int group = p.group;
    const int ngroups = (nkb + group - 1) / group;
    const uint64_t timeout_ns = p.timeout_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, kDrainEpiWarps);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), L::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tensormap(&tm_x);
            prefetch_tensormap(&tm_wa);
            const uint32_t tx = static_cast<uint32_t>(L::A_BYTES + p.bn * kBK * 2);
            int issued = 0;
            bool ok = true;
            for (int i = 0; i < nkb; ++i) {
                const int s = i % STAGES;
                const uint32_t ph = (i / STAGES) & 1;
                if (!mbar_wait(empty0 + 8 * s, ph ^ 1, timeout_ns, abort_flag)) { ok = false; break; }
                const uint32_t sa = base + s * L::STAGE;
                mbar_arrive_expect_tx(full0 + 8 * s, tx);
                tma_load_2d(sa, &tm_x, full0 + 8 * s, (kb0 + i) * kBK, m0);
                tma_load_2d(sa + L::A_BYTES, &tm_wa, full0 + 8 * s, (kb0 + i) * kBK, n0);
                ++issued;
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.status, kStatusWaitTimeout);
            }
            for (int i = issued > STAGES ? issued - STAGES : 0; i < issued; ++i)
                mbar_wait(full0 + 8 * (i % STAGES), (i / STAGES) & 1, timeout_ns, nullptr);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kBM, p.bn);
            bool ok = true;
            int i = 0;
            for (int g = 0; g < ngroups && ok; ++g) {
                const int b = g & 1;
                // wait until the epilogue drained this buffer's previous chain
                if (!mbar_wait(acce0 + 8 * b, ((g >> 1) & 1) ^ 1, timeout_ns, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t dacc = tmem + static_cast<uint32_t>(b * BN_MAX);
                const int iend = (g + 1) * group < nkb ? (g + 1) * group : nkb;
                for (int first = 1; i < iend; ++i, first = 0) {
                    const int s = i % STAGES;
                    const uint32_t ph = (i / STAGES) & 1;
                    if (!mbar_wait(full0 + 8 * s, ph, timeout_ns, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = base + s * L::STAGE;
                    const uint64_t ad = smem_desc_sw128(sa);
                    const uint64_t bd = smem_desc_sw128(sa + L::A_BYTES);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_bf16(dacc, ad + 2 * kk, bd + 2 * kk, idesc, (first && kk == 0) ? 0u : 1u);
                    mma_commit(empty0 + 8 * s);
                }
                if (ok) mma_commit(accf0 + 8 * b);
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.status, kStatusWaitTimeout);
            }
            // Every issued MMA must have finished before TMEM is released.
            mma_commit(mma_done);
            mbar_wait(mma_done, 0, timeout_ns, nullptr);
        }
    } else {
        const int ew = warp - 2;
        const int quarter = warp & 3;             // TMEM lane quarter this warp may access
        const int half = ew >> 2;                 // column half
        const int row = quarter * 32 + lane;
        const int t = m0 + row;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        float acc[HALF], cmp[HALF];
#pragma unroll
        for (int j = 0; j < HALF; ++j) acc[j] = cmp[j] = 0.0f;
        bool ok = true;
        for (int g = 0; g < ngroups; ++g) {
            const int b = g & 1;
            bool got = mbar_wait(accf0 + 8 * b, (g >> 1) & 1, timeout_ns, abort_flag);
            got = __all_sync(0xffffffffu, got);
            if (!got) { ok = false; break; }
            tc_fence_after();
            const uint32_t src = tmem + lane_off + static_cast<uint32_t>(b * BN_MAX + half * HALF);
#pragma unroll
            for (int j = 0; j < HALF; j += 16) {
                if (half * HALF + j < p.bn) {  // warp-uniform
                    float v[16];
                    tmem_ld16(src + j, v);
#pragma unroll
                    for (int e = 0; e < 16; ++e) two_sum_add(acc[j + e], cmp[j + e], v[e]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce0 + 8 * b);
        }
        if (!ok) {
            if (lane == 0) atomicOr(p.status, kStatusWaitTimeout);
        } else if (t < p.T) {
            float* dst = p.partials + (static_cast<size_t>(split) * p.T + t) * p.NA + n0 + half * HALF;
#pragma unroll
            for (int j = 0; j < HALF; j += 4) {
                const int col = n0 + half * HALF + j;
                if (half * HALF + j < p.bn && col < p.NA)
                    *reinterpret_cast<float4*>(dst + j) =
                        make_float4(__fadd_rn(acc[j], cmp[j]), __fadd_rn(acc[j + 1], cmp[j + 1]),
                                    __fadd_rn(acc[j + 2], cmp[j + 2]), __fadd_rn(acc[j + 3], cmp[j + 3]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

// -------------------------------------------------- expansion (normed W_b^T)

template <int BN_MAX, int STAGES>
__global__ void __launch_bounds__(kGemmThreads, 1)
    mla_expand_kernel(const __grid_constant__ CUtensorMap tm_aq,
                      const __grid_constant__ CUtensorMap tm_akv,
                      const __grid_constant__ CUtensorMap tm_bq,
                      const __grid_constant__ CUtensorMap tm_bkv, const ExpandParams p) {
    extern __shared__ uint8_t smem[];
    const int m0 = blockIdx.y * kBM;
    const int tile = blockIdx.x;
    const int Dn = p.Dn, R = p.R;

    if (tile < p.nq_tiles) {
        // q head h: FP32 q, RoPE on its rope slice, per-token running max |q|.
        const int h = tile;
        const TileJob job{&tm_aq, &tm_bq, m0, h * (Dn + R), 0, p.kb_q, Dn + R};
        gemm_tile<BN_MAX, STAGES>(smem, job, p.timeout_ns, p.status,
            [&](uint32_t tbase, int row) {
                const int t = m0 + row;
                const bool in = t < p.T;
                const int pos = in ? p.positions[t] : 0;
                const bool valid = in && pos >= 0 && pos < p.max_pos;
                float* qrow = p.qws + static_cast<size_t>(t) * p.NQ + static_cast<size_t>(h) * (Dn + R);
                float amax = 0.0f;
                for (int c = 0; c < Dn; c += 16) {
                    float v[16];
                    tmem_ld16(tbase + c, v);
                    if (in) {
                        float4* d4 = reinterpret_cast<float4*>(qrow + c);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            float4 o = valid ? make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3])
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(o.x), fabsf(o.y)), fmaxf(fabsf(o.z), fabsf(o.w))));
                            d4[q] = o;
                        }
                    }
                }
                const int half = R / 2;
                const float* cs = p.cos_sin + static_cast<size_t>(valid ? pos : 0) * R;
                for (int i = 0; i < half; i += 8) {
                    float a[8], b[8];
                    tmem_ld8(tbase + Dn + i, a);
                    tmem_ld8(tbase + Dn + half + i, b);
                    if (in) {
                        float o1[8], o2[8];
                        if (valid) {
                            const float4 c0 = *reinterpret_cast<const float4*>(cs + i);
                            const float4 c1 = *reinterpret_cast<const float4*>(cs + i + 4);
                            const float4 s0 = *reinterpret_cast<const float4*>(cs + half + i);
                            const float4 s1 = *reinterpret_cast<const float4*>(cs + half + i + 4);
                            const float cc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                            const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                // x*cos + rotate_half(x)*sin, rotate_half(x1, x2) = (-x2, x1)
                                o1[e] = __fadd_rn(__fmul_rn(a[e], cc[e]), __fmul_rn(-b[e], ss[e]));
                                o2[e] = __fadd_rn(__fmul_rn(b[e], cc[e]), __fmul_rn(a[e], ss[e]));
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) o1[e] = o2[e] = 0.0f;
                        }
#pragma unroll
                        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fmaxf(fabsf(o1[e]), fabsf(o2[e])));
                        float4* d1 = reinterpret_cast<float4*>(qrow + Dn + i);
                        float4* d2 = reinterpret_cast<float4*>(qrow + Dn + half + i);
                        d1[0] = make_float4(o1[0], o1[1], o1[2], o1[3]);
                        d1[1] = make_float4(o1[4], o1[5], o1[6], o1[7]);
                        d2[0] = make_float4(o2[0], o2[1], o2[2], o2[3]);
                        d2[1] = make_float4(o2[4], o2[5], o2[6], o2[7]);
                    }
                }
                // |q| >= 0, so the order of the float bit patterns is the order of the values.
                if (valid) atomicMax(p.amax + t, __float_as_uint(amax));
            });
    } else {
        // kv tile: columns [n0, n0 + bn_kv) of [T, H, Dn + Dv]; split into
        // k_nope (into K's first Dn columns) and value.
        const int n0 = (tile - p.nq_tiles) * p.bn_kv;
        const TileJob job{&tm_akv, &tm_bkv, m0, n0, 0, p.kb_kv, p.bn_kv};
        const int HD = Dn + p.Dv;
        gemm_tile<BN_MAX, STAGES>(smem, job, p.timeout_ns, p.status,
            [&](uint32_t tbase, int row) {
                const int t = m0 + row;
                const bool in = t < p.T;
                const int pos = in ? p.positions[t] : 0;
                const bool valid = in && pos >= 0 && pos < p.max_pos;
                for (int c = 0; c < p.bn_kv; c += 16) {
                    float v[16];
                    tmem_ld16(tbase + c, v);
                    const int n = n0 + c;
                    if (in && n < p.NKV) {
                        const int h = n / HD;
                        const int j = n - h * HD;
                        uint32_t w[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) w[e] = valid ? pack_bf16x2(v[2 * e], v[2 * e + 1]) : 0u;
                        uint16_t* dst = j < Dn
                            ? p.out_k + (static_cast<size_t>(t) * p.H + h) * (Dn + R) + j
                            : p.out_v + (static_cast<size_t>(t) * p.H + h) * p.Dv + (j - Dn);
                        uint4* d4 = reinterpret_cast<uint4*>(dst);
                        d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
            });
    }
}

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

using WideL = GemmLayout<256, 4>;
using NarrowL = GemmLayout<64, 4>;
using CWideL = DrainLayout<128, 6>;
using CNarrowL = DrainLayout<64, 4>;

int gemm_smem_bytes(GemmShape s) { return s == GemmShape::Wide ? WideL::BYTES : NarrowL::BYTES; }

cudaError_t gemm_set_attributes() {
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(mla_compress_kernel<128, 6>, cudaFuncAttributeMaxDynamicSharedMemorySize, CWideL::BYTES))) return e;
    if ((e = cudaFuncSetAttribute(mla_compress_kernel<64, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, CNarrowL::BYTES))) return e;
    if ((e = cudaFuncSetAttribute(mla_expand_kernel<256, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, WideL::BYTES))) return e;
    if ((e = cudaFuncSetAttribute(mla_expand_kernel<64, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, NarrowL::BYTES))) return e;
    return cudaSuccess;
}

cudaError_t launch_compress(GemmShape s, dim3 grid, const CUtensorMap& tm_x, const CUtensorMap& tm_wa,
                            const CompressParams& p, cudaStream_t st) {
    if (s == GemmShape::Wide)
        mla_compress_kernel<128, 6><<<grid, kCompressThreads, CWideL::BYTES, st>>>(tm_x, tm_wa, p);
    else
        mla_compress_kernel<64, 4><<<grid, kCompressThreads, CNarrowL::BYTES, st>>>(tm_x, tm_wa, p);
    return cudaGetLastError();
}

cudaError_t launch_expand(GemmShape s, dim3 grid, const CUtensorMap& tm_aq, const CUtensorMap& tm_akv,
                          const CUtensorMap& tm_bq, const CUtensorMap& tm_bkv, const ExpandParams& p,
                          cudaStream_t st) {
    if (s == GemmShape::Wide)
        return launch_kernel(mla_expand_kernel<256, 4>, grid, dim3(kGemmThreads), WideL::BYTES, st, true,
                             tm_aq, tm_akv, tm_bq, tm_bkv, p);
    return launch_kernel(mla_expand_kernel<64, 4>, grid, dim3(kGemmThreads), NarrowL::BYTES, st, true,
                         tm_aq, tm_akv, tm_bq, tm_bkv, p);
}

cudaError_t launch_wait_selftest(int* status, uint64_t timeout_ns, cudaStream_t st) {
    mla_wait_selftest_kernel<<<1, 32, 0, st>>>(status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace mlap
