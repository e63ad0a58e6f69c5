// The tcgen05 GEMM engine of the prolog, shared by the standalone
// compression / expansion kernels and the cooperative decode kernel.
//
// Roles inside a CTA:
//   warp 0       TMA producer: streams 128x64 A and BNx64 B tiles (128-byte
//                swizzle) into a STAGES-deep shared-memory ring;
//   warp 1       allocates TMEM and issues tcgen05.mma (M = 128, N = BN,
//                K = 16 per instruction) from one thread, committing each
//                ring stage back to the producer;
//   warps 2-9    epilogue: read their 32 TMEM lanes (one token row per
//                thread, two warps per lane quarter splitting the columns)
//                with tcgen05.ld and finish the tile.
// TMEM holds two accumulator buffers: the MMA warp fills one while the
// epilogue drains the other, so a tile's epilogue overlaps the next tile's
// main loop.  All three roles count ring slots and accumulator "chains" with
// CTA-global counters, so the barrier phases follow from the counters alone,
// across jobs and across phases.
//
// All waits are bounded (see ptx.cuh); a wait that gives up sets the status
// word, raises the CTA's abort flag, and the CTA still waits (bounded) for
// its own copies and MMAs before freeing TMEM.
#pragma once

#include "prolog.cuh"
#include "ptx.cuh"

namespace mlap {


// CG = 2: a CTA pair (cta_group::2) -- each CTA holds its 128 rows of A and
// half of the BN_MAX rows of B per stage.  EPI_STAGE bytes after the ring
// (1 KB aligned) stage the expansion epilogue's bulk tensor stores.
template <int BN_MAX, int STAGES, int CG = 1, int EPI_STAGE = 0>
struct Layout {
    static constexpr int A_BYTES = kBM * kBK * 2;
    static constexpr int B_BYTES = BN_MAX / CG * kBK * 2;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int RING = STAGES * STAGE;
    // full[S], empty[S], acc_full[2], acc_empty[2], mma_done
    static constexpr int MISC = RING + EPI_STAGE + (2 * STAGES + 5) * 8;
    static constexpr int BYTES = MISC + 16 + 1024;  // + slack to align the ring to 1 KB
    static constexpr uint32_t TMEM_COLS =
        2 * BN_MAX <= 32 ? 32 : 2 * BN_MAX <= 64 ? 64 : 2 * BN_MAX <= 128 ? 128 : 2 * BN_MAX <= 256 ? 256 : 512;
    static_assert(STAGE % 1024 == 0, "stages must keep 1 KB alignment for the swizzle atoms");
    static_assert(2 * BN_MAX <= 512, "two accumulators must fit in TMEM");
    static_assert(EPI_STAGE % 1024 == 0, "the staging area keeps 1 KB alignment");
};

struct Smem {
    uint32_t base;   // 1 KB aligned start of the ring
    uint32_t stage;  // the epilogue's store staging area (after the ring)
    uint32_t full0, empty0, accf0, acce0, done;
    uint32_t* tmem_slot;
    volatile int* abort_flag;
};

template <int BN_MAX, int STAGES, int CG = 1, int EPI_STAGE = 0>
__device__ __forceinline__ Smem carve(uint8_t* raw_ptr) {
    using L = Layout<BN_MAX, STAGES, CG, EPI_STAGE>;
    const uint32_t raw = smem_u32(raw_ptr);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    Smem s;
    s.base = raw + pad;
    s.stage = s.base + L::RING;
    s.full0 = s.stage + EPI_STAGE;
    s.empty0 = s.full0 + 8 * STAGES;
    s.accf0 = s.empty0 + 8 * STAGES;
    s.acce0 = s.accf0 + 16;
    s.done = s.acce0 + 16;
    s.tmem_slot = reinterpret_cast<uint32_t*>(raw_ptr + pad + L::MISC);
    s.abort_flag = reinterpret_cast<volatile int*>(raw_ptr + pad + L::MISC + 4);
    return s;
}

// Barrier init, TMEM allocation; returns the TMEM base address.  A pair
// allocates the same columns in both CTAs and leaves through a cluster
// barrier, so that every barrier of both CTAs exists before either uses it;
// the even CTA's accumulator-empty barriers count both CTAs' epilogue warps.
template <int BN_MAX, int STAGES, int CG = 1>
__device__ __forceinline__ uint32_t gemm_setup(const Smem& sm, int epi_warps) {
    using L = Layout<BN_MAX, STAGES, CG>;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(sm.full0 + 8 * s, 1);
            mbar_init(sm.empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(sm.accf0 + 8 * b, 1);
            mbar_init(sm.acce0 + 8 * b, epi_warps * CG);
        }
        mbar_init(sm.done, 1);
        *sm.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        if constexpr (CG == 2) {
            tmem_alloc_pair(smem_u32(sm.tmem_slot), L::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(sm.tmem_slot), L::TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (CG == 2) cluster_sync_all();
    tc_fence_after();
    return *sm.tmem_slot;
}

template <int BN_MAX, int STAGES, int CG = 1>
__device__ __forceinline__ void gemm_teardown(const Smem& sm, uint32_t tmem) {
    using L = Layout<BN_MAX, STAGES, CG>;
    tc_fence_before();
    __syncthreads();
    // a pair: no CTA frees TMEM or leaves while the other one's epilogue or
    // the even CTA's MMAs (which read both CTAs' shared memory) still run
    if constexpr (CG == 2) cluster_sync_all();
    if ((threadIdx.x >> 5) == 1) {
        tc_fence_after();
        if constexpr (CG == 2)
            tmem_dealloc_pair(tmem, L::TMEM_COLS);
        else
            tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

__device__ __forceinline__ void raise_abort(const Smem& sm, int* status) {
    *sm.abort_flag = 1;
    atomicOr(status, kStatusWaitTimeout);
}

// Producer: streams the nkb K blocks of one job.  `loads` counts ring slots
// filled so far by this CTA (slot = loads % STAGES, pass = loads / STAGES).
// With `weights_first` (the first job after a dependency: the previous
// kernel of a programmatic dependent launch, or an earlier phase of the
// same grid) the weight tiles of up to one ring pass are issued as their
// slots free up, then `dep()` waits for the activations to exist, then the
// activation tiles of those slots follow.
//
// A pair (CG = 2): each CTA's producer loads its own halves into its own
// ring -- A rows a_row + 128 * rank, B rows b_row + bn / 2 * rank -- and the
// copies of both CTAs complete on the even CTA's full barrier, whose expected
// byte count (both halves) only the even CTA sets.  Each CTA waits for its
// slots on its own empty barrier (the MMA commit arrives on both).
template <int BN_MAX, int STAGES, int CG = 1, class Dep>
__device__ __forceinline__ bool produce_job(const Smem& sm, uint32_t& loads, const CUtensorMap* tmA,
                                            const CUtensorMap* tmB, int a_row, int b_row, int kb0, int nkb,
                                            int bn, bool weights_first, uint64_t timeout_ns, Dep&& dep,
                                            uint64_t pol_a, uint64_t pol_b) {
    using L = Layout<BN_MAX, STAGES, CG>;
    const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    const int b_rows = bn / CG;
    const uint32_t tx = static_cast<uint32_t>(CG * (L::A_BYTES + b_rows * kBK * 2));
    a_row += static_cast<int>(rank) * kBM;
    b_row += static_cast<int>(rank) * b_rows;
    auto full_bar = [&](int s) -> uint32_t {
        if constexpr (CG == 2) return map_shared_rank(sm.full0 + 8 * s, 0);
        return sm.full0 + 8 * s;
    };
    auto load = [&](uint32_t dst, const CUtensorMap* map, int s, int c0, int c1, uint64_t pol) {
        if constexpr (CG == 2)
            tma_load_2d_pair_hint(dst, map, full_bar(s), c0, c1, pol);
        else
            tma_load_2d_hint(dst, map, full_bar(s), c0, c1, pol);
    };
    int i = 0;
    if (weights_first) {
        const int pre = nkb < STAGES ? nkb : STAGES;
        for (int k = 0; k < pre; ++k) {
            const uint32_t l = loads + k;
            const int s = l % STAGES;
            if (!mbar_wait(sm.empty0 + 8 * s, ((l / STAGES) & 1) ^ 1, timeout_ns, sm.abort_flag)) return false;
            if (leader) mbar_arrive_expect_tx(sm.full0 + 8 * s, tx);
            load(sm.base + s * L::STAGE + L::A_BYTES, tmB, s, (kb0 + k) * kBK, b_row, pol_b);
        }
        // The weight tiles above are in flight: their slots must still be
        // completed (the activation tiles) even when the wait gives up.
        const bool dep_ok = dep();
        for (int k = 0; k < pre; ++k) {
            const int s = (loads + k) % STAGES;
            load(sm.base + s * L::STAGE, tmA, s, (kb0 + k) * kBK, a_row, pol_a);
        }
        i = pre;
        loads += pre;
        if (!dep_ok) return false;
    }
    for (; i < nkb; ++i, ++loads) {
        const int s = loads % STAGES;
        const uint32_t ph = (loads / STAGES) & 1;
        if (!mbar_wait(sm.empty0 + 8 * s, ph ^ 1, timeout_ns, sm.abort_flag)) return false;
        const uint32_t sa = sm.base + s * L::STAGE;
        if (leader) mbar_arrive_expect_tx(sm.full0 + 8 * s, tx);
        load(sa, tmA, s, (kb0 + i) * kBK, a_row, pol_a);
        load(sa + L::A_BYTES, tmB, s, (kb0 + i) * kBK, b_row, pol_b);
    }
    return true;
}

// No copy may still be landing in shared memory when the CTA leaves.
template <int STAGES>
__device__ __forceinline__ void drain_loads(const Smem& sm, uint32_t loads, uint64_t timeout_ns) {
    for (uint32_t l = loads > STAGES ? loads - STAGES : 0; l < loads; ++l)
        mbar_wait(sm.full0 + 8 * (l % STAGES), (l / STAGES) & 1, timeout_ns, nullptr);
}

// MMA issuer: one accumulation chain of nkb K blocks into TMEM buffer
// (chain & 1), after the epilogue released that buffer's previous chain.  A
// pair's chain is issued by the even CTA (M = 256, idesc to match) and its
// commits arrive on the barriers of both CTAs.
template <int BN_MAX, int STAGES, int CG = 1>
__device__ __forceinline__ bool mma_chain(const Smem& sm, uint32_t& consumed, uint32_t chain, int nkb,
                                          uint32_t tmem, uint32_t idesc, uint64_t timeout_ns) {
    using L = Layout<BN_MAX, STAGES, CG>;
    const uint32_t b = chain & 1;
    if (!mbar_wait(sm.acce0 + 8 * b, ((chain >> 1) & 1) ^ 1, timeout_ns, sm.abort_flag)) return false;
    tc_fence_after();
    const uint32_t dacc = tmem + b * BN_MAX;
    for (int i = 0; i < nkb; ++i, ++consumed) {
        const int s = consumed % STAGES;
        const uint32_t ph = (consumed / STAGES) & 1;
        if (!mbar_wait(sm.full0 + 8 * s, ph, timeout_ns, sm.abort_flag)) return false;
        tc_fence_after();
        const uint32_t sa = sm.base + s * L::STAGE;
        const uint64_t ad = smem_desc_sw128(sa);
        const uint64_t bd = smem_desc_sw128(sa + L::A_BYTES);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {  // +32 bytes of K per instruction
            if constexpr (CG == 2)
                mma_bf16_pair(dacc, ad + 2 * kk, bd + 2 * kk, idesc, (i == 0 && kk == 0) ? 0u : 1u);
            else
                mma_bf16(dacc, ad + 2 * kk, bd + 2 * kk, idesc, (i == 0 && kk == 0) ? 0u : 1u);
        }
        if constexpr (CG == 2)
            mma_commit_pair(sm.empty0 + 8 * s, 0x3);
        else
            mma_commit(sm.empty0 + 8 * s);
    }
    if constexpr (CG == 2)
        mma_commit_pair(sm.accf0 + 8 * b, 0x3);
    else
        mma_commit(sm.accf0 + 8 * b);
    return true;
}

// Epilogue side of a chain: wait for it (warp-uniform result) ...
__device__ __forceinline__ bool epi_acquire(const Smem& sm, uint32_t chain, uint64_t timeout_ns) {
    bool got = mbar_wait(sm.accf0 + 8 * (chain & 1), (chain >> 1) & 1, timeout_ns, sm.abort_flag);
    got = __all_sync(0xffffffffu, got);
    tc_fence_after();
    return got;
}

// ... and hand the buffer back to the MMA warp (one arrival per warp; a
// pair's odd CTA arrives on the even CTA's barrier).
template <int CG = 1>
__device__ __forceinline__ void epi_release(const Smem& sm, uint32_t chain) {
    tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
        if (CG == 2 && cluster_ctarank() != 0)
            mbar_arrive_cluster(map_shared_rank(sm.acce0 + 8 * (chain & 1), 0));
        else
            mbar_arrive(sm.acce0 + 8 * (chain & 1));
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
// blocks, and the epilogue warps drain each chain into registers (TwoSum
// error-free accumulation, or plain FP32 adds) while the next chain runs.

constexpr int kDrainEpiWarps = 8;  // two warps per TMEM lane quarter, one per column half
constexpr int kCompressThreads = 64 + 32 * kDrainEpiWarps;


// -------------------------------------------------- expansion (normed W_b^T)

constexpr int kExpandEpiWarps = 8;  // two warps per TMEM lane quarter, one per column half
constexpr int kExpandThreads = 64 + 32 * kExpandEpiWarps;

// The epilogue warps as one thread group, threads [kEpiFirst, kExpandThreads),
// synchronised on named barrier 1 while the producer and MMA warps work on.
constexpr int kEpiFirst = 64;
constexpr int kEpiThreads = kExpandThreads - kEpiFirst;

// Epilogue-group arrival on a counter in global memory: the group meets at
// a named barrier, then one thread adds `n` with release semantics at GPU
// scope -- a release is cumulative, so it publishes every write the group
// made before the barrier.  Returns the AND of `ok` over the group, so that
// the group's next steps (and their named barriers) stay uniform even when
// one warp's wait gave up.
__device__ __forceinline__ bool epi_arrive(unsigned* counter, unsigned n, bool ok) {
    const bool all = named_bar_and(1, kEpiThreads, ok);
    if (threadIdx.x == kEpiFirst) red_release_gpu_add(counter, n);
    return all;
}

// Epilogue-group wait: one thread waits (bounded) until the counter reaches
// `target` (modulo 2^32), the group follows.  Returns, uniformly over the
// group, whether the count was reached; a wait that gives up sets
// kStatusWaitTimeout.  `ok_slot` is one int of shared memory.
__device__ __forceinline__ bool epi_wait(const unsigned* counter, unsigned target, uint64_t timeout_ns, int* status,
                                         const volatile int* abort_flag, int* ok_slot) {
    if (threadIdx.x == kEpiFirst) {
        const bool got = wait_counter(counter, target, timeout_ns, abort_flag);
        if (!got) atomicOr(status, kStatusWaitTimeout);
        *ok_slot = got;
    }
    named_bar_sync(1, kEpiThreads);
    return *ok_slot != 0;
}

// ---- epilogue stores through shared memory --------------------------------
//
// Each epilogue warp owns two 2 KB slots of the staging area.  A slot holds
// one box of an output tensor: the warp's 32 token rows x 64 bytes (16 FP32
// or 32 BF16 columns), row r at byte 64 r with its 16-byte chunk j at chunk
// j ^ ((r >> 1) & 3) -- the tensor map's 64-byte swizzle, under which the 32
// lanes' 16-byte writes hit distinct banks eight rows at a time.  The warp
// fills both slots, makes them visible to the async proxy with one fence,
// and lane 0 issues the two tensor stores as one bulk group; before the
// slots are filled again lane 0 waits until that group has read them.  The
// store writes whole 64-byte row pieces and clips rows past the tensor's end.
constexpr int kStoreSlotBytes = 32 * 64;
constexpr int kStoreStageBytes = kExpandEpiWarps * 2 * kStoreSlotBytes;

struct OutMaps {
    const CUtensorMap* q = nullptr;  // FP32 q workspace [T][NQ], boxes of 16 columns x 32 rows
    const CUtensorMap* k = nullptr;  // out_k [T][H (Dn + R)] BF16, boxes of 32 x 32
    const CUtensorMap* v = nullptr;  // out_v [T][H Dv] BF16, boxes of 32 x 32
};

struct StoreRing {
    uint32_t slots;   // this warp's two slots
    uint64_t policy;  // L2 priority of the stored lines (0: none)
};

// This lane's 16 words of one box row into slot `slot`.
__device__ __forceinline__ void stage_row(uint32_t slot, const uint32_t* w) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t row = slot + lane * 64u;
    const uint32_t sw = (lane >> 1) & 3u;
#pragma unroll
    for (uint32_t j = 0; j < 4; ++j)
        st_shared_v4(row + ((j ^ sw) << 4), w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
}

// Boxes (m0, x0, y) and, when m1 is not null, (m1, x1, y) -- elements, rows
// -- from this lane's words w0 / w1 of row y + lane.  Warp-uniform; boxes
// whose rows all lie past the end (`issue` false) are skipped.
__device__ __forceinline__ void store_boxes(const StoreRing& sr, const CUtensorMap* m0, int x0,
                                            const CUtensorMap* m1, int x1, int y, bool issue, const uint32_t* w0,
                                            const uint32_t* w1) {
    if (!issue) return;
    const int lane = threadIdx.x & 31;
    if (lane == 0) bulk_wait_read0();
    __syncwarp();
    stage_row(sr.slots, w0);
    if (m1) stage_row(sr.slots + kStoreSlotBytes, w1);
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d_hint(m0, sr.slots, x0, y, sr.policy);
        if (m1) tma_store_2d_hint(m1, sr.slots + kStoreSlotBytes, x1, y, sr.policy);
        bulk_commit();
    }
}

// FP32 values: 16 per box.
__device__ __forceinline__ void store_boxes_f32(const StoreRing& sr, const CUtensorMap* map, int x0, int x1,
                                                bool two, int y, bool issue, const float* v0, const float* v1) {
    uint32_t w0[16], w1[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) w0[e] = __float_as_uint(v0[e]), w1[e] = __float_as_uint(v1[e]);
    store_boxes(sr, map, x0, two ? map : nullptr, x1, y, issue, w0, w1);
}

// Job j -> (tile, token tile).  Tiles [0, nq_tiles) are q heads, the rest kv
// tiles.  Jobs go through the tiles in groups of group_n: all token tiles of
// a group before the next group, so the weights of a group stay in L2 while
// every token tile passes through them.
// With kv_halves, job ids from full - kv_halves on are half tiles: c0 is
// the first column within the tile and width the columns the job covers.
__device__ __forceinline__ void expand_job(const ExpandParams& p, int j, int& tile, int& m_tile, int& c0,
                                           int& width) {
    const int ntiles = p.nq_tiles + p.nkv_tiles;
    const int from = ntiles * p.m_tiles - p.kv_halves;
    c0 = 0;
    width = p.bn_kv;
    if (p.kv_halves > 0 && j >= from) {
        const int h = j - from;
        j = from + h / 2;
        width = p.bn_kv / 2;
        c0 = (h & 1) * width;
    }
    const int per_group = p.group_n * p.m_tiles;
    const int g = j / per_group, r = j - g * per_group;
    const int gw = ntiles - g * p.group_n < p.group_n ? ntiles - g * p.group_n : p.group_n;
    m_tile = r / gw;
    tile = g * p.group_n + (r - m_tile * gw);
}

__device__ __forceinline__ void expand_job(const ExpandParams& p, int j, int& tile, int& m_tile) {
    int c0, width;
    expand_job(p, j, tile, m_tile, c0, width);
}

// Jobs of the expansion (the half tiles count one each).
__device__ __forceinline__ int expand_njobs(const ExpandParams& p) {
    return (p.nq_tiles + p.nkv_tiles) * p.m_tiles + p.kv_halves;
}

// Per-row state of the expansion epilogue: the row's token, whether its
// position is valid, and (for the q path, R <= 64) its cos/sin row.  Loaded
// once per token tile, while the epilogue warps wait for the accumulator, so
// the RoPE does not wait on global loads between TMEM loads.
struct RowCtx {
    int t, pos;
    bool in, valid;
    float c[32], s[32];
};

__device__ __forceinline__ void load_row_ctx(const ExpandParams& p, int t, RowCtx& rc) {
    rc.t = t;
    rc.in = t < p.T;
    const int pos = rc.in ? p.positions[t] : 0;
    rc.valid = rc.in && pos >= 0 && pos < p.max_pos;
    rc.pos = rc.valid ? pos : 0;
    if (p.nq_tiles > 0 && p.R <= 64) {
        const int half = p.R / 2;
        const float* cs = p.cos_sin + static_cast<size_t>(rc.pos) * p.R;
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
            if (i < half) {
                const float4 c4 = *reinterpret_cast<const float4*>(cs + i);
                const float4 s4 = *reinterpret_cast<const float4*>(cs + half + i);
                rc.c[i] = c4.x, rc.c[i + 1] = c4.y, rc.c[i + 2] = c4.z, rc.c[i + 3] = c4.w;
                rc.s[i] = s4.x, rc.s[i + 1] = s4.y, rc.s[i + 2] = s4.z, rc.s[i + 3] = s4.w;
            }
        }
    }
}

// x*cos + rotate_half(x)*sin on 8 pairs, rotate_half(x1, x2) = (-x2, x1)
__device__ __forceinline__ void rope8(const float (&a)[8], const float (&b)[8], const float* cc, const float* ss,
                                      float (&o1)[8], float (&o2)[8]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        o1[e] = __fadd_rn(__fmul_rn(a[e], cc[e]), __fmul_rn(-b[e], ss[e]));
        o2[e] = __fadd_rn(__fmul_rn(b[e], cc[e]), __fmul_rn(a[e], ss[e]));
    }
}

// Rope pairs [i, i + 8) of a q head's rope slice, whose first column is the
// TMEM address `tr` (a head's column Dn): pair j is (j, R/2 + j), or,
// de-interleaved, (2j, 2j + 1); each value times rstd (the per-head norm)
// when `scaled`, then rotated with (cc, ss).  Zero for a row whose position
// is invalid.  Whole warp (TMEM loads).
__device__ __forceinline__ void q_rope8(const ExpandParams& p, uint32_t tr, bool valid, int i, bool scaled,
                                        float rstd, const float* cc, const float* ss, float (&o1)[8],
                                        float (&o2)[8]) {
    const int half = p.R / 2;
    float a[8], b[8];
    if (p.interleaved) {
        float v[16];
        tmem_ld16(tr + 2 * i, v);
#pragma unroll
        for (int e = 0; e < 8; ++e) a[e] = v[2 * e], b[e] = v[2 * e + 1];
    } else {
        tmem_ld8x2(tr + i, tr + half + i, a, b);
    }
    if (scaled) {
#pragma unroll
        for (int e = 0; e < 8; ++e) a[e] = __fmul_rn(a[e], rstd), b[e] = __fmul_rn(b[e], rstd);
    }
    if (valid) {
        rope8(a, b, cc, ss, o1, o2);
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) o1[e] = o2[e] = 0.0f;
    }
}

// Calls f(i, o1, o2) for every 8-pair chunk i of the row's rotated rope slice
// (see q_rope8); cos/sin from the row context (R <= 64) or the table.
template <class F>
__device__ __forceinline__ void q_rope_chunks(const ExpandParams& p, uint32_t tbase, const RowCtx& rc, bool scaled,
                                              float rstd, F&& f) {
    const int half = p.R / 2;
    if (p.R <= 64) {
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
            if (i < half) {  // warp-uniform
                float o1[8], o2[8];
                q_rope8(p, tbase + p.Dn, rc.valid, i, scaled, rstd, rc.c + i, rc.s + i, o1, o2);
                f(i, o1, o2);
            }
        }
    } else {
        const float* cs = p.cos_sin + static_cast<size_t>(rc.pos) * p.R;
        for (int i = 0; i < half; i += 8) {
            float cc[8], ss[8], o1[8], o2[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) cc[e] = cs[i + e], ss[e] = cs[half + i + e];
            q_rope8(p, tbase + p.Dn, rc.valid, i, scaled, rstd, cc, ss, o1, o2);
            f(i, o1, o2);
        }
    }
}

// Nope columns [c, c + 16) of the q head (times rstd when `scaled`; zero for
// an invalid position).  Whole warp.
__device__ __forceinline__ void q_nope16(uint32_t tbase, bool valid, int c, bool scaled, float rstd,
                                         float (&v)[16]) {
    tmem_ld16(tbase + c, v);
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = !valid ? 0.0f : scaled ? __fmul_rn(v[e], rstd) : v[e];
}

// Nope columns [c, c + 32) the same way, under one TMEM wait.
__device__ __forceinline__ void q_nope32(uint32_t tbase, bool valid, int c, bool scaled, float rstd,
                                         float (&v)[32]) {
    tmem_ld32(tbase + c, v);
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = !valid ? 0.0f : scaled ? __fmul_rn(v[e], rstd) : v[e];
}

// Symmetric INT8 code of one value: rint(v * inv) (ties to even), clamped to
// +-127, as one byte of a packed word.
__device__ __forceinline__ uint32_t q_code(float v, float inv) {
    int q = __float2int_rn(__fmul_rn(v, inv));
    q = q > 127 ? 127 : (q < -127 ? -127 : q);
    return static_cast<uint32_t>(q) & 0xFFu;
}

__device__ __forceinline__ uint32_t q_code4(const float* v, float inv) {
    return q_code(v[0], inv) | (q_code(v[1], inv) << 8) | (q_code(v[2], inv) << 16) | (q_code(v[3], inv) << 24);
}

// q head h of one token row.  Column half 0 writes the nope columns, half 1
// the rope slice.  Steps, as the q path defines them: the optional per-head
// RMSNorm (no gamma; x^2 times 1/(Dn + R), summed in column order, + eps,
// sqrt, reciprocal, x * rstd: both warps of the row compute the same rstd
// from the whole head), the RoPE of the rope slice, then either
//   per-token quant: FP32 q rows into the workspace and an atomic max of |q|
//     per token (the quant kernel finishes), or
//   per-(token, head) quant: amax of the head row (both warps, whole row),
//     inv = 127/amax, codes rint(q * inv) clamped to +-127, scale amax/127,
//     written straight from the epilogue (a zero row gives codes 0, scale 0).
// The per-head RMSNorm's 1/rms of the whole head row (1 without the norm).
// Whole warp (TMEM loads).
__device__ __forceinline__ float q_head_rstd(const ExpandParams& p, uint32_t tbase) {
    if (!p.head_norm) return 1.0f;
    float ms = 0.0f;
    for (int c = 0; c < p.Dn + p.R; c += 16) {
        float v[16];
        tmem_ld16(tbase + c, v);
#pragma unroll
        for (int e = 0; e < 16; ++e) ms = __fadd_rn(ms, __fmul_rn(__fmul_rn(v[e], v[e]), p.inv_hd));
    }
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, p.eps)));
}

__device__ __forceinline__ void expand_q_epilogue(const ExpandParams& p, uint32_t tbase, const RowCtx& rc, int h,
                                                  int half_idx) {
    const int Dn = p.Dn, R = p.R, HD = Dn + R, half = R / 2;
    const int t = rc.t;
    const bool in = rc.in, valid = rc.valid;
    const bool scaled = p.head_norm != 0;
    const float rstd = q_head_rstd(p, tbase);

    if (p.per_head) {
        float amax = 0.0f;
        for (int c = 0; c < Dn; c += 16) {
            float v[16];
            q_nope16(tbase, valid, c, scaled, rstd, v);
#pragma unroll
            for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(v[e]));
        }
        q_rope_chunks(p, tbase, rc, scaled, rstd, [&](int, const float (&o1)[8], const float (&o2)[8]) {
#pragma unroll
            for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fmaxf(fabsf(o1[e]), fabsf(o2[e])));
        });
        const float inv = amax > 0.0f ? __fdiv_rn(127.0f, amax) : 0.0f;
        int8_t* crow = p.q_codes + (static_cast<size_t>(t) * p.H + h) * HD;
        if (half_idx == 0) {
            for (int c = 0; c < Dn; c += 16) {
                float v[16];
                q_nope16(tbase, valid, c, scaled, rstd, v);
                if (in)
                    *reinterpret_cast<uint4*>(crow + c) =
                        make_uint4(q_code4(v, inv), q_code4(v + 4, inv), q_code4(v + 8, inv), q_code4(v + 12, inv));
            }
            if (in) p.q_scale[static_cast<size_t>(t) * p.H + h] = amax > 0.0f ? __fdiv_rn(amax, 127.0f) : 0.0f;
        } else {
            q_rope_chunks(p, tbase, rc, scaled, rstd, [&](int i, const float (&o1)[8], const float (&o2)[8]) {
                if (in) {
                    *reinterpret_cast<uint2*>(crow + Dn + i) = make_uint2(q_code4(o1, inv), q_code4(o1 + 4, inv));
                    *reinterpret_cast<uint2*>(crow + Dn + half + i) =
                        make_uint2(q_code4(o2, inv), q_code4(o2 + 4, inv));
                }
            });
        }
        return;
    }

    float* qrow = p.qws + static_cast<size_t>(t) * p.NQ + static_cast<size_t>(h) * HD;
    float amax = 0.0f;
    if (half_idx == 0) {
        int c = 0;
        for (; c + 32 <= Dn; c += 32) {
            float v[32];
            q_nope32(tbase, valid, c, scaled, rstd, v);
            if (in) {
#pragma unroll
                for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(v[e]));
#pragma unroll
                for (int e = 0; e < 32; e += 8)
                    st_v8(qrow + c + e, v[e], v[e + 1], v[e + 2], v[e + 3], v[e + 4], v[e + 5], v[e + 6], v[e + 7]);
            }
        }
        for (; c < Dn; c += 16) {
            float v[16];
            q_nope16(tbase, valid, c, scaled, rstd, v);
            if (in) {
#pragma unroll
                for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(v[e]));
                st_v8(qrow + c, v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7]);
                st_v8(qrow + c + 8, v[8], v[9], v[10], v[11], v[12], v[13], v[14], v[15]);
            }
        }
    } else {
        q_rope_chunks(p, tbase, rc, scaled, rstd, [&](int i, const float (&o1)[8], const float (&o2)[8]) {
            if (in) {
#pragma unroll
                for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fmaxf(fabsf(o1[e]), fabsf(o2[e])));
                st_v8(qrow + Dn + i, o1[0], o1[1], o1[2], o1[3], o1[4], o1[5], o1[6], o1[7]);
                st_v8(qrow + Dn + half + i, o2[0], o2[1], o2[2], o2[3], o2[4], o2[5], o2[6], o2[7]);
            }
        });
    }
    // |q| >= 0, so the order of the float bit patterns is the order of the values.
    if (valid) atomicMax(p.amax + t, __float_as_uint(amax));
}

// kv columns [n0, n0 + bn) of [T, H, Dn + Dv] for one token row: k_nope
// into K's first Dn columns, value into out_v, both BF16.  Column half h
// takes columns [h * bn / 2, (h + 1) * bn / 2).
__device__ __forceinline__ void expand_kv_epilogue(const ExpandParams& p, uint32_t tbase, const RowCtx& rc, int n0,
                                                   int half_idx, int width) {
    const int Dn = p.Dn, R = p.R, HD = p.Dn + p.Dv;
    const int t = rc.t;
    const int hw = width / 2;
    // 16 columns -> BF16 at K's nope slice or V (a 16-column group never
    // straddles the two: Dn and Dv are multiples of 16)
    auto store16 = [&](int c, const float* v) {
        const int n = n0 + c;
        if (rc.in && n < p.NKV) {
            const int h = n / HD;
            const int j = n - h * HD;
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = rc.valid ? pack_bf16x2(v[2 * e], v[2 * e + 1]) : 0u;
            uint16_t* dst = j < Dn ? p.out_k + (static_cast<size_t>(t) * p.H + h) * (Dn + R) + j
                                   : p.out_v + (static_cast<size_t>(t) * p.H + h) * p.Dv + (j - Dn);
            if (p.out_aligned32) {
                st_v8(dst, w);
            } else {
                uint4* d4 = reinterpret_cast<uint4*>(dst);
                d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
                d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
        }
    };
    const int c1 = (half_idx + 1) * hw;
    int c = half_idx * hw;
    for (; c + 32 <= c1; c += 32) {  // two 16-column groups per TMEM wait
        float v[32];
        tmem_ld32(tbase + c, v);
        store16(c, v);
        store16(c + 16, v + 16);
    }
    for (; c < c1; c += 16) {
        float v[16];
        tmem_ld16(tbase + c, v);
        store16(c, v);
    }
}

// The per-token q path through the store ring (R a multiple of 32, at most
// 64): the same values as expand_q_epilogue, with the columns split evenly --
// half 0 takes nope columns [0, ns), half 1 nope columns [ns, Dn) and the
// rope slice, ns = min(Dn, (Dn + R) / 2 rounded down to 16).  y0 is the
// warp's first token row.
__device__ __forceinline__ void expand_q_epilogue_ts(const ExpandParams& p, const OutMaps& om, const StoreRing& sr,
                                                     uint32_t tbase, const RowCtx& rc, int h, int half_idx, int y0) {
    const int Dn = p.Dn, R = p.R, HD = Dn + R, half = R / 2;
    const bool valid = rc.valid, issue = y0 < p.T;
    const bool scaled = p.head_norm != 0;
    const float rstd = q_head_rstd(p, tbase);
    const int ns = (HD / 2) / 16 * 16 < Dn ? (HD / 2) / 16 * 16 : Dn;
    const int c1 = half_idx ? Dn : ns;
    const int x0 = h * HD;
    float amax = 0.0f;
    int c = half_idx ? ns : 0;
    for (; c + 32 <= c1; c += 32) {
        float v[32];
        q_nope32(tbase, valid, c, scaled, rstd, v);
#pragma unroll
        for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(v[e]));
        store_boxes_f32(sr, om.q, x0 + c, x0 + c + 16, true, y0, issue, v, v + 16);
    }
    for (; c < c1; c += 16) {
        float v[16];
        q_nope16(tbase, valid, c, scaled, rstd, v);
#pragma unroll
        for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(v[e]));
        store_boxes_f32(sr, om.q, x0 + c, 0, false, y0, issue, v, v);
    }
    if (half_idx == 1) {
#pragma unroll
        for (int i = 0; i < 32; i += 16) {
            if (i < half) {  // warp-uniform
                float o1[16], o2[16];
                float a1[8], a2[8], b1[8], b2[8];
                q_rope8(p, tbase + Dn, valid, i, scaled, rstd, rc.c + i, rc.s + i, a1, a2);
                q_rope8(p, tbase + Dn, valid, i + 8, scaled, rstd, rc.c + i + 8, rc.s + i + 8, b1, b2);
#pragma unroll
                for (int e = 0; e < 8; ++e) o1[e] = a1[e], o1[8 + e] = b1[e], o2[e] = a2[e], o2[8 + e] = b2[e];
#pragma unroll
                for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fmaxf(fabsf(o1[e]), fabsf(o2[e])));
                store_boxes_f32(sr, om.q, x0 + Dn + i, x0 + Dn + half + i, true, y0, issue, o1, o2);
            }
        }
    }
    if (valid) atomicMax(p.amax + rc.t, __float_as_uint(amax));
}

// A q tile of kQWide columns starting at q column n0, across head
// boundaries (see ExpandParams::q_wide): each warp takes 128 columns as two
// 64-column pieces, either nope columns (copied) or one head's rope slice
// (rotated), through the store ring; one amax update per row.
__device__ __forceinline__ void expand_qw_epilogue_ts(const ExpandParams& p, const OutMaps& om, const StoreRing& sr,
                                                      uint32_t tbase, const RowCtx& rc, int n0, int half_idx,
                                                      int y0) {
    const int Dn = p.Dn, HD = Dn + p.R;
    const bool valid = rc.valid, issue = y0 < p.T;
    float amax = 0.0f;
#pragma unroll 1
    for (int s = 0; s < 2; ++s) {
        const int c = half_idx * (kQWide / 2) + s * 64;  // tile column
        const int g = n0 + c;                            // q column
        const int j = g - (g / HD) * HD;
        if (j >= Dn) {  // one head's rope slice: [o1 | o2], 32 pairs
#pragma unroll
            for (int side = 0; side < 2; ++side) {
                float o[32];
#pragma unroll
                for (int i = 0; i < 32; i += 8) {
                    float a1[8], a2[8];
                    q_rope8(p, tbase + c, valid, i, false, 1.0f, rc.c + i, rc.s + i, a1, a2);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        o[i + e] = side ? a2[e] : a1[e];
                        amax = fmaxf(amax, fabsf(o[i + e]));
                    }
                }
                store_boxes_f32(sr, om.q, g + 32 * side, g + 32 * side + 16, true, y0, issue, o, o + 16);
            }
        } else {
#pragma unroll
            for (int h2 = 0; h2 < 64; h2 += 32) {
                float v[32];
                q_nope32(tbase, valid, c + h2, false, 1.0f, v);
#pragma unroll
                for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(v[e]));
                store_boxes_f32(sr, om.q, g + h2, g + h2 + 16, true, y0, issue, v, v + 16);
            }
        }
    }
    if (valid) atomicMax(p.amax + rc.t, __float_as_uint(amax));
}

// The kv tile through the store ring (Dn, Dv multiples of 32, bn_kv a
// multiple of 64): 32-column groups, each all k_nope or all value.
__device__ __forceinline__ void expand_kv_epilogue_ts(const ExpandParams& p, const OutMaps& om, const StoreRing& sr,
                                                      uint32_t tbase, const RowCtx& rc, int n0, int half_idx, int y0,
                                                      int width) {
    const int Dn = p.Dn, HD = p.Dn + p.Dv, hw = width / 2;
    const bool issue = y0 < p.T;
    // 32-column group at n: its output tensor and first element
    auto dst = [&](int n, int& x) -> const CUtensorMap* {
        const int h = n / HD, j = n - h * HD;
        x = j < Dn ? h * (Dn + p.R) + j : h * p.Dv + (j - Dn);
        return j < Dn ? om.k : om.v;
    };
    const int c1 = (half_idx + 1) * hw;
    for (int c = half_idx * hw; c < c1; c += 64) {  // two 32-column groups per staging round
        const int n = n0 + c;
        if (n >= p.NKV) break;  // warp-uniform
        const bool two = c + 32 < c1 && n + 32 < p.NKV;
        float v[32];
        uint32_t w0[16], w1[16];
        tmem_ld32(tbase + c, v);
#pragma unroll
        for (int e = 0; e < 16; ++e) w0[e] = rc.valid ? pack_bf16x2(v[2 * e], v[2 * e + 1]) : 0u;
        if (two) {
            tmem_ld32(tbase + c + 32, v);
#pragma unroll
            for (int e = 0; e < 16; ++e) w1[e] = rc.valid ? pack_bf16x2(v[2 * e], v[2 * e + 1]) : 0u;
        } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) w1[e] = 0u;
        }
        int x0, x1 = 0;
        const CUtensorMap* m0 = dst(n, x0);
        const CUtensorMap* m1 = two ? dst(n + 32, x1) : nullptr;
        store_boxes(sr, m0, x0, m1, x1, y0, issue, w0, w1);
    }
}

// The jobs of this CTA (of this CTA pair when CG = 2: both CTAs of a pair
// run the same jobs): round robin over [0, njobs), or, when a balanced
// table is given, entries [table[c], table[c + 1]) of the id list that
// follows the units + 1 start offsets.
struct CtaJobs {
    const int* table;
    int unit, units;
    int begin, end;
    __device__ __forceinline__ CtaJobs(const int* t, int njobs, int cg = 1)
        : table(t), unit(static_cast<int>(blockIdx.x) / cg), units(static_cast<int>(gridDim.x) / cg) {
        if (t) {
            begin = t[unit];
            end = t[unit + 1];
        } else {
            begin = 0;
            end = (njobs - unit + units - 1) / units;
        }
    }
    __device__ __forceinline__ int operator[](int i) const {
        return table ? table[units + 1 + i] : unit + i * units;
    }
};


// Counters each role carries from one job (and one phase) to the next: ring
// slots filled (producer), ring slots consumed and accumulator chains issued
// (MMA), accumulator chains drained (epilogue).
struct RoleCounters {
    uint32_t loads = 0, consumed = 0, chain = 0;
};

// ---- compression phase: this CTA's jobs (round robin or balanced table) ---
//
// Job j = (token tile, weight tile, K split).  `first` / `stride` are this
// CTA's index and the grid size (they also split the L2 warm-up).  Returns
// false when a wait gave up (the CTA's abort flag is then raised).  With
// CG = 2 a CTA pair runs each job on a 256-token tile (M = 256, the even CTA
// issuing the MMAs), each CTA draining its own 128 rows.  COMP = false drops
// the TwoSum compensation registers (the drained chains are summed with plain
// FP32 adds whatever p.compensated says), which leaves room for 256 columns
// per tile.
template <int BN_MAX, int STAGES, int CBN, int CG = 1, bool COMP = true, bool W8 = false>
__device__ __forceinline__ bool compress_phase(const Smem& sm, uint32_t tmem, const CUtensorMap* tm_x,
                                               const CUtensorMap* tm_wa, const CompressParams& p, RoleCounters& rc,
                                               int first, int stride) {
    constexpr int HALF = CBN / 2;  // columns per epilogue thread
    const int rank = CG == 2 ? static_cast<int>(cluster_ctarank()) : 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int per_m = p.n_tiles * p.splits;
    const int njobs = p.m_tiles * per_m;
    const int group = p.group;
    auto job_of = [&](int j, int& m0, int& n0, int& split, int& kb0, int& nkb) {
        const int m = j / per_m, r = j - m * per_m;
        const int n = r / p.splits;
        split = r - n * p.splits;
        m0 = m * kBM * CG;
        n0 = n * p.bn;
        kb0 = split * p.kb_total / p.splits;
        nkb = (split + 1) * p.kb_total / p.splits - kb0;
    };
    bool ok = true;
    const CtaJobs jobs(p.job_table, njobs, CG);
    if (warp == 0 && lane != 0 && p.prefetch_l2) {
        // Warm L2 with the small inputs the norm and expansion read (cos/sin
        // rows of this batch's positions, gamma): when they run, HBM queues
        // are full of weight traffic and a miss there waits behind it.
        const int nthr = 31 * stride;
        for (int t = first * 31 + lane - 1; t < p.T; t += nthr) {
            const int pos = p.positions[t];
            if (pos >= 0 && pos < p.max_pos)
                bulk_prefetch_l2(p.cos_sin + static_cast<size_t>(pos) * p.R, static_cast<uint32_t>(p.R * 4));
        }
        if (first == 0 && lane == 1 && p.n_gamma > 0)
            bulk_prefetch_l2(p.gamma, static_cast<uint32_t>(p.n_gamma * 2));
    }
    if (warp == 0) {
        if (lane == 0) {
            prefetch_tensormap(tm_x);
            prefetch_tensormap(tm_wa);
            const uint64_t pol_a = l2_policy(p.l2_policy & kL2ActsLast ? 1 : 0);
            const uint64_t pol_w = l2_policy(p.l2_policy & kL2WeightsLast ? 1 : 0);
            for (int i = jobs.begin; i < jobs.end; ++i) {
                int m0, n0, split, kb0, nkb;
                job_of(jobs[i], m0, n0, split, kb0, nkb);
                if (!produce_job<BN_MAX, STAGES, CG>(sm, rc.loads, tm_x, tm_wa, m0, n0, kb0, nkb, p.bn, false,
                                                 p.timeout_ns, [] { return true; }, pol_a, pol_w)) {
                    raise_abort(sm, p.status);
                    ok = false;
                    break;
                }
            }
        }
        __syncwarp();
        if (p.l2_fetch_bytes > 0) {
            // Once this CTA's last operand load is issued, the expansion
            // weights stream into L2 from HBM while the compression drains
            // and the norm runs.
            constexpr uint64_t kPiece = 32768;
            const uint64_t pieces = (p.l2_fetch_bytes + kPiece - 1) / kPiece;
            for (uint64_t k = static_cast<uint64_t>(first) * 32 + lane; k < pieces;
                 k += 32ull * static_cast<uint64_t>(stride)) {
                const uint64_t off = k * kPiece;
                const uint64_t left = p.l2_fetch_bytes - off;
                bulk_prefetch_l2(p.l2_fetch + off, static_cast<uint32_t>(left < kPiece ? left : kPiece));
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {  // a pair's MMAs are issued by its even CTA
            const uint32_t idesc = idesc_bf16_f32(kBM * CG, p.bn);
            for (int i = jobs.begin; i < jobs.end && ok; ++i) {
                int m0, n0, split, kb0, nkb;
                job_of(jobs[i], m0, n0, split, kb0, nkb);
                for (int k = 0; k < nkb && ok; k += group, ++rc.chain)
                    ok = mma_chain<BN_MAX, STAGES, CG>(sm, rc.consumed, rc.chain, nkb - k < group ? nkb - k : group,
                                                       tmem, idesc, p.timeout_ns);
            }
            if (!ok) raise_abort(sm, p.status);
        }
    } else {
        const int ew = warp - 2;
        const int quarter = warp & 3;  // TMEM lane quarter this warp may access
        const int half = ew >> 2;      // column half
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        for (int i = jobs.begin; i < jobs.end && ok; ++i) {
            int m0, n0, split, kb0, nkb;
            job_of(jobs[i], m0, n0, split, kb0, nkb);
            // column pairs in packed f32x2 registers: half the drain instructions
            constexpr int NC = COMP ? HALF / 2 : 1;
            uint64_t acc[HALF / 2], cmp[NC];
#pragma unroll
            for (int c = 0; c < HALF / 2; ++c) acc[c] = 0ull;
#pragma unroll
            for (int c = 0; c < NC; ++c) cmp[c] = 0ull;
            const bool comp = COMP && p.compensated && !W8;
            constexpr bool LD32 = !COMP && HALF < 128;  // (no spills at 168 registers)
            // 16 drained columns into the sums (W8A8: each chain's sums are
            // exact integers, added in int32, two per register pair)
            auto drain16 = [&](int c, const float* v) {
                if constexpr (W8) {
#pragma unroll
                    for (int e = 0; e < 16; e += 2) {
                        const uint64_t a = acc[(c + e) / 2];
                        const uint32_t lo = static_cast<uint32_t>(a) + static_cast<uint32_t>(__float2int_rn(v[e]));
                        const uint32_t hi =
                            static_cast<uint32_t>(a >> 32) + static_cast<uint32_t>(__float2int_rn(v[e + 1]));
                        acc[(c + e) / 2] = (static_cast<uint64_t>(hi) << 32) | lo;
                    }
                } else if (comp) {
#pragma unroll
                    for (int e = 0; e < 16; e += 2)
                        two_sum_add2(acc[(c + e) / 2], cmp[COMP ? (c + e) / 2 : 0], pk2(v[e], v[e + 1]));
                } else {
#pragma unroll
                    for (int e = 0; e < 16; e += 2) acc[(c + e) / 2] = add2(acc[(c + e) / 2], pk2(v[e], v[e + 1]));
                }
            };
            for (int k = 0; k < nkb; k += group, ++rc.chain) {
                if (!epi_acquire(sm, rc.chain, p.timeout_ns)) { ok = false; break; }
                const uint32_t src = tmem + lane_off + (rc.chain & 1) * BN_MAX + half * HALF;
#pragma unroll
                for (int c = 0; c < HALF; c += 32) {
                    // warp-uniform: 32 columns under one wait where the registers allow
                    if (LD32 && c + 32 <= HALF && half * HALF + c + 32 <= p.bn) {
                        float v[32];
                        tmem_ld32(src + c, v);
                        drain16(c, v);
                        drain16(c + 16, v + 16);
                    } else {
#pragma unroll
                        for (int c2 = c; c2 < c + 32 && c2 < HALF; c2 += 16) {
                            if (half * HALF + c2 < p.bn) {
                                float v[16];
                                tmem_ld16(src + c2, v);
                                drain16(c2, v);
                            }
                        }
                    }
                }
                epi_release<CG>(sm, rc.chain);
            }
            if (!ok) break;
            const int t = m0 + rank * kBM + row;
            if (t < p.T && p.out_bf16) {  // one split: the BF16 row the norm reads
                uint16_t* dst = reinterpret_cast<uint16_t*>(p.partials) + static_cast<size_t>(t) * p.NA + n0 +
                                half * HALF;
#pragma unroll
                for (int c = 0; c < HALF; c += 8) {
                    if (half * HALF + c < p.bn && n0 + half * HALF + c < p.NA) {
                        float o[8];
                        if constexpr (W8) {  // AT-06: ((float)y * x_scale) * w_scale
                            const float sx = p.x_scale[t];
                            const float* ws = p.w_scale + n0 + half * HALF + c;
#pragma unroll
                            for (int e = 0; e < 8; e += 2) {
                                const uint64_t a = acc[(c + e) / 2];
                                o[e] = w8_dequant(static_cast<int>(static_cast<uint32_t>(a)), sx, ws[e]);
                                o[e + 1] = w8_dequant(static_cast<int>(static_cast<uint32_t>(a >> 32)), sx, ws[e + 1]);
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; e += 2)
                                upk2(COMP ? add2(acc[(c + e) / 2], cmp[COMP ? (c + e) / 2 : 0]) : acc[(c + e) / 2],
                                     o[e], o[e + 1]);
                        }
                        *reinterpret_cast<uint4*>(dst + c) = make_uint4(
                            pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                            pack_bf16x2(o[6], o[7]));
                    }
                }
            } else if (t < p.T) {
                float* dst = p.partials + (static_cast<size_t>(split) * p.T + t) * p.NA + n0 + half * HALF;
#pragma unroll
                for (int c = 0; c < HALF; c += 8) {
                    if (half * HALF + c < p.bn && n0 + half * HALF + c < p.NA) {
                        float o[8];
#pragma unroll
                        for (int e = 0; e < 8; e += 2) {
                            if constexpr (W8)  // int32 partials, summed and dequantised by the norm
                                o[e] = __uint_as_float(static_cast<uint32_t>(acc[(c + e) / 2])),
                                o[e + 1] = __uint_as_float(static_cast<uint32_t>(acc[(c + e) / 2] >> 32));
                            else
                                upk2(COMP ? add2(acc[(c + e) / 2], cmp[COMP ? (c + e) / 2 : 0]) : acc[(c + e) / 2],
                                     o[e], o[e + 1]);
                        }
                        st_v8(dst + c, o[0], o[1], o[2], o[3], o[4], o[5], o[6], o[7]);
                    }
                }
            }
        }
        if (!ok && lane == 0) atomicOr(p.status, kStatusWaitTimeout);
    }
    return ok;
}

// ---- W8A8 expansion: exact integer accumulators -> dequantised values ----
//
// Every code is an integer of magnitude <= 127, exact in BF16, so the
// tensor core's products are exact integers; a chain of at most kW8ChainKb
// K blocks keeps every partial sum an integer below 2^24, where each FP32
// add is exact.  A longer K runs as two chains into the two accumulator
// buffers (b0 first half, b1 second half).  This warp converts its share of
// the tile's columns in its lane quarter: y = int(b0) + int(b1), then
// ((float)y * a_scale) * w_scale[n] back into b0, for the epilogue to read
// as it reads a BF16-mode accumulator.  Columns past n_end (a ragged last
// tile) get scale 0.  Whole warp.
__device__ __forceinline__ void w8_dequant_tile(uint32_t tb0, uint32_t tb1, bool two, int width, int half_idx,
                                                float a_scale, const float* w_scale, int n0, int n_end) {
    const int hw = ((width + 31) / 32) * 16;  // columns per warp of the quarter, a multiple of 16
    const int c0 = half_idx * hw, c1 = c0 + hw < width ? c0 + hw : width;
    if (!two) {
        for (int c = c0; c < c1; c += 16) {
            float v[16];
            tmem_ld16(tb0 + c, v);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int n = n0 + c + e;
                v[e] = w8_dequant(__float2int_rn(v[e]), a_scale, n < n_end ? w_scale[n] : 0.0f);
            }
            tmem_st16(tb0 + c, v);
        }
        return;
    }
    for (int c = c0; c < c1; c += 8) {  // 8 columns at a time: the epilogue's row context stays in registers
        float v[8], u[8];
        tmem_ld8x2(tb0 + c, two ? tb1 + c : tb0 + c, v, u);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int y = __float2int_rn(v[e]) + (two ? __float2int_rn(u[e]) : 0);
            const int n = n0 + c + e;
            v[e] = w8_dequant(y, a_scale, n < n_end ? w_scale[n] : 0.0f);
        }
        tmem_st8(tb0 + c, v);
    }
}

// Whether the job of token tile m (CG 128-token tiles) runs its K as two
// chains: a K longer than kW8ChainKb blocks and a tile the norm step marked.
__device__ __forceinline__ bool w8_two_chains(const ExpandParams& p, int m, int cg, bool q) {
    if ((q ? p.kb_q : p.kb_kv) <= kW8ChainKb) return false;
    uint32_t bits = 0;
    for (int i = m * cg; i < (m + 1) * cg && i < p.n_tiles128; ++i) bits |= p.w8_split[i];
    return (bits & (q ? 1u : 2u)) != 0;
}

// ---- expansion phase: this CTA's jobs (round robin or balanced table) ----
//
// The normed activations come from an earlier step: `dep()` (called by the
// producer, after it has issued its first ring pass of weight tiles) waits
// for them.  With `pdl` the phase opens a programmatic dependent launch and
// the other roles also wait for the previous kernel right away (the
// epilogue's amax updates must follow the norm kernel's clearing).
//
// With CG = 2 the CTA pair runs one 256-token tile per job: token tile m
// covers rows [256 m, 256 m + 256), this CTA's epilogue rows 128 * rank on.
// With TS (a kernel with the store staging area) and p.tma_store the kv
// tiles and the per-token q tiles leave through the store ring.
template <int BN_MAX, int STAGES, int CG = 1, bool TS = false, bool W8 = false, class Dep>
__device__ __forceinline__ bool expand_phase(const Smem& sm, uint32_t tmem, const CUtensorMap* tm_aq,
                                             const CUtensorMap* tm_akv, const CUtensorMap* tm_bq,
                                             const CUtensorMap* tm_bkv, const CUtensorMap* tm_bkvh,
                                             const ExpandParams& p, RoleCounters& rc, const CtaJobs& jobs, bool pdl,
                                             const OutMaps& om, Dep&& dep) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Dn = p.Dn, R = p.R;
    const int rank = CG == 2 ? static_cast<int>(cluster_ctarank()) : 0;
    constexpr int TM = kBM * CG;  // token rows per job
    bool ok = true;
    if (pdl && warp != 0) pdl_wait();
    if (warp == 0) {
        if (lane == 0) {
            prefetch_tensormap(tm_aq);
            prefetch_tensormap(tm_akv);
            prefetch_tensormap(tm_bq);
            prefetch_tensormap(tm_bkv);
            const uint64_t pol_a = l2_policy(p.l2_policy & kL2ActsLast ? 1 : 0);
            const uint64_t pol_w = l2_policy(p.l2_policy & kL2WeightsLast ? 1 : 0);
            for (int i = jobs.begin; i < jobs.end && ok; ++i) {
                int tile, m, c0, w;
                expand_job(p, jobs[i], tile, m, c0, w);
                const bool first = i == jobs.begin;
                const int bq = p.q_wide ? kQWide : Dn + R;  // q tile width
                ok = tile < p.nq_tiles
                         ? produce_job<BN_MAX, STAGES, CG>(sm, rc.loads, tm_aq, tm_bq, m * TM, tile * bq, 0, p.kb_q,
                                                           bq, first, p.timeout_ns, dep, pol_a, pol_w)
                         : produce_job<BN_MAX, STAGES, CG>(sm, rc.loads, tm_akv, w < p.bn_kv ? tm_bkvh : tm_bkv,
                                                           m * TM, (tile - p.nq_tiles) * p.bn_kv + c0, 0, p.kb_kv, w,
                                                           first, p.timeout_ns, dep, pol_a, pol_w);
            }
            if (pdl && jobs.begin == jobs.end) pdl_wait();
            if (!ok) raise_abort(sm, p.status);
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {  // a pair's MMAs are issued by its even CTA
            const uint32_t idesc_q = idesc_bf16_f32(TM, p.q_wide ? kQWide : Dn + R);
            const uint32_t idesc_kv_full = idesc_bf16_f32(TM, p.bn_kv);
            const uint32_t idesc_kvh = idesc_bf16_f32(TM, p.bn_kv / 2);  // half tiles (kv_halves)
            for (int i = jobs.begin; i < jobs.end && ok; ++i) {
                int tile, m, c0, w;
                expand_job(p, jobs[i], tile, m, c0, w);
                const bool q = tile < p.nq_tiles;
                const uint32_t idesc_kv = w < p.bn_kv ? idesc_kvh : idesc_kv_full;
                const int nkb = q ? p.kb_q : p.kb_kv;
                if (W8 && w8_two_chains(p, m, CG, q)) {  // W8A8: two exact chains, one per accumulator buffer
                    ok = mma_chain<BN_MAX, STAGES, CG>(sm, rc.consumed, rc.chain, nkb / 2, tmem,
                                                       q ? idesc_q : idesc_kv, p.timeout_ns) &&
                         mma_chain<BN_MAX, STAGES, CG>(sm, rc.consumed, rc.chain + 1, nkb - nkb / 2, tmem,
                                                       q ? idesc_q : idesc_kv, p.timeout_ns);
                    rc.chain += 2;
                } else {
                    ok = mma_chain<BN_MAX, STAGES, CG>(sm, rc.consumed, rc.chain, nkb, tmem, q ? idesc_q : idesc_kv,
                                                       p.timeout_ns);
                    rc.chain += 1;
                }
            }
            if (!ok) raise_abort(sm, p.status);
        }
    } else {
        const int quarter = warp & 3;          // TMEM lane quarter this warp may access
        const int half_idx = (warp - 2) >> 2;  // column half
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        int cur_m = -1;
        RowCtx ctx;
        const StoreRing sr{sm.stage + static_cast<uint32_t>(warp - 2) * 2u * kStoreSlotBytes,
                           l2_policy(p.l2_policy & kL2StoresFirst ? 2 : 0)};
        for (int i = jobs.begin; i < jobs.end; ++i) {
            int tile, m, c0, kv_w;
            expand_job(p, jobs[i], tile, m, c0, kv_w);
            if (m != cur_m) {  // before waiting for the accumulator
                load_row_ctx(p, m * TM + rank * kBM + row, ctx);
                cur_m = m;
            }
            const bool is_q = tile < p.nq_tiles;
            const int chains = W8 && w8_two_chains(p, m, CG, is_q) ? 2 : 1;
            bool got = epi_acquire(sm, rc.chain, p.timeout_ns);
            if (chains == 2) got = got && epi_acquire(sm, rc.chain + 1, p.timeout_ns);
            const uint32_t tbase = tmem + lane_off + (rc.chain & 1) * BN_MAX;
            if constexpr (W8) {
                if (got) {
                    const int t = ctx.t;
                    const float as = t < p.T ? p.a_scale[2 * t + (is_q ? 0 : 1)] : 0.0f;
                    const int bq = p.q_wide ? kQWide : Dn + R;
                    if (is_q)
                        w8_dequant_tile(tbase, tmem + lane_off + ((rc.chain + 1) & 1) * BN_MAX, chains == 2, bq,
                                        half_idx, as, p.w_scale_q, tile * bq, p.NQ);
                    else
                        w8_dequant_tile(tbase, tmem + lane_off + ((rc.chain + 1) & 1) * BN_MAX, chains == 2,
                                        kv_w, half_idx, as, p.w_scale_kv, (tile - p.nq_tiles) * p.bn_kv + c0,
                                        p.NKV);
                }
                // Every warp's columns are converted before any warp reads
                // them.  The store-ring epilogues (wide q tiles, kv tiles, and
                // the per-token q tiles without the per-head norm) read only
                // the columns this warp converted; the others read across the
                // two column halves and meet first.
                // (expand_q_epilogue_ts splits a head at min(Dn, (Dn + R) / 2):
                // the pre-pass's split when Dn >= R, Dn + R a multiple of 32)
                const bool own_cols =
                    TS && (is_q ? (p.q_wide || (p.tma_store && !p.per_head && !p.head_norm && Dn >= R &&
                                                (Dn + R) % 32 == 0))
                                : p.tma_store != 0);
                if (!own_cols) {
                    tc_fence_before();
                    got = named_bar_and(2, kEpiThreads, got);
                    tc_fence_after();
                }
            }
            if (!got) {
                if (lane == 0) atomicOr(p.status, kStatusWaitTimeout);
                ok = false;
                break;
            }
            const int y0 = m * TM + rank * kBM + quarter * 32;
            if (TS && p.tma_store && tile >= p.nq_tiles)
                expand_kv_epilogue_ts(p, om, sr, tbase, ctx, (tile - p.nq_tiles) * p.bn_kv + c0, half_idx, y0,
                                      kv_w);
            else if (TS && p.q_wide)
                expand_qw_epilogue_ts(p, om, sr, tbase, ctx, tile * kQWide, half_idx, y0);
            else if (TS && p.tma_store && !p.per_head)
                expand_q_epilogue_ts(p, om, sr, tbase, ctx, tile, half_idx, y0);
            else if (tile < p.nq_tiles)
                expand_q_epilogue(p, tbase, ctx, tile, half_idx);
            else
                expand_kv_epilogue(p, tbase, ctx, (tile - p.nq_tiles) * p.bn_kv + c0, half_idx, kv_w);
            epi_release<CG>(sm, rc.chain);
            if (chains == 2) epi_release<CG>(sm, rc.chain + 1);
            rc.chain += chains;
        }
        // every tensor store has written its box before the CTA leaves
        if (TS && lane == 0) bulk_wait_all();
    }
    return ok;
}

// Teardown after the last phase: no TMA copy may still be landing and no MMA
// may still be running when TMEM is freed and the CTA leaves.
// A pair: the even CTA's full barriers count both CTAs' copies and its
// commits cover every MMA, so it alone drains and waits.
template <int BN_MAX, int STAGES, int CG = 1>
__device__ __forceinline__ void gemm_finish(const Smem& sm, uint32_t tmem, const RoleCounters& rc,
                                            uint64_t timeout_ns) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool leader = CG == 1 || cluster_ctarank() == 0;
    if (warp == 0 && lane == 0 && leader) drain_loads<STAGES>(sm, rc.loads, timeout_ns);
    if (warp == 1 && lane == 0 && leader) {
        if constexpr (CG == 2)
            mma_commit_pair(sm.done, 0x1);
        else
            mma_commit(sm.done);
        mbar_wait(sm.done, 0, timeout_ns, nullptr);
    }
    gemm_teardown<BN_MAX, STAGES, CG>(sm, tmem);
}

// ---- kv tiles of the prefill expansion on CTA pairs, activations resident --
//
// A kv tile has K = Lkv <= 512, so a pair's 256 token rows of normed c_kv
// (128 KB per CTA) fit in shared memory.  A super-job (pair token tile m,
// a group of kv tiles) loads them once and then streams only the weight
// halves (16 KB per CTA per K block) through a 4-stage ring, one TMEM
// accumulator chain per kv tile; the epilogue is the kv epilogue through the
// store ring.  The next super-job's activation K block k is loaded as soon as
// the last tile of the current one has consumed slot k, interleaved with the
// first weight blocks, so the switch costs no pipeline drain.
constexpr int kKvResKb = 8;              // resident K blocks (Lkv <= 8 * 64)
constexpr int kKvResStages = 4;          // weight ring
constexpr int kKvResA = kBM * kBK * 2;   // 16 KB: 128 token rows of one K block
constexpr int kKvResB = 128 * kBK * 2;   // 16 KB: half of a 256-row weight tile

struct KvResLayout {
    static constexpr int B_OFF = kKvResKb * kKvResA;                  // 128 KB of activations first
    static constexpr int STAGE_OFF = B_OFF + kKvResStages * kKvResB;  // then the ring (64 KB)
    static constexpr int BAR_OFF = STAGE_OFF + kStoreStageBytes;      // then the store staging (32 KB)
    // a_full[8], a_empty[8], b_full[4], b_empty[4], acc_full[2], acc_empty[2], done
    static constexpr int MISC = BAR_OFF + (2 * kKvResKb + 2 * kKvResStages + 5) * 8;
    static constexpr int BYTES = MISC + 16 + 1024;
    static constexpr uint32_t TMEM_COLS = 512;  // two 256-column accumulators
};

struct KvResSmem {
    Smem s;  // ring = weight stages (full0 / empty0), stage, accumulator barriers, TMEM slot
    uint32_t a, afull0, aempty0;
};

__device__ __forceinline__ KvResSmem kvres_carve(uint8_t* raw_ptr) {
    using L = KvResLayout;
    const uint32_t raw = smem_u32(raw_ptr);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    KvResSmem k;
    k.a = raw + pad;
    k.s.base = k.a + L::B_OFF;
    k.s.stage = k.a + L::STAGE_OFF;
    k.afull0 = k.a + L::BAR_OFF;
    k.aempty0 = k.afull0 + 8 * kKvResKb;
    k.s.full0 = k.aempty0 + 8 * kKvResKb;
    k.s.empty0 = k.s.full0 + 8 * kKvResStages;
    k.s.accf0 = k.s.empty0 + 8 * kKvResStages;
    k.s.acce0 = k.s.accf0 + 16;
    k.s.done = k.s.acce0 + 16;
    k.s.tmem_slot = reinterpret_cast<uint32_t*>(raw_ptr + pad + L::MISC);
    k.s.abort_flag = reinterpret_cast<volatile int*>(raw_ptr + pad + L::MISC + 4);
    return k;
}

__device__ __forceinline__ uint32_t kvres_setup(const KvResSmem& k) {
    if (threadIdx.x == 0) {
        for (int i = 0; i < kKvResKb; ++i) {
            mbar_init(k.afull0 + 8 * i, 1);
            mbar_init(k.aempty0 + 8 * i, 1);
        }
        for (int s = 0; s < kKvResStages; ++s) {
            mbar_init(k.s.full0 + 8 * s, 1);
            mbar_init(k.s.empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(k.s.accf0 + 8 * b, 1);
            mbar_init(k.s.acce0 + 8 * b, kExpandEpiWarps * 2);
        }
        mbar_init(k.s.done, 1);
        *k.s.abort_flag = 0;
        fence_barrier_init();
    }
    if ((threadIdx.x >> 5) == 1) {
        tmem_alloc_pair(smem_u32(k.s.tmem_slot), KvResLayout::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    return *k.s.tmem_slot;
}

// Super-job sj -> (pair token tile m, first kv tile, tiles in the group).
__device__ __forceinline__ void kvres_job(const ExpandParams& p, int group, int sj, int& m, int& t0, int& nt) {
    const int ngroups = (p.nkv_tiles + group - 1) / group;
    const int from = p.m_tiles * ngroups - p.kvres_halves;
    int half = -1;
    if (p.kvres_halves > 0 && sj >= from) {  // half super-jobs (ExpandParams::kvres_halves)
        half = (sj - from) & 1;
        sj = from + (sj - from) / 2;
    }
    m = sj / ngroups;
    t0 = (sj - m * ngroups) * group;
    nt = p.nkv_tiles - t0 < group ? p.nkv_tiles - t0 : group;
    if (half >= 0) {
        const int n0 = (nt + 1) / 2;
        t0 += half ? n0 : 0;
        nt = half ? nt - n0 : n0;
    }
}

// This pair's super-jobs: unit + i * units.  Returns false when a wait gave up.
// W8 (W8A8): the activations and weights are INT8 codes as BF16 integers; a
// kv tile's K (Lkv <= 8 * 64) is one exact chain, and each epilogue warp
// dequantises the columns it then stores (w8_dequant_tile) before the
// unchanged kv epilogue reads them.
template <bool W8 = false>
__device__ __forceinline__ bool expand_kvres_phase(const KvResSmem& k, uint32_t tmem, const CUtensorMap* tm_akv,
                                                   const CUtensorMap* tm_bkv, const ExpandParams& p,
                                                   const OutMaps& om, int group, RoleCounters& rc) {
    static_assert(!W8 || kKvResKb <= kW8ChainKb, "a kv tile's K must be one exact W8A8 chain");
    const Smem& sm = k.s;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = static_cast<int>(cluster_ctarank());
    const bool leader = rank == 0;
    const int unit = static_cast<int>(blockIdx.x) / 2, units = static_cast<int>(gridDim.x) / 2;
    const int n_sj = p.m_tiles * ((p.nkv_tiles + group - 1) / group) + p.kvres_halves;
    const int kb = p.kb_kv;
    bool ok = true;
    pdl_wait();  // the normed rows come from the norm kernel; amax clearing precedes the epilogue
    if (warp == 0) {
        if (lane == 0) {
            prefetch_tensormap(tm_akv);
            prefetch_tensormap(tm_bkv);
            const uint64_t pol_w = l2_policy(p.l2_policy & kL2WeightsLast ? 1 : 0);
            const uint64_t pol_a = l2_policy(p.l2_policy & kL2ActsLast ? 1 : 0);
            uint32_t sjn = 0;
            int a_last = 0;  // activation blocks issued for the latest super-job
            auto b_load = [&](int tile, int kk) -> bool {
                const uint32_t l = rc.loads;
                const int s = static_cast<int>(l % kKvResStages);
                if (!mbar_wait(sm.empty0 + 8 * s, ((l / kKvResStages) & 1) ^ 1, p.timeout_ns, sm.abort_flag))
                    return false;
                if (leader) mbar_arrive_expect_tx(sm.full0 + 8 * s, 2 * kKvResB);
                tma_load_2d_pair_hint(sm.base + s * kKvResB, tm_bkv, map_shared_rank(sm.full0 + 8 * s, 0),
                                      kk * kBK, tile * 256 + rank * 128, pol_w);
                ++rc.loads;
                return true;
            };
            for (int sj = unit; sj < n_sj && ok; sj += units, ++sjn) {
                int m, t0, nt;
                kvres_job(p, group, sj, m, t0, nt);
                a_last = 0;
                for (int kk = 0; kk < kb && ok; ++kk) {
                    // activation block kk, once the previous super-job's last tile is done with it
                    if (!mbar_wait(k.aempty0 + 8 * kk, (sjn & 1) ^ 1, p.timeout_ns, sm.abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(k.afull0 + 8 * kk, 2 * kKvResA);
                    tma_load_2d_pair_hint(k.a + kk * kKvResA, tm_akv, map_shared_rank(k.afull0 + 8 * kk, 0),
                                          kk * kBK, m * 256 + rank * 128, pol_a);
                    ++a_last;
                    ok = b_load(t0, kk);
                }
                for (int h = 1; h < nt && ok; ++h)
                    for (int kk = 0; kk < kb && ok; ++kk) ok = b_load(t0 + h, kk);
            }
            if (!ok) raise_abort(sm, p.status);
            // no activation copy may still be landing when the CTA leaves: the
            // last super-job's blocks (the leader's barriers count both CTAs)
            // (the loop's increment also runs after an abort: super-job sjn - 1
            // issued the latest blocks)
            if (leader && sjn > 0)
                for (int kk = 0; kk < a_last; ++kk)
                    mbar_wait(k.afull0 + 8 * kk, (sjn - 1) & 1, p.timeout_ns, nullptr);
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            const uint32_t idesc = idesc_bf16_f32(256, 256);
            uint32_t sjn = 0;
            for (int sj = unit; sj < n_sj && ok; sj += units, ++sjn) {
                int m, t0, nt;
                kvres_job(p, group, sj, m, t0, nt);
                for (int h = 0; h < nt && ok; ++h, ++rc.chain) {
                    const uint32_t b = rc.chain & 1;
                    if (!mbar_wait(sm.acce0 + 8 * b, ((rc.chain >> 1) & 1) ^ 1, p.timeout_ns, sm.abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t dacc = tmem + b * 256;
                    for (int kk = 0; kk < kb; ++kk, ++rc.consumed) {
                        if (h == 0 && !mbar_wait(k.afull0 + 8 * kk, sjn & 1, p.timeout_ns, sm.abort_flag)) {
                            ok = false;
                            break;
                        }
                        const int s = static_cast<int>(rc.consumed % kKvResStages);
                        if (!mbar_wait(sm.full0 + 8 * s, (rc.consumed / kKvResStages) & 1, p.timeout_ns,
                                       sm.abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t ad = smem_desc_sw128(k.a + kk * kKvResA);
                        const uint64_t bd = smem_desc_sw128(sm.base + s * kKvResB);
#pragma unroll
                        for (int q = 0; q < kBK / 16; ++q)
                            mma_bf16_pair(dacc, ad + 2 * q, bd + 2 * q, idesc, (kk == 0 && q == 0) ? 0u : 1u);
                        mma_commit_pair(sm.empty0 + 8 * s, 0x3);
                        if (h == nt - 1) mma_commit_pair(k.aempty0 + 8 * kk, 0x3);
                    }
                    if (ok) mma_commit_pair(sm.accf0 + 8 * b, 0x3);
                }
            }
            if (!ok) raise_abort(sm, p.status);
        }
    } else {
        const int quarter = warp & 3;
        const int half_idx = (warp - 2) >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        StoreRing sr{sm.stage + static_cast<uint32_t>(warp - 2) * 2u * kStoreSlotBytes,
                     l2_policy(p.l2_policy & kL2StoresFirst ? 2 : 0)};
        RowCtx ctx;
        for (int sj = unit; sj < n_sj && ok; sj += units) {
            int m, t0, nt;
            kvres_job(p, group, sj, m, t0, nt);
            load_row_ctx(p, m * 256 + rank * kBM + row, ctx);
            const int y0 = m * 256 + rank * kBM + quarter * 32;
            for (int h = 0; h < nt; ++h, ++rc.chain) {
                if (!epi_acquire(sm, rc.chain, p.timeout_ns)) {
                    if (lane == 0) atomicOr(p.status, kStatusWaitTimeout);
                    ok = false;
                    break;
                }
                const uint32_t tbase = tmem + lane_off + (rc.chain & 1) * 256;
                if constexpr (W8) {  // this warp's columns, which only it stores
                    const float as = ctx.t < p.T ? p.a_scale[2 * ctx.t + 1] : 0.0f;
                    w8_dequant_tile(tbase, tbase, false, p.bn_kv, half_idx, as, p.w_scale_kv, (t0 + h) * p.bn_kv,
                                    p.NKV);
                }
                expand_kv_epilogue_ts(p, om, sr, tbase, ctx, (t0 + h) * p.bn_kv, half_idx, y0, p.bn_kv);
                epi_release<2>(sm, rc.chain);
            }
        }
        if (lane == 0) bulk_wait_all();
    }
    return ok;
}

}  // namespace mlap
