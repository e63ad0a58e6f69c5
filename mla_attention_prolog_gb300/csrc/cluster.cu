// Compression projection, split, RMSNorm and k_pe RoPE of a small decode
// batch (one 128-token tile) in ONE thread-block cluster.
//
// With a few dozen tokens the split-K compression over every SM is cheap, but
// handing its FP32 partials to the norm costs a global-memory round trip and
// a kernel boundary, both latency.  Here the nc x ks CTAs of one cluster (at
// most 16) each compute one partial tile:
//   rank r -> column group g = r / ks (cgw weight rows of W_a), K split
//             s = r % ks (K blocks [s kb / ks, (s + 1) kb / ks)),
// with a TMA ring feeding tcgen05.mma into one TMEM accumulator (M = 128
// token rows, N = cgw as one or two instructions).  The epilogue warps stage
// the accumulator rows in the CTA's own shared memory; after a cluster
// barrier (every CTA's MMAs are done, so every ring is free to receive) the
// staged rows of each owner's tokens go to that CTA with one bulk copy
// (shared::cta -> shared::cluster), laid out [split][group][token][column]
// there and counted on its receive mbarrier.  Each CTA then runs the norm
// step of its tokens, two warps per token (splits summed in split order with
// TwoSum, BF16 cast, RMSNorm, RoPE, all outputs), with the positions,
// cos/sin rows and gamma loaded into shared memory while the MMAs ran.  The expansion kernel follows as a programmatic dependent launch and
// streams its weights meanwhile.
//
// Every mbarrier wait is bounded; a CTA whose wait gave up records
// MLA_STATUS_WAIT_TIMEOUT and still passes the cluster barriers, so the
// cluster always completes.  No CTA leaves before every CTA has received all
// of its rows (the last barrier is arrived at after the receive wait), so no
// bulk copy reads the shared memory of a CTA that has exited.
#include "engine.cuh"
#include "rows.cuh"

namespace mlap {

namespace {

// Bulk copy of `bytes` (multiple of 16) from this CTA's shared memory to a
// peer's (cluster address), completion counted on the peer's mbarrier.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst_cluster, uint32_t src, uint32_t bytes,
                                                  uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst_cluster),
        "r"(src), "r"(bytes), "r"(bar_cluster)
        : "memory");
}

__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

constexpr uint32_t kATile = kBM * kBK * 2;  // x tile of one K block (128 rows x 64 columns)
constexpr int kGroupThreads = kClusterThreads / kClusterNormGroups;  // 64: two warps per token

// The norm step of owned token t (local row lrow) by one group of two warps
// (gtid = 0..63, named barrier `bar`): each 4-column chunk's ks split rows
// are summed in split order with TwoSum and rounded to BF16; RMSNorm of c_q
// and c_kv (x^2 / L summed per thread in increasing chunk order, over each
// warp by butterfly, then warp 0 + warp 1), x * rstd * gamma, BF16; RoPE of
// k_pe; then the normed row, the cache row, out_kpe and K's rope slice of
// every head.  `pos`, `cs_row` and `gamma` are in shared memory.
__device__ __forceinline__ void cluster_norm_token(const ClusterNormParams& p, int lrow, int t, int gtid,
                                                   uint32_t bar, const float* recv, const uint16_t* gamma,
                                                   int pos, const float* cs_row, uint16_t* crow, float* red) {
    const NormRopeParams& n = p.n;
    const int NA = p.NA, Lq = n.Lq, Lkv = n.Lkv, R = n.R, half = R / 2, cgw = p.cgw;
    const int lane = gtid & 31, gw = gtid >> 5;
    uint16_t* rot = crow + NA;
    const bool valid = pos >= 0 && pos < n.max_pos;
    if (gtid == 0 && n.amax) n.amax[t] = 0u;
    uint16_t* nrow = n.normed + static_cast<size_t>(t) * (Lq + Lkv);
    uint16_t* cache_row = kv_cache_row(n, t, gtid == 0);
    const int nchunk = R / 8;
    const int ndst = n.H + (cache_row ? 2 : 1);  // rope-slice destinations (kpe_dst)
    if (!valid) {  // uniform over the group
        if (gtid == 0) atomicOr(n.status, kStatusPositionRange);
        const uint4 z = make_uint4(0, 0, 0, 0);
        for (int i = gtid * 8; i < Lq + Lkv; i += kGroupThreads * 8) {
            *reinterpret_cast<uint4*>(nrow + i) = z;
            if (cache_row && i >= Lq) *reinterpret_cast<uint4*>(cache_row + (i - Lq)) = z;
        }
        for (int k = gtid; k < ndst * nchunk; k += kGroupThreads) {
            const int h = k / nchunk, c = k - h * nchunk;
            *reinterpret_cast<uint4*>(kpe_dst(n, t, h, c, cache_row)) = z;
        }
        return;
    }
    const int sw = t & 7;  // the staging swizzle of this token's row
    const size_t split_stride = static_cast<size_t>(p.nc) * p.tpo * cgw;
    float ssq_q = 0.0f, ssq_kv = 0.0f;
    for (int j = gtid; j < NA / 4; j += kGroupThreads) {
        const int i = 4 * j, g = i / cgw, cj = (i - g * cgw) >> 2;
        const float* base = recv + (static_cast<size_t>(g) * p.tpo + lrow) * cgw + 4 * (cj ^ sw);
        float4 a = *reinterpret_cast<const float4*>(base), cmp = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int sp = 1; sp < p.ks; ++sp) {
            const float4 r = *reinterpret_cast<const float4*>(base + sp * split_stride);
            two_sum_add(a.x, cmp.x, r.x);
            two_sum_add(a.y, cmp.y, r.y);
            two_sum_add(a.z, cmp.z, r.z);
            two_sum_add(a.w, cmp.w, r.w);
        }
        if (p.ks > 1)
            a = make_float4(__fadd_rn(a.x, cmp.x), __fadd_rn(a.y, cmp.y), __fadd_rn(a.z, cmp.z), __fadd_rn(a.w, cmp.w));
        const uint32_t w0 = pack_bf16x2(a.x, a.y), w1 = pack_bf16x2(a.z, a.w);
        *reinterpret_cast<uint2*>(crow + i) = make_uint2(w0, w1);
        const float v[4] = {bf16_lo(w0), bf16_hi(w0), bf16_lo(w1), bf16_hi(w1)};
        if (i < Lq)
            ssq_q = __fadd_rn(ssq_q, chunk_ssq(v, n.inv_lq));
        else if (i < Lq + Lkv)
            ssq_kv = __fadd_rn(ssq_kv, chunk_ssq(v, n.inv_lkv));
    }
    ssq_q = lane_butterfly_sum(ssq_q);
    ssq_kv = lane_butterfly_sum(ssq_kv);
    if (lane == 0) red[2 * gw] = ssq_q, red[2 * gw + 1] = ssq_kv;
    named_bar_sync(bar, kGroupThreads);  // also publishes crow
    const float sq = __fadd_rn(red[0], red[2]), skv = __fadd_rn(red[1], red[3]);
    const float rstd_q = Lq > 0 ? __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(sq, n.eps))) : 0.0f;
    const float rstd_kv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(skv, n.eps)));
    for (int i = gtid * 8; i < Lq + Lkv; i += kGroupThreads * 8) {
        const uint4 xv = *reinterpret_cast<const uint4*>(crow + i);
        const uint4 gv = *reinterpret_cast<const uint4*>(gamma + i);
        const float rstd = i < Lq ? rstd_q : rstd_kv;
        const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
        const uint32_t gs[4] = {gv.x, gv.y, gv.z, gv.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float y0 = __fmul_rn(__fmul_rn(bf16_lo(xs[e]), rstd), bf16_lo(gs[e]));
            const float y1 = __fmul_rn(__fmul_rn(bf16_hi(xs[e]), rstd), bf16_hi(gs[e]));
            o[e] = pack_bf16x2(y0, y1);
        }
        const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(nrow + i) = ov;
        if (cache_row && i >= Lq) *reinterpret_cast<uint4*>(cache_row + (i - Lq)) = ov;
    }
    const uint16_t* kp = crow + Lq + Lkv;
    for (int i = gtid; i < half; i += kGroupThreads) {
        int j1, j2;
        kpe_pair(n.interleaved, i, half, j1, j2);
        const float x1 = __uint_as_float(static_cast<uint32_t>(kp[j1]) << 16);
        const float x2 = __uint_as_float(static_cast<uint32_t>(kp[j2]) << 16);
        const float c = cs_row[i], s = cs_row[half + i];
        const float o1 = __fadd_rn(__fmul_rn(x1, c), __fmul_rn(-x2, s));
        const float o2 = __fadd_rn(__fmul_rn(x2, c), __fmul_rn(x1, s));
        rot[i] = static_cast<uint16_t>(pack_bf16x2(o1, 0.0f) & 0xFFFFu);
        rot[i + half] = static_cast<uint16_t>(pack_bf16x2(o2, 0.0f) & 0xFFFFu);
    }
    named_bar_sync(bar, kGroupThreads);
    for (int k = gtid; k < ndst * nchunk; k += kGroupThreads) {
        const int h = k / nchunk, c = k - h * nchunk;
        *reinterpret_cast<uint4*>(kpe_dst(n, t, h, c, cache_row)) = *reinterpret_cast<const uint4*>(rot + c * 8);
    }
    named_bar_sync(bar, kGroupThreads);  // crow, rot and red are free for the group's next token
}

}  // namespace

__global__ void __launch_bounds__(kClusterThreads, 1)
    mla_compress_norm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_wa,
                             const ClusterNormParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t* area_ptr = smem_raw + pad;  // ring, then (once free) receive / norm / staging rows
    const uint32_t area = raw + pad;
    const int S = p.stages;
    const uint32_t full0 = area + p.area_bytes, empty0 = full0 + 8 * S, accf = empty0 + 8 * S, recvf = accf + 8;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(area_ptr + p.area_bytes + 8 * (2 * S + 2));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = static_cast<int>(cluster_ctarank());
    const int g = rank / p.ks, s = rank - g * p.ks;
    const int kb0 = s * p.kb_total / p.ks, nkb = (s + 1) * p.kb_total / p.ks - kb0;
    const int cgw = p.cgw, n1 = cgw < 256 ? cgw : 256, n2 = cgw - n1, NA = p.NA;
    const uint32_t stage_bytes = kATile + static_cast<uint32_t>(cgw) * kBK * 2;
    const int first = rank * p.tpo;
    const int count = p.T - first < p.tpo ? (p.T - first > 0 ? p.T - first : 0) : p.tpo;  // tokens owned
    const NormRopeParams& n = p.n;
    const int Lqkv = n.Lq + n.Lkv;
    uint16_t* gamma_s = reinterpret_cast<uint16_t*>(area_ptr + p.const_off);
    int* pos_s = reinterpret_cast<int*>(area_ptr + p.const_off + align16(static_cast<size_t>(Lqkv) * 2));
    float* cs_s = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(pos_s) + align16(p.tpo * 4));
    float* red_s = cs_s + p.tpo * n.R;  // kClusterNormGroups x 4 partial sums

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, 1);
        }
        mbar_init(accf, 1);
        mbar_init(recvf, 1);
        *abort_flag = 0;
        fence_barrier_init();
        // every (split, group) CTA sends the cgw-column rows of the owned tokens
        mbar_arrive_expect_tx(recvf, static_cast<uint32_t>(p.ks * p.nc * count * cgw * 4));
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();  // the expansion CTAs start streaming their weights

    bool ok = true;
    if (warp == 0) {
        if (lane == 0) {
            prefetch_tensormap(&tm_x);
            prefetch_tensormap(&tm_wa);
            const int rows_box = p.b_boxes == 2 ? cgw / 2 : cgw;
            int issued = 0;
            for (int i = 0; i < nkb; ++i, ++issued) {
                const int st = i % S;
                if (!mbar_wait(empty0 + 8 * st, ((i / S) & 1) ^ 1, p.timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t sa = area + st * stage_bytes;
                mbar_arrive_expect_tx(full0 + 8 * st, stage_bytes);
                tma_load_2d(sa, &tm_x, full0 + 8 * st, (kb0 + i) * kBK, 0);
                for (int b = 0; b < p.b_boxes; ++b)
                    tma_load_2d(sa + kATile + static_cast<uint32_t>(b * rows_box) * kBK * 2, &tm_wa, full0 + 8 * st,
                                (kb0 + i) * kBK, g * cgw + b * rows_box);
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.status, kStatusWaitTimeout);
            }
            // no copy may land in the ring once peers write into it
            for (int i = issued > S ? issued - S : 0; i < issued; ++i)
                mbar_wait(full0 + 8 * (i % S), (i / S) & 1, p.timeout_ns, nullptr);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc1 = idesc_bf16_f32(kBM, n1);
            const uint32_t idesc2 = idesc_bf16_f32(kBM, n2 > 0 ? n2 : 16);
            for (int i = 0; i < nkb; ++i) {
                const int st = i % S;
                if (!mbar_wait(full0 + 8 * st, (i / S) & 1, p.timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = area + st * stage_bytes;
                const uint64_t ad = smem_desc_sw128(sa);
                const uint64_t bd = smem_desc_sw128(sa + kATile);
                const uint64_t bd2 = smem_desc_sw128(sa + kATile + 256u * kBK * 2);
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {  // +32 bytes of K per instruction
                    const uint32_t acc = (i == 0 && kk == 0) ? 0u : 1u;
                    mma_bf16(tmem, ad + 2 * kk, bd + 2 * kk, idesc1, acc);
                    if (n2 > 0) mma_bf16(tmem + 256, ad + 2 * kk, bd2 + 2 * kk, idesc2, acc);
                }
                mma_commit(empty0 + 8 * st);
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.status, kStatusWaitTimeout);
            }
            mma_commit(accf);  // arrives once every MMA issued above has completed
            // no MMA may still read the ring once peers write into it, nor
            // use TMEM when it is freed
            mbar_wait(accf, 0, p.timeout_ns, nullptr);
        }
    } else {
        // While the MMAs run: the norm constants of the owned tokens (gamma,
        // positions, cos/sin rows) into shared memory.
        const int et = threadIdx.x - 64, ent = kClusterThreads - 64;
        for (int i = et * 8; i < Lqkv; i += ent * 8)
            *reinterpret_cast<uint4*>(gamma_s + i) = *reinterpret_cast<const uint4*>(n.gamma + i);
        for (int l = et; l < count; l += ent) pos_s[l] = n.positions[first + l];
        for (int k = et; k < count * (n.R / 4); k += ent) {
            const int l = k / (n.R / 4), c = (k - l * (n.R / 4)) * 4;
            const int pos = n.positions[first + l];
            const bool valid = pos >= 0 && pos < n.max_pos;
            *reinterpret_cast<float4*>(cs_s + l * n.R + c) =
                valid ? *reinterpret_cast<const float4*>(n.cos_sin + static_cast<size_t>(pos) * n.R + c)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // the accumulator is complete (warp-uniform result)
        bool got = mbar_wait(accf, 0, p.timeout_ns, abort_flag);
        got = __all_sync(0xffffffffu, got);
        tc_fence_after();
        if (!got) {
            if (lane == 0) atomicOr(p.status, kStatusWaitTimeout);
            ok = false;
        }
        // stage this warp's token rows (its column half) in the CTA's own
        // shared memory: the MMAs are done, so the staging rows are free
        const int quarter = warp & 3, half_idx = (warp - 2) >> 2;
        const int t = quarter * 32 + lane;
        const int hw = cgw / 2;
        const uint32_t src = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        float* srow = reinterpret_cast<float*>(area_ptr + p.stg_off) + static_cast<size_t>(t) * cgw;
        const int sw = t & 7;  // 16-byte chunk j of row t sits at chunk j ^ (t & 7): no bank conflicts
        for (int c = half_idx * hw; c < (half_idx + 1) * hw; c += 16) {
            if (g * cgw + c >= NA) break;  // warp-uniform: columns past NA hold zero weights
            float v[16];
            tmem_ld16(src + c, v);
            if (t < p.T) {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    *reinterpret_cast<float4*>(srow + 4 * (((c >> 2) + e) ^ sw)) =
                        make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
            }
        }
        fence_proxy_async_shared();
        tc_fence_before();
    }
    __syncwarp();
    cluster_arrive();  // every CTA's MMAs are done: every ring is free to receive
    cluster_wait();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, p.tmem_cols);
    }

    if (warp == 2 && ok) {
        // one bulk copy per owner: the staged rows of its tokens (contiguous)
        const int owner = lane, ctas = p.nc * p.ks;
        const int cnt = p.T - owner * p.tpo < p.tpo ? p.T - owner * p.tpo : p.tpo;
        if (owner < ctas && cnt > 0) {
            const uint32_t src = area + p.stg_off + static_cast<uint32_t>(owner * p.tpo * cgw) * 4u;
            const uint32_t dst = area + static_cast<uint32_t>((s * p.nc + g) * p.tpo * cgw) * 4u;
            bulk_copy_to_peer(map_shared_rank(dst, static_cast<uint32_t>(owner)), src,
                              static_cast<uint32_t>(cnt * cgw) * 4u, map_shared_rank(recvf, static_cast<uint32_t>(owner)));
        }
    }

    // Every row this CTA owns has arrived; only then may the cluster's last
    // barrier complete (no CTA exits while a copy still reads its staging).
    const bool rcv = mbar_wait(recvf, 0, p.timeout_ns, nullptr);
    if (!rcv && threadIdx.x == 0) atomicOr(p.status, kStatusWaitTimeout);
    __syncwarp();
    cluster_arrive();

    // The norm step of this CTA's tokens, two warps per token.
    const int grp = warp >> 1, gtid = threadIdx.x - grp * kGroupThreads;
    const size_t row_bytes = align16(static_cast<size_t>(NA + n.R) * 2);
    uint16_t* crow = reinterpret_cast<uint16_t*>(area_ptr + p.recv_bytes + grp * row_bytes);
    const float* recv = reinterpret_cast<const float*>(area_ptr);
    for (int lrow = grp; lrow < count; lrow += kClusterNormGroups)
        cluster_norm_token(p, lrow, first + lrow, gtid, 1 + grp, recv, gamma_s, pos_s[lrow], cs_s + lrow * n.R,
                           crow, red_s + 4 * grp);
    cluster_wait();
}

cudaError_t cluster_set_attributes(size_t smem, int ctas) {
    cudaError_t e = cudaFuncSetAttribute(mla_compress_norm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (ctas > 8)
        e = cudaFuncSetAttribute(mla_compress_norm_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

namespace {
cudaLaunchConfig_t cluster_config(int ctas, size_t smem, cudaStream_t st, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(kClusterThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ctas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}
}  // namespace

cudaError_t cluster_max_active(size_t smem, int ctas, int* clusters) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = cluster_config(ctas, smem, nullptr, attr);
    return cudaOccupancyMaxActiveClusters(clusters, mla_compress_norm_kernel, &cfg);
}

cudaError_t launch_compress_norm_cluster(int ctas, size_t smem, const CUtensorMap& tm_x, const CUtensorMap& tm_wa,
                                         const ClusterNormParams& p, cudaStream_t st) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = cluster_config(ctas, smem, st, attr);
    return cudaLaunchKernelEx(&cfg, mla_compress_norm_kernel, tm_x, tm_wa, p);
}

}  // namespace mlap
