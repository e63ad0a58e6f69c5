// Row-wise steps of the prolog as device functions, shared by the
// standalone kernels (rowwise.cu) and the cooperative decode kernel.
#pragma once

#include "prolog.cuh"
#include "ptx.cuh"

namespace mlap {

// The thread group that runs a row step: FIRST == 0 is the whole CTA (NT
// threads, __syncthreads); otherwise threads [FIRST, FIRST + NT), whole
// warps, synchronised on named barrier 1 while the other warps work on.
template <int NT, int FIRST>
__device__ __forceinline__ void group_sync() {
    if constexpr (FIRST == 0)
        __syncthreads();
    else
        named_bar_sync(1, NT);
}

// Sum of squares of a normed block in the one order every norm kernel uses,
// whatever its thread count: 4-column chunk j contributes
// ((t0 + t1) + t2) + t3 (t = x^2 / L of its BF16 values), lane j % 32 of a
// warp adds its chunks in increasing j, and a butterfly over the 32 lanes
// (every lane ends with the same sum) finishes.  So a token's normed row is
// the same bits in the decode, prefill and cooperative kernels.
__device__ __forceinline__ float chunk_ssq(const float (&v)[4], float inv_l) {
    float c = __fmul_rn(__fmul_rn(v[0], v[0]), inv_l);
#pragma unroll
    for (int e = 1; e < 4; ++e) c = __fadd_rn(c, __fmul_rn(__fmul_rn(v[e], v[e]), inv_l));
    return c;
}

__device__ __forceinline__ float lane_butterfly_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ------------------------------------------------------------------ W8A8

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ uint32_t warp_sum(uint32_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Codes of eight normed BF16 values (code_bf16x2), as BF16 integers.
__device__ __forceinline__ uint4 codes_bf16x8(uint4 y, float inv) {
    return make_uint4(code_bf16x2(bf16_lo(y.x), bf16_hi(y.x), inv), code_bf16x2(bf16_lo(y.y), bf16_hi(y.y), inv),
                      code_bf16x2(bf16_lo(y.z), bf16_hi(y.z), inv), code_bf16x2(bf16_lo(y.w), bf16_hi(y.w), inv));
}

// Sum of |code| of eight codes held as BF16 integers.
__device__ __forceinline__ uint32_t abs_sum_bf16x8(uint4 c) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    uint32_t s = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e)
        s += static_cast<uint32_t>(fabsf(bf16_lo(w[e]))) + static_cast<uint32_t>(fabsf(bf16_hi(w[e])));
    return s;
}

// One token's normed-row scales (amax / 127, 0 for a zero row) and, where
// a row's codes could drive an expansion's partial sums to 2^24 (sum |code|
// * 127 >= 2^24, the largest weight code being 127), the mark that makes
// the expansion split that token tile's K into two exact chains (bit 0: the
// q expansion, bit 1: the kv expansion).
__device__ __forceinline__ void w8_finish_token(const NormRopeParams& p, int t, float amax_q, float amax_kv,
                                                uint32_t sum_q, uint32_t sum_kv) {
    p.nscale[2 * t] = amax_q > 0.0f ? __fdiv_rn(amax_q, 127.0f) : 0.0f;
    p.nscale[2 * t + 1] = amax_kv > 0.0f ? __fdiv_rn(amax_kv, 127.0f) : 0.0f;
    const uint32_t bits = (sum_q > kW8SumLimit ? 1u : 0u) | (sum_kv > kW8SumLimit ? 2u : 0u);
    if (bits) atomicOr(p.w8_split + t / kBM, bits);
}

// The latent KV-cache row of token t: null without a cache, for a negative
// (padding) slot, and for a slot past the cache, which also sets
// kStatusSlotRange (when `report`, i.e. from one thread of the token).
__device__ __forceinline__ uint16_t* kv_cache_row(const NormRopeParams& p, int t, bool report) {
    if (!p.cache) return nullptr;
    const long long slot = p.slots[t];
    if (slot < 0) return nullptr;
    if (slot >= p.num_slots) {
        if (report) atomicOr(p.status, kStatusSlotRange);
        return nullptr;
    }
    return p.cache + slot * static_cast<long long>(p.Lkv + p.R);
}

// Destination of 8-column chunk c of the rotated k_pe: the rope slice of K's
// head h (h < H), out_kpe (h == H), or the latent cache row (h == H + 1).
__device__ __forceinline__ uint16_t* kpe_dst(const NormRopeParams& p, int t, int h, int c, uint16_t* cache_row) {
    if (h < p.H) return p.out_k + (static_cast<size_t>(t) * p.H + h) * (p.Dn + p.R) + p.Dn + c * 8;
    if (h == p.H) return p.out_kpe + static_cast<size_t>(t) * p.R + c * 8;
    return cache_row + p.Lkv + c * 8;
}

// Rope pair i of a k_pe row: (i, i + R/2), or, de-interleaved, (2i, 2i + 1).
__device__ __forceinline__ void kpe_pair(int interleaved, int i, int half, int& j1, int& j2) {
    j1 = interleaved ? 2 * i : i;
    j2 = interleaved ? 2 * i + 1 : i + half;
}

// Shared memory a norm group needs per token: the BF16 row (NA + R) and the
// FP32 chunk sums ((Lq + Lkv) / 4), 16-byte aligned.
__host__ __device__ inline size_t norm_token_smem_bytes(int NA, int R, int Lq, int Lkv) {
    return ((static_cast<size_t>(NA + R) * 2 + 15) & ~static_cast<size_t>(15)) +
           static_cast<size_t>((Lq + Lkv) / 4) * 4;
}

// Step 1 of the norm for one group of a thread's 4-column chunks (CPG of
// them, NT * 4 columns apart, the first at column i0): every split's partial
// of every chunk, BATCH loads in flight at a time, summed in split order
// with TwoSum, rounded to BF16 into `crow`, chunk sums of x^2 / L into
// `csum` (see chunk_ssq).
template <int CPG, int BATCH, int NT, bool W8 = false>
__device__ __forceinline__ void norm_chunk_group(const NormRopeParams& p, const float* prow, int i0,
                                                 uint16_t* crow, float* csum, float sx = 0.0f) {
    constexpr int SPB = BATCH / CPG;  // splits per chunk and batch
    const size_t sstride = static_cast<size_t>(p.T) * p.NA;
    const int NA = p.NA, Lq = p.Lq, Lkv = p.Lkv, splits = p.splits;
    float4 acc[CPG], cmp[CPG];
    for (int s0 = 0; s0 < splits; s0 += SPB) {
        float4 r[BATCH];
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            const int sp = s0 + u % SPB, i = i0 + (u / SPB) * NT * 4;
            if (sp < splits && i < NA) r[u] = *reinterpret_cast<const float4*>(prow + sp * sstride + i);
        }
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            const int c = u / SPB, sp = s0 + u % SPB, i = i0 + c * NT * 4;
            if (sp < splits && i < NA) {
                if constexpr (W8) {  // exact int32 partials: integer sums
                    if (sp == 0) {
                        acc[c] = r[u];
                    } else {
                        acc[c].x = __int_as_float(__float_as_int(acc[c].x) + __float_as_int(r[u].x));
                        acc[c].y = __int_as_float(__float_as_int(acc[c].y) + __float_as_int(r[u].y));
                        acc[c].z = __int_as_float(__float_as_int(acc[c].z) + __float_as_int(r[u].z));
                        acc[c].w = __int_as_float(__float_as_int(acc[c].w) + __float_as_int(r[u].w));
                    }
                } else if (sp == 0) {
                    acc[c] = r[u];
                    cmp[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                } else {
                    two_sum_add(acc[c].x, cmp[c].x, r[u].x);
                    two_sum_add(acc[c].y, cmp[c].y, r[u].y);
                    two_sum_add(acc[c].z, cmp[c].z, r[u].z);
                    two_sum_add(acc[c].w, cmp[c].w, r[u].w);
                }
            }
        }
    }
#pragma unroll
    for (int c = 0; c < CPG; ++c) {
        const int i = i0 + c * NT * 4;
        if (i < NA) {
            float4 a;
            if constexpr (W8) {  // AT-06 on the integer sums
                const float4 ws = *reinterpret_cast<const float4*>(p.w_scale + i);
                a = make_float4(w8_dequant(__float_as_int(acc[c].x), sx, ws.x),
                                w8_dequant(__float_as_int(acc[c].y), sx, ws.y),
                                w8_dequant(__float_as_int(acc[c].z), sx, ws.z),
                                w8_dequant(__float_as_int(acc[c].w), sx, ws.w));
            } else {
                a = make_float4(__fadd_rn(acc[c].x, cmp[c].x), __fadd_rn(acc[c].y, cmp[c].y),
                                __fadd_rn(acc[c].z, cmp[c].z), __fadd_rn(acc[c].w, cmp[c].w));
            }
            const uint32_t w0 = pack_bf16x2(a.x, a.y), w1 = pack_bf16x2(a.z, a.w);
            *reinterpret_cast<uint2*>(crow + i) = make_uint2(w0, w1);
            const float v[4] = {bf16_lo(w0), bf16_hi(w0), bf16_lo(w1), bf16_hi(w1)};
            if (i < Lq + Lkv) csum[i / 4] = chunk_ssq(v, i < Lq ? p.inv_lq : p.inv_lkv);
        }
    }
}

// One token of the norm step, by a group of NT threads (see group_sync):
// reduce the token's split-K partials in split order (TwoSum), round to
// BF16, RMSNorm of c_q and c_kv (x^2/L summed as chunk_ssq describes,
// + eps, sqrt, reciprocal, x * rstd, * gamma, BF16), rotate-half RoPE of
// k_pe, and write the normed row, out_kpe, K's rope slice of every head and
// (with a cache) the token's latent cache row [normed c_kv | k_pe_rot].
// `crow` is norm_token_smem_bytes of shared memory, `red` 2 floats (W8: 6
// words; the integer split-K partials are summed exactly and dequantised,
// and the normed rows leave as per-token codes, see norm_token_warp).
template <int NT, int BATCH, int FIRST = 0, bool W8 = false>
__device__ __forceinline__ void norm_token(const NormRopeParams& p, int t, uint16_t* crow, float* red) {
    constexpr int kNormThreads = NT;
    const int tid = static_cast<int>(threadIdx.x) - FIRST;
    const int NA = p.NA, Lq = p.Lq, Lkv = p.Lkv, R = p.R, half = R / 2;
    uint16_t* rot = crow + NA;
    float* csum = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(crow) +
                                           ((static_cast<size_t>(NA + R) * 2 + 15) & ~static_cast<size_t>(15)));

    const int pos = p.positions[t];
    const bool valid = pos >= 0 && pos < p.max_pos;
    if (tid == 0 && p.amax) p.amax[t] = 0u;
    uint16_t* nrow = p.normed + static_cast<size_t>(t) * (Lq + Lkv);
    uint16_t* cache_row = kv_cache_row(p, t, tid == 0);
    const int nchunk = R / 8;
    const int ndst = p.H + (cache_row ? 2 : 1);  // rope-slice destinations (kpe_dst)
    if (!valid) {  // CTA-uniform
        if (tid == 0) atomicOr(p.status, kStatusPositionRange);
        if (W8 && tid == 0) p.nscale[2 * t] = p.nscale[2 * t + 1] = 0.0f;
        const uint4 z = make_uint4(0, 0, 0, 0);
        for (int i = tid * 8; i < Lq + Lkv; i += kNormThreads * 8) {
            *reinterpret_cast<uint4*>(nrow + i) = z;
            if (cache_row && i >= Lq) *reinterpret_cast<uint4*>(cache_row + (i - Lq)) = z;
        }
        for (int k = tid; k < ndst * nchunk; k += kNormThreads) {
            const int h = k / nchunk, c = k - h * nchunk;
            *reinterpret_cast<uint4*>(kpe_dst(p, t, h, c, cache_row)) = z;
        }
        return;
    }

    // 0) Loads that do not wait for the partials: gamma for step 2 and this
    //    token's cos/sin row for step 3, in flight with step 1's loads.
    constexpr int kGammaPre = 2;
    uint4 gpre[kGammaPre];
#pragma unroll
    for (int u = 0; u < kGammaPre; ++u) {
        const int i = (tid + u * kNormThreads) * 8;
        if (i < Lq + Lkv) gpre[u] = *reinterpret_cast<const uint4*>(p.gamma + i);
    }
    const float* cs = p.cos_sin + static_cast<size_t>(pos) * R;
    float c_pre = 0.0f, s_pre = 0.0f;
    if (tid < half) c_pre = cs[tid], s_pre = cs[half + tid];

    // 1) Reduce the split-K partials in split order (TwoSum), round to BF16,
    //    and the chunk sums of x^2 / L of the c_q and c_kv blocks.  A thread's
    //    chunks go in groups whose loads (every split of up to two chunks,
    //    BATCH at most) are all in flight before the first sum.
    const float* prow = p.partials + static_cast<size_t>(t) * NA;
    uint32_t* ured = reinterpret_cast<uint32_t*>(red) + 2;  // W8: max |normed| and sum |code| of c_q, c_kv
    if (W8 && tid < 4) ured[tid] = 0u;
    const float sx = W8 ? p.x_scale[t] : 0.0f;
    if (2 * p.splits <= BATCH) {
        for (int i0 = tid * 4; i0 < NA; i0 += 2 * kNormThreads * 4)
            norm_chunk_group<2, BATCH, NT, W8>(p, prow, i0, crow, csum, sx);
    } else {
        for (int i0 = tid * 4; i0 < NA; i0 += kNormThreads * 4)
            norm_chunk_group<1, BATCH, NT, W8>(p, prow, i0, crow, csum, sx);
    }
    group_sync<NT, FIRST>();  // also publishes crow
    if (tid < 32) {
        float sq = 0.0f, skv = 0.0f;
        for (int j = tid; j < (Lq + Lkv) / 4; j += 32) {
            if (j < Lq / 4)
                sq = __fadd_rn(sq, csum[j]);
            else
                skv = __fadd_rn(skv, csum[j]);
        }
        sq = lane_butterfly_sum(sq);
        skv = lane_butterfly_sum(skv);
        if (tid == 0) red[0] = sq, red[1] = skv;
    }
    group_sync<NT, FIRST>();
    const float ssq_q = red[0], ssq_kv = red[1];
    // Variant B of the pages' RMSNorm: std = sqrt(ms + eps), rstd = 1 / std,
    // both correctly rounded.
    const float rstd_q = Lq > 0 ? __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ssq_q, p.eps))) : 0.0f;
    const float rstd_kv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ssq_kv, p.eps)));

    // 2) y = bf16((x * rstd) * gamma) for c_q and c_kv, 8 columns per thread.
    float amax_q = 0.0f, amax_kv = 0.0f;  // W8
    auto norm8 = [&](int i, const uint4 gv) {
        const uint4 xv = *reinterpret_cast<const uint4*>(crow + i);
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
        if constexpr (W8) {  // the normed values stay here until their codes are known
            *reinterpret_cast<uint4*>(crow + i) = ov;
            float m = 0.0f;
#pragma unroll
            for (int e = 0; e < 4; ++e) m = fmaxf(m, fmaxf(fabsf(bf16_lo(o[e])), fabsf(bf16_hi(o[e]))));
            if (i < Lq)
                amax_q = fmaxf(amax_q, m);
            else
                amax_kv = fmaxf(amax_kv, m);
        } else {
            *reinterpret_cast<uint4*>(nrow + i) = ov;
        }
        if (cache_row && i >= Lq) *reinterpret_cast<uint4*>(cache_row + (i - Lq)) = ov;
    };
#pragma unroll
    for (int u = 0; u < kGammaPre; ++u) {
        const int i = (tid + u * kNormThreads) * 8;
        if (i < Lq + Lkv) norm8(i, gpre[u]);
    }
    for (int i = (tid + kGammaPre * kNormThreads) * 8; i < Lq + Lkv; i += kNormThreads * 8)
        norm8(i, *reinterpret_cast<const uint4*>(p.gamma + i));
    if constexpr (W8) {
        // AT-11: per-token codes of the normed c_q and c_kv rows (group-wide
        // max |y| through shared memory: non-negative floats order as their bits)
        amax_q = warp_max(amax_q);
        amax_kv = warp_max(amax_kv);
        if ((tid & 31) == 0) {
            atomicMax(&ured[0], __float_as_uint(amax_q));
            atomicMax(&ured[1], __float_as_uint(amax_kv));
        }
        group_sync<NT, FIRST>();
        const float mq = __uint_as_float(ured[0]), mkv = __uint_as_float(ured[1]);
        const float inv_q = mq > 0.0f ? __fdiv_rn(127.0f, mq) : 0.0f;
        const float inv_kv = mkv > 0.0f ? __fdiv_rn(127.0f, mkv) : 0.0f;
        uint32_t sq = 0, skv = 0;
        for (int i = tid * 8; i < Lq + Lkv; i += kNormThreads * 8) {
            const uint4 yv = *reinterpret_cast<const uint4*>(crow + i);
            const uint4 cv = codes_bf16x8(yv, i < Lq ? inv_q : inv_kv);
            *reinterpret_cast<uint4*>(nrow + i) = cv;
            (i < Lq ? sq : skv) += abs_sum_bf16x8(cv);
        }
        sq = warp_sum(sq);
        skv = warp_sum(skv);
        if ((tid & 31) == 0) {
            atomicAdd(&ured[2], sq);
            atomicAdd(&ured[3], skv);
        }
        group_sync<NT, FIRST>();
        if (tid == 0) w8_finish_token(p, t, mq, mkv, ured[2], ured[3]);
    }

    // 3) k_pe RoPE (rotate-half) in FP32 with this token's cos/sin row; the
    //    interleaved variant pairs (2i, 2i + 1) and stores the pair at
    //    (i, i + R/2) (de-interleaved order).
    const uint16_t* kp = crow + Lq + Lkv;
    for (int i = tid; i < half; i += kNormThreads) {
        int j1, j2;
        kpe_pair(p.interleaved, i, half, j1, j2);
        const float x1 = __uint_as_float(static_cast<uint32_t>(kp[j1]) << 16);
        const float x2 = __uint_as_float(static_cast<uint32_t>(kp[j2]) << 16);
        const float c = i == tid ? c_pre : cs[i], s = i == tid ? s_pre : cs[half + i];
        const float o1 = __fadd_rn(__fmul_rn(x1, c), __fmul_rn(-x2, s));
        const float o2 = __fadd_rn(__fmul_rn(x2, c), __fmul_rn(x1, s));
        rot[i] = static_cast<uint16_t>(pack_bf16x2(o1, 0.0f) & 0xFFFFu);
        rot[i + half] = static_cast<uint16_t>(pack_bf16x2(o2, 0.0f) & 0xFFFFu);
    }
    group_sync<NT, FIRST>();

    // 4) out_kpe[t], the shared rope slice of K for every head and the
    //    cache row's k_pe.
    for (int k = tid; k < ndst * nchunk; k += kNormThreads) {
        const int h = k / nchunk, c = k - h * nchunk;
        *reinterpret_cast<uint4*>(kpe_dst(p, t, h, c, cache_row)) = *reinterpret_cast<const uint4*>(rot + c * 8);
    }
}

// One token of the norm step by one warp: reduce the token's `splits`
// partial rows (prow + sp * sstride, FP32, global or shared memory) in split
// order with TwoSum, round to BF16, RMSNorm of c_q and c_kv, RoPE of k_pe,
// and write the normed row, out_kpe, K's rope slice of every head and the
// cache row -- the arithmetic of norm_token, with the chunk sums of x^2 / L
// on lane (i / 4) % 32 in increasing chunk order, so the bits agree with it
// for equal partials.  `pos` is the token's position, `cs_row` its cos/sin
// row (read only when pos is valid; c_pre, s_pre: its entries lane and
// R/2 + lane, loaded by the caller) and `gamma` the Lq + Lkv weights, from
// global or shared memory.  `crow` is (NA + R) BF16 of this warp's shared
// memory.
__device__ __forceinline__ void norm_token_warp(const NormRopeParams& p, int t, int pos, const float* cs_row,
                                                const uint16_t* gamma, const float* prow, size_t sstride,
                                                int splits, uint16_t* crow, float c_pre, float s_pre) {
    const int lane = threadIdx.x & 31;
    const int NA = p.NA, Lq = p.Lq, Lkv = p.Lkv, R = p.R, half = R / 2;
    uint16_t* rot = crow + NA;
    const bool valid = pos >= 0 && pos < p.max_pos;
    if (lane == 0 && p.amax) p.amax[t] = 0u;
    uint16_t* nrow = p.normed + static_cast<size_t>(t) * (Lq + Lkv);
    uint16_t* cache_row = kv_cache_row(p, t, lane == 0);
    const int nchunk = R / 8;
    const int ndst = p.H + (cache_row ? 2 : 1);  // rope-slice destinations (kpe_dst)
    if (!valid) {
        if (lane == 0) atomicOr(p.status, kStatusPositionRange);
        if (lane == 0 && p.w8a8) p.nscale[2 * t] = p.nscale[2 * t + 1] = 0.0f;
        const uint4 z = make_uint4(0, 0, 0, 0);
        for (int i = lane * 8; i < Lq + Lkv; i += 256) {
            *reinterpret_cast<uint4*>(nrow + i) = z;
            if (cache_row && i >= Lq) *reinterpret_cast<uint4*>(cache_row + (i - Lq)) = z;
        }
        for (int k = lane; k < ndst * nchunk; k += 32) {
            const int h = k / nchunk, c = k - h * nchunk;
            *reinterpret_cast<uint4*>(kpe_dst(p, t, h, c, cache_row)) = z;
        }
        return;
    }
    float ssq_q = 0.0f, ssq_kv = 0.0f;
    // 4 columns -> BF16 row in shared memory and the sums of squares (chunk
    // i / 4 on lane (i / 4) % 32, in increasing order: chunk_ssq)
    auto take4 = [&](int i, float4 a) {
        const uint32_t w0 = pack_bf16x2(a.x, a.y), w1 = pack_bf16x2(a.z, a.w);
        *reinterpret_cast<uint2*>(crow + i) = make_uint2(w0, w1);
        const float v[4] = {bf16_lo(w0), bf16_hi(w0), bf16_lo(w1), bf16_hi(w1)};
        if (i < Lq)
            ssq_q = __fadd_rn(ssq_q, chunk_ssq(v, p.inv_lq));
        else if (i < Lq + Lkv)
            ssq_kv = __fadd_rn(ssq_kv, chunk_ssq(v, p.inv_lkv));
    };
    // One split: kB of the lane's loads in flight before any is used (the
    // shared-memory stores would otherwise keep each load behind the last).
    constexpr int kB = 6;
    if (p.in_bf16) {  // the compression already rounded the row to BF16
        const uint16_t* brow = reinterpret_cast<const uint16_t*>(prow);
        for (int i0 = lane * 4; i0 < NA; i0 += 128 * kB) {
            uint2 a[kB];
#pragma unroll
            for (int u = 0; u < kB; ++u)
                if (i0 + 128 * u < NA) a[u] = *reinterpret_cast<const uint2*>(brow + i0 + 128 * u);
#pragma unroll
            for (int u = 0; u < kB; ++u)
                if (i0 + 128 * u < NA)
                    take4(i0 + 128 * u, make_float4(bf16_lo(a[u].x), bf16_hi(a[u].x), bf16_lo(a[u].y), bf16_hi(a[u].y)));
        }
    }
    for (int i0 = lane * 4; splits == 1 && !p.in_bf16 && i0 < NA; i0 += 128 * kB) {
        float4 a[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u)
            if (i0 + 128 * u < NA) a[u] = *reinterpret_cast<const float4*>(prow + i0 + 128 * u);
#pragma unroll
        for (int u = 0; u < kB; ++u)
            if (i0 + 128 * u < NA) take4(i0 + 128 * u, a[u]);
    }
    for (int i = lane * 4; splits > 1 && p.w8a8 && i < NA; i += 128) {
        // W8A8: exact int32 partials, summed exactly, then dequantised
        int4 a = *reinterpret_cast<const int4*>(prow + i);
        for (int sp = 1; sp < splits; ++sp) {
            const int4 r = *reinterpret_cast<const int4*>(prow + sp * sstride + i);
            a.x += r.x, a.y += r.y, a.z += r.z, a.w += r.w;
        }
        const float sx = p.x_scale[t];
        const float4 ws = *reinterpret_cast<const float4*>(p.w_scale + i);
        take4(i, make_float4(w8_dequant(a.x, sx, ws.x), w8_dequant(a.y, sx, ws.y), w8_dequant(a.z, sx, ws.z),
                             w8_dequant(a.w, sx, ws.w)));
    }
    for (int i = lane * 4; splits > 1 && !p.w8a8 && i < NA; i += 128) {
        float4 a = *reinterpret_cast<const float4*>(prow + i), cmp = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int sp = 1; sp < splits; ++sp) {
            const float4 r = *reinterpret_cast<const float4*>(prow + sp * sstride + i);
            two_sum_add(a.x, cmp.x, r.x);
            two_sum_add(a.y, cmp.y, r.y);
            two_sum_add(a.z, cmp.z, r.z);
            two_sum_add(a.w, cmp.w, r.w);
        }
        a = make_float4(__fadd_rn(a.x, cmp.x), __fadd_rn(a.y, cmp.y), __fadd_rn(a.z, cmp.z), __fadd_rn(a.w, cmp.w));
        take4(i, a);
    }
    ssq_q = lane_butterfly_sum(ssq_q);
    ssq_kv = lane_butterfly_sum(ssq_kv);
    const float rstd_q = Lq > 0 ? __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ssq_q, p.eps))) : 0.0f;
    const float rstd_kv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ssq_kv, p.eps)));
    __syncwarp();
    float amax_q = 0.0f, amax_kv = 0.0f;  // W8A8: max |normed| of c_q and c_kv
    auto norm8 = [&](int i, const uint4 gv) {
        const uint4 xv = *reinterpret_cast<const uint4*>(crow + i);
        const float rstd = i < Lq ? rstd_q : rstd_kv;
        const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
        const uint32_t gs[4] = {gv.x, gv.y, gv.z, gv.w};
        uint32_t o[4];
        float m = 0.0f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float y0 = __fmul_rn(__fmul_rn(bf16_lo(xs[e]), rstd), bf16_lo(gs[e]));
            const float y1 = __fmul_rn(__fmul_rn(bf16_hi(xs[e]), rstd), bf16_hi(gs[e]));
            o[e] = pack_bf16x2(y0, y1);
            m = fmaxf(m, fmaxf(fabsf(bf16_lo(o[e])), fabsf(bf16_hi(o[e]))));
        }
        const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
        if (p.w8a8) {  // the normed values stay here until their codes are known
            *reinterpret_cast<uint4*>(crow + i) = ov;
            if (i < Lq)
                amax_q = fmaxf(amax_q, m);
            else
                amax_kv = fmaxf(amax_kv, m);
        } else {
            *reinterpret_cast<uint4*>(nrow + i) = ov;
        }
        if (cache_row && i >= Lq) *reinterpret_cast<uint4*>(cache_row + (i - Lq)) = ov;
    };
    for (int i = lane * 8; i < Lq + Lkv; i += 256) norm8(i, *reinterpret_cast<const uint4*>(gamma + i));
    if (p.w8a8) {
        // AT-11: the normed c_q and c_kv rows quantised per token, the
        // expansions' INT8 inputs (each lane re-reads its own chunks)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            amax_q = fmaxf(amax_q, __shfl_xor_sync(0xffffffffu, amax_q, o));
            amax_kv = fmaxf(amax_kv, __shfl_xor_sync(0xffffffffu, amax_kv, o));
        }
        const float inv_q = amax_q > 0.0f ? __fdiv_rn(127.0f, amax_q) : 0.0f;
        const float inv_kv = amax_kv > 0.0f ? __fdiv_rn(127.0f, amax_kv) : 0.0f;
        uint32_t sq = 0, skv = 0;
        for (int i = lane * 8; i < Lq + Lkv; i += 256) {
            const uint4 yv = *reinterpret_cast<const uint4*>(crow + i);
            const uint4 cv = codes_bf16x8(yv, i < Lq ? inv_q : inv_kv);
            *reinterpret_cast<uint4*>(nrow + i) = cv;
            (i < Lq ? sq : skv) += abs_sum_bf16x8(cv);
        }
        sq = warp_sum(sq);
        skv = warp_sum(skv);
        if (lane == 0) w8_finish_token(p, t, amax_q, amax_kv, sq, skv);
    }
    const uint16_t* kp = crow + Lq + Lkv;
    for (int i = lane; i < half; i += 32) {
        int j1, j2;
        kpe_pair(p.interleaved, i, half, j1, j2);
        const float x1 = __uint_as_float(static_cast<uint32_t>(kp[j1]) << 16);
        const float x2 = __uint_as_float(static_cast<uint32_t>(kp[j2]) << 16);
        const float c = i == lane ? c_pre : cs_row[i], s = i == lane ? s_pre : cs_row[half + i];
        const float o1 = __fadd_rn(__fmul_rn(x1, c), __fmul_rn(-x2, s));
        const float o2 = __fadd_rn(__fmul_rn(x2, c), __fmul_rn(x1, s));
        rot[i] = static_cast<uint16_t>(pack_bf16x2(o1, 0.0f) & 0xFFFFu);
        rot[i + half] = static_cast<uint16_t>(pack_bf16x2(o2, 0.0f) & 0xFFFFu);
    }
    __syncwarp();
    if (32 % nchunk == 0) {
        // Each lane keeps one 16-byte chunk c of the rotated row and writes
        // it to every (32 / nchunk)-th head's rope slice from head lane /
        // nchunk on, then out_kpe and the cache row (lanes below nchunk):
        // the same bytes as the destination loop below, without its
        // per-chunk division and destination choice.
        const int c = lane % nchunk, step = 32 / nchunk;
        const uint4 v = *reinterpret_cast<const uint4*>(rot + c * 8);
        const size_t hstride = static_cast<size_t>(p.Dn + R);
        uint16_t* dst = p.out_k + (static_cast<size_t>(t) * p.H + lane / nchunk) * hstride + p.Dn + c * 8;
        for (int h = lane / nchunk; h < p.H; h += step, dst += step * hstride) *reinterpret_cast<uint4*>(dst) = v;
        if (lane < nchunk) {
            *reinterpret_cast<uint4*>(kpe_dst(p, t, p.H, c, cache_row)) = v;
            if (cache_row) *reinterpret_cast<uint4*>(kpe_dst(p, t, p.H + 1, c, cache_row)) = v;
        }
        return;
    }
    for (int k = lane; k < ndst * nchunk; k += 32) {
        const int h = k / nchunk, c = k - h * nchunk;
        *reinterpret_cast<uint4*>(kpe_dst(p, t, h, c, cache_row)) = *reinterpret_cast<const uint4*>(rot + c * 8);
    }
}

// Quantises columns [c0, c1) of one row with the row's amax, by `nthr`
// threads (this one is `tid`): inv = 127/amax, rint(y*inv) ties to even,
// clamp +-127, all correctly rounded; the chunk holding column 0 writes the
// scale amax/127.  A zero row gives codes 0 and scale 0.
template <int kB = 8>  // 16-byte loads in flight per thread
__device__ __forceinline__ void quant_span(const QuantParams& p, int row, int c0, int c1, float amax, int tid,
                                           int nthr) {
    const float* y = p.y + static_cast<size_t>(row) * p.row_len;
    int8_t* out = p.codes + static_cast<size_t>(row) * p.row_len;
    if (amax == 0.0f) {
        for (int i = c0 + tid * 4; i < c1; i += nthr * 4) *reinterpret_cast<char4*>(out + i) = make_char4(0, 0, 0, 0);
        if (tid == 0 && c0 == 0) p.scale[row] = 0.0f;
        return;
    }
    const float inv = __fdiv_rn(127.0f, amax);
    // kB loads in flight per thread before any store
    for (int i0 = c0 + tid * 4; i0 < c1; i0 += kB * nthr * 4) {
        float4 v[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u) {
            const int i = i0 + u * nthr * 4;
            if (i < c1) v[u] = *reinterpret_cast<const float4*>(y + i);
        }
#pragma unroll
        for (int u = 0; u < kB; ++u) {
            const int i = i0 + u * nthr * 4;
            if (i < c1) {
                const float f[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                signed char c[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int q = __float2int_rn(__fmul_rn(f[e], inv));  // round to nearest, ties to even
                    q = q > 127 ? 127 : (q < -127 ? -127 : q);
                    c[e] = static_cast<signed char>(q);
                }
                *reinterpret_cast<char4*>(out + i) = make_char4(c[0], c[1], c[2], c[3]);
            }
        }
    }
    if (tid == 0 && c0 == 0) p.scale[row] = __fdiv_rn(amax, 127.0f);
}

}  // namespace mlap
