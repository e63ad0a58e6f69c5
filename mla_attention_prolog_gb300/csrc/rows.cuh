// Row-wise steps of the prolog as device functions, shared by the
// standalone kernels (rowwise.cu) and the cooperative decode kernel.
#pragma once

#include "prolog.cuh"
#include "ptx.cuh"

namespace mlap {

// Sum of a per-thread value over the CTA in a fixed order (deterministic).
template <int NW>
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < NW; ++w) s = __fadd_rn(s, red[w]);
    return s;
}

// One token of the norm step, by a CTA of NT threads (threadIdx.x < NT):
// reduce the token's split-K partials in split order (TwoSum), round to
// BF16, RMSNorm of c_q and c_kv (x^2/L summed, + eps, sqrt, reciprocal,
// x * rstd, * gamma, BF16), rotate-half RoPE of k_pe, and write the normed
// row, out_kpe and K's rope slice of every head.  `crow` is NA + R BF16
// values of shared memory, `red` 2 * NT / 32 floats.
template <int NT, int BATCH>
__device__ __forceinline__ void norm_token(const NormRopeParams& p, int t, uint16_t* crow, float* red) {
    constexpr int kNormThreads = NT;
    constexpr int kNormWarps = NT / 32;
    const int tid = threadIdx.x;
    const int NA = p.NA, Lq = p.Lq, Lkv = p.Lkv, R = p.R, half = R / 2;
    uint16_t* rot = crow + NA;

    const int pos = p.positions[t];
    const bool valid = pos >= 0 && pos < p.max_pos;
    if (tid == 0 && p.amax) p.amax[t] = 0u;
    uint16_t* nrow = p.normed + static_cast<size_t>(t) * (Lq + Lkv);
    const int nchunk = R / 8;
    if (!valid) {  // CTA-uniform
        if (tid == 0) atomicOr(p.status, kStatusPositionRange);
        const uint4 z = make_uint4(0, 0, 0, 0);
        for (int i = tid * 8; i < Lq + Lkv; i += kNormThreads * 8) *reinterpret_cast<uint4*>(nrow + i) = z;
        for (int k = tid; k < (p.H + 1) * nchunk; k += kNormThreads) {
            const int h = k / nchunk, c = k - h * nchunk;
            uint16_t* dst = h < p.H ? p.out_k + (static_cast<size_t>(t) * p.H + h) * (p.Dn + R) + p.Dn + c * 8
                                    : p.out_kpe + static_cast<size_t>(t) * R + c * 8;
            *reinterpret_cast<uint4*>(dst) = z;
        }
        return;
    }

    // 1) Reduce the split-K partials in split order (TwoSum), round to BF16,
    //    and accumulate x^2 / L of the c_q and c_kv blocks.
    float ssq_q = 0.0f, ssq_kv = 0.0f;
    const size_t sstride = static_cast<size_t>(p.T) * NA;
    const float* prow = p.partials + static_cast<size_t>(t) * NA;
    for (int i = tid * 4; i < NA; i += kNormThreads * 4) {
        float4 a = *reinterpret_cast<const float4*>(prow + i);
        if (BATCH > 1 && p.splits > 1) {
            // every split's load in flight first (up to BATCH at a time),
            // then the sums in split order with TwoSum
            float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int s0 = 1; s0 < p.splits; s0 += BATCH) {
                float4 b[BATCH];
#pragma unroll
                for (int u = 0; u < BATCH; ++u)
                    if (s0 + u < p.splits) b[u] = *reinterpret_cast<const float4*>(prow + (s0 + u) * sstride + i);
#pragma unroll
                for (int u = 0; u < BATCH; ++u) {
                    if (s0 + u < p.splits) {
                        two_sum_add(a.x, c.x, b[u].x);
                        two_sum_add(a.y, c.y, b[u].y);
                        two_sum_add(a.z, c.z, b[u].z);
                        two_sum_add(a.w, c.w, b[u].w);
                    }
                }
            }
            a = make_float4(__fadd_rn(a.x, c.x), __fadd_rn(a.y, c.y), __fadd_rn(a.z, c.z), __fadd_rn(a.w, c.w));
        }
        const uint32_t w0 = pack_bf16x2(a.x, a.y), w1 = pack_bf16x2(a.z, a.w);
        *reinterpret_cast<uint2*>(crow + i) = make_uint2(w0, w1);
        const float v[4] = {bf16_lo(w0), bf16_hi(w0), bf16_lo(w1), bf16_hi(w1)};
        if (i < Lq) {
#pragma unroll
            for (int e = 0; e < 4; ++e) ssq_q = __fadd_rn(ssq_q, __fmul_rn(__fmul_rn(v[e], v[e]), p.inv_lq));
        } else if (i < Lq + Lkv) {
#pragma unroll
            for (int e = 0; e < 4; ++e) ssq_kv = __fadd_rn(ssq_kv, __fmul_rn(__fmul_rn(v[e], v[e]), p.inv_lkv));
        }
    }
    ssq_q = block_sum<kNormWarps>(ssq_q, red);
    ssq_kv = block_sum<kNormWarps>(ssq_kv, red + kNormWarps);  // its __syncthreads also publishes crow
    // Variant B of the pages' RMSNorm: std = sqrt(ms + eps), rstd = 1 / std,
    // both correctly rounded.
    const float rstd_q = Lq > 0 ? __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ssq_q, p.eps))) : 0.0f;
    const float rstd_kv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ssq_kv, p.eps)));

    // 2) y = bf16((x * rstd) * gamma) for c_q and c_kv, 8 columns per thread.
    for (int i = tid * 8; i < Lq + Lkv; i += kNormThreads * 8) {
        const uint4 xv = *reinterpret_cast<const uint4*>(crow + i);
        const uint4 gv = *reinterpret_cast<const uint4*>(p.gamma + i);
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
        *reinterpret_cast<uint4*>(nrow + i) = make_uint4(o[0], o[1], o[2], o[3]);
    }

    // 3) k_pe RoPE (rotate-half) in FP32 with this token's cos/sin row.
    const uint16_t* kp = crow + Lq + Lkv;
    const float* cs = p.cos_sin + static_cast<size_t>(pos) * R;
    for (int i = tid; i < half; i += kNormThreads) {
        const float x1 = __uint_as_float(static_cast<uint32_t>(kp[i]) << 16);
        const float x2 = __uint_as_float(static_cast<uint32_t>(kp[i + half]) << 16);
        const float c = cs[i], s = cs[half + i];
        const float o1 = __fadd_rn(__fmul_rn(x1, c), __fmul_rn(-x2, s));
        const float o2 = __fadd_rn(__fmul_rn(x2, c), __fmul_rn(x1, s));
        rot[i] = static_cast<uint16_t>(pack_bf16x2(o1, 0.0f) & 0xFFFFu);
        rot[i + half] = static_cast<uint16_t>(pack_bf16x2(o2, 0.0f) & 0xFFFFu);
    }
    __syncthreads();

    // 4) out_kpe[t] and the shared rope slice of K for every head.
    for (int k = tid; k < (p.H + 1) * nchunk; k += kNormThreads) {
        const int h = k / nchunk, c = k - h * nchunk;
        const uint4 v = *reinterpret_cast<const uint4*>(rot + c * 8);
        uint16_t* dst = h < p.H ? p.out_k + (static_cast<size_t>(t) * p.H + h) * (p.Dn + R) + p.Dn + c * 8
                                : p.out_kpe + static_cast<size_t>(t) * R + c * 8;
        *reinterpret_cast<uint4*>(dst) = v;
    }
}

// Quantises columns [c0, c1) of one row with the row's amax, by `nthr`
// threads (this one is `tid`): inv = 127/amax, rint(y*inv) ties to even,
// clamp +-127, all correctly rounded; the chunk holding column 0 writes the
// scale amax/127.  A zero row gives codes 0 and scale 0.
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
#pragma unroll 4
    for (int i = c0 + tid * 4; i < c1; i += nthr * 4) {
        const float4 v = *reinterpret_cast<const float4*>(y + i);
        const float f[4] = {v.x, v.y, v.z, v.w};
        signed char c[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            int q = __float2int_rn(__fmul_rn(f[e], inv));  // round to nearest, ties to even
            q = q > 127 ? 127 : (q < -127 ? -127 : q);
            c[e] = static_cast<signed char>(q);
        }
        *reinterpret_cast<char4*>(out + i) = make_char4(c[0], c[1], c[2], c[3]);
    }
    if (tid == 0 && c0 == 0) p.scale[row] = __fdiv_rn(amax, 127.0f);
}

}  // namespace mlap
