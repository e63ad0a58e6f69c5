// Row-wise kernels of the prolog.
//
// mla_norm_rope_kernel  one warp per token: sums the split-K partials of the
//   compression projection in split order (deterministic), rounds each value
//   to BF16, splits the row into c_q | c_kv | k_pe, applies RMSNorm in FP32
//   (sum of x^2/L, + eps, sqrt, reciprocal, x * rstd, * gamma, cast to BF16:
//   PyPTO-Gym AT-10 article, section 三 variant B and section 五) and
//   rotate-half RoPE to k_pe, and writes out_kpe plus the rope slice of every
//   head of out_k (the "assemble" step of the V2-Lite migration guide).
//
// mla_quant_kernel  one CTA per token row: per-token symmetric INT8 with
//   correctly rounded FP32 operations (inv = 127/amax, rint(y*inv) ties to
//   even, clamp +-127, scale = amax/127), as in the PrologQuant section of the
//   DeepSeek-V3.2-Exp PyPTO article.
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

// One CTA per token.  Launched as a programmatic dependent of the compression
// kernel: it waits for the partials, then lets the expansion kernel launch.
// With split-K partials (decode) the CTA is wider and keeps every split's
// load of its columns in flight at once: the step is latency bound.
template <bool SPLIT, int NT>
__global__ void __launch_bounds__(NT) mla_norm_rope_kernel(const NormRopeParams p) {
    constexpr int kNormThreads = NT;
    constexpr int kNormWarps = NT / 32;
    constexpr int kBatch = SPLIT ? 16 : 1;
    extern __shared__ __align__(16) uint16_t crow[];  // BF16 row of C [NA], then rotated k_pe [R]
    __shared__ float red[2][kNormWarps];
    pdl_wait();
    pdl_launch_dependents();
    const int t = blockIdx.x, tid = threadIdx.x;
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
        if (SPLIT) {
            // every split's load in flight first (up to kBatch at a time),
            // then the sums in split order with TwoSum
            float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int s0 = 1; s0 < p.splits; s0 += kBatch) {
                float4 b[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; ++u)
                    if (s0 + u < p.splits) b[u] = *reinterpret_cast<const float4*>(prow + (s0 + u) * sstride + i);
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
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
    ssq_q = block_sum<kNormWarps>(ssq_q, red[0]);
    ssq_kv = block_sum<kNormWarps>(ssq_kv, red[1]);  // its __syncthreads also publishes crow
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

// Prefill variant (no split-K partials): one warp per token, eight tokens
// per CTA, so many tokens' loads are in flight per SM and no CTA-wide
// barrier sits between the steps.  Same arithmetic as mla_norm_rope_kernel.
constexpr int kNormWarpTokens = 8;

__global__ void __launch_bounds__(32 * kNormWarpTokens) mla_norm_rope_warp_kernel(const NormRopeParams p) {
    extern __shared__ __align__(16) uint16_t wsm[];
    pdl_wait();
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * kNormWarpTokens + warp;
    if (t >= p.T) return;  // warp-uniform
    const int NA = p.NA, Lq = p.Lq, Lkv = p.Lkv, R = p.R, half = R / 2;
    uint16_t* crow = wsm + static_cast<size_t>(warp) * (NA + R);
    uint16_t* rot = crow + NA;
    const int pos = p.positions[t];
    const bool valid = pos >= 0 && pos < p.max_pos;
    if (lane == 0 && p.amax) p.amax[t] = 0u;
    uint16_t* nrow = p.normed + static_cast<size_t>(t) * (Lq + Lkv);
    const int nchunk = R / 8;
    if (!valid) {
        if (lane == 0) atomicOr(p.status, kStatusPositionRange);
        const uint4 z = make_uint4(0, 0, 0, 0);
        for (int i = lane * 8; i < Lq + Lkv; i += 256) *reinterpret_cast<uint4*>(nrow + i) = z;
        for (int k = lane; k < (p.H + 1) * nchunk; k += 32) {
            const int h = k / nchunk, c = k - h * nchunk;
            uint16_t* dst = h < p.H ? p.out_k + (static_cast<size_t>(t) * p.H + h) * (p.Dn + R) + p.Dn + c * 8
                                    : p.out_kpe + static_cast<size_t>(t) * R + c * 8;
            *reinterpret_cast<uint4*>(dst) = z;
        }
        return;
    }
    float ssq_q = 0.0f, ssq_kv = 0.0f;
    const float* prow = p.partials + static_cast<size_t>(t) * NA;
    for (int i = lane * 4; i < NA; i += 128) {
        const float4 a = *reinterpret_cast<const float4*>(prow + i);
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
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ssq_q = __fadd_rn(ssq_q, __shfl_xor_sync(0xffffffffu, ssq_q, o));
        ssq_kv = __fadd_rn(ssq_kv, __shfl_xor_sync(0xffffffffu, ssq_kv, o));
    }
    const float rstd_q = Lq > 0 ? __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ssq_q, p.eps))) : 0.0f;
    const float rstd_kv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ssq_kv, p.eps)));
    __syncwarp();
    for (int i = lane * 8; i < Lq + Lkv; i += 256) {
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
    const uint16_t* kp = crow + Lq + Lkv;
    const float* cs = p.cos_sin + static_cast<size_t>(pos) * R;
    for (int i = lane; i < half; i += 32) {
        const float x1 = __uint_as_float(static_cast<uint32_t>(kp[i]) << 16);
        const float x2 = __uint_as_float(static_cast<uint32_t>(kp[i + half]) << 16);
        const float c = cs[i], s = cs[half + i];
        const float o1 = __fadd_rn(__fmul_rn(x1, c), __fmul_rn(-x2, s));
        const float o2 = __fadd_rn(__fmul_rn(x2, c), __fmul_rn(x1, s));
        rot[i] = static_cast<uint16_t>(pack_bf16x2(o1, 0.0f) & 0xFFFFu);
        rot[i + half] = static_cast<uint16_t>(pack_bf16x2(o2, 0.0f) & 0xFFFFu);
    }
    __syncwarp();
    for (int k = lane; k < (p.H + 1) * nchunk; k += 32) {
        const int h = k / nchunk, c = k - h * nchunk;
        const uint4 v = *reinterpret_cast<const uint4*>(rot + c * 8);
        uint16_t* dst = h < p.H ? p.out_k + (static_cast<size_t>(t) * p.H + h) * (p.Dn + R) + p.Dn + c * 8
                                : p.out_kpe + static_cast<size_t>(t) * R + c * 8;
        *reinterpret_cast<uint4*>(dst) = v;
    }
}

// ---------------------------------------------------------------- quant

constexpr int kQuantThreads = 256;
constexpr int kQuantChunk = 4096;  // elements per CTA when amax is known

// blockIdx.x = row, blockIdx.y = chunk of the row.  With a known amax the
// chunks of a row are independent; without one, one CTA takes the whole row
// and first reduces max |y|.
__global__ void __launch_bounds__(kQuantThreads) mla_quant_kernel(const QuantParams p) {
    pdl_wait();
    const int row = blockIdx.x;
    const float* y = p.y + static_cast<size_t>(row) * p.row_len;
    const int c0 = blockIdx.y * p.chunk;
    const int c1 = c0 + p.chunk < p.row_len ? c0 + p.chunk : p.row_len;
    float amax;
    if (p.amax) {
        amax = __uint_as_float(p.amax[row]);
    } else {
        __shared__ float red[kQuantThreads / 32];
        float m = 0.0f;
        for (int i = threadIdx.x * 4; i < p.row_len; i += kQuantThreads * 4) {
            const float4 v = *reinterpret_cast<const float4*>(y + i);
            m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
        __syncthreads();
        m = 0.0f;
#pragma unroll
        for (int w = 0; w < kQuantThreads / 32; ++w) m = fmaxf(m, red[w]);
        amax = m;
    }
    int8_t* out = p.codes + static_cast<size_t>(row) * p.row_len;
    if (amax == 0.0f) {
        for (int i = c0 + threadIdx.x * 4; i < c1; i += kQuantThreads * 4)
            *reinterpret_cast<char4*>(out + i) = make_char4(0, 0, 0, 0);
        if (threadIdx.x == 0 && blockIdx.y == 0) p.scale[row] = 0.0f;
        return;
    }
    const float inv = __fdiv_rn(127.0f, amax);
#pragma unroll 4
    for (int i = c0 + threadIdx.x * 4; i < c1; i += kQuantThreads * 4) {
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
    if (threadIdx.x == 0 && blockIdx.y == 0) p.scale[row] = __fdiv_rn(amax, 127.0f);
}

// ------------------------------------------------------------ launchers

cudaError_t launch_norm_rope(const NormRopeParams& p, cudaStream_t st) {
    if (p.T == 0) return cudaSuccess;
    const size_t smem = static_cast<size_t>(p.NA + p.R) * sizeof(uint16_t);
    if (p.splits > 1)
        return launch_kernel(mla_norm_rope_kernel<true, 512>, dim3(p.T), dim3(512), smem, st, true, p);
    return launch_kernel(mla_norm_rope_warp_kernel, dim3((p.T + kNormWarpTokens - 1) / kNormWarpTokens),
                         dim3(32 * kNormWarpTokens), smem * kNormWarpTokens, st, true, p);
}

cudaError_t launch_quant(const QuantParams& p_in, cudaStream_t st, bool pdl) {
    if (p_in.rows == 0) return cudaSuccess;
    QuantParams p = p_in;
    p.chunk = p.amax ? kQuantChunk : p.row_len;
    const int chunks = (p.row_len + p.chunk - 1) / p.chunk;
    return launch_kernel(mla_quant_kernel, dim3(p.rows, chunks), dim3(kQuantThreads), 0, st, pdl, p);
}

}  // namespace mlap
