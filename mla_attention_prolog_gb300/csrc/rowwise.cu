// Row-wise kernels of the prolog.
//
// mla_norm_rope_kernel  one warp per token: sums the split-K partials of the
//   compression projection in split order (deterministic), rounds each value
//   to BF16, splits the row into c_q | c_kv | k_pe, applies RMSNorm in FP32
//   (sum of x^2/L, + eps, sqrt, reciprocal, x * rstd, * gamma, cast to BF16:
//   PyPTO-Gym AT-10 article, section 三 variant B and section 五) and
//   rotate-half RoPE to k_pe, and writes out_kpe plus the rope slice of every
//   head of out_k (the "assemble" step of the V2-Lite migration guide) and,
//   when a latent KV cache is given, the token's cache row [normed c_kv |
//   k_pe_rot] (the ScatterUpdate into the KV cache of the DeepSeek-V3.2-Exp
//   PyPTO article).
//
// mla_quant_kernel  one CTA per token row: per-token symmetric INT8 with
//   correctly rounded FP32 operations (inv = 127/amax, rint(y*inv) ties to
//   even, clamp +-127, scale = amax/127), as in the PrologQuant section of the
//   DeepSeek-V3.2-Exp PyPTO article.
#include "rows.cuh"

namespace mlap {

// One CTA per token.  Launched as a programmatic dependent of the compression
// kernel: it waits for the partials, then lets the expansion kernel launch.
// With split-K partials (decode) the CTA is wide and keeps every split's load
// of its columns in flight at once: the step is latency bound.
template <int NT, int BATCH>
__global__ void __launch_bounds__(NT) mla_norm_rope_kernel(const NormRopeParams p) {
    extern __shared__ __align__(16) uint16_t crow[];  // BF16 row of C [NA], then rotated k_pe [R]
    __shared__ float red[2];
    pdl_wait();
    pdl_launch_dependents();
    norm_token<NT, BATCH>(p, blockIdx.x, crow, red);
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
    uint16_t* cache_row = kv_cache_row(p, t, lane == 0);
    const int nchunk = R / 8;
    const int ndst = p.H + (cache_row ? 2 : 1);  // rope-slice destinations (kpe_dst)
    if (!valid) {
        if (lane == 0) atomicOr(p.status, kStatusPositionRange);
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
    const float* prow = p.partials + static_cast<size_t>(t) * NA;
    for (int i = lane * 4; i < NA; i += 128) {
        const float4 a = *reinterpret_cast<const float4*>(prow + i);
        const uint32_t w0 = pack_bf16x2(a.x, a.y), w1 = pack_bf16x2(a.z, a.w);
        *reinterpret_cast<uint2*>(crow + i) = make_uint2(w0, w1);
        const float v[4] = {bf16_lo(w0), bf16_hi(w0), bf16_lo(w1), bf16_hi(w1)};
        // chunk i / 4 on lane (i / 4) % 32, in increasing order (chunk_ssq)
        if (i < Lq)
            ssq_q = __fadd_rn(ssq_q, chunk_ssq(v, p.inv_lq));
        else if (i < Lq + Lkv)
            ssq_kv = __fadd_rn(ssq_kv, chunk_ssq(v, p.inv_lkv));
    }
    ssq_q = lane_butterfly_sum(ssq_q);
    ssq_kv = lane_butterfly_sum(ssq_kv);
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
        const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(nrow + i) = ov;
        if (cache_row && i >= Lq) *reinterpret_cast<uint4*>(cache_row + (i - Lq)) = ov;
    }
    const uint16_t* kp = crow + Lq + Lkv;
    const float* cs = p.cos_sin + static_cast<size_t>(pos) * R;
    for (int i = lane; i < half; i += 32) {
        int j1, j2;
        kpe_pair(p.interleaved, i, half, j1, j2);
        const float x1 = __uint_as_float(static_cast<uint32_t>(kp[j1]) << 16);
        const float x2 = __uint_as_float(static_cast<uint32_t>(kp[j2]) << 16);
        const float c = cs[i], s = cs[half + i];
        const float o1 = __fadd_rn(__fmul_rn(x1, c), __fmul_rn(-x2, s));
        const float o2 = __fadd_rn(__fmul_rn(x2, c), __fmul_rn(x1, s));
        rot[i] = static_cast<uint16_t>(pack_bf16x2(o1, 0.0f) & 0xFFFFu);
        rot[i + half] = static_cast<uint16_t>(pack_bf16x2(o2, 0.0f) & 0xFFFFu);
    }
    __syncwarp();
    for (int k = lane; k < ndst * nchunk; k += 32) {
        const int h = k / nchunk, c = k - h * nchunk;
        *reinterpret_cast<uint4*>(kpe_dst(p, t, h, c, cache_row)) = *reinterpret_cast<const uint4*>(rot + c * 8);
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
    const int c0 = blockIdx.y * p.chunk;
    const int c1 = c0 + p.chunk < p.row_len ? c0 + p.chunk : p.row_len;
    float amax;
    if (p.amax) {
        amax = __uint_as_float(p.amax[row]);
    } else {
        __shared__ float red[kQuantThreads / 32];
        const float* y = p.y + static_cast<size_t>(row) * p.row_len;
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
    quant_span(p, row, c0, c1, amax, threadIdx.x, kQuantThreads);
}

// ------------------------------------------------------------ launchers

cudaError_t launch_norm_rope(const NormRopeParams& p, cudaStream_t st) {
    if (p.T == 0) return cudaSuccess;
    if (p.splits > 1)
        return launch_kernel(mla_norm_rope_kernel<512, 16>, dim3(p.T), dim3(512),
                             norm_token_smem_bytes(p.NA, p.R, p.Lq, p.Lkv), st, true, p);
    const size_t smem = static_cast<size_t>(p.NA + p.R) * sizeof(uint16_t);
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
