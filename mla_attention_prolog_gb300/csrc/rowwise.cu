// Row-wise kernels of the prolog.
//
// mla_norm_rope_kernel  one CTA per token (split-K partials) or one warp per
//   token (mla_norm_rope_warp_kernel, prefill): sums the split-K partials of the
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
template <int NT, int BATCH, bool W8 = false>
__global__ void __launch_bounds__(NT) mla_norm_rope_kernel(const NormRopeParams p) {
    extern __shared__ __align__(16) uint16_t crow[];  // BF16 row of C [NA], then rotated k_pe [R]
    __shared__ float red[6];
    // The dependent expansion may start launching now: its CTAs prefetch their
    // first weight tiles while this grid runs, and wait for it before reading
    // the normed rows.
    pdl_launch_dependents();
    pdl_wait();
    norm_token<NT, BATCH, 0, W8>(p, blockIdx.x, crow, red);
}

// Prefill variant (no split-K partials): one warp per token, eight tokens
// per CTA, so many tokens' loads are in flight per SM and no CTA-wide
// barrier sits between the steps.  Same arithmetic as mla_norm_rope_kernel.
constexpr int kNormWarpTokens = 8;

// Shared memory: gamma (Lq + Lkv BF16, 16-byte aligned), then each warp's
// BF16 row and rotated k_pe.  Everything that does not come from the
// previous kernel (gamma, the token's position and its cos/sin pair) is
// loaded before the dependency wait, so after it only the row's loads stand
// between the wait and the first result.
__global__ void __launch_bounds__(32 * kNormWarpTokens) mla_norm_rope_warp_kernel(const NormRopeParams p) {
    extern __shared__ __align__(16) uint16_t wsm[];
    pdl_launch_dependents();  // as in mla_norm_rope_kernel
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ng = p.Lq + p.Lkv, gpad = (ng + 7) & ~7;
    for (int i = threadIdx.x * 8; i < ng; i += 32 * kNormWarpTokens * 8)
        *reinterpret_cast<uint4*>(wsm + i) = *reinterpret_cast<const uint4*>(p.gamma + i);
    const int t = blockIdx.x * kNormWarpTokens + warp;
    int pos = 0;
    float c_pre = 0.0f, s_pre = 0.0f;
    const float* cs_row = p.cos_sin;
    if (t < p.T) {
        pos = p.positions[t];
        if (pos >= 0 && pos < p.max_pos) {
            cs_row = p.cos_sin + static_cast<size_t>(pos) * p.R;
            if (lane < p.R / 2) c_pre = cs_row[lane], s_pre = cs_row[p.R / 2 + lane];
        }
    }
    __syncthreads();  // gamma staged
    pdl_wait();
    if (t >= p.T) return;  // warp-uniform
    // the row of token t: FP32 partials, or (in_bf16) the BF16 row, at element t * NA of its type
    const float* prow = p.in_bf16 ? reinterpret_cast<const float*>(reinterpret_cast<const uint16_t*>(p.partials) +
                                                                   static_cast<size_t>(t) * p.NA)
                                  : p.partials + static_cast<size_t>(t) * p.NA;
    norm_token_warp(p, t, pos, cs_row, wsm, prow, static_cast<size_t>(p.T) * p.NA, p.splits,
                    wsm + gpad + static_cast<size_t>(warp) * (p.NA + p.R), c_pre, s_pre);
}

// ---------------------------------------------------------------- quant

constexpr int kQuantThreads = 256;
// Elements per CTA when the amax is known: one batch of KB 16-byte loads in
// flight per thread, 256 * KB * 4 elements.  Measured on GB300 (V3 prefill,
// 16384 rows of 24576, the kernel alone): 4096 -> 338 us, 8192 and 12288 ->
// 291 us (the copy rate), 16384 -> 343 us (a ragged second chunk per row).
// Beside the kv-resident kernel (one quant CTA per SM) 12 or 16 loads in
// flight per thread measured no faster than 8.
constexpr int kQuantLoads = 8;

// blockIdx.x = row, blockIdx.y = chunk of the row.  With a known amax the
// chunks of a row are independent; without one, one CTA takes the whole row
// and first reduces max |y|.
template <int KB>
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
    quant_span<KB>(p, row, c0, c1, amax, threadIdx.x, kQuantThreads);
}

// ------------------------------------------------------------ W8A8

// One CTA per row of x: the per-token symmetric INT8 quantisation of the
// BF16 row (amax = max |x|, inv = 127/amax, code = rint(x * inv) ties to
// even, clamped to +-127, scale = amax/127, all correctly rounded FP32;
// AT-05 in the PyPTO-Gym AT-10 article, section 四).  The codes are written
// as BF16, which holds every integer of magnitude <= 127 exactly: the form
// the BF16 tensor-core path multiplies.  A zero row gives codes 0, scale 0.
constexpr int kQuantXThreads = 256;

__global__ void __launch_bounds__(kQuantXThreads) mla_quant_x_kernel(const QuantXParams p) {
    __shared__ float red[kQuantXThreads / 32];
    const int row = blockIdx.x;
    if (threadIdx.x == 0 && row < p.n_split) p.w8_split[row] = 0u;  // (rows >= tiles)
    const uint16_t* x = p.x + static_cast<size_t>(row) * p.cols;
    uint16_t* out = p.codes + static_cast<size_t>(row) * p.cols;
    float m = 0.0f;
    for (int i = threadIdx.x * 8; i < p.cols; i += kQuantXThreads * 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(x + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[e])), fabsf(bf16_hi(w[e]))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    float amax = 0.0f;
#pragma unroll
    for (int w = 0; w < kQuantXThreads / 32; ++w) amax = fmaxf(amax, red[w]);
    const float inv = amax > 0.0f ? __fdiv_rn(127.0f, amax) : 0.0f;
    for (int i = threadIdx.x * 8; i < p.cols; i += kQuantXThreads * 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(x + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) o[e] = code_bf16x2(bf16_lo(w[e]), bf16_hi(w[e]), inv);
        *reinterpret_cast<uint4*>(out + i) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (threadIdx.x == 0) p.scale[row] = amax > 0.0f ? __fdiv_rn(amax, 127.0f) : 0.0f;
}

// INT8 weight codes -> BF16 integers, 16 per thread step.
__global__ void __launch_bounds__(256) mla_widen_i8_kernel(const int8_t* src, uint16_t* dst, size_t n) {
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x * 16;
    for (size_t i = (static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 16; i < n; i += stride) {
        if (i + 16 <= n) {
            const int4 v = *reinterpret_cast<const int4*>(src + i);
            const uint32_t w[4] = {static_cast<uint32_t>(v.x), static_cast<uint32_t>(v.y),
                                   static_cast<uint32_t>(v.z), static_cast<uint32_t>(v.w)};
            uint32_t o[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float b0 = static_cast<float>(static_cast<int8_t>(w[e] & 0xFF));
                const float b1 = static_cast<float>(static_cast<int8_t>((w[e] >> 8) & 0xFF));
                const float b2 = static_cast<float>(static_cast<int8_t>((w[e] >> 16) & 0xFF));
                const float b3 = static_cast<float>(static_cast<int8_t>(w[e] >> 24));
                o[2 * e] = pack_bf16x2(b0, b1);
                o[2 * e + 1] = pack_bf16x2(b2, b3);
            }
            *reinterpret_cast<uint4*>(dst + i) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(dst + i + 8) = make_uint4(o[4], o[5], o[6], o[7]);
        } else {
            for (size_t k = i; k < n; ++k)
                dst[k] = static_cast<uint16_t>(pack_bf16x2(static_cast<float>(src[k]), 0.0f) & 0xFFFFu);
        }
    }
}

// ------------------------------------------------------------ launchers

cudaError_t launch_norm_rope(const NormRopeParams& p, cudaStream_t st) {
    if (p.T == 0) return cudaSuccess;
    // split-K partials of a decode batch: a wide CTA per token keeps every
    // split's load in flight; prefill (many tokens): one warp per token
    if (p.splits > 1 && p.T <= 2 * kBM)
        return launch_kernel(p.w8a8 ? mla_norm_rope_kernel<512, 16, true> : mla_norm_rope_kernel<512, 16>, dim3(p.T),
                             dim3(512), norm_token_smem_bytes(p.NA, p.R, p.Lq, p.Lkv), st, true, p);
    const size_t smem = static_cast<size_t>(p.NA + p.R) * sizeof(uint16_t);
    const size_t gsmem = static_cast<size_t>((p.Lq + p.Lkv + 7) & ~7) * sizeof(uint16_t);
    return launch_kernel(mla_norm_rope_warp_kernel, dim3((p.T + kNormWarpTokens - 1) / kNormWarpTokens),
                         dim3(32 * kNormWarpTokens), gsmem + smem * kNormWarpTokens, st, true, p);
}

cudaError_t launch_quant(const QuantParams& p_in, cudaStream_t st, bool pdl) {
    if (p_in.rows == 0) return cudaSuccess;
    QuantParams p = p_in;
    p.chunk = p.amax ? kQuantThreads * kQuantLoads * 4 : p.row_len;
    const int chunks = (p.row_len + p.chunk - 1) / p.chunk;
    return launch_kernel(mla_quant_kernel<kQuantLoads>, dim3(p.rows, chunks), dim3(kQuantThreads), 0, st, pdl, p);
}

cudaError_t launch_quant_x(const QuantXParams& p, cudaStream_t st) {
    if (p.rows == 0) return cudaSuccess;
    return launch_kernel(mla_quant_x_kernel, dim3(p.rows), dim3(kQuantXThreads), 0, st, false, p);
}

cudaError_t launch_widen_i8(const int8_t* src, uint16_t* dst, size_t n, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const size_t threads = (n + 15) / 16;
    const size_t blocks = std::min<size_t>((threads + 255) / 256, 152 * 8);
    return launch_kernel(mla_widen_i8_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, false, src, dst,
                         n);
}

}  // namespace mlap
