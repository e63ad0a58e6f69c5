// mla_prolog_run_noalloc: the whole prolog pass without a handle and
// without any device allocation, for callers that must not call cudaMalloc
// themselves or through this library -- for example a plugin inside an
// inference runtime that reserves the device memory pool up front (a
// cudaMalloc there fails or fragments the pool), or a latency-critical path
// where cudaMalloc's implicit device synchronisation is not acceptable.
//
// The scratch that mla_prolog_run() keeps in its handle's workspace (split-K
// partials, normed rows, FP32 q rows, per-token amax, status word) lives here
// in one file-scope __device__ array of kNoallocScratchBytes.  Every GPU that
// loads the library holds its own copy of that array until the process
// exits.  All calls on one device share it and it keeps the last call's
// contents, so two calls whose kernels overlap on the same GPU (for example
// on two streams) race on it.
//
// The math and the schedule rules are those of mla_prolog_run() (the same
// tile widths and split-K factors; jobs in round-robin order instead of the
// handle's balanced job tables, which does not change any job's result),
// but this entry launches only a subset of its kernels: the one-CTA split-K
// or wide compression, the norm kernel, the one-CTA expansion and the quant
// kernel.
// A handle may pick other kernels for the same dims (the cluster compression
// + norm for tiny batches, CTA pairs for prefills with a q path), so results
// agree with mla_prolog_run() within the parity tolerances; where both paths
// launch the same kernels (the V2-Lite and V3 decode shapes, the V2-Lite
// prefill shape) they agree bit for bit.
#include <cmath>
#include <cstdio>
#include <mutex>

#include "../../include/mla_prolog.h"
#include "prolog.cuh"

namespace mlap {
namespace {

constexpr size_t kNoallocScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};   // device address of g_noalloc_scratch, per device
int g_sms[kMaxDevices] = {};

// A failed CUDA call; `what` names it for a reader of this file (the entry
// point reports MLA_ERR_CUDA without recording the text).
int set_error(const char* what) {
    (void)what;
    return MLA_ERR_CUDA;
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool encode(EncodeFn fn, CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t stride_elems,
            uint32_t box_rows) {
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {stride_elems * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
int cdiv(int a, int b) { return (a + b - 1) / b; }
size_t al256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

// Once per device, with that device current: the device address of the
// static scratch, the kernel attributes and the SM count.
int setup_device(int dev, void** scratch, int* sms) {
    if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return set_error("cudaGetDeviceProperties");
        if (prop.major != 10 || prop.minor != 3) return MLA_ERR_DEVICE;
        if (gemm_set_attributes() != cudaSuccess) return set_error("cudaFuncSetAttribute");
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return set_error("cudaGetSymbolAddress");
        g_sms[dev] = prop.multiProcessorCount;
        g_scratch_ptr[dev] = p;
    }
    *scratch = g_scratch_ptr[dev];
    *sms = g_sms[dev];
    return MLA_OK;
}

}  // namespace
}  // namespace mlap

using namespace mlap;

extern "C" int mla_prolog_run_noalloc(const mla_prolog_dims* dims, const void* x, const void* gamma,
                                      const void* W_a, const void* W_b, const int32_t* positions,
                                      const float* cos_sin, void* out_k, void* out_v, void* out_kpe,
                                      int8_t* out_q_int8, float* out_scale, int32_t* status, void* stream) {
    if (!dims) return MLA_ERR_INVALID_ARG;
    const mla_prolog_dims d = *dims;
    // size rules of mla_prolog_dims
    auto m16 = [](int v) { return v > 0 && v % 16 == 0; };
    if (!m16(d.D) || !m16(d.kv_lora_rank) || !m16(d.rope_dim) || !m16(d.nope_dim) || !m16(d.v_dim) ||
        d.q_lora_rank < 0 || d.q_lora_rank % 16 || d.rope_dim > 128 || d.T < 0 || d.num_heads < 1 ||
        d.max_pos < 1 || !std::isfinite(d.eps) || d.eps < 0.0f)
        return MLA_ERR_UNSUPPORTED_DIMS;
    if ((d.flags & ~MLA_PROLOG_QUANT_Q) != 0 || ((d.flags & MLA_PROLOG_QUANT_Q) != 0) != (d.q_lora_rank > 0))
        return MLA_ERR_INVALID_ARG;
    if (d.q_lora_rank > 0 && d.nope_dim + d.rope_dim > 256) return MLA_ERR_UNSUPPORTED_DIMS;
    const int Lq = d.q_lora_rank, Lkv = d.kv_lora_rank, R = d.rope_dim, H = d.num_heads;
    const int NA = Lq + Lkv + R, NQ = H * (d.nope_dim + R), NKV = H * (d.nope_dim + d.v_dim);
    const int m_tiles = cdiv(d.T, kBM);

    // The schedule mla_prolog_create() picks for these dims.
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return set_error("cudaGetDevice");
    void* scratch = nullptr;
    int sms = 0;
    int rc = setup_device(dev, &scratch, &sms);
    if (rc != MLA_OK) return rc;
    const Schedule sc = plan_schedule(d.T, d.D, Lq, Lkv, R, H, d.nope_dim, d.v_dim, sms);
    const bool decode = sc.decode;
    const GemmShape shape_b = sc.shape_b;
    GemmShape shape_a = sc.shape_a;
    int bn_a = sc.bn_a, splits_a = sc.splits_a;
    const int bn_kv = sc.bn_kv, group_a = sc.group_a;
    const int kb_a = cdiv(d.D, kBK);
    if (!decode) {  // the prefill compression tile a handle selects (jobs in round-robin order here)
        CompressTilePlan plans[kNumCompressTiles];
        bn_a = plan_compress_tiles(d.T, NA, kb_a, sms, plans);
        for (const auto& ct : plans)
            if (ct.bn == bn_a) splits_a = ct.splits;
        shape_a = bn_a == 128 ? GemmShape::Wide : bn_a <= 192 ? GemmShape::Wide192 : GemmShape::Wide256;
    }

    // Scratch layout (same order as the handle's workspace) and its limit.
    const size_t T = static_cast<size_t>(d.T);
    const size_t b_part = al256(static_cast<size_t>(splits_a) * T * NA * 4);
    const size_t b_norm = al256(T * (Lq + Lkv) * 2);
    const size_t b_q = Lq > 0 ? al256(T * NQ * 4) : 0;
    const size_t b_amax = al256(T * 4);
    const size_t need = b_part + b_norm + b_q + b_amax + 256;
    if (need > kNoallocScratchBytes) return MLA_ERR_UNSUPPORTED_DIMS;  // beyond the 32 MiB static scratch
    if (d.T == 0) return MLA_OK;

    const void* p16[] = {x, gamma, W_a, W_b, cos_sin, out_k, out_v, out_kpe};
    for (const void* p : p16)
        if (!p || !aligned(p, 16)) return MLA_ERR_INVALID_ARG;
    if (!positions || !aligned(positions, 4)) return MLA_ERR_INVALID_ARG;
    if (status && !aligned(status, 4)) return MLA_ERR_INVALID_ARG;
    if (Lq > 0) {
        if (!out_q_int8 || !out_scale || !aligned(out_q_int8, 16) || !aligned(out_scale, 4))
            return MLA_ERR_INVALID_ARG;
    } else if (out_q_int8 || out_scale) {
        return MLA_ERR_INVALID_ARG;
    }

    char* w = static_cast<char*>(scratch);
    float* partials = reinterpret_cast<float*>(w);
    uint16_t* normed = reinterpret_cast<uint16_t*>(w + b_part);
    float* qws = Lq > 0 ? reinterpret_cast<float*>(w + b_part + b_norm) : nullptr;
    uint32_t* amax = reinterpret_cast<uint32_t*>(w + b_part + b_norm + b_q);
    int* dstatus = reinterpret_cast<int*>(w + b_part + b_norm + b_q + b_amax);

    // Tensor maps are encoded on the host for every call (no device memory).
    void* fnp = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fnp, 12000, cudaEnableDefault, &q) !=
            cudaSuccess || q != cudaDriverEntryPointSuccess || !fnp)
        return set_error("cuTensorMapEncodeTiled entry point");
    const EncodeFn fn = reinterpret_cast<EncodeFn>(fnp);
    CUtensorMap tm_x, tm_wa, tm_nq, tm_nkv, tm_wqb, tm_wkvb;
    const uint16_t* wb = static_cast<const uint16_t*>(W_b);
    bool ok = encode(fn, &tm_x, x, d.D, d.T, d.D, kBM) && encode(fn, &tm_wa, W_a, d.D, NA, d.D, bn_a) &&
              encode(fn, &tm_nkv, normed + Lq, Lkv, d.T, Lq + Lkv, kBM) &&
              encode(fn, &tm_wkvb, wb + static_cast<size_t>(NQ) * Lq, Lkv, NKV, Lkv, bn_kv);
    if (ok && Lq > 0)
        ok = encode(fn, &tm_nq, normed, Lq, d.T, Lq + Lkv, kBM) &&
             encode(fn, &tm_wqb, wb, Lq, NQ, Lq, d.nope_dim + R);
    if (!ok) return set_error("cuTensorMapEncodeTiled");
    if (Lq == 0) {
        tm_nq = tm_nkv;
        tm_wqb = tm_wkvb;
    }

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint64_t timeout_ns = 1000000000ull;
    // The status word must start at zero; partials, normed rows and q are
    // overwritten in full and amax is cleared by the norm kernel.
    if (cudaMemsetAsync(dstatus, 0, sizeof(int), st) != cudaSuccess) return set_error("cudaMemsetAsync");

    CompressParams pa{};
    pa.partials = partials;
    pa.T = d.T;
    pa.NA = NA;
    pa.bn = bn_a;
    pa.kb_total = kb_a;
    pa.splits = splits_a;
    pa.group = group_a;
    pa.n_tiles = cdiv(NA, bn_a);
    pa.m_tiles = m_tiles;
    pa.compensated = 1;
    pa.prefetch_l2 = decode ? 1 : 0;
    pa.positions = positions;
    pa.cos_sin = cos_sin;
    pa.R = R;
    pa.max_pos = d.max_pos;
    pa.gamma = static_cast<const uint16_t*>(gamma);
    pa.n_gamma = Lq + Lkv;
    pa.status = dstatus;
    pa.timeout_ns = timeout_ns;
    const int jobs_a = pa.n_tiles * m_tiles * splits_a;
    if (launch_compress(shape_a, jobs_a < sms ? jobs_a : sms, tm_x, tm_wa, pa, st) != cudaSuccess)
        return set_error("launch mla_compress_kernel");

    NormRopeParams pn{};
    pn.partials = partials;
    pn.splits = splits_a;
    pn.T = d.T;
    pn.NA = NA;
    pn.Lq = Lq;
    pn.Lkv = Lkv;
    pn.R = R;
    pn.H = H;
    pn.Dn = d.nope_dim;
    pn.inv_lq = Lq > 0 ? static_cast<float>(1.0 / Lq) : 0.0f;
    pn.inv_lkv = static_cast<float>(1.0 / Lkv);
    pn.eps = d.eps;
    pn.gamma = static_cast<const uint16_t*>(gamma);
    pn.positions = positions;
    pn.cos_sin = cos_sin;
    pn.max_pos = d.max_pos;
    pn.normed = normed;
    pn.out_k = static_cast<uint16_t*>(out_k);
    pn.out_kpe = static_cast<uint16_t*>(out_kpe);
    pn.amax = Lq > 0 ? amax : nullptr;
    pn.status = dstatus;
    if (launch_norm_rope(pn, st) != cudaSuccess) return set_error("launch mla_norm_rope_kernel");

    ExpandParams pb{};
    pb.T = d.T;
    pb.H = H;
    pb.Dn = d.nope_dim;
    pb.Dv = d.v_dim;
    pb.R = R;
    pb.NQ = NQ;
    pb.NKV = NKV;
    pb.nq_tiles = Lq > 0 ? H : 0;
    pb.nkv_tiles = cdiv(NKV, bn_kv);
    pb.bn_kv = bn_kv;
    pb.m_tiles = m_tiles;
    pb.group_n = 16;
    pb.job_table = nullptr;  // round robin: same per-job results as the balanced order
    pb.Lq = Lq;
    pb.Lkv = Lkv;
    pb.kb_q = cdiv(Lq, kBK);
    pb.kb_kv = cdiv(Lkv, kBK);
    pb.positions = positions;
    pb.cos_sin = cos_sin;
    pb.max_pos = d.max_pos;
    pb.out_k = static_cast<uint16_t*>(out_k);
    pb.out_v = static_cast<uint16_t*>(out_v);
    pb.out_aligned32 = (reinterpret_cast<uintptr_t>(out_k) % 32 == 0) && (reinterpret_cast<uintptr_t>(out_v) % 32 == 0);
    pb.qws = qws;
    pb.amax = amax;
    pb.status = dstatus;
    pb.timeout_ns = timeout_ns;
    const int jobs_b = (pb.nq_tiles + pb.nkv_tiles) * m_tiles;
    if (launch_expand(shape_b, jobs_b < sms ? jobs_b : sms, tm_nq, tm_nkv, tm_wqb, tm_wkvb, OutTensorMaps{}, pb, st) != cudaSuccess)
        return set_error("launch mla_expand_kernel");
    if (Lq > 0) {
        QuantParams pq{qws, amax, d.T, NQ, NQ, out_q_int8, out_scale};
        if (launch_quant(pq, st, true) != cudaSuccess) return set_error("launch mla_quant_kernel");
    }
    if (status && cudaMemcpyAsync(status, dstatus, sizeof(int), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return set_error("cudaMemcpyAsync(status)");
    return MLA_OK;
}
