// Host side of the C ABI declared in include/mla_prolog.h: argument checks,
// the schedule chosen at create time, the device workspace, TMA tensor maps,
// and the kernel launches of one run.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <new>
#include <utility>
#include <vector>

#include "../../include/mla_prolog.h"
#include "prolog.cuh"

using namespace mlap;

namespace {

thread_local char g_last_cuda_error[256] = "";

int cuda_fail(cudaError_t e, const char* where) {
    std::snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "%s: %s", where, cudaGetErrorString(e));
    return e == cudaErrorMemoryAllocation ? MLA_ERR_OOM : MLA_ERR_CUDA;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// K-major BF16 operand [rows, cols] with row stride `stride_elems`, loaded as
// boxes of 64 columns (one 128-byte swizzle atom) x box_rows rows.  Reads
// outside [rows, cols] are filled with zeros.
bool encode_bf16(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t stride_elems,
                 uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {stride_elems * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output tensor [rows, cols] (row pitch `row_bytes`) written by bulk tensor
// stores in boxes of box_cols x 32 rows of 64 bytes, 64-byte swizzle.
bool encode_store(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows,
                  uint64_t row_bytes, uint32_t box_cols) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_cols, 32};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
int cdiv(int a, int b) { return (a + b - 1) / b; }

constexpr int kKernelCount = 6;  // most kernels one run launches (timing-hook events: + 1)
constexpr int kPairCompressBN = 256;                // the compression pair kernel's tile width

const char* const kClusterKernelNames[3] = {"mla_compress_norm_kernel", "mla_expand_kernel", "mla_quant_kernel"};
const char* const kFusedKernelName = "mla_decode_kernel";

}  // namespace

struct mla_prolog {
    mla_prolog_dims d{};
    int device = 0;
    int NA = 0, NQ = 0, NKV = 0;
    // schedule
    bool decode = false;
    GemmShape shape_a = GemmShape::Wide, shape_b = GemmShape::Wide;
    int bn_a = 0, splits_a = 1, bn_kv = 0, m_tiles = 0;
    int group_a = 1;      // K blocks per tensor-core accumulation chain (compression)
    int compensated = 1;  // TwoSum accumulation of the drained chains
    int sms = 0;
    // workspace
    void* ws = nullptr;
    size_t ws_bytes = 0;
    float* partials = nullptr;
    uint16_t* normed = nullptr;
    float* qws = nullptr;
    uint32_t* amax = nullptr;
    int* status = nullptr;
    int* job_table = nullptr;  // balanced expansion job lists (decode)
    int* compress_table = nullptr;  // balanced compression job lists (prefill)
    // prefill compression: one plan per weight-tile width (128, 192, 256)
    struct CompressTile {
        int bn = 0;
        GemmShape shape = GemmShape::Wide;
        int splits = 1;
        int* table = nullptr;
    };
    CompressTile ctile[kNumCompressTiles];
    int expand_grid = 0;
    // KV-only prefill on one CTA per tile: the last jobs as half tiles
    // (ExpandParams::kv_halves; tunable)
    int kv_halves = 0;
    int kvres_halves = 0;  // the same for the kv-resident kernel's super-jobs
    bool kv_halves_on = false;
    // cooperative decode kernel (one launch for the whole pass)
    bool fused_ok = false;     // the dims and the device allow it
    bool fused = false;        // in use (tunable)
    size_t decode_smem = 0;
    unsigned* sync = nullptr;  // its hand-over counters (kSyncWords words)
    uint64_t timeout_ns = 1000000000ull;
    // prefill expansion on CTA pairs (cta_group::2, 256-token tiles)
    bool pair_ok = false;
    bool pair = false;
    int pair_grid = 0, pair_m_tiles = 0;
    // prefill compression on CTA pairs
    bool cpair_ok = false;
    bool cpair = false;
    int cpair_grid = 0, cpair_m_tiles = 0, cpair_splits = 1;
    int* cpair_table = nullptr;
    // compression + norm in one thread-block cluster (small decode batches)
    bool cluster_ok = false;   // the dims and the device allow it
    bool cluster = false;      // in use (tunable; on by default where allowed)
    ClusterPlan cplan;
    int cluster_ctas = 0, cluster_expand_grid = 0;
    GemmShape cluster_shape_b = GemmShape::Narrow;
    // tensor maps: workspace ones are fixed, caller ones are re-encoded when a pointer changes
    CUtensorMap tm_nq{}, tm_nkv{}, tm_x{}, tm_wa{}, tm_wa_c{}, tm_wqb{}, tm_wkvb{};
    CUtensorMap tm_wqb2{}, tm_wkvb2{}, tm_wa2{};  // half-tile weight boxes of the pair kernels
    CUtensorMap tm_wqbw{};  // W_q_b in boxes of half a wide q tile (pairs with q_wide)
    bool q_wide_ok = false;  // pairs: q tiles of kQWide columns across heads possible
    bool q_wide = false;     // in use (tunable)
    bool kvres_ok = false;   // pairs: kv tiles with the activations resident possible
    bool kvres = false;      // in use (tunable)
    int kvres_group = 8;     // kv tiles per super-job (tunable)
    int l2_policy = 0;       // MLA_TUNE_L2_POLICY bits (kL2WeightsLast, kL2ActsLast, kL2StoresFirst)
    int kvres_grid = 0;      // CTA pairs of that kernel
    // the expansion epilogue's bulk tensor stores (kernels with a staging area)
    bool l2_fetch = false;  // decode: the compression kernel fetches W_b into L2 (tunable)
    bool ts_ok = false;     // the dims allow them
    bool tma_store = false;  // in use (tunable)
    OutTensorMaps tm_out{};  // q workspace (fixed), out_k / out_v (re-encoded per pointer)
    const void* last_out_k = nullptr;
    const void* last_out_v = nullptr;
    const void* last_x = nullptr;
    const void* last_wa = nullptr;
    const void* last_wb = nullptr;
    cudaEvent_t events[kKernelCount + 1] = {};
    // The per-token quant beside the kv-resident kernel: an internal
    // low-priority stream, forked from and joined back to the caller's.
    bool quant_overlap = false;  // in use (tunable; needs the kv-resident kernel)
    cudaStream_t side = nullptr;
    cudaEvent_t fork_ev = nullptr, join_ev = nullptr;
    int n_events = 0;
    // W8A8 (MLA_PROLOG_W8A8): the weights as BF16 integers with their row
    // scales (filled by mla_prolog_load_w8a8), x's codes and scales, and the
    // normed rows' scales, in one allocation of their own.
    bool w8a8 = false;
    bool w8_loaded = false;
    void* w8mem = nullptr;
    uint16_t* wa16 = nullptr;
    uint16_t* wb16 = nullptr;
    float* wscale = nullptr;
    uint16_t* xq = nullptr;
    float* xscale = nullptr;
    float* nscale = nullptr;
    uint32_t* w8_split = nullptr;  // per 128-token tile: the expansions' chain split marks
    size_t wa_elems = 0, wb_elems = 0, n_wscale = 0;
};

namespace {

// Puts the prefill compression plan of weight-tile width `bn` in use; false
// when there is none of that width.  The W_a tensor map is re-encoded (its
// box is one tile high) on the next run.
// Whether the kv tiles run on the kv-resident pair kernel (with the pair
// expansion): its epilogue writes through tensor stores.
bool kvres_active(mla_prolog_t h) { return h->kvres && h->tma_store; }

// The kv-resident kernel's last round of super-jobs as half super-jobs when
// that round is shorter than half the pairs and every group is whole.
void plan_kvres_halves(mla_prolog_t h) {
    const int nkv_tiles = cdiv(h->NKV, h->bn_kv);
    const int n_sj = h->pair_m_tiles * cdiv(nkv_tiles, h->kvres_group);
    h->kvres_halves = h->kvres_group >= 2 && nkv_tiles % h->kvres_group == 0
                          ? plan_last_round_halves(n_sj, h->kvres_grid)
                          : 0;
}

bool select_compress_tile(mla_prolog_t h, int bn) {
    for (const auto& ct : h->ctile) {
        if (ct.bn != bn || bn == 0) continue;
        h->bn_a = ct.bn;
        h->shape_a = ct.shape;
        h->splits_a = ct.splits;
        h->compress_table = ct.table;
        h->last_wa = nullptr;
        return true;
    }
    return false;
}

int check_dims(const mla_prolog_dims& d) {
    auto m16 = [](int v) { return v > 0 && v % 16 == 0; };
    if (!m16(d.D) || !m16(d.kv_lora_rank) || !m16(d.rope_dim) || !m16(d.nope_dim) || !m16(d.v_dim))
        return MLA_ERR_UNSUPPORTED_DIMS;
    if (d.q_lora_rank < 0 || d.q_lora_rank % 16) return MLA_ERR_UNSUPPORTED_DIMS;
    if (d.rope_dim > 128 || d.T < 0 || d.num_heads < 1 || d.max_pos < 1) return MLA_ERR_UNSUPPORTED_DIMS;
    if (!std::isfinite(d.eps) || d.eps < 0.0f) return MLA_ERR_UNSUPPORTED_DIMS;
    const bool quant = (d.flags & MLA_PROLOG_QUANT_Q) != 0;
    const uint32_t known = MLA_PROLOG_QUANT_Q | MLA_PROLOG_ROPE_INTERLEAVED | MLA_PROLOG_Q_HEAD_NORM |
                           MLA_PROLOG_QUANT_PER_HEAD | MLA_PROLOG_W8A8;
    if ((d.flags & ~known) != 0) return MLA_ERR_INVALID_ARG;
    if (quant != (d.q_lora_rank > 0)) return MLA_ERR_INVALID_ARG;
    // the per-head norm and the per-head quant act on the q path
    if ((d.flags & (MLA_PROLOG_Q_HEAD_NORM | MLA_PROLOG_QUANT_PER_HEAD)) && d.q_lora_rank == 0)
        return MLA_ERR_INVALID_ARG;
    if (d.q_lora_rank > 0 && d.nope_dim + d.rope_dim > 256) return MLA_ERR_UNSUPPORTED_DIMS;
    // W8A8: an expansion's K runs as at most two exact accumulation chains
    if ((d.flags & MLA_PROLOG_W8A8) && (d.q_lora_rank > 2 * kW8ChainKb * kBK || d.kv_lora_rank > 2 * kW8ChainKb * kBK))
        return MLA_ERR_UNSUPPORTED_DIMS;
    // 32-bit index headroom of the kernels' row arithmetic
    const double big = static_cast<double>(d.T) * d.num_heads * (d.nope_dim + d.rope_dim + d.v_dim);
    if (big > 4.0e9 || static_cast<double>(d.T) * d.D > 4.0e9) return MLA_ERR_UNSUPPORTED_DIMS;
    return MLA_OK;
}

}  // namespace

extern "C" {

const char* mla_prolog_strerror(int code) {
    switch (code) {
        case MLA_OK: return "ok";
        case MLA_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, or bad flags)";
        case MLA_ERR_UNSUPPORTED_DIMS: return "unsupported dims (see the size rules of mla_prolog_dims)";
        case MLA_ERR_CUDA: return "CUDA error (see mla_prolog_last_cuda_error)";
        case MLA_ERR_OOM: return "device memory allocation failed";
        case MLA_ERR_DEVICE: return "current device is not an sm_103 GPU";
        default: return "unknown error code";
    }
}

const char* mla_prolog_last_cuda_error(void) { return g_last_cuda_error; }

int mla_prolog_create(const mla_prolog_dims* dims, mla_prolog_t* out) {
    if (!dims || !out) return MLA_ERR_INVALID_ARG;
    *out = nullptr;
    int rc = check_dims(*dims);
    if (rc != MLA_OK) return rc;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    cudaDeviceProp prop;
    if ((e = cudaGetDeviceProperties(&prop, dev)) != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
    if (prop.major != 10 || prop.minor != 3) return MLA_ERR_DEVICE;
    if (!encode_fn()) return cuda_fail(cudaErrorNotSupported, "cuTensorMapEncodeTiled entry point");
    if ((e = gemm_set_attributes()) != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");

    mla_prolog* h = new (std::nothrow) mla_prolog();
    if (!h) return MLA_ERR_OOM;
    h->d = *dims;
    h->device = dev;
    const mla_prolog_dims& d = h->d;
    const int Lq = d.q_lora_rank, Lkv = d.kv_lora_rank, R = d.rope_dim;
    h->NA = Lq + Lkv + R;
    h->NQ = d.num_heads * (d.nope_dim + R);
    h->NKV = d.num_heads * (d.nope_dim + d.v_dim);
    h->m_tiles = cdiv(d.T, kBM);
    const int sms = prop.multiProcessorCount;
    h->sms = sms;

    const Schedule sc = plan_schedule(d.T, d.D, Lq, Lkv, R, d.num_heads, d.nope_dim, d.v_dim, sms);
    h->decode = sc.decode;
    h->shape_a = sc.shape_a;
    h->bn_a = sc.bn_a;
    h->splits_a = sc.splits_a;
    h->group_a = sc.group_a;
    h->compensated = 1;
    h->shape_b = sc.shape_b;
    h->bn_kv = sc.bn_kv;

    // Decode expansion: jobs of unequal size (a q head streams (Dn+R)*Lq
    // weights, a kv tile bn_kv*Lkv); assign them to the CTAs longest first,
    // each to the least loaded CTA, so every SM streams about the same bytes.
    const int njobs_b = ((Lq > 0 ? d.num_heads : 0) + cdiv(h->NKV, h->bn_kv)) * h->m_tiles;
    h->expand_grid = njobs_b < sms ? njobs_b : sms;
    // A KV-only prefill whose jobs leave a last round shorter than half the
    // grid runs those jobs as half tiles (128 of 256 columns) on twice as
    // many CTAs: measured on GB300, V2-Lite prefill (512 jobs, 152 SMs).
    if (!h->decode && Lq == 0 && h->bn_kv % 128 == 0) {
        h->kv_halves = plan_last_round_halves(njobs_b, sms);
        h->kv_halves_on = h->kv_halves > 0;
    }
    // The cooperative decode kernel takes one token tile, heads of at most
    // kDecodeMaxBN columns and needs one resident CTA per SM.
    if (h->m_tiles == 1 && h->bn_kv <= kDecodeMaxBN && (Lq == 0 || d.nope_dim + R <= kDecodeMaxBN)) {
        int coop = 0, blocks = 0;
        h->decode_smem = decode_smem_bytes(h->NA, R, Lq, Lkv);
        if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && coop &&
            decode_set_attributes(h->decode_smem) == cudaSuccess &&
            decode_occupancy(h->decode_smem, &blocks) == cudaSuccess && blocks >= 1)
            h->fused_ok = true;
        cudaGetLastError();
    }
    // Off by default: a grid-wide barrier across 152 CTAs costs about 2 us on
    // GB300 (both dies' L2s take part), so the kernel's three barriers cost
    // more than the overlapped (PDL) hand-offs of the four-kernel path.
    h->fused = false;
    // Small decode batches: compression + norm in one cluster of up to 16
    // CTAs (8 where 16 cannot be co-scheduled), the expansion on the other
    // SMs with every K block of its weights in flight before the hand-off.
    if (h->m_tiles == 1) {
        for (int ctas_max : {kClusterMaxCtas, 8}) {
            const ClusterPlan cp = plan_cluster(d.T, d.D, Lq, Lkv, R, ctas_max);
            if (!cp.ok) break;
            const int ctas = cp.nc * cp.ks;
            int active = 0;
            if (cluster_set_attributes(cp.smem, ctas) == cudaSuccess &&
                cluster_max_active(cp.smem, ctas, &active) == cudaSuccess && active >= 1 && ctas < sms) {
                h->cluster_ok = true;
                h->cplan = cp;
                h->cluster_ctas = ctas;
                break;
            }
            cudaGetLastError();
        }
        cudaGetLastError();
    }
    // Prefill: the expansion on CTA pairs (half of each weight tile per SM).
    if (!h->decode && h->bn_kv == 256 && (Lq == 0 || (d.nope_dim + R <= 256 && (d.nope_dim + R) % 16 == 0))) {
        int active = 0;
        if (expand_pair_max_active(&active) == cudaSuccess && active >= 1) {
            h->pair_ok = true;
            // Measured on GB300: the V3 prefill expansion 1440 vs 1539 us on
            // pairs; the KV-only V2-Lite prefill 28.0 vs 25.6 us (slower).
            h->pair = Lq > 0;
            h->pair_m_tiles = cdiv(d.T, 2 * kBM);
            const int pjobs = ((Lq > 0 ? d.num_heads : 0) + cdiv(h->NKV, h->bn_kv)) * h->pair_m_tiles;
            h->pair_grid = pjobs < sms / 2 ? pjobs : sms / 2;
        }
        cudaGetLastError();
    }
    // Prefill: the compression on CTA pairs (half of each W_a tile per SM).
    std::vector<int> cptable;
    if (!h->decode) {
        int active = 0;
        if (!(d.flags & MLA_PROLOG_W8A8) && compress_pair_max_active(&active) == cudaSuccess && active >= 1) {
            const int kb = cdiv(d.D, kBK);
            h->cpair_ok = true;
            // Measured on GB300: slower on pairs (256-wide tiles, plain FP32
            // drain: V3 prefill step 2257 vs 2187 us, V2-Lite 47.4 vs 42.5
            // us; 128-wide with TwoSum earlier: compression 831 vs 640 us):
            // the accumulators drain every few K blocks and each drain waits
            // for both CTAs' epilogues.
            h->cpair = false;
            h->cpair_splits = prefill_compress_splits(d.T, h->NA, kb, sms, 2, kPairCompressBN);
            h->cpair_m_tiles = cdiv(d.T, 2 * kBM);
            const int cjobs = cdiv(h->NA, kPairCompressBN) * h->cpair_m_tiles * h->cpair_splits;
            h->cpair_grid = cjobs < sms / 2 ? cjobs : sms / 2;
            if (cjobs > sms / 2)
                lpt_assign(compress_job_bytes(d.T, h->NA, kb, kPairCompressBN, h->cpair_splits, 2), sms / 2,
                           &cptable, true);
        }
        cudaGetLastError();
    }
    if (h->cluster_ok) {
        h->cluster = h->cplan.est_us <= kClusterDefaultUs;
        h->cluster_expand_grid = njobs_b < sms - h->cluster_ctas ? njobs_b : sms - h->cluster_ctas;
        h->cluster_shape_b = h->shape_b == GemmShape::Narrow ? GemmShape::Deep : h->shape_b;
    }
    // W8A8 runs on the split-K / per-tile and pair kernels, whose epilogues
    // turn the exact integer accumulators into dequantised values; the
    // cooperative and cluster kernels do not take it.
    h->w8a8 = (d.flags & MLA_PROLOG_W8A8) != 0;
    if (h->w8a8) {
        h->fused_ok = h->fused = false;
        h->cluster_ok = h->cluster = false;
        if (h->group_a > kW8ChainKb) h->group_a = kW8ChainKb;
    }
    // A table is needed only when there are more jobs than SMs; the expansion
    // grid and the cooperative grid are then both one CTA per SM, so one
    // table serves either path.
    std::vector<int> table;
    if (h->decode && njobs_b > sms) {
        const int nq = Lq > 0 ? d.num_heads : 0;
        const int ntiles = nq + cdiv(h->NKV, h->bn_kv), gn = 16;
        std::vector<long long> cost;
        for (int j = 0; j < njobs_b; ++j) {
            // the job -> tile order of the kernel (groups of gn tiles, token tiles inside)
            const int g = j / (gn * h->m_tiles), r = j - g * gn * h->m_tiles;
            const int gw = ntiles - g * gn < gn ? ntiles - g * gn : gn;
            const int tile = g * gn + (r - (r / gw) * gw);
            cost.push_back(tile < nq ? 2LL * (d.nope_dim + R) * Lq : 2LL * h->bn_kv * Lkv);
        }
        lpt_assign(cost, sms, &table);
    }
    // Prefill compression, for each weight-tile width: its split-K factor and
    // its jobs (of unequal size: ragged token and weight tiles) longest
    // first, each to the least-loaded CTA.
    std::vector<int> ctable[kNumCompressTiles];
    int part_splits = h->cpair_splits > h->splits_a ? h->cpair_splits : h->splits_a;
    int ctile_default = 128;
    if (!h->decode) {
        CompressTilePlan plans[kNumCompressTiles];
        ctile_default = plan_compress_tiles(d.T, h->NA, cdiv(d.D, kBK), sms, plans, ctable);
        for (int i = 0; i < kNumCompressTiles; ++i) {
            auto& ct = h->ctile[i];
            ct.bn = plans[i].bn;
            ct.shape = ct.bn == 128 ? GemmShape::Wide : ct.bn <= 192 ? GemmShape::Wide192 : GemmShape::Wide256;
            ct.splits = plans[i].splits;
            if (ct.splits > part_splits) part_splits = ct.splits;
        }
    }

    // Workspace: partials | normed | q | amax | status | job tables, each 256-byte aligned.
    auto al = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
    const size_t T = static_cast<size_t>(d.T);
    const size_t b_part = al(static_cast<size_t>(part_splits) * T * h->NA * 4);
    const size_t b_norm = al(T * (Lq + Lkv) * 2);
    const bool per_head = (d.flags & MLA_PROLOG_QUANT_PER_HEAD) != 0;  // no FP32 q round trip
    const size_t b_q = Lq > 0 && !per_head ? al(T * h->NQ * 4) : 0;
    const size_t b_amax = al(T * 4);
    const size_t b_stat = 1024;  // status word, then the cooperative kernel's counters
    const size_t b_tab = al(table.size() * sizeof(int));
    size_t b_ctab = 0;
    for (const auto& t : ctable) b_ctab += al(t.size() * sizeof(int));
    const size_t b_cptab = al(cptable.size() * sizeof(int));
    h->ws_bytes = b_part + b_norm + b_q + b_amax + b_stat + b_tab + b_ctab + b_cptab;
    if ((e = cudaMalloc(&h->ws, h->ws_bytes)) != cudaSuccess) {
        delete h;
        return cuda_fail(e, "cudaMalloc(workspace)");
    }
    char* w = static_cast<char*>(h->ws);
    h->partials = reinterpret_cast<float*>(w);
    h->normed = reinterpret_cast<uint16_t*>(w + b_part);
    h->qws = b_q > 0 ? reinterpret_cast<float*>(w + b_part + b_norm) : nullptr;
    h->amax = reinterpret_cast<uint32_t*>(w + b_part + b_norm + b_q);
    h->status = reinterpret_cast<int*>(w + b_part + b_norm + b_q + b_amax);
    h->sync = reinterpret_cast<unsigned*>(w + b_part + b_norm + b_q + b_amax + 128);

    if ((e = cudaMemset(h->ws, 0, h->ws_bytes)) != cudaSuccess) {
        cudaFree(h->ws);
        delete h;
        return cuda_fail(e, "cudaMemset(workspace)");
    }
    if (!table.empty()) {
        h->job_table = reinterpret_cast<int*>(w + b_part + b_norm + b_q + b_amax + b_stat);
        if ((e = cudaMemcpy(h->job_table, table.data(), table.size() * sizeof(int), cudaMemcpyHostToDevice)) !=
            cudaSuccess) {
            cudaFree(h->ws);
            delete h;
            return cuda_fail(e, "cudaMemcpy(job table)");
        }
    }
    if (!cptable.empty()) {
        h->cpair_table = reinterpret_cast<int*>(w + b_part + b_norm + b_q + b_amax + b_stat + b_tab + b_ctab);
        if ((e = cudaMemcpy(h->cpair_table, cptable.data(), cptable.size() * sizeof(int),
                            cudaMemcpyHostToDevice)) != cudaSuccess) {
            cudaFree(h->ws);
            delete h;
            return cuda_fail(e, "cudaMemcpy(pair compression job table)");
        }
    }
    char* ct_base = w + b_part + b_norm + b_q + b_amax + b_stat + b_tab;
    for (int i = 0; i < kNumCompressTiles; ++i) {
        if (ctable[i].empty()) continue;
        h->ctile[i].table = reinterpret_cast<int*>(ct_base);
        ct_base += al(ctable[i].size() * sizeof(int));
        if ((e = cudaMemcpy(h->ctile[i].table, ctable[i].data(), ctable[i].size() * sizeof(int),
                            cudaMemcpyHostToDevice)) != cudaSuccess) {
            cudaFree(h->ws);
            delete h;
            return cuda_fail(e, "cudaMemcpy(compression job table)");
        }
    }
    if (!h->decode) select_compress_tile(h, ctile_default);
    const uint64_t Tm = d.T > 0 ? static_cast<uint64_t>(d.T) : 1;
    bool ok = encode_bf16(&h->tm_nkv, h->normed + Lq, Lkv, Tm, Lq + Lkv, kBM);
    if (Lq > 0) ok = ok && encode_bf16(&h->tm_nq, h->normed, Lq, Tm, Lq + Lkv, kBM);
    else h->tm_nq = h->tm_nkv;
    // Bulk tensor stores in the expansion epilogue: 32-column BF16 groups
    // that never straddle k_nope / value, and (per-token q path) a rope slice
    // of 32 or 64 columns in 16-column boxes.
    h->ts_ok = d.nope_dim % 32 == 0 && d.v_dim % 32 == 0 && h->bn_kv % 64 == 0 &&
               (Lq == 0 || per_head || (R % 32 == 0 && R <= 64));
    if (h->ts_ok && h->qws)
        ok = ok && encode_store(&h->tm_out.q, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, h->qws, h->NQ, Tm,
                                static_cast<uint64_t>(h->NQ) * 4, 16);
    h->tma_store = h->ts_ok;
    // Pairs: q tiles of kQWide columns across head boundaries (the
    // per-token q path through the store ring; 64-column pieces all nope or
    // one head's whole rope slice).
    h->q_wide_ok = h->pair_ok && h->ts_ok && Lq > 0 && !per_head && !(d.flags & MLA_PROLOG_Q_HEAD_NORM) &&
                   R == 64 && d.nope_dim % 64 == 0 && h->NQ % kQWide == 0;
    // Measured on GB300: V3 prefill step 2189 -> 2073 us (interleaved RoPE
    // 2191 -> 2066 us): 32 KB of operands per SM per 4.2 MFLOP K block
    // instead of 28 KB per 3.1 MFLOP, and a quarter fewer q jobs.
    h->q_wide = h->q_wide_ok;
    // Pairs: the kv tiles on their own kernel with the normed c_kv rows of a
    // 256-token tile resident in shared memory (K = Lkv <= 512).
    if (h->pair_ok && h->ts_ok && Lkv <= 512 && Lkv % kBK == 0 && h->bn_kv == 256) {
        int active = 0;
        if (expand_kv_pair_max_active(&active) == cudaSuccess && active >= 1) {
            h->kvres_ok = true;
            const int nkv_tiles = cdiv(h->NKV, h->bn_kv);
            h->kvres_group = plan_kv_group(h->pair_m_tiles, nkv_tiles, sms / 2);
            const int n_sj = h->pair_m_tiles * cdiv(nkv_tiles, h->kvres_group);
            h->kvres_grid = n_sj < sms / 2 ? n_sj : sms / 2;
            plan_kvres_halves(h);
            if (h->kvres_halves > 0) h->kv_halves_on = true;
            // Measured on GB300 with groups of 8: V3 prefill step 2044 -> 2009
            // us, with the per-head quant 1872 -> 1827 us.  On when every pair
            // gets at least two super-jobs (the kv-only V2-Lite prefill runs
            // one CTA per tile by default: 42.2 us, vs 41.5 us here).
            h->kvres = n_sj >= sms;
        }
        cudaGetLastError();
    }
    // Decode: W_b fetched into L2 behind the compression's last loads (off
    // by default).  First measured on GB300 at V3 decode (110 MB of W_b)
    // 49.1 -> 48.1 us and V2-Lite decode (4 MB) 16.4 -> 18.6 us; with the
    // norm kernels' early dependent launch the V3 decode measures 49.1 us
    // without it and 50.5 us with it.  Issued from the compression's start,
    // or by the norm kernel's CTAs at their start, it was slower still
    // (56.9 / 57.1 us): the fetch delays that kernel's own loads.
    h->l2_fetch = false;
    // Prefill: weight tiles loaded evict-last.  Measured on GB300 (ncu, V3
    // prefill at full size): kv-resident kernel DRAM reads 459 -> 373 MB,
    // 463 -> 443 us; q expansion 421 -> 404 MB, 747 -> 741 us; compression
    // 546 -> 531 MB.  Decode batches measured no change and keep no hint.
    h->l2_policy = h->decode ? 0 : kL2WeightsLast;
    if (!ok) {
        cudaFree(h->ws);
        delete h;
        return cuda_fail(cudaErrorInvalidValue, "cuTensorMapEncodeTiled(workspace)");
    }
    if (h->w8a8) {
        const size_t NQw = Lq > 0 ? static_cast<size_t>(h->NQ) : 0;
        h->wa_elems = static_cast<size_t>(h->NA) * d.D;
        h->wb_elems = NQw * Lq + static_cast<size_t>(h->NKV) * Lkv;
        h->n_wscale = h->NA + NQw + h->NKV;
        const size_t b_wa = al(h->wa_elems * 2), b_wb = al(h->wb_elems * 2), b_ws = al(h->n_wscale * 4);
        const size_t b_xq = al(T * d.D * 2), b_xs = al(T * 4), b_ns = al(T * 8), b_sp = al(h->m_tiles * 4 + 4);
        if ((e = cudaMalloc(&h->w8mem, b_wa + b_wb + b_ws + b_xq + b_xs + b_ns + b_sp)) != cudaSuccess) {
            cudaFree(h->ws);
            delete h;
            return cuda_fail(e, "cudaMalloc(W8A8 weights)");
        }
        char* q = static_cast<char*>(h->w8mem);
        h->wa16 = reinterpret_cast<uint16_t*>(q);
        h->wb16 = reinterpret_cast<uint16_t*>(q + b_wa);
        h->wscale = reinterpret_cast<float*>(q + b_wa + b_wb);
        h->xq = reinterpret_cast<uint16_t*>(q + b_wa + b_wb + b_ws);
        h->xscale = reinterpret_cast<float*>(q + b_wa + b_wb + b_ws + b_xq);
        h->nscale = reinterpret_cast<float*>(q + b_wa + b_wb + b_ws + b_xq + b_xs);
        h->w8_split = reinterpret_cast<uint32_t*>(q + b_wa + b_wb + b_ws + b_xq + b_xs + b_ns);
        if ((e = cudaMemset(h->w8_split, 0, b_sp)) != cudaSuccess) {
            cudaFree(h->w8mem);
            cudaFree(h->ws);
            delete h;
            return cuda_fail(e, "cudaMemset(W8A8 marks)");
        }
    }
    if (h->kvres_ok && Lq > 0 && !per_head) {
        int least = 0, greatest = 0;
        if ((e = cudaDeviceGetStreamPriorityRange(&least, &greatest)) != cudaSuccess ||
            (e = cudaStreamCreateWithPriority(&h->side, cudaStreamNonBlocking, least)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&h->fork_ev, cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&h->join_ev, cudaEventDisableTiming)) != cudaSuccess) {
            if (h->side) cudaStreamDestroy(h->side);
            if (h->fork_ev) cudaEventDestroy(h->fork_ev);
            cudaFree(h->ws);
            if (h->w8mem) cudaFree(h->w8mem);
            delete h;
            return cuda_fail(e, "side stream for the quant");
        }
        h->quant_overlap = true;
    }
    *out = h;
    return MLA_OK;
}

int mla_prolog_destroy(mla_prolog_t h) {
    if (!h) return MLA_OK;
    int dev = -1;
    cudaGetDevice(&dev);
    if (dev != h->device) cudaSetDevice(h->device);
    cudaDeviceSynchronize();
    if (h->side) cudaStreamDestroy(h->side);
    if (h->fork_ev) cudaEventDestroy(h->fork_ev);
    if (h->join_ev) cudaEventDestroy(h->join_ev);
    if (h->ws) cudaFree(h->ws);
    if (h->w8mem) cudaFree(h->w8mem);
    if (dev >= 0 && dev != h->device) cudaSetDevice(dev);
    delete h;
    return MLA_OK;
}

}  // extern "C"

namespace {

// One pass of the prolog (mla_prolog_run, and mla_prolog_run_cached when
// `cache` is not null).
int run_pass(mla_prolog_t h, const void* x, const void* gamma, const void* W_a, const void* W_b,
             const int32_t* positions, const float* cos_sin, void* out_k, void* out_v, void* out_kpe,
             int8_t* out_q_int8, float* out_scale, const int32_t* slot_mapping, void* cache, int64_t num_slots,
             void* stream) {
    if (!h) return MLA_ERR_INVALID_ARG;
    const mla_prolog_dims& d = h->d;
    const int Lq = d.q_lora_rank, Lkv = d.kv_lora_rank, R = d.rope_dim;
    const bool interleaved = (d.flags & MLA_PROLOG_ROPE_INTERLEAVED) != 0;
    const bool head_norm = (d.flags & MLA_PROLOG_Q_HEAD_NORM) != 0;
    const bool per_head = (d.flags & MLA_PROLOG_QUANT_PER_HEAD) != 0;
    if (cache && (!slot_mapping || !aligned(slot_mapping, 4) || !aligned(cache, 16) || num_slots < 0))
        return MLA_ERR_INVALID_ARG;
    if (h->w8a8) {  // the weights live in the handle (mla_prolog_load_w8a8)
        if (W_a || W_b || !h->w8_loaded) return MLA_ERR_INVALID_ARG;
        W_a = h->wa16;
        W_b = h->wb16;
    }
    if (d.T == 0) return MLA_OK;
    const void* p16[] = {x, gamma, W_a, W_b, cos_sin, out_k, out_v, out_kpe};
    for (const void* p : p16)
        if (!p || !aligned(p, 16)) return MLA_ERR_INVALID_ARG;
    if (!positions || !aligned(positions, 4)) return MLA_ERR_INVALID_ARG;
    if (Lq > 0) {
        if (!out_q_int8 || !out_scale || !aligned(out_q_int8, 16) || !aligned(out_scale, 4))
            return MLA_ERR_INVALID_ARG;
    } else if (out_q_int8 || out_scale) {
        return MLA_ERR_INVALID_ARG;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint16_t* wb = static_cast<const uint16_t*>(W_b);
    const void* x_mma = h->w8a8 ? static_cast<const void*>(h->xq) : x;  // the compression's A operand
    if (x_mma != h->last_x) {
        if (!encode_bf16(&h->tm_x, x_mma, d.D, d.T, d.D, kBM)) return cuda_fail(cudaErrorInvalidValue, "tensor map x");
        h->last_x = x_mma;
    }
    if (W_a != h->last_wa) {
        if (!encode_bf16(&h->tm_wa, W_a, d.D, h->NA, d.D, h->bn_a))
            return cuda_fail(cudaErrorInvalidValue, "tensor map W_a");
        if (h->cpair_ok && !encode_bf16(&h->tm_wa2, W_a, d.D, h->NA, d.D, kPairCompressBN / 2))
            return cuda_fail(cudaErrorInvalidValue, "tensor map W_a (pairs)");
        if (h->cluster_ok) {
            const int cgw = h->cplan.cgw;
            if (!encode_bf16(&h->tm_wa_c, W_a, d.D, h->NA, d.D, cgw <= 256 ? cgw : cgw / 2))
                return cuda_fail(cudaErrorInvalidValue, "tensor map W_a (cluster)");
        }
        h->last_wa = W_a;
    }
    if (W_b != h->last_wb) {
        const uint16_t* wkvb = wb + static_cast<size_t>(h->NQ) * Lq;
        if (!encode_bf16(&h->tm_wkvb, wkvb, Lkv, h->NKV, Lkv, h->bn_kv))
            return cuda_fail(cudaErrorInvalidValue, "tensor map W_kv_b");
        if (Lq > 0) {
            if (!encode_bf16(&h->tm_wqb, wb, Lq, h->NQ, Lq, d.nope_dim + R))
                return cuda_fail(cudaErrorInvalidValue, "tensor map W_q_b");
        } else {
            h->tm_wqb = h->tm_wkvb;
        }
        if (h->pair_ok || h->kv_halves > 0) {  // boxes of bn_kv / 2 rows: pairs, half tiles
            if (!encode_bf16(&h->tm_wkvb2, wkvb, Lkv, h->NKV, Lkv, h->bn_kv / 2))
                return cuda_fail(cudaErrorInvalidValue, "tensor map W_kv_b (pairs)");
        }
        if (h->pair_ok) {
            if (Lq > 0) {
                if (h->q_wide_ok && !encode_bf16(&h->tm_wqbw, wb, Lq, h->NQ, Lq, kQWide / 2))
                    return cuda_fail(cudaErrorInvalidValue, "tensor map W_q_b (wide pairs)");
                if (!encode_bf16(&h->tm_wqb2, wb, Lq, h->NQ, Lq, (d.nope_dim + R) / 2))
                    return cuda_fail(cudaErrorInvalidValue, "tensor map W_q_b (pairs)");
            } else {
                h->tm_wqb2 = h->tm_wkvb2;
            }
        }
        h->last_wb = W_b;
    }
    if (h->ts_ok && (out_k != h->last_out_k || out_v != h->last_out_v)) {
        const uint64_t HK = static_cast<uint64_t>(d.num_heads) * (d.nope_dim + R);
        const uint64_t HV = static_cast<uint64_t>(d.num_heads) * d.v_dim;
        if (!encode_store(&h->tm_out.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, out_k, HK, d.T, HK * 2, 32) ||
            !encode_store(&h->tm_out.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, out_v, HV, d.T, HV * 2, 32))
            return cuda_fail(cudaErrorInvalidValue, "tensor map out_k / out_v");
        h->last_out_k = out_k;
        h->last_out_v = out_v;
    }
    const bool timed = h->n_events > 0;
    cudaError_t e;
    // Inside a stream capture the records must be external event nodes to time graph replays.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (timed && cudaStreamIsCapturing(st, &cap) != cudaSuccess) return cuda_fail(cudaGetLastError(), "cudaStreamIsCapturing");
    const unsigned rec_flags = cap == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
    auto mark = [&](int i) -> cudaError_t {
        return timed ? cudaEventRecordWithFlags(h->events[i], st, rec_flags) : cudaSuccess;
    };

    CompressParams pa{};
    pa.partials = h->partials;
    pa.T = d.T;
    pa.NA = h->NA;
    pa.bn = h->bn_a;
    pa.kb_total = cdiv(d.D, kBK);
    pa.splits = h->splits_a;
    pa.group = h->group_a;
    pa.n_tiles = cdiv(h->NA, h->bn_a);
    pa.m_tiles = h->m_tiles;
    pa.compensated = h->compensated;
    pa.prefetch_l2 = h->decode ? 1 : 0;
    pa.positions = positions;
    pa.cos_sin = cos_sin;
    pa.R = R;
    pa.max_pos = d.max_pos;
    pa.gamma = static_cast<const uint16_t*>(gamma);
    pa.n_gamma = Lq + Lkv;
    pa.status = h->status;
    pa.timeout_ns = h->timeout_ns;
    pa.job_table = h->compress_table;
    pa.w8a8 = h->w8a8 ? 1 : 0;
    pa.x_scale = h->xscale;
    pa.w_scale = h->wscale;
    pa.l2_policy = h->l2_policy;
    if (h->decode && h->l2_fetch) {
        pa.l2_fetch = static_cast<const uint8_t*>(W_b);
        pa.l2_fetch_bytes = (static_cast<uint64_t>(h->NQ) * Lq + static_cast<uint64_t>(h->NKV) * Lkv) * 2;
    }

    NormRopeParams pn{};
    pn.partials = h->partials;
    pn.splits = h->splits_a;
    pn.T = d.T;
    pn.NA = h->NA;
    pn.Lq = Lq;
    pn.Lkv = Lkv;
    pn.R = R;
    pn.H = d.num_heads;
    pn.Dn = d.nope_dim;
    pn.inv_lq = Lq > 0 ? static_cast<float>(1.0 / Lq) : 0.0f;
    pn.inv_lkv = static_cast<float>(1.0 / Lkv);
    pn.eps = d.eps;
    pn.gamma = static_cast<const uint16_t*>(gamma);
    pn.positions = positions;
    pn.cos_sin = cos_sin;
    pn.max_pos = d.max_pos;
    pn.normed = h->normed;
    pn.out_k = static_cast<uint16_t*>(out_k);
    pn.out_kpe = static_cast<uint16_t*>(out_kpe);
    pn.amax = Lq > 0 && !per_head ? h->amax : nullptr;
    pn.status = h->status;
    pn.interleaved = interleaved;
    pn.cache = static_cast<uint16_t*>(cache);
    pn.slots = slot_mapping;
    pn.num_slots = num_slots;
    pn.w8a8 = h->w8a8 ? 1 : 0;
    pn.x_scale = h->xscale;
    pn.w_scale = h->wscale;
    pn.nscale = h->nscale;
    pn.w8_split = h->w8_split;

    ExpandParams pb{};
    pb.T = d.T;
    pb.H = d.num_heads;
    pb.Dn = d.nope_dim;
    pb.Dv = d.v_dim;
    pb.R = R;
    pb.NQ = h->NQ;
    pb.NKV = h->NKV;
    pb.nq_tiles = Lq > 0 ? d.num_heads : 0;
    pb.nkv_tiles = cdiv(h->NKV, h->bn_kv);
    pb.bn_kv = h->bn_kv;
    pb.m_tiles = h->m_tiles;
    pb.group_n = 16;
    pb.job_table = h->job_table;
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
    pb.qws = h->qws;
    pb.amax = h->amax;
    pb.status = h->status;
    pb.timeout_ns = h->timeout_ns;
    pb.interleaved = interleaved;
    pb.head_norm = head_norm;
    pb.inv_hd = 1.0f / static_cast<float>(d.nope_dim + R);
    pb.eps = d.eps;
    pb.per_head = per_head;
    pb.q_codes = out_q_int8;
    pb.q_scale = out_scale;
    pb.tma_store = h->tma_store ? 1 : 0;
    pb.w8a8 = h->w8a8 ? 1 : 0;
    pb.a_scale = h->nscale;
    pb.w_scale_q = h->wscale ? h->wscale + h->NA : nullptr;
    pb.w_scale_kv = h->wscale ? h->wscale + h->NA + (Lq > 0 ? h->NQ : 0) : nullptr;
    pb.w8_split = h->w8_split;
    pb.n_tiles128 = h->m_tiles;
    pb.l2_policy = h->l2_policy;

    // the per-token quant kernel (the per-head quant runs in the q epilogue)
    QuantParams pq{h->qws, h->amax, Lq > 0 && !per_head ? d.T : 0, h->NQ, h->NQ, out_q_int8, out_scale};

    if ((e = mark(0)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(timing hook)");
    if (h->fused) {
        DecodeParams pd{};
        pd.a = pa;
        pd.n = pn;
        pd.b = pb;
        pd.q = pq;
        pd.q.chunk = 8192;  // one batch of eight loads per epilogue thread
        pd.sync = h->sync;
        pd.status = h->status;
        pd.timeout_ns = h->timeout_ns;
        if ((e = launch_decode(h->sms, h->decode_smem, h->tm_x, h->tm_wa, h->tm_nq, h->tm_nkv, h->tm_wqb,
                               h->tm_wkvb, pd, st)) != cudaSuccess)
            return cuda_fail(e, "launch mla_decode_kernel");
        if ((e = mark(1)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(timing hook)");
        return MLA_OK;
    }
    if (h->cluster) {
        ClusterNormParams pc{};
        const ClusterPlan& cp = h->cplan;
        pc.T = d.T;
        pc.NA = h->NA;
        pc.kb_total = cdiv(d.D, kBK);
        pc.nc = cp.nc;
        pc.ks = cp.ks;
        pc.cgw = cp.cgw;
        pc.tpo = cp.tpo;
        pc.stages = cp.stages;
        pc.b_boxes = cp.cgw <= 256 ? 1 : 2;
        pc.tmem_cols = cp.cgw <= 32 ? 32 : cp.cgw <= 64 ? 64 : cp.cgw <= 128 ? 128 : cp.cgw <= 256 ? 256 : 512;
        pc.area_bytes = cp.area;
        pc.recv_bytes = cp.recv;
        pc.stg_off = cp.stg_off;
        pc.const_off = cp.const_off;
        pc.n = pn;
        pc.status = h->status;
        pc.timeout_ns = h->timeout_ns;
        pb.job_table = nullptr;  // one job per CTA, or round robin
        if ((e = launch_compress_norm_cluster(h->cluster_ctas, cp.smem, h->tm_x, h->tm_wa_c, pc, st)) != cudaSuccess)
            return cuda_fail(e, "launch mla_compress_norm_kernel");
        if ((e = mark(1)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(timing hook)");
        if ((e = launch_expand(h->cluster_shape_b, h->cluster_expand_grid, h->tm_nq, h->tm_nkv, h->tm_wqb,
                               h->tm_wkvb, h->tm_out, pb, st)) != cudaSuccess)
            return cuda_fail(e, "launch mla_expand_kernel");
        if ((e = mark(2)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(timing hook)");
        if (pq.rows > 0) {
            if ((e = launch_quant(pq, st, true)) != cudaSuccess) return cuda_fail(e, "launch mla_quant_kernel");
            if ((e = mark(3)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(timing hook)");
        }
        return MLA_OK;
    }
    int ev = 1;  // next timing-hook event
    if (h->w8a8) {  // AT-05 on x: the compression's INT8 input
        QuantXParams px{static_cast<const uint16_t*>(x), d.T, d.D, h->xq, h->xscale, h->w8_split, h->m_tiles};
        if ((e = launch_quant_x(px, st)) != cudaSuccess) return cuda_fail(e, "launch mla_quant_x_kernel");
        if ((e = mark(ev++)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(timing hook)");
    }
    const int jobs_a = pa.n_tiles * pa.m_tiles * pa.splits;
    // one split: the compression writes the BF16 row and the norm reads it
    if (h->cpair) {
        CompressParams pp = pa;
        pp.bn = kPairCompressBN;
        pp.n_tiles = cdiv(h->NA, kPairCompressBN);
        pp.m_tiles = h->cpair_m_tiles;
        pp.splits = h->cpair_splits;
        pp.job_table = h->cpair_table;
        pp.out_bf16 = pp.splits == 1;
        pn.splits = h->cpair_splits;
        pn.in_bf16 = pp.out_bf16;
        if ((e = launch_compress_pair(h->cpair_grid, h->tm_x, h->tm_wa2, pp, st)) != cudaSuccess)
            return cuda_fail(e, "launch mla_compress_pair_kernel");
    } else {
        pa.out_bf16 = pa.splits == 1;
        pn.in_bf16 = pa.out_bf16;
        if ((e = launch_compress(h->shape_a, jobs_a < h->sms ? jobs_a : h->sms, h->tm_x, h->tm_wa, pa, st)) !=
            cudaSuccess)
            return cuda_fail(e, "launch mla_compress_kernel");
    }
    if ((e = mark(ev++)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(timing hook)");
    if ((e = launch_norm_rope(pn, st)) != cudaSuccess) return cuda_fail(e, "launch mla_norm_rope_kernel");
    if ((e = mark(ev++)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(timing hook)");
    if (h->pair) {
        ExpandParams pp = pb;
        pp.m_tiles = h->pair_m_tiles;
        pp.job_table = nullptr;
        const bool kvres = kvres_active(h);
        if (kvres) pp.nkv_tiles = 0;  // the kv tiles go to the kv-resident kernel
        const bool wide = h->q_wide && h->tma_store;
        if (wide) {
            pp.q_wide = 1;
            pp.nq_tiles = h->NQ / kQWide;
        }
        const int jobs = (pp.nq_tiles + pp.nkv_tiles) * pp.m_tiles;
        const int grid = jobs < h->sms / 2 ? jobs : h->sms / 2;
        if (jobs > 0) {
            if ((e = launch_expand_pair(grid, h->tm_nq, h->tm_nkv, wide ? h->tm_wqbw : h->tm_wqb2, h->tm_wkvb2,
                                        h->tm_out, pp, st)) != cudaSuccess)
                return cuda_fail(e, "launch mla_expand_pair_kernel");
            if ((e = mark(ev++)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(timing hook)");
        }
        // With the kv tiles on their own kernel the quant needs only the q
        // tiles: it runs on the side stream beside the kv kernel (not with
        // the timing hook, whose events time the kernels one after another).
        const bool overlap = kvres && pq.rows > 0 && h->quant_overlap && h->side && !timed && jobs > 0;
        if (overlap) {
            if ((e = cudaEventRecord(h->fork_ev, st)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(fork)");
            if ((e = cudaStreamWaitEvent(h->side, h->fork_ev, 0)) != cudaSuccess)
                return cuda_fail(e, "cudaStreamWaitEvent(fork)");
        }
        if (kvres) {
            ExpandParams pk = pb;
            pk.m_tiles = h->pair_m_tiles;
            pk.nq_tiles = 0;
            pk.job_table = nullptr;
            pk.kvres_halves = h->kv_halves_on ? h->kvres_halves : 0;
            if ((e = launch_expand_kv_pair(h->kvres_grid, h->tm_nkv, h->tm_wkvb2, h->tm_out, pk, h->kvres_group, st)) !=
                cudaSuccess)
                return cuda_fail(e, "launch mla_expand_kv_pair_kernel");
            if ((e = mark(ev++)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(timing hook)");
        }
        if (overlap) {
            if ((e = launch_quant(pq, h->side, false)) != cudaSuccess) return cuda_fail(e, "launch mla_quant_kernel");
            if ((e = cudaEventRecord(h->join_ev, h->side)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(join)");
            if ((e = cudaStreamWaitEvent(st, h->join_ev, 0)) != cudaSuccess)
                return cuda_fail(e, "cudaStreamWaitEvent(join)");
            return MLA_OK;
        }
    } else {
        pb.kv_halves = h->kv_halves_on ? h->kv_halves : 0;
        if ((e = launch_expand(h->shape_b, h->expand_grid, h->tm_nq, h->tm_nkv, h->tm_wqb, h->tm_wkvb, h->tm_out, pb,
                               st, &h->tm_wkvb2)) != cudaSuccess)
            return cuda_fail(e, "launch mla_expand_kernel");
        if ((e = mark(ev++)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(timing hook)");
    }
    if (pq.rows > 0) {
        if ((e = launch_quant(pq, st, true)) != cudaSuccess) return cuda_fail(e, "launch mla_quant_kernel");
        if ((e = mark(ev++)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord(timing hook)");
    }
    return MLA_OK;
}

}  // namespace

extern "C" {

int mla_prolog_run(mla_prolog_t h, const void* x, const void* gamma, const void* W_a, const void* W_b,
                   const int32_t* positions, const float* cos_sin, void* out_k, void* out_v, void* out_kpe,
                   int8_t* out_q_int8, float* out_scale, void* stream) {
    return run_pass(h, x, gamma, W_a, W_b, positions, cos_sin, out_k, out_v, out_kpe, out_q_int8, out_scale,
                    nullptr, nullptr, 0, stream);
}

int mla_prolog_run_cached(mla_prolog_t h, const void* x, const void* gamma, const void* W_a, const void* W_b,
                          const int32_t* positions, const float* cos_sin, void* out_k, void* out_v, void* out_kpe,
                          int8_t* out_q_int8, float* out_scale, const int32_t* slot_mapping, void* kv_cache,
                          int64_t num_slots, void* stream) {
    if (!kv_cache) return MLA_ERR_INVALID_ARG;
    return run_pass(h, x, gamma, W_a, W_b, positions, cos_sin, out_k, out_v, out_kpe, out_q_int8, out_scale,
                    slot_mapping, kv_cache, num_slots, stream);
}

int mla_prolog_device_status(mla_prolog_t h, void* stream, int32_t* status) {
    if (!h || !status) return MLA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    int v = 0;
    if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    if ((e = cudaMemcpy(&v, h->status, sizeof v, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e, "cudaMemcpy(status)");
    if ((e = cudaMemset(h->status, 0, sizeof v)) != cudaSuccess) return cuda_fail(e, "cudaMemset(status)");
    // After a wait that gave up, start the cooperative kernel's counters over.
    if ((v & MLA_STATUS_WAIT_TIMEOUT) && (e = cudaMemset(h->sync, 0, kSyncWords * sizeof(unsigned))) != cudaSuccess)
        return cuda_fail(e, "cudaMemset(sync)");
    *status = v;
    return MLA_OK;
}

int mla_prolog_quant_rows(const float* y, int32_t rows, int32_t row_len, int8_t* codes, float* scale,
                          void* stream) {
    if (rows < 0 || row_len <= 0 || row_len % 4) return MLA_ERR_INVALID_ARG;
    if (rows == 0) return MLA_OK;
    if (!y || !codes || !scale || !aligned(y, 16) || !aligned(codes, 4) || !aligned(scale, 4))
        return MLA_ERR_INVALID_ARG;
    QuantParams p{y, nullptr, rows, row_len, row_len, codes, scale};
    cudaError_t e = launch_quant(p, static_cast<cudaStream_t>(stream), false);
    return e == cudaSuccess ? MLA_OK : cuda_fail(e, "launch mla_quant_kernel");
}

int mla_prolog_load_w8a8(mla_prolog_t h, const int8_t* W_a, const int8_t* W_b, const float* w_scale, void* stream) {
    if (!h || !h->w8a8 || !W_a || !W_b || !w_scale) return MLA_ERR_INVALID_ARG;
    if (!aligned(W_a, 16) || !aligned(W_b, 16) || !aligned(w_scale, 4)) return MLA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if ((e = launch_widen_i8(W_a, h->wa16, h->wa_elems, st)) != cudaSuccess) return cuda_fail(e, "widen W_a");
    if ((e = launch_widen_i8(W_b, h->wb16, h->wb_elems, st)) != cudaSuccess) return cuda_fail(e, "widen W_b");
    if ((e = cudaMemcpyAsync(h->wscale, w_scale, h->n_wscale * 4, cudaMemcpyDefault, st)) != cudaSuccess)
        return cuda_fail(e, "cudaMemcpyAsync(w_scale)");
    h->w8_loaded = true;
    return MLA_OK;
}

int mla_prolog_set_wait_timeout(mla_prolog_t h, uint64_t timeout_ns) {
    if (!h || timeout_ns == 0) return MLA_ERR_INVALID_ARG;
    h->timeout_ns = timeout_ns;
    return MLA_OK;
}

int mla_prolog_selftest_wait_timeout(mla_prolog_t h, uint64_t timeout_ns, void* stream) {
    if (!h || timeout_ns == 0 || timeout_ns > 10000000000ull) return MLA_ERR_INVALID_ARG;
    cudaError_t e = launch_wait_selftest(h->status, timeout_ns, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : cuda_fail(e, "launch mla_wait_selftest_kernel");
}

int mla_prolog_set_timing_events(mla_prolog_t h, void* const* events, int32_t n_events) {
    if (!h || n_events < 0) return MLA_ERR_INVALID_ARG;
    if (n_events == 0) {
        h->n_events = 0;
        return MLA_OK;
    }
    const int need = mla_prolog_kernel_count(h) + 1;
    if (!events || n_events < need) return MLA_ERR_INVALID_ARG;
    for (int i = 0; i < need; ++i) {
        if (!events[i]) return MLA_ERR_INVALID_ARG;
        h->events[i] = static_cast<cudaEvent_t>(events[i]);
    }
    h->n_events = need;
    return MLA_OK;
}

namespace {
// Whether a run launches the per-token quant kernel (no q path and the
// per-head quant, which runs in the q epilogue, do without it).
bool quant_kernel_runs(mla_prolog_t h) {
    const bool per_head = (h->d.flags & MLA_PROLOG_QUANT_PER_HEAD) != 0;
    return h->d.q_lora_rank > 0 && !per_head;
}

// The kernels of the standard path (compression, norm, expansion, quant),
// in launch order, with the current tuning; returns how many.
int standard_kernels(mla_prolog_t h, const char* (&names)[kKernelCount]) {
    int n = 0;
    if (h->w8a8) names[n++] = "mla_quant_x_kernel";
    names[n++] = h->cpair ? "mla_compress_pair_kernel" : "mla_compress_kernel";
    names[n++] = "mla_norm_rope_kernel";
    if (h->pair && kvres_active(h)) {
        if (h->d.q_lora_rank > 0) names[n++] = "mla_expand_pair_kernel";
        names[n++] = "mla_expand_kv_pair_kernel";
    } else {
        names[n++] = h->pair ? "mla_expand_pair_kernel" : "mla_expand_kernel";
    }
    if (quant_kernel_runs(h)) names[n++] = "mla_quant_kernel";
    return n;
}
}  // namespace

int32_t mla_prolog_kernel_count(mla_prolog_t h) {
    if (!h) return 0;
    if (h->fused) return 1;
    if (h->cluster) return 2 + (quant_kernel_runs(h) ? 1 : 0);
    const char* names[kKernelCount];
    return standard_kernels(h, names);
}

const char* mla_prolog_kernel_name(mla_prolog_t h, int32_t i) {
    if (!h || i < 0 || i >= mla_prolog_kernel_count(h)) return "";
    if (h->fused) return kFusedKernelName;
    if (h->cluster) return kClusterKernelNames[i];
    const char* names[kKernelCount];
    standard_kernels(h, names);
    return names[i];
}

int mla_prolog_copy_tap(mla_prolog_t h, int32_t which, void* dst, size_t bytes, void* stream) {
    if (!h || !dst) return MLA_ERR_INVALID_ARG;
    const mla_prolog_dims& d = h->d;
    const size_t T = static_cast<size_t>(d.T);
    const void* src = nullptr;
    size_t n = 0;
    switch (which) {
        case MLA_TAP_NORMED:
            src = h->normed;
            n = T * (d.q_lora_rank + d.kv_lora_rank) * 2;
            break;
        case MLA_TAP_Q:  // absent with the per-head quant (q never leaves the epilogue)
            src = h->qws;
            n = T * h->NQ * 4;
            break;
        case MLA_TAP_AMAX:
            src = h->qws ? h->amax : nullptr;
            n = T * 4;
            break;
        case MLA_TAP_X_CODES:
            src = h->xq;
            n = T * d.D * 2;
            break;
        case MLA_TAP_X_SCALE:
            src = h->xscale;
            n = T * 4;
            break;
        case MLA_TAP_NORM_SCALE:
            src = h->nscale;
            n = T * 8;
            break;
        default: return MLA_ERR_INVALID_ARG;
    }
    if (!src || bytes != n) return MLA_ERR_INVALID_ARG;
    if (n == 0) return MLA_OK;
    cudaError_t e = cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : cuda_fail(e, "cudaMemcpyAsync(tap)");
}

int mla_prolog_set_tuning(mla_prolog_t h, int32_t key, int32_t value) {
    if (!h) return MLA_ERR_INVALID_ARG;
    switch (key) {
        case MLA_TUNE_COMPRESS_GROUP:
            if (value < 1 || value > (h->w8a8 ? kW8ChainKb : 64)) return MLA_ERR_INVALID_ARG;
            h->group_a = value;
            return MLA_OK;
        case MLA_TUNE_COMPRESS_COMPENSATED:
            if (value != 0 && value != 1) return MLA_ERR_INVALID_ARG;
            h->compensated = value;
            return MLA_OK;
        case MLA_TUNE_DECODE_FUSED:
            if (value != 0 && value != 1) return MLA_ERR_INVALID_ARG;
            if (value == 1 && !h->fused_ok) return MLA_ERR_INVALID_ARG;
            h->fused = value == 1;
            if (h->fused) h->cluster = false;
            h->n_events = 0;  // the kernel count changed: re-arm the timing hook
            return MLA_OK;
        case MLA_TUNE_PAIR_COMPRESS:
            if (value != 0 && value != 1) return MLA_ERR_INVALID_ARG;
            if (value == 1 && !h->cpair_ok) return MLA_ERR_INVALID_ARG;
            h->cpair = value == 1;
            return MLA_OK;
        case MLA_TUNE_PAIR_EXPAND:
            if (value != 0 && value != 1) return MLA_ERR_INVALID_ARG;
            if (value == 1 && !h->pair_ok) return MLA_ERR_INVALID_ARG;
            h->pair = value == 1;
            h->n_events = 0;
            return MLA_OK;
        case MLA_TUNE_COMPRESS_TILE:
            if (h->decode || h->cluster || h->fused) return MLA_ERR_INVALID_ARG;
            return select_compress_tile(h, value) ? MLA_OK : MLA_ERR_INVALID_ARG;
        case MLA_TUNE_L2_FETCH:
            if (value != 0 && value != 1) return MLA_ERR_INVALID_ARG;
            if (value == 1 && !h->decode) return MLA_ERR_INVALID_ARG;
            h->l2_fetch = value == 1;
            return MLA_OK;
        case MLA_TUNE_Q_WIDE:
            if (value != 0 && value != 1) return MLA_ERR_INVALID_ARG;
            if (value == 1 && !h->q_wide_ok) return MLA_ERR_INVALID_ARG;
            h->q_wide = value == 1;
            return MLA_OK;
        case MLA_TUNE_KV_GROUP: {
            if (value < 1 || !h->kvres_ok) return MLA_ERR_INVALID_ARG;
            const int nkv_tiles = cdiv(h->NKV, h->bn_kv);
            if (value > nkv_tiles) return MLA_ERR_INVALID_ARG;
            h->kvres_group = value;
            const int n_sj = h->pair_m_tiles * cdiv(nkv_tiles, value);
            h->kvres_grid = n_sj < h->sms / 2 ? n_sj : h->sms / 2;
            plan_kvres_halves(h);
            return MLA_OK;
        }
        case MLA_TUNE_QUANT_OVERLAP:
            if (value != 0 && value != 1) return MLA_ERR_INVALID_ARG;
            if (value == 1 && !h->side) return MLA_ERR_INVALID_ARG;
            h->quant_overlap = value == 1;
            return MLA_OK;
        case MLA_TUNE_KV_RESIDENT:
            if (value != 0 && value != 1) return MLA_ERR_INVALID_ARG;
            if (value == 1 && !h->kvres_ok) return MLA_ERR_INVALID_ARG;
            h->kvres = value == 1;
            h->n_events = 0;  // the kernel count may change: re-arm the timing hook
            return MLA_OK;
        case MLA_TUNE_TMA_STORE:
            if (value != 0 && value != 1) return MLA_ERR_INVALID_ARG;
            if (value == 1 && !h->ts_ok) return MLA_ERR_INVALID_ARG;
            h->tma_store = value == 1;
            h->n_events = 0;  // the kernel count may change: re-arm the timing hook
            return MLA_OK;
        case MLA_TUNE_L2_POLICY:
            if (value < 0 || value > 7) return MLA_ERR_INVALID_ARG;
            h->l2_policy = value;
            return MLA_OK;
        case MLA_TUNE_KV_HALVES:
            if (value != 0 && value != 1) return MLA_ERR_INVALID_ARG;
            if (value == 1 && h->kv_halves == 0 && h->kvres_halves == 0) return MLA_ERR_INVALID_ARG;
            h->kv_halves_on = value == 1;
            return MLA_OK;
        case MLA_TUNE_CLUSTER_NORM:
            if (value != 0 && value != 1) return MLA_ERR_INVALID_ARG;
            if (value == 1 && !h->cluster_ok) return MLA_ERR_INVALID_ARG;
            h->cluster = value == 1;
            if (h->cluster) h->fused = false;
            h->n_events = 0;
            return MLA_OK;
        default: return MLA_ERR_INVALID_ARG;
    }
}

int mla_prolog_workspace_bytes(mla_prolog_t h, size_t* bytes) {
    if (!h || !bytes) return MLA_ERR_INVALID_ARG;
    *bytes = h->ws_bytes;
    return MLA_OK;
}

int mla_prolog_schedule(mla_prolog_t h, int32_t* bn_a, int32_t* splits_a, int32_t* bn_kv, int32_t* bn_q) {
    if (!h) return MLA_ERR_INVALID_ARG;
    if (bn_a) *bn_a = h->cluster ? h->cplan.cgw : h->bn_a;
    if (splits_a) *splits_a = h->cluster ? h->cplan.ks : h->splits_a;
    if (bn_kv) *bn_kv = h->bn_kv;
    if (bn_q)
        *bn_q = h->d.q_lora_rank == 0              ? 0
                : h->pair && h->q_wide && h->tma_store ? kQWide
                                                       : h->d.nope_dim + h->d.rope_dim;
    return MLA_OK;
}

int mla_prolog_plan(const mla_prolog_dims* dims, int32_t sms, mla_prolog_plan_info* out) {
    if (!dims || !out || sms < 1) return MLA_ERR_INVALID_ARG;
    const int rc = check_dims(*dims);
    if (rc != MLA_OK) return rc;
    const mla_prolog_dims& d = *dims;
    const int Lq = d.q_lora_rank, Lkv = d.kv_lora_rank, R = d.rope_dim;
    const int NA = Lq + Lkv + R, kb = cdiv(d.D, kBK);
    const Schedule sc = plan_schedule(d.T, d.D, Lq, Lkv, R, d.num_heads, d.nope_dim, d.v_dim, sms);
    int bn_a = sc.bn_a, splits = sc.splits_a;
    if (!sc.decode) {
        CompressTilePlan plans[kNumCompressTiles];
        bn_a = plan_compress_tiles(d.T, NA, kb, sms, plans);
        for (const auto& ct : plans)
            if (ct.bn == bn_a) splits = ct.splits;
    }
    const auto cost = compress_job_bytes(d.T, NA, kb, bn_a, splits);
    *out = mla_prolog_plan_info{};
    out->decode = sc.decode ? 1 : 0;
    out->bn_a = bn_a;
    out->splits_a = splits;
    out->group_a = sc.group_a;
    out->compress_jobs = static_cast<int32_t>(cost.size());
    out->bn_kv = sc.bn_kv;
    out->busiest_bytes = cost.empty() ? 0 : lpt_assign(cost, sms);
    // a KV-only prefill's last expansion round as half tiles (one CTA per tile)
    const int njobs_b = cdiv(d.num_heads * (d.nope_dim + d.v_dim), sc.bn_kv) * cdiv(d.T, kBM);
    out->kv_halves = !sc.decode && Lq == 0 && sc.bn_kv % 128 == 0 ? plan_last_round_halves(njobs_b, sms) : 0;
    return MLA_OK;
}

int mla_prolog_lpt(const int64_t* cost, int32_t n, int32_t groups, int32_t* table, int64_t* busiest) {
    if (n < 0 || groups < 1 || (n > 0 && !cost)) return MLA_ERR_INVALID_ARG;
    std::vector<long long> c(cost, cost + n);
    for (long long v : c)
        if (v < 0) return MLA_ERR_INVALID_ARG;
    std::vector<int> t;
    const long long b = n > 0 ? lpt_assign(c, groups, &t) : 0;
    if (table) {
        if (n == 0) t.assign(static_cast<size_t>(groups) + 1, 0);
        std::copy(t.begin(), t.end(), table);
    }
    if (busiest) *busiest = b;
    return MLA_OK;
}

}  // extern "C"
