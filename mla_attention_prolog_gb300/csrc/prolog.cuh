// Kernel parameter blocks and host-side launchers of the prolog kernels.
// Included by the kernel translation units and by the C-ABI host code.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <utility>
#include <vector>

namespace mlap {

constexpr int kStatusPositionRange = 0x1;
constexpr int kStatusWaitTimeout = 0x2;
constexpr int kStatusSlotRange = 0x4;

constexpr int kBM = 128;  // MMA M: token rows per tile (one TMEM lane per row)
constexpr int kBK = 64;   // K per pipeline stage: one 128-byte swizzle atom of BF16

inline int cdiv_host(int a, int b) { return (a + b - 1) / b; }

// Compression projection: partial[split][t][n] = sum over the split's K range
// of x[t, k] * W_a[n, k] (FP32).  Jobs: m_tiles x n_tiles x splits.
struct CompressParams {
    float* partials;  // [splits][T][NA]
    int T, NA;
    int bn;           // tile width over the NA weight rows
    int kb_total;     // K blocks of 64 over D
    int splits;       // split-K factor
    int group;        // K blocks per tensor-core accumulation chain (>= 1)
    int n_tiles, m_tiles;
    int compensated;  // drained chains summed with TwoSum (1) or plain FP32 adds (0)
    int prefetch_l2;  // warm L2 with the later kernels' small inputs (decode)
    const int32_t* positions;
    const float* cos_sin;
    int R, max_pos;
    const uint16_t* gamma;
    int n_gamma;
    int* status;
    uint64_t timeout_ns;
    const int* job_table;  // balanced per-CTA job lists (null: round robin)
    // One split (splits == 1): write the sums as the BF16 row the norm would
    // round them to, [T][NA] BF16 in the partials buffer, instead of FP32.
    int out_bf16;
    // A byte range the kernel asks L2 to fetch from HBM while it runs (the
    // expansion weights of a decode batch; null: none), in pieces of 32 KB
    // issued by the producer warp's spare lanes.
    const uint8_t* l2_fetch;
    uint64_t l2_fetch_bytes;
    // W8A8: x and W_a hold INT8 codes as BF16 integers; each chain's sums are
    // exact integers, added in int32, and leave as AT-06 dequantised BF16
    // ((float)y * x_scale[t]) * w_scale[n] (one split) or as int32 partials.
    int w8a8;
    const float* x_scale;  // [T]
    const float* w_scale;  // [NA]
    int l2_policy;  // L2 eviction priority of the operand loads (kL2WeightsLast, kL2ActsLast)
};

// Per-token reduction of the partials, BF16 cast, RMSNorm of c_q and c_kv,
// RoPE of k_pe; writes the normed rows, out_kpe and the rope slice of out_k.
struct NormRopeParams {
    const float* partials;  // [splits][T][NA]
    int splits, T, NA, Lq, Lkv, R, H, Dn;
    int in_bf16;            // one split written as BF16 [T][NA] (CompressParams::out_bf16)
    float inv_lq, inv_lkv, eps;
    const uint16_t* gamma;  // [Lq + Lkv]
    const int32_t* positions;
    const float* cos_sin;
    int max_pos;
    uint16_t* normed;   // [T][Lq + Lkv]
    uint16_t* out_k;    // [T][H][Dn + R]
    uint16_t* out_kpe;  // [T][R]
    uint32_t* amax;     // [T] (cleared here when the per-token q quant is on)
    int* status;
    int interleaved;    // k_pe de-interleaved (pairs (2i, 2i+1)) before the RoPE
    // latent KV cache (null: none): row slots[t] of [num_slots][Lkv + R]
    // receives [normed c_kv | k_pe_rot]; a negative slot is skipped
    uint16_t* cache;
    const int32_t* slots;
    long long num_slots;
    // W8A8: split-K partials are int32 (dequantised here with x_scale and
    // w_scale), and the normed c_q and c_kv rows leave as per-token INT8
    // codes (as BF16 integers) with their scales in nscale[t] = (c_q, c_kv).
    int w8a8;
    const float* x_scale;  // [T]
    const float* w_scale;  // [NA]
    float* nscale;         // [T][2]
    uint32_t* w8_split;    // [ceil(T / 128)]: token tiles whose expansion K must split (w8_finish_token)
};

// Expansion projections.  Tiles [0, nq_tiles) are q heads (one head of
// Dn + R columns each), the rest are kv tiles of bn_kv columns.
struct ExpandParams {
    int T, H, Dn, Dv, R;
    int NQ, NKV;
    int nq_tiles, nkv_tiles, bn_kv;
    int m_tiles, group_n;  // token tiles; weight tiles per L2 group of the job order
    const int* job_table;  // balanced per-CTA job lists (null: round robin)
    int Lq, Lkv;
    int kb_q, kb_kv;
    const int32_t* positions;
    const float* cos_sin;
    int max_pos;
    uint16_t* out_k;  // [T][H][Dn + R]
    uint16_t* out_v;  // [T][H][Dv]
    int out_aligned32;  // out_k and out_v 32-byte aligned: 256-bit stores
    float* qws;       // [T][NQ] FP32 q after RoPE (per-token quant)
    uint32_t* amax;   // [T] bits of max |q| per token (per-token quant)
    int* status;
    uint64_t timeout_ns;
    int interleaved;  // rope slices de-interleaved before the RoPE
    int head_norm;    // per-head RMSNorm (no gamma) of q before its RoPE
    float inv_hd, eps;  // 1 / (Dn + R) and the norm's epsilon
    int per_head;     // INT8 codes and one scale per (token, head) in the epilogue
    int8_t* q_codes;  // [T][H][Dn + R] (per_head)
    float* q_scale;   // [T][H] (per_head)
    // Epilogue stores through shared memory and bulk tensor stores (the
    // kernels built with a staging area; the kv tiles and the per-token q
    // path): the output tensor maps are kernel parameters.
    int tma_store;
    // q tiles of kQWide columns that run across head boundaries (nq_tiles =
    // NQ / kQWide) instead of one head per tile: the per-token q path through
    // the store ring, R = 64 and Dn a multiple of 64, so every 64-column piece
    // of a tile is nope columns or one head's whole rope slice.
    int q_wide;
    // W8A8: the activations are INT8 codes (as BF16 integers) with a scale
    // per token (a_scale[2t] for c_q, a_scale[2t + 1] for c_kv), the weights
    // INT8 codes with one scale per output row.  The epilogue first turns
    // the exact integer accumulator into ((float)y * a_scale) * w_scale.
    int w8a8;
    const float* a_scale;     // [T][2]
    const float* w_scale_q;   // [NQ]
    const float* w_scale_kv;  // [NKV]
    // Per 128-token tile: bit 0 / bit 1 set when the q / kv expansion of
    // that tile runs as two exact chains (a K longer than kW8ChainKb blocks
    // and some row's codes large enough to need it).
    const uint32_t* w8_split;
    int n_tiles128;
    int l2_policy;  // L2 eviction priorities: kL2WeightsLast, kL2ActsLast, kL2StoresFirst
    // A KV-only prolog on one CTA per tile: the last kv_halves jobs of the
    // job order run as two jobs each over the columns [0, bn_kv / 2) and
    // [bn_kv / 2, bn_kv) of their tile, appended after the others (job ids
    // full - kv_halves .. full + kv_halves - 1), so that a last round of
    // jobs shorter than the grid spreads over twice as many CTAs.
    int kv_halves;
    // The same for the kv-resident pair kernel's super-jobs (a token tile and
    // a group of kv tiles): its last kvres_halves super-jobs run as two
    // super-jobs of half the group each, appended after the others (every
    // group whole, of at least two tiles).
    int kvres_halves;
};

// Bits of CompressParams / ExpandParams::l2_policy (MLA_TUNE_L2_POLICY):
// weight tiles and activation tiles loaded with the evict-last priority,
// tensor stores of the outputs with the evict-first priority.
constexpr int kL2WeightsLast = 1, kL2ActsLast = 2, kL2StoresFirst = 4;

constexpr int kQWide = 256;
// W8A8: K blocks of one exact accumulation chain.  A chain of k blocks sums
// 64 k products of magnitude <= 127^2, so every partial sum is an integer
// below 2^24 (exact in FP32) while 64 k * 127^2 < 2^24, i.e. k <= 16.
constexpr int kW8ChainKb = 16;
// W8A8: a token tile whose activation rows all have sum |code| <= this
// bound needs no chain split whatever its K: every partial sum is then at
// most 127 * 132104 = 16,777,208 < 2^24 in magnitude.
constexpr uint32_t kW8SumLimit = 132104;

// W8A8: per-token INT8 codes of a BF16 matrix (x), written as BF16 integers.
struct QuantXParams {
    const uint16_t* x;  // [rows][cols] BF16
    int rows, cols;
    uint16_t* codes;    // [rows][cols] BF16 integers in [-127, 127]
    float* scale;       // [rows]
    uint32_t* w8_split;  // [n_split] cleared here for the norm step to mark
    int n_split;
};

struct QuantParams {
    const float* y;          // [rows][row_len]
    const uint32_t* amax;    // [rows] bits of max|y| (null: the kernel finds it)
    int rows, row_len;
    int chunk;               // elements per CTA (row_len when amax is null)
    int8_t* codes;
    float* scale;
};

// The cooperative decode kernel: the four steps as phases of one launch,
// handing over through counters (word offsets into `sync`, one 128-byte line
// each): runs completed, and per run one arrival per CTA after the
// compression, one per token after the norm, one per CTA after the
// expansion and one per CTA at exit.
constexpr int kSyncEpoch = 0;
constexpr int kSyncCompressed = 32;
constexpr int kSyncNormed = 64;
constexpr int kSyncExpanded = 96;
constexpr int kSyncFinished = 128;
constexpr int kSyncWords = 160;

struct DecodeParams {
    CompressParams a;
    NormRopeParams n;
    ExpandParams b;
    QuantParams q;   // q.rows == 0 without a q path
    unsigned* sync;  // kSyncWords words, zero at creation
    int* status;
    uint64_t timeout_ns;
};

// Compression + split + RMSNorm + k_pe RoPE of one token tile in one
// thread-block cluster (small decode batches): CTA rank r computes the
// split-K partial of column group r / ks over K-split r % ks, stages it in
// its own shared memory and copies each token's row (bulk copies, completed
// on the owner's mbarrier) into the shared memory of the CTA that owns the
// token (tokens [o * tpo, (o + 1) * tpo) belong to rank o), which then runs
// the norm step for its tokens.
//
// Shared memory (from a 1 KB aligned base): the ring [0, area); once the
// ring is free, the receive buffer [0, recv) ([split][group][token][cgw]
// FP32), the norm groups' rows [recv, stg_off) and the staging rows
// [stg_off, ...) (T rows of cgw FP32, 16-byte chunks XOR-swizzled by the
// token's row); then the barriers, and from const_off the norm constants of
// the owned tokens (gamma, positions, cos/sin rows) and the groups' partial
// sums.
struct ClusterNormParams {
    int T, NA, kb_total;
    int nc, ks, cgw, tpo;  // column groups, K splits, group width, tokens per owner
    int stages;            // ring stages
    int b_boxes;           // TMA boxes per weight tile (cgw > 256: two of cgw / 2 rows)
    uint32_t tmem_cols;
    uint32_t area_bytes;   // ring / receive area (1 KB aligned) before the barriers
    uint32_t recv_bytes;   // receive buffer at the start of the area
    uint32_t stg_off;      // staging rows (cgw floats each)
    uint32_t const_off;    // norm constants
    NormRopeParams n;      // outputs and norm constants (partials unused)
    int* status;
    uint64_t timeout_ns;
};

// The cluster layout for a problem, or ok = false when it does not pay
// (more than one token tile, or too many weight bytes for a dozen SMs).
// Measured on GB300, the cluster path beats the split-K path only when its
// estimated loads + exchange stay near a microsecond (tiny batches): each of
// its phases (cluster barriers, the exchange, the norm) costs 0.3-0.8 us of
// latency whatever its size, and the 16 SMs receive weights at ~100 GB/s
// each.  It is the default below kClusterDefaultUs and opt-in above.
struct ClusterPlan {
    bool ok = false;
    int nc = 0, ks = 0, cgw = 0, tpo = 0, stages = 0;
    double est_us = 0.0;  // estimated loads + exchange time
    size_t smem = 0;
    uint32_t area = 0, recv = 0, stg_off = 0, const_off = 0;
};

constexpr int kClusterThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 drain; all ten warps norm
constexpr int kClusterNormGroups = 5;  // norm groups of two warps, one token each at a time
constexpr int kClusterMaxCtas = 16;
constexpr size_t kClusterSmemBudget = 216 * 1024;  // ring or receive area (+ barriers < 227 KB)
constexpr size_t kClusterSmemMax = 227 * 1024;
constexpr double kClusterDefaultUs = 1.5;

__host__ __device__ inline size_t align16(size_t b) { return (b + 15) & ~static_cast<size_t>(15); }

inline ClusterPlan plan_cluster(int T, int D, int Lq, int Lkv, int R, int max_ctas) {
    ClusterPlan best;
    const int NA = Lq + Lkv + R, kb = cdiv_host(D, kBK);
    if (T < 1 || T > kBM) return best;
    long long best_bytes = 0;
    for (int nc = 1; nc <= max_ctas; ++nc) {
        const int cgw = cdiv_host(cdiv_host(NA, nc), 32) * 32;
        if (cgw > 512) continue;
        const int ks = max_ctas / nc < kb ? max_ctas / nc : kb;
        if (ks < 1) break;
        const int kbps = cdiv_host(kb, ks);
        const size_t stage = static_cast<size_t>(kBM) * kBK * 2 + static_cast<size_t>(cgw) * kBK * 2;
        int stages = static_cast<int>(kClusterSmemBudget / stage);
        if (stages > kbps) stages = kbps;
        if (stages < 1 || (stages < 2 && kbps > 1)) continue;
        const int ctas = nc * ks, tpo = cdiv_host(T, ctas);
        const size_t recv = static_cast<size_t>(ks) * nc * tpo * cgw * 4;
        const size_t rows = kClusterNormGroups * align16(static_cast<size_t>(NA + R) * 2);
        const size_t stg_off = (recv + rows + 127) & ~static_cast<size_t>(127);
        const size_t need = stg_off + static_cast<size_t>(T) * cgw * 4;
        if (need > kClusterSmemBudget) continue;
        const size_t ring = static_cast<size_t>(stages) * stage;
        const size_t area = ((ring > need ? ring : need) + 1023) & ~static_cast<size_t>(1023);
        const size_t const_off = area + 8 * (2 * stages + 2) + 16;
        const size_t smem = const_off + align16(static_cast<size_t>(Lq + Lkv) * 2) + align16(tpo * 4) +
                            static_cast<size_t>(tpo) * R * 4 + kClusterNormGroups * 4 * 4 + 1024;
        if (smem > kClusterSmemMax) continue;
        // Estimated time: the bytes one CTA must receive (its weight rows and
        // the token rows of x) at ~100 GB/s per SM, plus the split partials
        // exchanged inside the cluster at ~450 GB/s for the whole cluster
        // (both rates measured on GB300).
        const double t_load = static_cast<double>(kbps) * kBK * 2 * (cgw + T) / 100e3;
        const double t_swap = static_cast<double>(ks - 1) * T * NA * 4 / 450e3;
        const long long bytes = static_cast<long long>((t_load + t_swap) * 1e3);  // ns
        if (!best.ok || bytes < best_bytes) {
            best.ok = true;
            best_bytes = bytes;
            best.nc = nc, best.ks = ks, best.cgw = cgw, best.tpo = tpo, best.stages = stages;
            best.area = static_cast<uint32_t>(area);
            best.recv = static_cast<uint32_t>(recv);
            best.stg_off = static_cast<uint32_t>(stg_off);
            best.const_off = static_cast<uint32_t>(const_off);
            best.smem = smem;
            best.est_us = t_load + t_swap;
        }
    }
    // Worth it while the loads and the exchange take a few microseconds;
    // beyond that the split-K path over every SM wins.
    if (best.ok && best_bytes > 5000) best.ok = false;
    return best;
}

cudaError_t cluster_set_attributes(size_t smem, int ctas);
cudaError_t cluster_max_active(size_t smem, int ctas, int* clusters);
cudaError_t launch_compress_norm_cluster(int ctas, size_t smem, const CUtensorMap& tm_x, const CUtensorMap& tm_wa,
                                         const ClusterNormParams& p, cudaStream_t st);

size_t decode_smem_bytes(int NA, int R, int Lq, int Lkv);
cudaError_t decode_set_attributes(size_t smem);
cudaError_t decode_occupancy(size_t smem, int* blocks_per_sm);
cudaError_t launch_decode(int grid, size_t smem, const CUtensorMap& tm_x, const CUtensorMap& tm_wa,
                          const CUtensorMap& tm_aq, const CUtensorMap& tm_akv, const CUtensorMap& tm_bq,
                          const CUtensorMap& tm_bkv, const DecodeParams& p, cudaStream_t st);
constexpr int kDecodeMaxBN = 192;  // widest expansion tile the decode kernel takes

// Shapes of the GEMM kernel instantiations.
// Expansion kernel: Wide = BN_MAX 256, 4 stages; Mid = BN_MAX 192, 5 stages
// (decode with a q path: one head of Dn + R <= 192 columns per tile);
// Narrow = BN_MAX 64, 4 stages; Deep = BN_MAX 64, 8 stages (after the
// cluster compression: every K block of a narrow kv tile's weights is in
// flight before the normed rows exist).
// Compression kernel: Wide = BN_MAX 128, 6 stages; Narrow = BN_MAX 64, 4 stages.
// The narrow (decode) shapes use half the shared memory so that a compression
// CTA and an expansion CTA fit on one SM and the expansion can start
// streaming its weights while the compression is still running.
// Kernel shapes: Wide / Mid / Narrow / Deep for both projections; Wide192 and
// Wide256 are the compression's 192- and 256-column tiles (plain FP32 drain).
enum class GemmShape { Wide, Mid, Narrow, Deep, Wide192, Wide256 };

// Tile shapes and work split of one problem size, chosen on the host.
struct Schedule {
    bool decode;          // few token tiles: weights streamed once by split-K / narrow tiles
    int m_tiles;          // 128-token tiles
    GemmShape shape_a;    // compression kernel shape
    int bn_a, splits_a;   // compression weight-tile width, split-K factor
    int group_a;          // K blocks per tensor-core accumulation chain (compression)
    GemmShape shape_b;    // expansion kernel shape
    int bn_kv;            // expansion kv tile width
};

// Jobs of unequal cost over G CTAs, longest first, each to the least-loaded
// CTA.  Returns the busiest CTA's load and, when `table` is given, the job
// table the kernels read: G + 1 start offsets, then every CTA's job ids --
// in the order assigned, or (by_index) each CTA's jobs in job-id order, so
// that CTAs that progress alike work on neighbouring job ids at any time.
inline long long lpt_assign(const std::vector<long long>& cost, int G, std::vector<int>* table = nullptr,
                            bool by_index = false) {
    std::vector<std::pair<long long, int>> w;
    w.reserve(cost.size());
    for (size_t j = 0; j < cost.size(); ++j) w.push_back({-cost[j], static_cast<int>(j)});
    std::sort(w.begin(), w.end());
    std::vector<long long> load(G, 0);
    std::vector<std::vector<int>> lists(G);
    for (const auto& e : w) {
        int best = 0;
        for (int c = 1; c < G; ++c)
            if (load[c] < load[best]) best = c;
        load[best] -= e.first;
        lists[best].push_back(e.second);
    }
    if (by_index)
        for (auto& l : lists) std::sort(l.begin(), l.end());
    if (table) {
        table->clear();
        table->push_back(0);
        for (int c = 0; c < G; ++c) table->push_back(table->back() + static_cast<int>(lists[c].size()));
        for (int c = 0; c < G; ++c) table->insert(table->end(), lists[c].begin(), lists[c].end());
    }
    return *std::max_element(load.begin(), load.end());
}

// Operand bytes of each compression job, in the kernel's job order (token
// tile, weight tile, K split): its K blocks x (the token rows of x + the
// weight rows of its tile), 128 bytes per row per K block.
//
// With CTA pairs (cg = 2) token tiles are 256 rows and the cost is that of the
// busier CTA of the pair: up to 128 token rows and bn / 2 weight rows.
inline std::vector<long long> compress_job_bytes(int T, int NA, int kb, int bn, int splits, int cg = 1) {
    const int tm = kBM * cg;
    const int m_tiles = cdiv_host(T, tm), n_tiles = cdiv_host(NA, bn);
    std::vector<long long> c;
    c.reserve(static_cast<size_t>(m_tiles) * n_tiles * splits);
    for (int m = 0; m < m_tiles; ++m)
        for (int n = 0; n < n_tiles; ++n)
            for (int sp = 0; sp < splits; ++sp) {
                const int nkb = (sp + 1) * kb / splits - sp * kb / splits;
                const int rows = T - m * tm < kBM ? T - m * tm : kBM;
                const int width = NA - n * bn < bn ? NA - n * bn : bn;
                c.push_back(static_cast<long long>(nkb) * 128 * (rows + (width + cg - 1) / cg));
            }
    return c;
}

// Prefill compression: the split-K factor (1, 2 or 4) whose busiest CTA,
// jobs assigned longest first, finishes first -- its operand bytes at ~100
// GB/s per SM, plus the extra FP32 partials written and read back by the
// norm at ~8 TB/s (both rates measured on GB300).  cg = 2: CTA pairs; bn:
// the weight-tile width.
inline int prefill_compress_splits(int T, int NA, int kb, int sms, int cg, int bn = 128) {
    double best_us = 0.0;
    int best = 1;
    for (int k = 1; k <= 4 && k <= kb / 4; k *= 2) {
        const long long busiest = lpt_assign(compress_job_bytes(T, NA, kb, bn, k, cg), sms / cg);
        const double us = busiest / 100e3 + (k - 1) * static_cast<double>(T) * NA * 8 / 8e6;
        if (k == 1 || us < best_us) best_us = us, best = k;
    }
    return best;
}

// Prefill compression plans for each weight-tile width of
// kCompressTileWidths: split-K factor and the operand bytes of the busiest
// CTA (jobs longest first, each to the least-loaded CTA; the job tables into
// `tables` when given and there are more jobs than CTAs).  Returns the
// default width: the wide tile (144, 192 or 256) that needs no split-K and
// brings its busiest SM the fewest operand bytes, else 128.  (A 144-wide
// tile runs on the 192-wide kernel: 4 tiles of 144 cover the 576 rows of a
// KV-only prolog with 33 % more jobs than 3 tiles of 192.)  Measured on GB300
// (step time): V3 prefill 16384 tokens 2441 / 2245 / 2173 us (128 / 192 /
// 256), V2-Lite prefill 4096 tokens 52.3 / 43.5 / 48.1 us (256 needs
// split-K 2 there), V3 prefill 385 tokens 109.5 / 127.3 / 120.0 us (the
// wide ones need split-K 4).
constexpr int kNumCompressTiles = 4;
constexpr int kCompressTileWidths[kNumCompressTiles] = {128, 144, 192, 256};
struct CompressTilePlan {
    int bn, splits, jobs;
    long long busiest;
};
inline int plan_compress_tiles(int T, int NA, int kb, int sms, CompressTilePlan (&out)[kNumCompressTiles],
                               std::vector<int>* tables = nullptr) {
    int def = 128;
    long long best = -1;
    for (int i = 0; i < kNumCompressTiles; ++i) {
        CompressTilePlan& ct = out[i];
        ct.bn = kCompressTileWidths[i];
        ct.splits = prefill_compress_splits(T, NA, kb, sms, 1, ct.bn);
        const auto cost = compress_job_bytes(T, NA, kb, ct.bn, ct.splits);
        ct.jobs = static_cast<int>(cost.size());
        ct.busiest = lpt_assign(cost, sms, tables && ct.jobs > sms ? &tables[i] : nullptr, true);
        if (ct.bn > 128 && ct.splits == 1 && (best < 0 || ct.busiest < best)) {
            best = ct.busiest;
            def = ct.bn;
        }
    }
    return def;
}

// Jobs of a last round to run as two half jobs each on twice as many
// workers: the remainder r of `jobs` over `grid` workers when there is more
// than one round and 2 r workers are free in the last one, else 0 (the
// busiest worker then does rounds - 1/2 jobs' work instead of rounds).
inline int plan_last_round_halves(int jobs, int grid) {
    if (grid <= 0 || jobs <= grid) return 0;
    const int r = jobs % grid;
    return r > 0 && 2 * r <= grid ? r : 0;
}

// kv tiles per super-job of the kv-resident pair kernel: the largest of 8,
// 4, 2 that still gives every CTA pair a super-job, else 1.  Measured on
// GB300 (step time): V3 prefill 1932 / 1870 / 1897 / 1893 us with groups of
// 4 / 8 / 16 / 32; V2-Lite prefill 41.7 / 41.5 / 53.2 us with 2 / 4 / 8 (32
// super-jobs for 76 pairs at 8).
inline int plan_kv_group(int pair_m_tiles, int nkv_tiles, int pairs) {
    for (int g = 8; g > 1; g /= 2)
        if (g <= nkv_tiles && static_cast<long long>(pair_m_tiles) * cdiv_host(nkv_tiles, g) >= pairs) return g;
    return 1;
}

// T tokens, D model width, Lq / Lkv / R ranks, H heads of Dn + R (q) and
// Dn + Dv (kv) columns, on a device with `sms` SMs.
inline Schedule plan_schedule(int T, int D, int Lq, int Lkv, int R, int H, int Dn, int Dv, int sms) {
    Schedule s{};
    const int NA = Lq + Lkv + R, NKV = H * (Dn + Dv);
    const int kb_a = cdiv_host(D, kBK);
    s.m_tiles = cdiv_host(T, kBM);
    s.decode = s.m_tiles <= 2;
    s.shape_a = GemmShape::Wide;
    s.bn_a = 128;
    s.splits_a = 1;
    if (s.decode) {
        // Split-K over weight tiles of 128 columns or a little less: the
        // width (multiple of 16) that puts the most CTAs to work, the widest
        // on a tie (more weight bytes in flight per ring stage).
        int best = 0;
        for (int bn = 128; bn >= 96; bn -= 16) {
            const int tiles = cdiv_host(NA, bn) * s.m_tiles;
            int k = tiles > 0 ? sms / tiles : 1;
            if (k > kb_a / 2) k = kb_a / 2;
            if (k < 1) k = 1;
            const int ctas = tiles * k <= sms ? tiles * k : 0;
            if (ctas > best) best = ctas, s.bn_a = bn, s.splits_a = k;
        }
    } else {
        s.splits_a = prefill_compress_splits(T, NA, kb_a, sms, 1);
    }
    // Accumulation chain length (K blocks) of the compression projection:
    // each drained chain costs the tensor core ~0.4 us, and longer chains
    // flip more INT8 q codes.  Measured on GB300 (flips vs the oracle, bar
    // 1e-3): V3 prefill 4.2e-4 / 5.8e-4 / 1.07e-3 at 4 / 8 / 16; V3 decode
    // 3.2e-4 / 4.5e-4 / 9.95e-4 at 2 / 4 / 14, 50.4 / 49.8 / 49.0 us per step.
    s.group_a = 4;
    // Expansion: prefill uses 256-wide kv tiles (one head of V2/V3); decode
    // without a q path uses the narrow kernel with enough tiles to cover the
    // SMs; decode with a q path puts one q head per tile (the 192-wide,
    // 5-stage shape when the head fits) and kv tiles as wide as the ring, so
    // a kv K block moves as many weight bytes as a q one and the per-CTA job
    // lists balance by bytes and by K blocks alike.
    if (!s.decode) {
        s.shape_b = GemmShape::Wide;
        s.bn_kv = 256;
    } else if (Lq == 0) {
        s.shape_b = GemmShape::Narrow;
        s.bn_kv = cdiv_host(NKV, 64) * s.m_tiles >= sms ? 64 : 32;
    } else {
        s.shape_b = Dn + R <= 192 ? GemmShape::Mid : GemmShape::Wide;
        s.bn_kv = s.shape_b == GemmShape::Mid ? 192 : 256;
    }
    return s;
}


// Launches `kernel`; with `pdl` the launch may overlap the tail of the
// previous kernel in the stream (programmatic dependent launch): the kernel
// must call pdl_wait() before touching anything that kernel produced.
template <class... KArgs, class... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t st, bool pdl, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

cudaError_t gemm_set_attributes();
cudaError_t launch_compress(GemmShape s, int grid, const CUtensorMap& tm_x,
                            const CUtensorMap& tm_wa, const CompressParams& p, cudaStream_t st);
// The expansion's output tensor maps for its bulk tensor stores (used when
// ExpandParams::tma_store is set, by the kernels that stage stores): the FP32
// q workspace in boxes of 16 columns x 32 rows, out_k and out_v in boxes of
// 32 x 32, all with the 64-byte swizzle.
struct OutTensorMaps {
    CUtensorMap q, k, v;
};
// tm_bkvh: W_kv_b in boxes of bn_kv / 2 rows, for the half tiles of
// ExpandParams::kv_halves (null: no half tiles).
cudaError_t launch_expand(GemmShape s, int grid, const CUtensorMap& tm_aq,
                          const CUtensorMap& tm_akv, const CUtensorMap& tm_bq,
                          const CUtensorMap& tm_bkv, const OutTensorMaps& om, const ExpandParams& p,
                          cudaStream_t st, const CUtensorMap* tm_bkvh = nullptr);
// Prefill expansion on CTA pairs: 256-token tiles, kv tiles of 256 columns,
// q heads of at most 256 columns; the B tensor maps' boxes are half a tile
// (bn / 2 rows) and m_tiles counts 256-token tiles.
cudaError_t expand_pair_max_active(int* clusters);
cudaError_t compress_pair_max_active(int* clusters);
// Prefill compression on CTA pairs: 256-token tiles of 128 weight rows (the
// W_a tensor map's box is 64 rows), m_tiles counting 256-token tiles.
cudaError_t launch_compress_pair(int pairs, const CUtensorMap& tm_x, const CUtensorMap& tm_wa,
                                 const CompressParams& p, cudaStream_t st);
cudaError_t launch_expand_pair(int pairs, const CUtensorMap& tm_aq, const CUtensorMap& tm_akv,
                               const CUtensorMap& tm_bq, const CUtensorMap& tm_bkv, const OutTensorMaps& om,
                               const ExpandParams& p, cudaStream_t st);
// The kv tiles of the prefill expansion on CTA pairs with the normed c_kv
// rows resident in shared memory (Lkv <= 512, 256-wide kv tiles, kv outputs
// through tensor stores): super-jobs of `group` kv tiles per 256-token tile.
cudaError_t expand_kv_pair_max_active(int* clusters);
cudaError_t launch_expand_kv_pair(int pairs, const CUtensorMap& tm_akv, const CUtensorMap& tm_bkv,
                                  const OutTensorMaps& om, const ExpandParams& p, int group, cudaStream_t st);
cudaError_t launch_expand_kv_pair_w8(int pairs, const CUtensorMap& tm_akv, const CUtensorMap& tm_bkv,
                                     const OutTensorMaps& om, const ExpandParams& p, int group, cudaStream_t st);
// The W8A8 instantiations (gemm_w8a8.cu), chosen by the launchers above
// when the parameters ask for W8A8.
cudaError_t gemm_w8a8_set_attributes();
cudaError_t launch_compress_w8(GemmShape s, int grid, const CUtensorMap& tm_x, const CUtensorMap& tm_wa,
                               const CompressParams& p, cudaStream_t st);
cudaError_t launch_expand_w8(GemmShape s, int grid, const CUtensorMap& tm_aq, const CUtensorMap& tm_akv,
                             const CUtensorMap& tm_bq, const CUtensorMap& tm_bkv, const OutTensorMaps& om,
                             const ExpandParams& p, cudaStream_t st, const CUtensorMap* tm_bkvh = nullptr);
cudaError_t launch_expand_pair_w8(int pairs, const CUtensorMap& tm_aq, const CUtensorMap& tm_akv,
                                  const CUtensorMap& tm_bq, const CUtensorMap& tm_bkv, const OutTensorMaps& om,
                                  const ExpandParams& p, cudaStream_t st);
cudaError_t launch_norm_rope(const NormRopeParams& p, cudaStream_t st);
cudaError_t launch_quant(const QuantParams& p, cudaStream_t st, bool pdl);
cudaError_t launch_quant_x(const QuantXParams& p, cudaStream_t st);
// INT8 codes -> the same integers as BF16 (exact), n elements.
cudaError_t launch_widen_i8(const int8_t* src, uint16_t* dst, size_t n, cudaStream_t st);
cudaError_t launch_wait_selftest(int* status, uint64_t timeout_ns, cudaStream_t st);

}  // namespace mlap
