/*
 * mla_prolog.h -- C ABI of the GB300 (sm_103a) fused MLA attention prolog.
 *
 * The prolog turns the hidden states of T tokens into the per-head K and V
 * of Multi-head Latent Attention (and, optionally, an INT8 per-token q):
 *
 *   1. compression projection  C = x . W_a^T, rounded to BF16
 *      (DeepSeek-V2-Lite-Chat MLA KV Prolog migration guide, section 背景,
 *       step "kv_a_proj"; PyPTO-Gym AT-10 article, section 五, q_a_proj);
 *   2. split C into c_q | c_kv | k_pe (migration guide, step "split");
 *   3. RMSNorm of c_q and c_kv in FP32 with gamma, cast to BF16
 *      (AT-10 article, sections 二 and 三, variant B);
 *   4. rotate-half RoPE of k_pe with the token's row of the cos/sin table
 *      (migration guide, step "RoPE" and section 精度验证; DeepSeek-V3.2-Exp
 *       PyPTO article, section 3.3);
 *   5. KV expansion projection of the normed c_kv (migration guide, "kv_b_proj");
 *   6. reshape to [T, H, Dn + Dv], split into k_nope | value, and assemble
 *      K = [k_nope | k_pe_rot] per head (migration guide, "reshape split" and
 *      "assemble");
 *   7. q path (when q_lora_rank > 0): q expansion of the normed c_q, RoPE on
 *      each head's rope slice, then per-token symmetric INT8 quantisation:
 *      amax = max|q_row|, code = clamp(rint_half_even(q * (127/amax)), +-127),
 *      scale = amax/127 (DeepSeek-V3.2-Exp PyPTO article, section 3.1
 *      PrologQuant; grouped_matmul_swiglu_quant article, section 数学公式).
 *
 * Notation: T tokens, D hidden size, Lq = q_lora_rank (0: no q path),
 * Lkv = kv_lora_rank, R = rope_dim, H = num_heads, Dn = nope_dim, Dv = v_dim.
 *
 * Conventions for every call below
 *   - Tensor arguments are DEVICE pointers on the handle's device, owned by
 *     the caller, contiguous row-major, and 16-byte aligned (positions:
 *     4-byte aligned).  BF16 tensors are passed as raw 16-bit storage.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls enqueue work and return without synchronising, except
 *     where a call says it synchronises.
 *   - Return value: MLA_OK (0) or a negative MLA_ERR_* code.  A failed call
 *     enqueues nothing.  Faults found on the device (a position outside the
 *     table, a wait that ran out) never trap: they set bits of the handle's
 *     device status word, read with mla_prolog_device_status().
 */
#ifndef MLA_PROLOG_H_
#define MLA_PROLOG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ------------------------------------------------------ */
#define MLA_OK                    0
#define MLA_ERR_INVALID_ARG      -1  /* null / misaligned pointer, bad flag combination   */
#define MLA_ERR_UNSUPPORTED_DIMS -2  /* a size rule below is broken                        */
#define MLA_ERR_CUDA             -3  /* a CUDA runtime call or launch failed               */
#define MLA_ERR_OOM              -4  /* workspace allocation failed                        */
#define MLA_ERR_DEVICE           -5  /* current device is not an sm_103 (GB300) GPU       */

/* ---- device status bits (mla_prolog_device_status) --------------------- */
#define MLA_STATUS_POSITION_RANGE 0x1 /* some positions[t] was outside [0, max_pos): that
                                         token's outputs were zero-filled                  */
#define MLA_STATUS_WAIT_TIMEOUT   0x2 /* a bounded in-kernel wait gave up; outputs of the
                                         affected tile are undefined                       */
#define MLA_STATUS_SLOT_RANGE     0x4 /* mla_prolog_run_cached: some slot_mapping[t] was
                                         >= num_slots; that token's cache row was skipped  */

/* ---- dims flags --------------------------------------------------------- */
#define MLA_PROLOG_QUANT_Q 0x1u /* q path emits INT8 codes + FP32 per-token scales.
                                   Required exactly when q_lora_rank > 0.               */
/*
 * Interleaved RoPE (QuantRope3D, DeepSeek-V3.2-Exp PyPTO article, sections
 * 2.3 and 3.3: the rope slice viewed as [R/2, 2] chunks and transposed before
 * the rotation).  Every rope slice -- k_pe and each q head's -- is first
 * de-interleaved, x'[i] = x[2i], x'[R/2 + i] = x[2i + 1], then rotated as
 * above; the rotated values stay in the de-interleaved order (out_kpe, K's
 * rope slice, the q codes).  The pages do not print the chunk size: 2 is the
 * reading taken, the one that turns adjacent pairs into rotate-half pairs.
 */
#define MLA_PROLOG_ROPE_INTERLEAVED 0x2u
/*
 * Per-head q RMSNorm (the DeepSeek-V4 q path, PyPTO-Gym AT-10 article,
 * section 九: q_b_proj, reshape to (heads, head_dim), RMSNorm again).  Each
 * head's Dn + R FP32 values of q are normalised before the RoPE, without a
 * gamma: ms = sum(x^2 / (Dn + R)), rstd = 1/sqrt(ms + eps), x * rstd, all
 * FP32.  Requires q_lora_rank > 0.
 */
#define MLA_PROLOG_Q_HEAD_NORM 0x4u
/*
 * Per-(token, head) INT8 quantisation of q: the quantisation formula of the
 * q path applied to each head row of Dn + R values, so out_scale is FP32
 * [T, H].  Runs inside the expansion kernel (no FP32 q round trip through
 * memory); the MLA_TAP_Q and MLA_TAP_AMAX taps are then absent.  Requires
 * q_lora_rank > 0.
 */
#define MLA_PROLOG_QUANT_PER_HEAD 0x8u
/*
 * W8A8 projections: the INT8 mode of the Linear step (PyPTO-Gym AT-10
 * article, section 四, AT-09 "INT8 W8A8"): every projection takes its input
 * row quantised per token (the formula of the q path: AT-05), multiplies
 * INT8 codes by INT8 weight codes exactly (an int32 result), and
 * dequantises it (AT-06) in FP32 as ((float)y * input_scale) * w_scale[row].
 *   - compression: x (BF16) -> codes; the dequantised sums are rounded to
 *     BF16 as in the BF16 mode;
 *   - expansions: the normed c_q and c_kv rows (after their BF16 cast) are
 *     quantised per token, each with its own scale (AT-11, RMSNorm + Linear
 *     + Quant); k_nope and value are the dequantised sums rounded to BF16,
 *     q the dequantised FP32 sums (then RoPE and the q quantisation).
 * The weights live in the handle: load them once with
 * mla_prolog_load_w8a8(), then call mla_prolog_run() / _run_cached() with
 * W_a = W_b = NULL.  Extra size rules: Lq <= 2048 and Lkv <= 2048.  Not
 * available through mla_prolog_run_noalloc().
 *
 * On sm_103a the tensor cores have no INT8 MMA kind, so the codes are kept
 * as BF16 integers (exact) and multiplied on the BF16 path with FP32
 * accumulation; accumulation chains are kept short enough (at most 1024 K
 * per chain) that every partial sum is an integer below 2^24 and so exact,
 * and chains are added in int32: the integer product is exact.
 */
#define MLA_PROLOG_W8A8 0x10u

/*
 * Problem sizes, fixed for the life of a handle.
 * Size rules (else MLA_ERR_UNSUPPORTED_DIMS):
 *   D, Lkv, R, Dn, Dv  positive multiples of 16;  Lq = 0 or a multiple of 16;
 *   R <= 128;  Dn + R <= 256 when Lq > 0;  T >= 0;  H >= 1;  max_pos >= 1;
 *   eps finite and >= 0;  T * H * (Dn + R + Dv) <= 4e9 and T * D <= 4e9 (the
 *   kernels keep row offsets in 32 bits: the DeepSeek-V3 shapes take up to
 *   T = 69 754 tokens per run).
 */
typedef struct mla_prolog_dims {
    int32_t  T;            /* tokens per run (rows of x)                         */
    int32_t  D;            /* hidden size                                        */
    int32_t  q_lora_rank;  /* Lq; 0 = KV prolog only                             */
    int32_t  kv_lora_rank; /* Lkv                                                */
    int32_t  rope_dim;     /* R                                                  */
    int32_t  num_heads;    /* H                                                  */
    int32_t  nope_dim;     /* Dn                                                 */
    int32_t  v_dim;        /* Dv                                                 */
    int32_t  max_pos;      /* rows of the cos/sin table                          */
    float    eps;          /* RMSNorm epsilon (1e-6 in the DeepSeek shapes)      */
    uint32_t flags;        /* OR of MLA_PROLOG_* flags                           */
} mla_prolog_dims;

typedef struct mla_prolog* mla_prolog_t;

/*
 * Creates a handle for the CURRENT CUDA device: validates dims, picks the
 * decode (small T) or prefill schedule, and allocates the handle's device
 * workspace (split-K partials, the normed c_q | c_kv rows, the FP32 q rows,
 * per-token amax, the status word).  *out receives the handle.
 * Errors: INVALID_ARG (null pointers), UNSUPPORTED_DIMS, DEVICE, OOM, CUDA.
 */
int mla_prolog_create(const mla_prolog_dims* dims, mla_prolog_t* out);

/*
 * Enqueues one prolog pass over T tokens on `stream`.
 *
 * Inputs (device, read only):
 *   x          BF16 [T, D]
 *   gamma      BF16 [Lq + Lkv]              = [gamma_q ; gamma_kv]
 *   W_a        BF16 [Lq + Lkv + R, D]       = rows [W_q_a ; W_kv_a], W_kv_a rows
 *                                             ordered [c_kv (Lkv) ; k_pe (R)]
 *   W_b        BF16, W_q_b [H(Dn+R), Lq] followed by W_kv_b [H(Dn+Dv), Lkv]
 *              (both [N, K] row-major; W_q_b empty when Lq = 0)
 *              (W_a and W_b: NULL with MLA_PROLOG_W8A8, whose weights are
 *              loaded into the handle by mla_prolog_load_w8a8)
 *   positions  int32 [T], each in [0, max_pos)
 *   cos_sin    FP32 [max_pos, R]: columns [0, R/2) = cos(p * theta_i),
 *              [R/2, R) = sin(p * theta_i)
 * Outputs (device, written in full):
 *   out_k      BF16 [T, H, Dn + R]  = [k_nope | k_pe_rot] per head
 *   out_v      BF16 [T, H, Dv]
 *   out_kpe    BF16 [T, R]          rotated k_pe (shared by every head)
 *   out_q_int8 int8 [T, H, Dn + R]  q codes (NULL iff Lq == 0)
 *   out_scale  FP32 [T]             per-token q scale (NULL iff Lq == 0);
 *              FP32 [T, H] with MLA_PROLOG_QUANT_PER_HEAD
 * One run at a time per handle (the workspace is shared): use one handle per
 * concurrent stream.  Inputs and outputs must not overlap.
 * Errors: INVALID_ARG, CUDA.
 */
int mla_prolog_run(mla_prolog_t h,
                   const void* x, const void* gamma, const void* W_a, const void* W_b,
                   const int32_t* positions, const float* cos_sin,
                   void* out_k, void* out_v, void* out_kpe,
                   int8_t* out_q_int8, float* out_scale,
                   void* stream);

/*
 * mla_prolog_run() plus the write of the MLA latent KV cache.  The
 * DeepSeek-V3.2-Exp PyPTO article (section 2.3 and its step 2) caches the
 * prolog's results in the KV cache with a ScatterUpdate; the cache layout is
 * not printed, and this library reads it as one BF16 row per slot:
 *   kv_cache      BF16 [num_slots, Lkv + R], 16-byte aligned (device)
 *   slot_mapping  int32 [T] (device): token t writes row slot_mapping[t] =
 *                 [normed c_kv (Lkv, the expansion's input) | k_pe_rot (R)]
 * A negative slot marks a padding token: nothing is written.  A slot
 * >= num_slots is skipped and sets MLA_STATUS_SLOT_RANGE.  A token whose
 * position is out of range writes a zero row (as for its other outputs).
 * Two tokens with the same slot leave one of their rows (which one is not
 * specified).  Every other output and argument is that of mla_prolog_run().
 * Errors: INVALID_ARG (null cache or slot_mapping, misalignment,
 * num_slots < 0), CUDA.
 */
int mla_prolog_run_cached(mla_prolog_t h,
                          const void* x, const void* gamma, const void* W_a, const void* W_b,
                          const int32_t* positions, const float* cos_sin,
                          void* out_k, void* out_v, void* out_kpe,
                          int8_t* out_q_int8, float* out_scale,
                          const int32_t* slot_mapping, void* kv_cache, int64_t num_slots,
                          void* stream);

/*
 * W8A8 handles only: loads the INT8 weights into the handle (enqueued on
 * `stream`; the inputs may be freed once the stream has passed this call).
 *   W_a      int8 [Lq + Lkv + R, D]   codes, the layout of the BF16 W_a
 *   W_b      int8                     codes, the layout of the BF16 W_b
 *   w_scale  FP32 [Lq + Lkv + R + (Lq > 0 ? H(Dn+R) : 0) + H(Dn+Dv)]
 *            one scale per weight row: W_a rows, then W_q_b rows, then
 *            W_kv_b rows
 * All device pointers; W_a and W_b 16-byte aligned.  The handle keeps the
 * codes as BF16 integers (2 bytes per weight; see MLA_PROLOG_W8A8).
 * Errors: INVALID_ARG (not a W8A8 handle, null or misaligned), CUDA.
 */
int mla_prolog_load_w8a8(mla_prolog_t h, const int8_t* W_a, const int8_t* W_b, const float* w_scale, void* stream);

/* Frees the workspace and the handle.  NULL-safe.  Synchronises the device. */
int mla_prolog_destroy(mla_prolog_t h);

/*
 * Synchronises `stream`, copies the handle's device status word (an OR of
 * MLA_STATUS_* bits accumulated since the last call) into *status, and clears
 * it (after a wait timeout it also resets the decode kernel's grid barrier).
 * Errors: INVALID_ARG, CUDA.
 */
int mla_prolog_device_status(mla_prolog_t h, void* stream, int32_t* status);

/* Static English text for a return code (never NULL). */
const char* mla_prolog_strerror(int code);

/* Text of the last CUDA error seen by this library in the calling thread ("" if none). */
const char* mla_prolog_last_cuda_error(void);

/*
 * Per-token symmetric INT8 quantisation of `rows` FP32 rows of `row_len`
 * values (device): codes int8 [rows, row_len], scale FP32 [rows].  The same
 * quantisation step the q path of mla_prolog_run() ends with (DeepSeek-V3.2-Exp
 * PyPTO article, section 3.1 PrologQuant): amax = max|y|, inv = 127/amax,
 * code = clamp(rint_half_even(y * inv), +-127), scale = amax/127; a zero row
 * gives codes 0 and scale 0.  Every FP32 operation is correctly rounded, so
 * the result is bit-exact for a given input.  `y` 16-byte aligned, codes
 * 4-byte aligned.  Errors: INVALID_ARG (row_len not a multiple of 4, bad
 * pointers), CUDA.
 */
int mla_prolog_quant_rows(const float* y, int32_t rows, int32_t row_len,
                          int8_t* codes, float* scale, void* stream);

/*
 * Sets the limit, in nanoseconds, after which an in-kernel wait of this
 * handle gives up (default 1e9 = 1 s).  A wait that gives up sets
 * MLA_STATUS_WAIT_TIMEOUT and lets its CTA finish cleanly.
 */
int mla_prolog_set_wait_timeout(mla_prolog_t h, uint64_t timeout_ns);

/*
 * Self-test of the bounded-wait path: launches one CTA that waits on a
 * barrier phase that nothing completes, for at most `timeout_ns`.  Expected
 * result: MLA_STATUS_WAIT_TIMEOUT in the handle's status word, a clean return
 * and a usable context.  No fault, trap or hang is involved.
 */
int mla_prolog_selftest_wait_timeout(mla_prolog_t h, uint64_t timeout_ns, void* stream);

/*
 * Profiling hook.  With n_events >= mla_prolog_kernel_count(h) + 1 CUDA
 * events (cudaEvent_t passed as void*), each later run records events[0]
 * before its first kernel and events[i + 1] after its kernel i, on the run's
 * stream; n_events = 0 turns the hook off.  Events stay owned by the caller.
 */
int mla_prolog_set_timing_events(mla_prolog_t h, void* const* events, int32_t n_events);

/* Number of kernels one run launches (with the current tuning), and the
 * name of kernel i in launch order. */
int32_t mla_prolog_kernel_count(mla_prolog_t h);
const char* mla_prolog_kernel_name(mla_prolog_t h, int32_t i);

/*
 * Copies an intermediate of the handle's most recent run out of its device
 * workspace into `dst` (device memory, `bytes` long), enqueued on `stream`.
 * For checking each step of the path on its own:
 *   MLA_TAP_NORMED  BF16 [T, Lq + Lkv]  normed c_q | c_kv (after gamma and the
 *                                       BF16 cast: input of the expansion)
 *   MLA_TAP_Q       FP32 [T, H(Dn+R)]   q after its projection and RoPE (the
 *                                       quantisation input; Lq > 0 and no
 *                                       MLA_PROLOG_QUANT_PER_HEAD)
 *   MLA_TAP_AMAX    FP32 [T]            max |q| per token (as MLA_TAP_Q)
 * Errors: INVALID_ARG (unknown tap, tap absent, size mismatch), CUDA.
 */
#define MLA_TAP_NORMED 1
#define MLA_TAP_Q      2
#define MLA_TAP_AMAX   3
/* W8A8 handles (with them MLA_TAP_NORMED holds the normed rows' INT8 codes,
 * as BF16 integers):
 *   MLA_TAP_X_CODES    BF16 [T, D]  x's per-token codes, as BF16 integers
 *   MLA_TAP_X_SCALE    FP32 [T]     x's per-token scales
 *   MLA_TAP_NORM_SCALE FP32 [T, 2]  scales of the normed (c_q, c_kv) codes */
#define MLA_TAP_X_CODES    4
#define MLA_TAP_X_SCALE    5
#define MLA_TAP_NORM_SCALE 6
int mla_prolog_copy_tap(mla_prolog_t h, int32_t which, void* dst, size_t bytes, void* stream);

/*
 * Tuning knobs; create() picks the defaults.
 *   MLA_TUNE_COMPRESS_GROUP  K blocks of 64 summed by one tensor-core
 *                            accumulation chain of the compression projection
 *                            before the chain is drained into exactly
 *                            compensated FP32 registers (1 .. 64).  Shorter
 *                            chains round closer to the exact sum.
 * Errors: INVALID_ARG (unknown key or value out of range).
 */
#define MLA_TUNE_COMPRESS_GROUP 1
/*   MLA_TUNE_COMPRESS_COMPENSATED  1: the drained chains are summed with
 *                            error-free TwoSum; 0: with plain FP32 adds.   */
#define MLA_TUNE_COMPRESS_COMPENSATED 2
/*   MLA_TUNE_DECODE_FUSED    1: batches of at most 128 tokens run as one
 *                            cooperative kernel (where the dims and the
 *                            device allow it); 0 (the default): as four
 *                            kernels.  INVALID_ARG when 1 is not available. */
#define MLA_TUNE_DECODE_FUSED 3
/*   MLA_TUNE_CLUSTER_NORM    1: the compression projection and the norm run
 *                            in one thread-block cluster of up to 16 CTAs
 *                            that sum the split-K partials in distributed
 *                            shared memory, then the expansion kernel
 *                            (available for batches of at most 128 tokens
 *                            with small compression weights, e.g. the
 *                            DeepSeek-V2-Lite KV prolog; the default only for
 *                            tiny problems, where it measured faster); 0:
 *                            split-K compression over every SM, norm kernel,
 *                            expansion.  INVALID_ARG when 1 is not available.
 *                            Setting 1 turns MLA_TUNE_DECODE_FUSED off, and
 *                            the reverse. */
#define MLA_TUNE_CLUSTER_NORM 4
/*   MLA_TUNE_PAIR_EXPAND     1 (the default for prefill batches with a q
 *                            path, where it measured faster): the
 *                            expansion projections run on CTA pairs
 *                            (tcgen05 cta_group::2, 256-token tiles, each SM
 *                            streaming half of every weight tile); 0: one CTA
 *                            per 128-token tile.  INVALID_ARG when 1 is not
 *                            available (decode batches, or heads wider than
 *                            256 columns). */
#define MLA_TUNE_PAIR_EXPAND 6
/*   MLA_TUNE_PAIR_COMPRESS   1: the compression projection runs on CTA pairs
 *                            (256-token tiles of 256 weight rows, each SM
 *                            streaming half of every weight tile, plain FP32
 *                            sums of the drained chains); 0 (the default,
 *                            measured faster): one CTA per 128-token tile.
 *                            INVALID_ARG when 1 is not available (decode
 *                            batches). */
#define MLA_TUNE_PAIR_COMPRESS 7
/*   MLA_TUNE_TMA_STORE       1 (the default where the dims allow it: nope
 *                            and value widths multiples of 32, and with the
 *                            per-token quant a rope width of 32 or 64): the
 *                            prefill expansion kernels write their kv outputs
 *                            and FP32 q rows through shared memory with bulk
 *                            tensor stores; 0: each thread stores its own
 *                            row.  Same values either way.  INVALID_ARG when
 *                            1 is not available. */
#define MLA_TUNE_TMA_STORE 8
/*   MLA_TUNE_COMPRESS_TILE   prefill batches: the width of the compression
 *                            projection's weight tiles, 128, 144, 192 or
 *                            256 columns.  Wider tiles bring fewer operand
 *                            bytes per tensor-core FLOP into each SM; the
 *                            144-, 192- and 256-wide tiles sum the drained
 *                            chains with plain FP32 adds
 *                            (MLA_TUNE_COMPRESS_COMPENSATED applies to
 *                            128-wide tiles).  Default: the wide
 *                            tile that needs no split-K and brings the
 *                            busiest SM the fewest operand bytes, else 128.
 *                            INVALID_ARG for decode batches (and the
 *                            cluster or cooperative paths) or another
 *                            width. */
#define MLA_TUNE_COMPRESS_TILE 9
/*   MLA_TUNE_L2_FETCH        decode batches: 1: once the compression kernel
 *                            has issued its last operand loads it asks L2 to
 *                            fetch the expansion weights W_b from HBM while
 *                            it drains and the norm runs, so the expansion
 *                            reads them from L2; 0 (the default, measured
 *                            faster): the expansion streams them from HBM.
 *                            INVALID_ARG for prefill batches. */
#define MLA_TUNE_L2_FETCH 10
/*   MLA_TUNE_Q_WIDE          prefill on CTA pairs with the per-token q path
 *                            (rope width 64, nope width a multiple of 64, no
 *                            per-head norm or quant): 1 (the default there,
 *                            measured faster): q tiles of 256 columns that
 *                            run across head boundaries (fewer operand bytes
 *                            per tensor-core FLOP than one 192-column head
 *                            per tile); 0: one head per tile.  Same values either way (the tensor
 *                            stores must be on for 1 to take effect).
 *                            INVALID_ARG when 1 is not available. */
#define MLA_TUNE_Q_WIDE 11
/*   MLA_TUNE_KV_RESIDENT     prefill on CTA pairs with kv tiles of 256 columns
 *                            and Lkv <= 512: 1 (the default when there are at
 *                            least as many groups of 8 kv tiles x 256-token
 *                            tiles as SMs, where it measured faster): the kv
 *                            tiles run on their own kernel, which keeps a
 *                            256-token tile's normed c_kv rows in shared
 *                            memory and streams only the weights for a group
 *                            of 8 kv tiles; 0: the kv
 *                            tiles share the pair expansion kernel with the q
 *                            tiles.  Same values either way (the tensor
 *                            stores must be on for 1 to take effect).
 *                            INVALID_ARG when 1 is not available. */
#define MLA_TUNE_KV_RESIDENT 12
/*   MLA_TUNE_QUANT_OVERLAP   with the kv-resident kernel and the per-token
 *                            quant: 1 (the default): the quant kernel, which
 *                            needs only the q tiles, runs on an internal
 *                            low-priority stream beside the kv kernel (forked
 *                            from and joined back to the caller's stream
 *                            with events, which stream capture follows);
 *                            0: after it on the caller's stream.  Not used
 *                            while the timing hook is armed.  INVALID_ARG
 *                            when 1 is not available. */
#define MLA_TUNE_QUANT_OVERLAP 13
/*   MLA_TUNE_KV_GROUP        kv tiles per super-job of the kv-resident kernel
 *                            (1 .. the kv tile count; the default minimises
 *                            the operand bytes of the busiest CTA pair).
 *                            INVALID_ARG when that kernel is not available. */
#define MLA_TUNE_KV_GROUP 14
/*   MLA_TUNE_L2_POLICY       L2 eviction priorities of the projections' bulk
 *                            copies, an OR of: 1 the weight tiles load with
 *                            the evict-last priority, 2 the activation tiles
 *                            load with the evict-last priority, 4 the output
 *                            tensor stores of the expansions write with the
 *                            evict-first priority; 0: no priority hint on
 *                            any copy.  Default: 1 for prefill batches (the
 *                            kv expansion reads ~20 % fewer DRAM bytes), 0
 *                            for decode batches.  Values are unchanged; only
 *                            which lines L2 keeps.  INVALID_ARG outside
 *                            0..7. */
#define MLA_TUNE_L2_POLICY 15
/*   MLA_TUNE_KV_HALVES       when the kv jobs leave a last round shorter
 *                            than half the grid: 1 (the default there):
 *                            those jobs run as two half jobs each on twice
 *                            as many CTAs -- half tiles (bn_kv / 2 columns)
 *                            for a KV-only prefill on one CTA per tile, half
 *                            groups of kv tiles on the kv-resident kernel;
 *                            0: whole.  Same values either way.  INVALID_ARG
 *                            when not available. */
#define MLA_TUNE_KV_HALVES 16
int mla_prolog_set_tuning(mla_prolog_t h, int32_t key, int32_t value);

/*
 * mla_prolog_run() without a handle and without allocating device memory.
 * The pages have no counterpart of this entry point: it exists for callers
 * that cannot call cudaMalloc, such as a plugin inside an inference runtime
 * that reserves the whole device memory pool up front, or a latency-critical
 * caller that cannot accept cudaMalloc's implicit synchronisation.
 *
 * Arguments and outputs are those of mla_prolog_run(), with the dims passed
 * in directly.  The scratch that a handle keeps in its workspace is instead a
 * static 32 MiB device array inside the library (each GPU that loads the
 * library holds it until the process exits); dims whose workspace would not
 * fit (split-K partials + normed rows + FP32 q rows + amax) are rejected with
 * MLA_ERR_UNSUPPORTED_DIMS before anything runs.  On a 152-SM GB300 that
 * admits the V2-Lite KV shape up to about 10 000 tokens (decode and prefill
 * schedules) and the V3 shape with its q path up to about 246 tokens; the
 * exact limit follows from the schedule mla_prolog_plan() reports.  The
 * kernels are a subset of mla_prolog_run()'s (no cluster, cooperative or
 * CTA-pair kernels), so results agree with it within the parity tolerances,
 * and bit for bit where both launch the same kernels.
 * `status` (device int32, may be NULL) receives the run's device status word
 * (MLA_STATUS_* bits).  Of the dims flags only MLA_PROLOG_QUANT_Q is taken
 * (the variant flags give MLA_ERR_INVALID_ARG).
 *
 * The first call on a device looks up the array's device address and sets
 * the kernels' attributes; make that first call before any stream capture.
 * All calls on one device share the array and it keeps the previous call's
 * contents (this entry clears what must start at zero), so calls whose
 * kernels overlap on one GPU -- e.g. on two streams -- race on it: order them
 * on one stream.  No cudaMalloc, cudaFree or allocating library routine is
 * called.  Errors: INVALID_ARG, UNSUPPORTED_DIMS, DEVICE, CUDA.
 */
int mla_prolog_run_noalloc(const mla_prolog_dims* dims,
                           const void* x, const void* gamma, const void* W_a, const void* W_b,
                           const int32_t* positions, const float* cos_sin,
                           void* out_k, void* out_v, void* out_kpe,
                           int8_t* out_q_int8, float* out_scale, int32_t* status,
                           void* stream);

/* Bytes of device workspace the handle holds. */
int mla_prolog_workspace_bytes(mla_prolog_t h, size_t* bytes);

/*
 * Schedule chosen at create time, for reports: tile widths and split-K of the
 * two projections (with the cluster compression: the column-group width and
 * the K splits of the cluster).  Any pointer may be NULL.
 */
int mla_prolog_schedule(mla_prolog_t h, int32_t* bn_a, int32_t* splits_a,
                        int32_t* bn_kv, int32_t* bn_q);

/*
 * The schedule mla_prolog_create() chooses for `dims` on a device with `sms`
 * SMs, computed on the host without touching the GPU (the rules in one place,
 * for tests and reports).  decode: 1 for the decode schedule (at most two
 * 128-token tiles); bn_a, splits_a, group_a: the compression's weight-tile
 * width (prefill: the default of MLA_TUNE_COMPRESS_TILE), split-K factor and
 * accumulation-chain length in K blocks of 64; compress_jobs: its jobs (token
 * tiles x weight tiles x splits); busiest_bytes: the operand bytes (token rows
 * + weight rows, 128 bytes per row per K block) that the busiest CTA streams
 * in the compression; bn_kv: the expansion's kv tile width; kv_halves: for
 * a KV-only prefill, the last-round expansion jobs that run as two half
 * tiles each (MLA_TUNE_KV_HALVES; 0: none).
 * Errors: INVALID_ARG (a NULL pointer, sms < 1), UNSUPPORTED_DIMS as
 * mla_prolog_create().
 */
typedef struct mla_prolog_plan_info {
    int32_t decode, bn_a, splits_a, group_a, compress_jobs, bn_kv;
    int32_t kv_halves;
    int64_t busiest_bytes;
} mla_prolog_plan_info;
int mla_prolog_plan(const mla_prolog_dims* dims, int32_t sms, mla_prolog_plan_info* out);

/*
 * Longest-processing-time assignment of n jobs of the given costs to `groups`
 * workers, the way the kernels' balanced job tables are built: jobs by
 * decreasing cost (ties by index), each to the least-loaded worker (the lowest
 * index on a tie).  table (groups + 1 + n int32s, may be NULL): groups + 1
 * start offsets, then the job indices of worker 0, worker 1, ...; *busiest
 * (may be NULL): the largest worker load.  Host only.
 * Errors: INVALID_ARG (n < 0, groups < 1, cost NULL with n > 0, a negative
 * cost).
 */
int mla_prolog_lpt(const int64_t* cost, int32_t n, int32_t groups, int32_t* table, int64_t* busiest);

#ifdef __cplusplus
}
#endif

#endif /* MLA_PROLOG_H_ */
