/*
 * lora_gemm.h - C ABI of the GB300 (sm_103a) batched multi-adapter LoRA branch.
 *
 * The library computes, for a batch of T tokens where token t carries an adapter
 * slot id slot_ids[t] (-1 = no adapter):
 *
 *     y[t, o_i + m] += scale_s * sum_j ( sum_c x[t, c] * A_s,i[j, c] ) * B_s,i[m, j]
 *
 * for s = slot_ids[t], every output slice i and column m < d_i.  This is the
 * unmerged LoRA side branch h = W0 x + (alpha/r) B A x (llama.cpp LoRA adapter
 * page, section "why the low-rank increment can be added afterwards"; vLLM book
 * ch. 16, section 16.1.3, Y = xW + s (xA)B), batched over tokens that use
 * different adapters (vLLM book ch. 16, section 16.4.2, token_lora_mapping with
 * -1 = no LoRA), with packed projections (QKV, gate_up) as output slices
 * (vLLM LoRA deep-dive page, section 5.4 packed modules).
 *
 * Layouts (PEFT orientation, vLLM LoRA deep-dive page section 4: lora_a is
 * (r, k), lora_b is (d, r)); all matrices row-major, bf16 unless stated:
 *   x        [T, ldx]       input rows, first k columns used
 *   y        [T, ldy]       output rows, first d = slice_offsets[n] columns used
 *   A_s,i    [r_s, k]       contiguous, one per slot s and slice i
 *   B_s,i    [d_i, r_s]     contiguous, one per slot s and slice i
 *   ws       float32        caller-owned workspace, see lora_workspace_bytes()
 *
 * Conventions for every call:
 *   - Asynchronous on the caller's stream.  The library allocates nothing,
 *     never synchronises the device and never reads device memory back, so a
 *     step of calls can be captured in a CUDA graph.  (lora_set_slot_table
 *     copies from host memory; see its notes.)
 *   - Host-side argument checks return a lora_status_t before anything is
 *     enqueued.  Errors found in device data (a slot id outside [-1, S), a
 *     timed-out wait) are written to the caller's device word `err` as the first
 *     error code (compare-and-swap from 0); the library never clears it.  Zero
 *     it before a step and read it after synchronising.
 *   - Device pointers to bf16 data and leading dimensions must be 16-byte
 *     aligned / multiples of 8 elements; k and every slice width must be
 *     multiples of 8.  Ranks are 0 or multiples of 8 up to LORA_MAX_RANK
 *     (TensorRT-LLM pads ranks below 8 for the same alignment reason: TensorRT-LLM
 *     LoRA serving page, "path 1: CUDA Graph mode", min_kn).  A rank-0 slot is an
 *     empty slot; its pointers may be null and it contributes nothing
 *     (TensorRT-LLM's base sentinel slot has rank 0: same page, "adapter pool").
 *   - Nothing is thread-safe beyond what the stream order gives: calls that run
 *     concurrently on different streams must not share ws, err or y.
 */
#ifndef LORA_GEMM_H
#define LORA_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; a null stream is the legacy default stream. */
typedef struct CUstream_st *lora_stream_t;

#define LORA_ABI_VERSION 1
#define LORA_MAX_SLICES 4
#define LORA_MAX_RANK 512
#define LORA_MAX_SLOTS 1024

typedef enum {
    LORA_OK = 0,
    LORA_ERR_INVALID_ARG = 1,   /* null pointer with nonzero size, negative size, bad shape */
    LORA_ERR_ALIGNMENT = 2,     /* pointer / leading dimension / width not 16-byte aligned */
    LORA_ERR_RANK = 3,          /* rank not 0 or a multiple of 8, or above r_max / LORA_MAX_RANK */
    LORA_ERR_SLOT_RANGE = 4,    /* device: a slot id outside [-1, S) (token left unchanged) */
    LORA_ERR_NULL_WEIGHT = 5,   /* a slot with rank > 0 has a null A or B pointer */
    LORA_ERR_WORKSPACE = 6,     /* workspace missing or smaller than lora_workspace_bytes() */
    LORA_ERR_TIMEOUT = 7,       /* device: a bounded wait between thread blocks gave up */
    LORA_ERR_CUDA = 8,          /* a CUDA runtime call failed (e.g. launch) */
    LORA_ERR_UNSUPPORTED = 9    /* no kernel for this device or configuration */
} lora_status_t;

/* Kernel path of lora_apply_ex. */
typedef enum {
    LORA_PATH_AUTO = 0,          /* the prefill kernels if max_seg_hint > LORA_DECODE_MAX_SEG and
                                    r_max <= 64; otherwise, above 64 tokens, the warp-streaming
                                    decode kernels (LORA_PATH_DECODE_DIRECT) when they take the
                                    shape, else the fused decode path when it does; at 64 tokens
                                    and fewer LORA_PATH_DECODE_CLUSTER when it takes the shape;
                                    otherwise the split decode kernels */
    LORA_PATH_DECODE_FUSED = 1,  /* one launch: shrink, per-(slot, slice) wait, expand, on warp-level
                                    MMA; needs T <= 2048, r_max <= 128 and k % 16 == 0 (else
                                    LORA_ERR_UNSUPPORTED) */
    LORA_PATH_DECODE_SPLIT = 2,  /* two launches: shrink then expand (programmatic dependent launch);
                                    any rank up to LORA_MAX_RANK; sums reduced in a fixed order, so
                                    results are bit-identical over runs (the deterministic choice:
                                    the other decode paths add split-K partials with fp32 atomics
                                    whose order varies) */
    LORA_PATH_PREFILL = 3,       /* two launches: tcgen05/TMEM tensor-core shrink (split-K over a
                                    thread-block cluster) and expand, on 128-token tiles of
                                    one slot's segment; needs r_max <= 64
                                    (else LORA_ERR_UNSUPPORTED) */
    LORA_PATH_DECODE_TC = 4,     /* retired (slower than LORA_PATH_DECODE_DIRECT on every measured
                                    shape): always LORA_ERR_UNSUPPORTED */
    LORA_PATH_DECODE_STREAM = 5, /* retired, as LORA_PATH_DECODE_TC: always LORA_ERR_UNSUPPORTED */
    LORA_PATH_DECODE_DIRECT = 6, /* two launches on warp-level MMA in which every warp streams its
                                    own byte-balanced share through a private cp.async ring (no
                                    barriers between warps): a split-K shrink adding into an fp32
                                    accumulator, then an expand launched as its programmatic
                                    dependent; needs T <= 2048, r_max <= 64, S <= 512 and
                                    S * n_slices <= 512 (else LORA_ERR_UNSUPPORTED) */
    LORA_PATH_DECODE_DIRECT_FP8 = 7, /* LORA_PATH_DECODE_DIRECT with FP8 adapters (TensorRT-LLM LoRA
                                    serving page, "第五步:FP8 特判" and the input-dtype check of the
                                    forward pass): every A and B pointer of the slot table
                                    addresses float8_e4m3fn codes in the same row-major layouts
                                    (A_s,i [r][k], B_s,i [d_i][r], one byte each); x and y stay
                                    bf16.  x is clamped to +-448 and rounded to e4m3 (nearest,
                                    ties to even) inside the shrink, whose products are exact
                                    and summed in fp32; the sums enter the expand as two bf16
                                    parts (hi and the remainder, about 2^-17 of each sum, no
                                    overflow) against B converted exactly to bf16, and
                                    y = bf16(y + s * acc) as for bf16 adapters.
                                    Scale B at load time with lora_premultiply on its bf16
                                    values, then clamp and round to e4m3.  Same limits as
                                    LORA_PATH_DECODE_DIRECT plus k % 16 == 0; never chosen by
                                    LORA_PATH_AUTO, whose table is bf16 */
    LORA_PATH_DECODE_TMA = 8     /* one persistent kernel per call (one CTA per SM): the adapter
                                    tiles arrive as TMA boxes through the tensor maps of a table
                                    set with lora_set_slot_table_tma, x and y rows are gathered
                                    beside them, and the expand of a slot starts in the same
                                    kernel once a per-slot counter says its shrink sums are
                                    complete.  Launched as a programmatic dependent of the
                                    previous kernel on the stream: it loads adapter weights (and
                                    its plan) before that kernel has finished, so neither may be
                                    written by the kernel directly before it.  Needs r_max <= 64,
                                    n_slices * r_max <= 192 and k % 64 == 0 (else
                                    LORA_ERR_UNSUPPORTED); every CTA of the call must be resident
                                    at once (a slot whose sums are not complete within 200 ms is
                                    reported as LORA_ERR_TIMEOUT).  Without a plan, lora_apply_ex
                                    builds one in the workspace first (two launches); with
                                    lora_build_plan(s) / lora_apply_plan it is one launch per call.
                                    Never chosen by LORA_PATH_AUTO, whose table may lack the
                                    tensor maps */,
    LORA_PATH_DECODE_CLUSTER = 9 /* small batches in one launch: one thread-block cluster of 16
                                    CTAs per slot.  Each CTA multiplies the slot's x rows by A
                                    over 1/16 of k (warp MMA, fp32), the partial sums meet in
                                    distributed shared memory (added in CTA-rank order), and
                                    each CTA applies B to 1/16 of every slice's columns, y read and
                                    written once.  Tokens are taken 16 at a time.  Launched as a
                                    programmatic dependent of the previous kernel on the stream:
                                    it reads the slot table, the index and the adapter weights
                                    before that kernel has finished (x and y after), so none of
                                    those may be written by the kernel directly before it
                                    (lora_build_index and the plan builders never start a
                                    dependent early).  Needs r_max <= 256 and a CTA's tiles
                                    (A and x over its share of k, B and y over its share of the
                                    columns) within 227 KB of shared memory (else
                                    LORA_ERR_UNSUPPORTED).  Uses no workspace */
} lora_path_t;

#define LORA_DECODE_MAX_SEG 256

/*
 * Shape of one packed projection, passed by the host to every branch call.
 *   S              number of resident slots in the slot table (1..LORA_MAX_SLOTS)
 *   r_max          upper bound on every slot's rank (multiple of 8, <= LORA_MAX_RANK);
 *                  it sets the workspace row stride
 *   k              input width (multiple of 8)
 *   n_slices       number of output slices (1..LORA_MAX_SLICES)
 *   slice_offsets  slice i owns y columns [slice_offsets[i], slice_offsets[i+1]);
 *                  slice_offsets[0] = 0, strictly increasing, widths multiples of 8
 */
typedef struct {
    int32_t S;
    int32_t r_max;
    int32_t k;
    int32_t n_slices;
    int32_t slice_offsets[LORA_MAX_SLICES + 1];
} lora_shape_t;

/* Library ABI version (LORA_ABI_VERSION of the build). */
int32_t lora_abi_version(void);

/* Human-readable name of a status code; never null. */
const char *lora_status_string(lora_status_t status);

/*
 * Per-slot scale rule (host).  llama.cpp's get_scale (llama.cpp LoRA adapter
 * page, section "where the scale is applied"): adapter_scale * alpha / rank, or
 * adapter_scale alone when alpha == 0 (a file without alpha).  With rslora != 0
 * the rank enters as sqrt(rank) (vLLM LoRA deep-dive page, section 1, rsLoRA).
 * Returns adapter_scale for rank <= 0.
 */
double lora_scale(double alpha, int32_t rank, int32_t rslora, double adapter_scale);

/*
 * Fold a scale into B on load, in place on the device: w[e] = bf16(scale * w[e])
 * with the product in fp32 and round-to-nearest-even (vLLM LoRA deep-dive page,
 * section 1, LoRALayerWeights.optimize(): lora_b *= scaling, scaling = 1).  The
 * slot is then used with scale 1.  w: device bf16, n elements, 2-byte aligned.
 */
lora_status_t lora_premultiply(void *w, int64_t n, float scale, lora_stream_t stream);

/*
 * The same for an FP8 B (TensorRT-LLM LoRA serving page, "第五步:FP8 特判": FP8 has
 * no scalar multiply, so the scale is applied in bf16 and the result clamped back
 * into the FP8 range): w[e] = e4m3(clamp(bf16(value(w[e]) * scale), -448, 448)),
 * the product exact (fp64) and rounded once to bf16, then rounded to the nearest
 * e4m3 code with ties to even; NaN codes become 0x7F.  w: device float8_e4m3fn
 * codes, n bytes, any alignment.  For LORA_PATH_DECODE_DIRECT_FP8 slots.
 */
lora_status_t lora_premultiply_e4m3(void *w, int64_t n, float scale, lora_stream_t stream);

/*
 * Slot table: per slot s its rank r_s, runtime scale s_s and, per slice i, the
 * device addresses of A_s,i and B_s,i as 64-bit integers (TensorRT-LLM LoRA
 * serving page, "a decode batch's route", step 3: one row per slot, int64
 * pointers, refreshed only when slot ownership changes).  The packed table lives
 * in caller-owned device memory of lora_slot_table_bytes(S, n_slices) bytes
 * (16-byte aligned).  Ranks of one slot are shared by all its slices.
 */
size_t lora_slot_table_bytes(int32_t S, int32_t n_slices);

/*
 * Validate the host arrays and pack them into host_buf (lora_slot_table_bytes
 * bytes).  ranks[S], scales[S], A_ptrs[S * n_slices] and B_ptrs[S * n_slices]
 * are host arrays; entry s * n_slices + i is slot s, slice i.  Checks: 1 <= S <=
 * LORA_MAX_SLOTS, 1 <= n_slices <= LORA_MAX_SLICES, r_max a multiple of 8 in
 * [8, LORA_MAX_RANK], every rank 0 or a multiple of 8 <= r_max (LORA_ERR_RANK),
 * every pointer of a rank>0 slot non-null (LORA_ERR_NULL_WEIGHT) and 16-byte
 * aligned (LORA_ERR_ALIGNMENT).  Pure host code; usable without a GPU.
 */
lora_status_t lora_pack_slot_table(void *host_buf, int32_t S, int32_t n_slices, int32_t r_max,
                                   const int32_t *ranks, const float *scales,
                                   const uint64_t *A_ptrs, const uint64_t *B_ptrs);

/*
 * lora_pack_slot_table into host_staging, then an asynchronous host-to-device
 * copy of the packed bytes into dev_table on `stream`.  host_staging must stay
 * unchanged until the copy has executed (pinned memory recommended; with
 * pageable memory the CUDA runtime stages the bytes before returning).  Call it
 * only when the slot-to-adapter assignment changes.
 */
lora_status_t lora_set_slot_table(void *dev_table, void *host_staging, int32_t S, int32_t n_slices,
                                  int32_t r_max, const int32_t *ranks, const float *scales,
                                  const uint64_t *A_ptrs, const uint64_t *B_ptrs,
                                  lora_stream_t stream);

/*
 * Slot table with TMA tensor maps, for LORA_PATH_DECODE_TMA: the table of
 * lora_set_slot_table (every path accepts it), aligned to 128 bytes, then a
 * 128-byte block header, S int32 slot flags (padded to 128 bytes) and eight
 * 128-byte tensor maps per slot: for a slot s with rank r_s > 0, tensor maps
 * of A (bf16, 128-byte swizzle, read in k-blocks of 64 columns) and of every
 * B_s,i as [d_i][r_s], encoded on the host with the driver's
 * cuTensorMapEncodeTiled (no allocation; the CUDA runtime must be able to
 * reach the driver).  When the slot's A slices are one packed block
 * (A_ptrs[s n + i] = A_ptrs[s n] + i r_s k 2 bytes for every i, n r_s <= 256)
 * the A maps cover all n r_s rows and a stage of k-blocks takes one to four
 * copies; otherwise each slice has its own map.  The maps are tied to this
 * shape's k and slice widths (a plan built with another shape is refused on
 * the device).
 *
 * lora_slot_table_tma_bytes: the table's size for S slots and this shape (0 for
 * a bad shape or S outside [1, LORA_MAX_SLOTS]).
 *
 * lora_set_slot_table_tma: checks as lora_pack_slot_table (with S and n_slices
 * from the shape), dev_table 128-byte aligned (LORA_ERR_ALIGNMENT), then packs
 * host_staging (lora_slot_table_tma_bytes bytes) and copies it to dev_table on
 * `stream` as lora_set_slot_table does.  LORA_ERR_UNSUPPORTED if the driver's
 * encoder is unavailable or rejects a map (e.g. a rank above 256).
 */
size_t lora_slot_table_tma_bytes(int32_t S, const lora_shape_t *shape);
lora_status_t lora_set_slot_table_tma(void *dev_table, void *host_staging, const lora_shape_t *shape,
                                      const int32_t *ranks, const float *scales, const uint64_t *A_ptrs,
                                      const uint64_t *B_ptrs, lora_stream_t stream);

/*
 * Per-step token index (TensorRT-LLM LoRA serving page, "a decode batch's
 * route", steps 2 and 4: sorted ids, bincount, cumsum with a final total; vLLM
 * book ch. 16, section 16.4.3, the LoRAKernelMeta tensors).  Device arrays:
 *   slot_ids    int32 [T]      input; -1 = no adapter
 *   sorted_ids  int32 [T]      tokens ordered by key = slot (no-adapter and
 *                              out-of-range ids keyed S, i.e. last), ties in
 *                              ascending token index (a stable sort)
 *   seg_offsets int32 [S + 2]  seg_offsets[b] = number of tokens with key < b;
 *                              slot s owns sorted positions [seg_offsets[s],
 *                              seg_offsets[s+1]); seg_offsets[S+1] = T
 *   active      int32 [S + 1]  active[0] = number of slots with at least one
 *                              token and rank > 0; active[1..] those slots, ascending
 *   err         int32 [1]      first error; LORA_ERR_SLOT_RANGE for ids outside [-1, S)
 * Ranks come from dev_table (any module's table: ranks are per slot).  Built once
 * per step and shared by every projection of the step.  T may be 0.
 */
lora_status_t lora_build_index(const int32_t *slot_ids, int32_t T, int32_t S, const void *dev_table,
                               int32_t *sorted_ids, int32_t *seg_offsets, int32_t *active,
                               int32_t *err, lora_stream_t stream);

/*
 * Token index for speculative decoding, where every sequence carries the same
 * number of tokens (TensorRT-LLM LoRA serving page, section "一次 decode 批次的
 * 路由": with tokens_per_seq > 1 the sequence order is expanded to the token
 * order as sorted * tokens_per_seq + arange(tokens_per_seq)).
 *   seq_slot_ids   device int32[n_seq], the slot of each sequence (-1: none)
 *   tokens_per_seq >= 1; sequence b owns tokens b*tokens_per_seq ..
 *                  b*tokens_per_seq + tokens_per_seq - 1 of x and y (T =
 *                  n_seq * tokens_per_seq tokens, at most INT32_MAX)
 * The outputs are exactly lora_build_index's for the token-level slot ids
 * (each sequence's slot repeated tokens_per_seq times): sorted_ids int32[T],
 * seg_offsets int32[S + 2] (seg_offsets[S + 1] = T), active int32[S + 1],
 * the same error reporting.  One launch; nothing is allocated.  Host checks:
 * LORA_ERR_INVALID_ARG for n_seq < 0, tokens_per_seq < 1, T above INT32_MAX,
 * S outside [1, LORA_MAX_SLOTS] or missing pointers, LORA_ERR_ALIGNMENT for an
 * unaligned table.
 */
lora_status_t lora_build_index_seq(const int32_t *seq_slot_ids, int32_t n_seq, int32_t tokens_per_seq, int32_t S,
                                   const void *dev_table, int32_t *sorted_ids, int32_t *seg_offsets,
                                   int32_t *active, int32_t *err, lora_stream_t stream);

/*
 * Workspace size for T tokens of a projection, in order: a control block of
 * per-slot counters and a call counter; the fp32 shrink output
 * xa[n_slices][T][r_max] (row t = token t); the fused decode kernel's fp32
 * accumulator (same size); and, when r_max <= 64, the prefill kernels' xa as two
 * bf16 parts hi + lo, each [n_slices][T][RP] in sorted-token order (RP = 16, 32
 * or 64, the rank padded up); then, when r_max <= 128, two more fp32
 * accumulators the size of xa that LORA_PATH_DECODE_DIRECT uses in turn (a call
 * adds into one and clears the other); then, when r_max <= 64,
 * LORA_PATH_DECODE_TMA's two fp32 sum sets (the size of xa, used in turn), its
 * control block (2 S per-slot counters, a call counter and an exit counter) and
 * room for the plan such a call without one builds.  Regions start on 256-byte
 * boundaries, at offsets that depend on T and the shape: use one workspace for
 * one (T, shape) pair.  The whole buffer must be zero before the first call that
 * uses it (e.g. one cudaMemsetAsync), and again after a call whose error word
 * reads LORA_ERR_TIMEOUT.  Otherwise every call leaves what the next call of any
 * path needs: the per-slot counters and the fused accumulator zero, each call
 * counter matching the clear accumulator or sum set of its path.
 */
lora_status_t lora_workspace_bytes(int32_t T, const lora_shape_t *shape, size_t *bytes);

/*
 * Byte offset of xa inside the workspace (xa is float32 [n_slices][T][r_max]);
 * 0 if the shape is invalid.  Host only.
 */
size_t lora_workspace_xa_offset(const lora_shape_t *shape);

/*
 * Shrink: xa[i][t][j] = sum_c x[t, c] * A_s,i[j, c] for tokens t of active slots s,
 * j < r_s, accumulated in fp32 (vLLM book ch. 16, section 16.4.2: lora_shrink
 * writes buffer[num_tokens, r] from lora_a).  Other rows of xa are not written.
 */
lora_status_t lora_shrink(const void *x, int64_t ldx, int32_t T, const lora_shape_t *shape,
                          const void *dev_table, const int32_t *sorted_ids,
                          const int32_t *seg_offsets, const int32_t *active,
                          float *ws, size_t ws_bytes, int32_t *err, lora_stream_t stream);

/*
 * Expand: y[t, o_i + m] = bf16( y[t, o_i + m] + scale_s * sum_j xa[i][t][j] * B_s,i[m, j] ),
 * the sum in fp32, one round-to-nearest-even per element (vLLM book ch. 16,
 * section 16.4.2: lora_expand accumulates into the output slices; TensorRT-LLM
 * LoRA serving page, add_lora_result: output.add_(lora_result)).  Rows of tokens
 * without an active slot are neither read nor written.
 */
lora_status_t lora_expand(const float *ws, size_t ws_bytes, void *y, int64_t ldy, int32_t T,
                          const lora_shape_t *shape, const void *dev_table,
                          const int32_t *sorted_ids, const int32_t *seg_offsets,
                          const int32_t *active, int32_t *err, lora_stream_t stream);

/*
 * Shrink followed by expand on the same workspace: the whole branch for one
 * projection.  max_seg_hint is a host-known upper bound on the tokens of any one
 * slot in this step (T is always valid); LORA_PATH_AUTO picks the decode kernels
 * when it is <= LORA_DECODE_MAX_SEG and the tensor-core prefill kernels
 * otherwise.  When no token has an active slot the kernels exit early on the
 * device (the no-LoRA step).
 */
lora_status_t lora_apply(const void *x, int64_t ldx, void *y, int64_t ldy, int32_t T,
                         const lora_shape_t *shape, const void *dev_table,
                         const int32_t *sorted_ids, const int32_t *seg_offsets,
                         const int32_t *active, int32_t max_seg_hint,
                         float *ws, size_t ws_bytes, int32_t *err, lora_stream_t stream);

/*
 * The path lora_apply takes for this max_seg_hint (and T) in this library
 * version, for r_max <= 64 and k % 16 == 0: requested itself unless it is
 * LORA_PATH_AUTO.  *launches receives the number of kernel launches the path
 * makes per call (may be null).  Host only.
 */
lora_path_t lora_resolve_path(lora_path_t requested, int32_t T, int32_t max_seg_hint, int32_t *launches);

/* lora_apply with an explicit kernel path. */
lora_status_t lora_apply_ex(const void *x, int64_t ldx, void *y, int64_t ldy, int32_t T,
                            const lora_shape_t *shape, const void *dev_table,
                            const int32_t *sorted_ids, const int32_t *seg_offsets,
                            const int32_t *active, int32_t max_seg_hint, lora_path_t path,
                            float *ws, size_t ws_bytes, int32_t *err, lora_stream_t stream);

/*
 * The branch overlapped with the producer of y (TensorRT-LLM LoRA serving page,
 * section "与基座并行:forward_with_base": the LoRA branch runs on an auxiliary
 * stream next to the base projection y = x W0^T and the two join on events).
 * Same arguments and result as lora_apply_ex, plus:
 *   y_ready   a CUDA event (cudaEvent_t) the caller records once y holds its
 *             input values (e.g. after the base GEMM on another stream), or
 *             null when y is already ready on `stream`.
 * On `stream`, the x-only half of the branch (the shrink: reads x, A and the
 * index, writes the workspace) is launched first, then the stream waits for
 * y_ready, then the half that reads and writes y (the expand).  So the shrink
 * runs while the other stream computes y, and y is touched only after it is
 * ready.  The two-kernel decode paths (LORA_PATH_DECODE_DIRECT,
 * LORA_PATH_DECODE_SPLIT, and LORA_PATH_AUTO where it picks them) split this
 * way; on the other paths the stream waits for y_ready before the whole call.
 * The caller joins `stream` back (an event) before using y.  Nothing is
 * allocated; host checks and errors as lora_apply_ex.  The event must stay
 * valid until the call's work has run.
 */
typedef void *lora_event_t;
lora_status_t lora_apply_overlap(const void *x, int64_t ldx, void *y, int64_t ldy, int32_t T,
                                 const lora_shape_t *shape, const void *dev_table, const int32_t *sorted_ids,
                                 const int32_t *seg_offsets, const int32_t *active, int32_t max_seg_hint,
                                 lora_path_t path, float *ws, size_t ws_bytes, int32_t *err, lora_stream_t stream,
                                 lora_event_t y_ready);

/*
 * lora_apply without a workspace argument, for callers that cannot allocate
 * device memory where they run the branch: for example a plug-in inside a host
 * engine that owns all device memory through its own pool and gives plug-ins no
 * allocator, or code that must not call cudaMalloc because it synchronises the
 * device.  The pages describe no counterpart of this call; it is a service of
 * this library.
 *
 * It runs the same shrink and expand kernels as LORA_PATH_DECODE_SPLIT, with the
 * fp32 shrink output kept in a fixed array inside the library's device image:
 * LORA_NOALLOC_WS_BYTES (4 MiB) on every device that loads the library, held
 * until the process exits.  It calls no allocating routine.
 *   - Limit: n_slices * T * r_max * 4 bytes must fit in LORA_NOALLOC_WS_BYTES,
 *     else the call returns LORA_ERR_WORKSPACE and enqueues nothing.
 *   - Set-up: the first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current and keeps it for the
 *     process; make that first call before any stream capture.  The address
 *     belongs to the device's context: do not reset the device
 *     (cudaDeviceReset) between calls.
 *   - Sharing: every call on a device uses the same array, and the array keeps
 *     the last call's contents.  Calls whose kernels overlap on the GPU (calls
 *     on different streams, or from threads that do not order their streams)
 *     race on it and give wrong results; issue them on one stream.  Nothing in
 *     the array has to start at zero: the shrink writes every entry the expand
 *     reads.
 * Other arguments, checks and errors are those of lora_apply.
 */
#define LORA_NOALLOC_WS_BYTES (4u << 20)
lora_status_t lora_apply_noalloc(const void *x, int64_t ldx, void *y, int64_t ldy, int32_t T,
                                 const lora_shape_t *shape, const void *dev_table,
                                 const int32_t *sorted_ids, const int32_t *seg_offsets,
                                 const int32_t *active, int32_t *err, lora_stream_t stream);

/*
 * Token index with activated-LoRA (aLoRA) enablement (llama.cpp LoRA adapter
 * page, "aLoRA:让适配器在 prompt 中间生效": a request runs without its adapter
 * before its invocation point and with it from there on).  Token t belongs to
 * sequence q = seq_ids[t] (device int32 [T], in [0, n_seq)) at position
 * positions[t] (device int32 [T]); its slot is seq_slot[q] (device int32
 * [n_seq], -1 for none) when positions[t] >= invocation_start[q] (device int32
 * [n_seq]) and -1 before it.  invocation_start 0 is a plain LoRA; a start past
 * the sequence's last position leaves the sequence without its adapter (the
 * pages' "invocation not found" case).  Outputs, limits and errors as
 * lora_build_index; a sequence id outside [0, n_seq) is reported as
 * LORA_ERR_SLOT_RANGE and the token keeps its y.
 */
lora_status_t lora_build_index_activated(const int32_t *seq_ids, const int32_t *positions, int32_t T,
                                         const int32_t *seq_slot, const int32_t *invocation_start, int32_t n_seq,
                                         int32_t S, const void *dev_table, int32_t *sorted_ids, int32_t *seg_offsets,
                                         int32_t *active, int32_t *err, lora_stream_t stream);

/*
 * A plan: the tables the two warp-streaming kernels otherwise build at the start
 * of every call (the active slots, their token ranges and ranks, the split of
 * the work over the warps), built once per batch and shape and then read by
 * every call of that shape (one table image per kernel, loaded with one pass of
 * 16-byte copies).  A plan holds the slot table's ranks, scales and weight
 * pointers: build one per slot table (per layer), and rebuild it whenever the
 * index or that table changes.
 *
 * lora_plan_bytes: the plan's size for T tokens and this shape, enough for
 * either kind of plan (0 for T < 1 or a bad shape).
 *
 * lora_build_plan: one launch on `stream` that reads the slot table and the
 * index (after lora_build_index) and writes the plan (device, 16-byte aligned,
 * plan_bytes >= lora_plan_bytes).  path: LORA_PATH_DECODE_DIRECT,
 * LORA_PATH_DECODE_DIRECT_FP8 or LORA_PATH_DECODE_TMA (the kernels the plan is
 * for; else LORA_ERR_UNSUPPORTED, also when those kernels do not take the
 * shape).  Device data errors of the index are reported here, as lora_apply
 * would.  A LORA_PATH_DECODE_TMA plan holds, per active slot, its token groups
 * and, per CTA, its share of the call's work (split by bytes moved) and a copy
 * of sorted_ids; it needs a table from lora_set_slot_table_tma of this shape
 * (else LORA_ERR_INVALID_ARG in err and a plan every call refuses), and is
 * built for the current device's SM count.  The plan kernel is never launched
 * as a programmatic dependent, so a LORA_PATH_DECODE_TMA call right after it
 * (which reads the plan before waiting for its predecessor) sees it complete.
 *
 * lora_apply_plan: lora_apply_ex on that path with the plan instead of the table
 * and the index.  A plan built for another T, slot count, slice count or path is
 * reported as LORA_ERR_INVALID_ARG in err and the call leaves y unchanged; the
 * plan must also have been built with this shape's k and slice widths (not
 * checked on the device).  Other arguments, checks and errors as lora_apply_ex.
 */
size_t lora_plan_bytes(int32_t T, const lora_shape_t *shape);
lora_status_t lora_build_plan(int32_t T, const lora_shape_t *shape, const void *dev_table, const int32_t *sorted_ids,
                              const int32_t *seg_offsets, const int32_t *active, lora_path_t path, void *plan,
                              size_t plan_bytes, int32_t *err, lora_stream_t stream);
lora_status_t lora_apply_plan(const void *x, int64_t ldx, void *y, int64_t ldy, int32_t T, const lora_shape_t *shape,
                              const void *plan, size_t plan_bytes, lora_path_t path, float *ws, size_t ws_bytes,
                              int32_t *err, lora_stream_t stream);

/*
 * The plans of `count` slot tables that share the shape and the index (the
 * layers of one step, each with its own weights), in one launch: dev_tables and
 * plans are host arrays of `count` device pointers, each plan plan_bytes long.
 * Checks and errors as lora_build_plan, for every table and plan.
 */
lora_status_t lora_build_plans(int32_t T, const lora_shape_t *shape, int32_t count, const void *const *dev_tables,
                               void *const *plans, size_t plan_bytes, const int32_t *sorted_ids,
                               const int32_t *seg_offsets, const int32_t *active, lora_path_t path, int32_t *err,
                               lora_stream_t stream);

/*
 * Routed-expert (MoE) LoRA.  llama.cpp LoRA adapter page, "MoE 专属的
 * build_lora_mm_id": in an expert layer both the A and the B product are routed
 * by the token's expert ids, like the base weights, so each (token, chosen
 * expert) pair uses that expert's A and B; TensorRT-LLM LoRA serving page, "MoE
 * LoRA: per-expert 布局": an adapter's expert weights are stored as
 * A [E][r][k] and B [E][d_i][r], and expert e's pair starts e * dim * rank
 * elements into each.
 *
 * The branch for pairs: with T tokens each routed to K experts, pair
 * p = t K + j (token t, its j-th choice, expert e = expert_ids[p]) of a token
 * with adapter s computes
 *     y[p, o_i + m] = bf16( f32(y[p, o_i + m]) + scale_s * sum_j xa_j B_{s,e,i}[m, j] ),
 *     xa_j = sum_c x[row(p), c] A_{s,e,i}[j, c],
 * row(p) = t when the x rows are per token (x_per_token != 0, the layer's
 * input shared by a token's experts) and p when they are per pair (the second
 * projection of an expert MLP).  Pairs of tokens with slot -1 keep y.
 *
 * The library serves it as the batched branch over n_adapters * E virtual slots
 * (slot s E + e) and T K rows: build the virtual table with
 * lora_moe_slot_pointers and lora_set_slot_table (S = n_adapters * E), the
 * index with lora_build_index_moe, and run lora_apply_moe.  The workspace is
 * lora_workspace_bytes(T * K, shape).
 */

/*
 * Virtual slot table entries (host only, no device access): for adapter a in
 * [0, n_adapters) and expert e in [0, E), slot v = a E + e gets rank ranks[a],
 * scale scales[a] and, for slice i, A_ptrs[v n + i] = A_base[a n + i] +
 * e * r_a * k * elem_bytes and B_ptrs[v n + i] = B_base[a n + i] +
 * e * d_i * r_a * elem_bytes (a zero base stays zero).  shape->S must equal
 * n_adapters * E; elem_bytes is 2 (bf16).  Outputs: v_ranks and v_scales
 * [n_adapters E], A_ptrs and B_ptrs [n_adapters E n_slices], caller-allocated.
 * Errors: LORA_ERR_INVALID_ARG (null pointers, counts, S mismatch), the shape
 * checks of lora_workspace_bytes.
 */
lora_status_t lora_moe_slot_pointers(int32_t n_adapters, int32_t E, const lora_shape_t *shape, int32_t elem_bytes,
                                     const int32_t *ranks, const float *scales, const uint64_t *A_base,
                                     const uint64_t *B_base, int32_t *v_ranks, float *v_scales, uint64_t *A_ptrs,
                                     uint64_t *B_ptrs);

/*
 * Index over the T K (token, choice) pairs: slot_ids [T] (device int32, the
 * token's adapter or -1), expert_ids [T K] (device int32, token-major: the K
 * experts of token t at t K .. t K + K - 1).  Pair p is keyed by the virtual
 * slot slot_ids[p / K] E + expert_ids[p]; outputs as lora_build_index with S
 * the virtual slot count (a multiple of E, at most LORA_MAX_SLOTS) and T K
 * items.  A slot id outside [-1, S / E) or an expert id outside [0, E) for a
 * token with an adapter writes LORA_ERR_SLOT_RANGE to err and the pair keeps
 * its y.
 */
lora_status_t lora_build_index_moe(const int32_t *slot_ids, const int32_t *expert_ids, int32_t T, int32_t K,
                                   int32_t E, int32_t S, const void *dev_table, int32_t *sorted_ids,
                                   int32_t *seg_offsets, int32_t *active, int32_t *err, lora_stream_t stream);

/*
 * The routed-expert branch on the warp-streaming decode kernels: y has T K rows
 * (one per pair, ldy), x has T rows when x_per_token != 0 and T K rows
 * otherwise (ldx); index from lora_build_index_moe; ws of
 * lora_workspace_bytes(T * K, shape) bytes.  Needs T K <= 2048, r_max <= 64 and
 * the virtual table within the limits of LORA_PATH_DECODE_DIRECT (else
 * LORA_ERR_UNSUPPORTED).  Checks and errors otherwise as lora_apply.
 */
lora_status_t lora_apply_moe(const void *x, int64_t ldx, int32_t x_per_token, void *y, int64_t ldy, int32_t T,
                             int32_t K, const lora_shape_t *shape, const void *dev_table, const int32_t *sorted_ids,
                             const int32_t *seg_offsets, const int32_t *active, float *ws, size_t ws_bytes,
                             int32_t *err, lora_stream_t stream);

/*
 * lora_apply_moe with a plan instead of the virtual table and the pair index: the
 * plan built by lora_build_plan(s) for T * K rows, the virtual table and the
 * pair index (path LORA_PATH_DECODE_DIRECT).  Checks and errors as
 * lora_apply_moe and lora_apply_plan.
 */
lora_status_t lora_apply_moe_plan(const void *x, int64_t ldx, int32_t x_per_token, void *y, int64_t ldy, int32_t T,
                                  int32_t K, const lora_shape_t *shape, const void *plan, size_t plan_bytes, float *ws,
                                  size_t ws_bytes, int32_t *err, lora_stream_t stream);

/*
 * lora_apply_moe on an explicit path: LORA_PATH_DECODE_DIRECT (what
 * lora_apply_moe runs), LORA_PATH_DECODE_TMA, the one-kernel tensor-map
 * decode over the pairs, or LORA_PATH_DECODE_CLUSTER, one cluster per virtual
 * slot (its limits as in lora_apply_ex; the workspace is not used).  The TMA
 * path needs dev_table to be a table of
 * lora_set_slot_table_tma over the virtual slots (the entries of
 * lora_moe_slot_pointers), x 16-byte aligned with ldx a multiple of 8, and
 * T K and the shape within the limits of LORA_PATH_DECODE_TMA in lora_apply_ex;
 * it builds its plan in the workspace, like lora_apply_ex.  Any other path:
 * LORA_ERR_UNSUPPORTED.  Checks and errors otherwise as lora_apply_moe.
 */
lora_status_t lora_apply_moe_ex(const void *x, int64_t ldx, int32_t x_per_token, void *y, int64_t ldy, int32_t T,
                                int32_t K, const lora_shape_t *shape, const void *dev_table, const int32_t *sorted_ids,
                                const int32_t *seg_offsets, const int32_t *active, lora_path_t path, float *ws,
                                size_t ws_bytes, int32_t *err, lora_stream_t stream);

/*
 * lora_apply_moe_plan on an explicit path (LORA_PATH_DECODE_DIRECT or
 * LORA_PATH_DECODE_TMA); the plan must have been built by lora_build_plan(s)
 * for T * K rows with the same path (a TMA plan on a table of
 * lora_set_slot_table_tma).  Checks and errors as lora_apply_moe_ex and
 * lora_apply_plan.
 */
lora_status_t lora_apply_moe_plan_ex(const void *x, int64_t ldx, int32_t x_per_token, void *y, int64_t ldy,
                                     int32_t T, int32_t K, const lora_shape_t *shape, const void *plan,
                                     size_t plan_bytes, lora_path_t path, float *ws, size_t ws_bytes, int32_t *err,
                                     lora_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LORA_GEMM_H */
