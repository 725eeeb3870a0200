/*
 * dsa.h -- C ABI of a GB300 (sm_103a) library for DeepSeek-V4.1 top-k sparse
 * attention.
 *
 * The operation (akol1 TensorFold PR #4, first commit message; TensorFold
 * PR #1206, "What changes"): for each query row r and head h, gather the
 * n_sel[r] latent KV rows x_j = kv[slot(r)][idx[r][j]] that an indexer
 * selected, score them, and return the softmax-weighted sum of the same rows
 * with one extra per-head sink logit in the denominator:
 *
 *   s_j = scale * <q[r][h][:], x_j>          (the 512-wide row is key and value)
 *   out[r][h][:] = sum_j e^{s_j} x_j / (e^{sink[h]} + sum_j e^{s_j})
 *
 * computed tile by tile with a running maximum, a running sum and a running
 * value sum.  The sink is a logit (it is not multiplied by scale) and has no
 * value row.  The latent row is 512 wide, handled as sixteen 32-wide column
 * groups on the pages; here it is one contiguous row.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All array arguments are DEVICE pointers owned by the caller.  The
 *   library never frees or retains them.  Row-major, contiguous:
 *     q     [R][H][512]    dtype (float32, or bfloat16 bit patterns)
 *     kv    prefill: [N][512] (one cache shared by all rows)
 *           decode:  [B][N][512] (row b reads only slot b)
 *     idx   [R][k_max] int32; only the first n_sel[r] entries are used (the
 *           rest may be read ahead but are ignored; they need no valid value)
 *     n_sel [R] int32
 *     sink  [H] float32 (any value, including +-inf)
 *     out   [R][H][512] float32; must not overlap any input
 *   q, kv and out must be 16-byte aligned.
 * - 1 <= H <= 64 (the pages use 64 heads, 16 or 32 a rank under tensor
 *   parallelism); the row width is fixed at 512.
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *   default stream) and run on the current device.  The library allocates
 *   nothing per call: a small device block (the error word and up to 64
 *   two-int row queues) and, for decode, one scratch buffer for split partial
 *   results are allocated once per device on first use (the scratch grows
 *   when a larger batch needs it; dsa_topk_select has one of its own) and
 *   released by dsa_shutdown().  Do not
 *   issue the first call of a device inside a CUDA graph capture.  Decode
 *   calls whose work overlaps on the GPU (other streams, other threads) share
 *   that scratch and race; order them on one stream.
 * - A bf16 prefill call with more rows than the GPU has SMs hands its rows to
 *   the SMs from a row queue owned by its stream (calls on one stream run in
 *   order; calls on different streams use different queues), so that faster
 *   SMs take more rows.  It falls back to a fixed round-robin assignment on
 *   the per-thread default stream, while its stream is being captured into
 *   a CUDA graph, and once 64 streams of the device hold a queue (until
 *   dsa_shutdown()).  Which SM runs a row does not change its result.
 * - The kernels are launched with programmatic stream serialisation: a
 *   kernel may start its set-up while the previous work on the stream is
 *   finishing, but it touches no global memory before that work has
 *   completed, so stream order holds as for an ordinary launch.
 * - Host-side errors return before anything is launched.
 * - Device-side errors: an index in idx[r][0..n_sel[r]) outside [0, N), or an
 *   n_sel[r] outside [0, k_max], sets a bit in a sticky device error word and
 *   writes NaN to every output of that row; the kernels never trap.  Read
 *   (and clear) the word with dsa_get_device_error().
 * - Numerics: float32 inputs run on CUDA cores in fp32 with precise expf; bf16
 *   inputs run on the tensor cores (bf16 products, fp32 accumulation, the
 *   softmax weights split into two bf16 terms), fp32 softmax.  Results are
 *   bit-identical from run to run and do not depend on the other rows of the
 *   batch.  The bf16 path weighs keys against a per-head reference that may
 *   lag the running maximum by up to 2^32, so its fp32 sums overflow (to
 *   +-inf or NaN) only when a selected kv value exceeds about 1e26 in
 *   magnitude.
 */
#ifndef DSA_H
#define DSA_H

#include <stdint.h>

#if defined(__GNUC__)
#define DSA_API __attribute__((visibility("default")))
#else
#define DSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, bad alignment        */
    DSA_ERR_UNSUPPORTED = 2,   /* H > 64, unknown dtype, not an sm_103 GPU     */
    DSA_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed         */
    DSA_ERR_DEVICE_CHECK = 4   /* reserved: returned by no call at present     */
} dsa_status;

typedef enum {
    DSA_F32 = 0,               /* q and kv are float32                         */
    DSA_BF16 = 1               /* q and kv are bfloat16                        */
} dsa_dtype;

/* Bits of the device error word. */
#define DSA_DEVERR_IDX_RANGE  0x1u  /* an idx entry outside [0, N)                */
#define DSA_DEVERR_NSEL_RANGE 0x2u  /* an n_sel entry outside [0, k_max]          */
#define DSA_DEVERR_TIMEOUT    0x4u  /* a bounded in-kernel wait gave up; the
                                       outputs of that launch are undefined      */
#define DSA_DEVERR_LAYOUT     0x8u  /* shared memory not 1024-byte aligned; the
                                       kernel did no work                        */
#define DSA_DEVERR_NVALID_RANGE 0x10u /* dsa_topk_select: an n_valid entry outside
                                       [0, ld]; that row selects nothing         */

/*
 * Decode: B slots with one query row each.  Row b attends to k <= k_max
 * positions of its own cache kv[b] (N positions).  On the pages this is a
 * decode step's attention call (akol1 TensorFold PR #4; "warm attention call"
 * timings at positions 128 and 8191).
 *   q [B][H][512], kv [B][N][512], idx [B][k_max], n_sel [B], out [B][H][512].
 * Returns DSA_OK after queueing the work (B == 0 queues nothing).
 */
DSA_API dsa_status dsa_sparse_attn_decode(const void* q, const void* kv_cache,
                                          const int32_t* idx, const int32_t* n_sel,
                                          const float* sink, float scale, float* out,
                                          int B, int H, int N, int k_max,
                                          dsa_dtype dtype, void* stream);

/*
 * Decode with T query rows a slot: B slots, each with T rows that attend to
 * the slot's own cache (several tokens of one sequence decoded together, as
 * when a step's draft tokens are verified).  Row r = b*T + t reads only
 * kv[b]; every row has its own selection.  T = 1 is dsa_sparse_attn_decode.
 *   q [B*T][H][512], kv [B][N][512], idx [B*T][k_max], n_sel [B*T],
 *   out [B*T][H][512].
 * A row's result is bit-identical to the same row in a one-row-a-slot call
 * over that slot's cache.  DSA_ERR_INVALID_ARG for T < 1 or B*T beyond int
 * range; otherwise as dsa_sparse_attn_decode (the split scratch included).
 */
DSA_API dsa_status dsa_sparse_attn_decode_rows(const void* q, const void* kv_cache,
                                               const int32_t* idx, const int32_t* n_sel,
                                               const float* sink, float scale, float* out,
                                               int B, int T, int H, int N, int k_max,
                                               dsa_dtype dtype, void* stream);

/*
 * Prefill: R query rows of one segment attend to one shared cache of N
 * positions (TensorFold PR #1206: 2048-row prefill segments; a row at
 * position p selects min(p+1, k) positions in [0, p]).
 *   q [R][H][512], kv [N][512], idx [R][k_max], n_sel [R], out [R][H][512].
 * Returns DSA_OK after queueing the work (R == 0 queues nothing).
 */
DSA_API dsa_status dsa_sparse_attn_prefill(const void* q, const void* kv_cache,
                                           const int32_t* idx, const int32_t* n_sel,
                                           const float* sink, float scale, float* out,
                                           int R, int H, int N, int k_max,
                                           dsa_dtype dtype, void* stream);

/*
 * The three calls above in one, with the output type chosen:
 *   rows_per_slot 0   prefill: every row reads the one cache kv [N][512];
 *   rows_per_slot T   decode: row r reads slot r / T of kv [R/T][N][512]
 *                     (R a multiple of T).
 *   out_dtype DSA_F32   out [R][H][512] float32, as the calls above;
 *   out_dtype DSA_BF16  out [R][H][512] bfloat16: each element is the float32
 *                       result of the same call rounded to nearest even,
 *                       bit for bit.  Half the bytes, and the A operand of
 *                       dsa_oproj as it stands.
 * Otherwise as dsa_sparse_attn_prefill / _decode_rows (out 16-byte aligned).
 */
DSA_API dsa_status dsa_sparse_attn(const void* q, const void* kv_cache,
                                   const int32_t* idx, const int32_t* n_sel,
                                   const float* sink, float scale, void* out,
                                   int R, int rows_per_slot, int H, int N, int k_max,
                                   dsa_dtype dtype, dsa_dtype out_dtype, void* stream);

/*
 * Decode without the key split, for batches large enough to fill the GPU:
 * row r (rows_per_slot >= 1 rows a slot, R a multiple of it) reads slot
 * r / rows_per_slot of kv [R / rows_per_slot][N][512], and each row's keys
 * run from first to last in one CTA, as a prefill row's do, with rows handed
 * out by the stream's row queue.  dsa_sparse_attn_decode splits every row
 * into 128-key chunks on separate SMs and merges their partials (128 KB of
 * fp32 each) in a second kernel: at 8 rows that spreads the work over 40 SMs,
 * but once there are about as many rows as SMs the partials only add traffic
 * (and stop fitting in the L2).  This call writes no partials and launches
 * one kernel.
 * Results: the same computation as dsa_sparse_attn_decode (running maximum,
 * tile sum and value sum over the selected keys, the sink folded into the
 * denominator), with one running softmax over the whole row instead of
 * chunks merged, so the bits differ from that call's within the same
 * tolerance.  They do not depend on the batch, and they equal, bit for bit,
 * dsa_sparse_attn_prefill's over the slots' caches viewed as one cache
 * [R / rows_per_slot * N][512] with each row's indices offset by its slot
 * times N.  fp32 inputs run the fp32 kernel, which never splits (the same
 * bits as dsa_sparse_attn_decode_rows).  Arguments, layouts, ownership and
 * errors as dsa_sparse_attn (out_dtype DSA_F32 or DSA_BF16); rows_per_slot
 * < 1 or R not a multiple of it is DSA_ERR_INVALID_ARG.
 */
DSA_API dsa_status dsa_sparse_attn_decode_whole_rows(const void* q, const void* kv_cache,
                                                     const int32_t* idx, const int32_t* n_sel,
                                                     const float* sink, float scale, void* out,
                                                     int R, int rows_per_slot, int H, int N, int k_max,
                                                     dsa_dtype dtype, dsa_dtype out_dtype, void* stream);

/*
 * Output projection of attention rows (the step after the attention: the
 * heads' outputs of a row, concatenated, times the projection matrix):
 *   attn [R][K] bfloat16 (for this library's output, K = H*512 and the
 *        [R][H][512] bf16 out of dsa_sparse_attn),
 *   w_o  [K][d_out] bfloat16, row-major,
 *   out  [R][d_out] float32 = attn . w_o, accumulated in float32.
 * Run by this library's own tensor-core kernel (tcgen05 MMAs fed by TMA, two
 * TMEM accumulators; no split of K, so every output is one fp32 sum in a
 * fixed order and repeated calls give the same bits).  The pages give no
 * shape for this projection; d_out is the caller's.  All three 16-byte
 * aligned, K and d_out multiples of 8.  Allocates nothing beyond the
 * per-device error word.  A wait that gives up sets DSA_DEVERR_TIMEOUT
 * (outputs undefined).  DSA_ERR_INVALID_ARG for null pointers or bad
 * sizes, DSA_ERR_CUDA if the launch fails.
 */
DSA_API dsa_status dsa_oproj(const void* attn, const void* w_o, float* out,
                             int R, int K, int d_out, void* stream);

/*
 * Prefill attention with its output projection: dsa_sparse_attn with bf16
 * inputs, rows_per_slot 0 and out_dtype DSA_BF16 into the caller's buffer
 * attn [R][H][512] bfloat16, then dsa_oproj(attn, w_o, out, R, H*512, d_out)
 * on the same stream.  The attention's rows go to the GEMM as bf16, half the
 * bytes of the float32 output.
 */
DSA_API dsa_status dsa_sparse_attn_prefill_oproj(const void* q, const void* kv_cache,
                                                 const int32_t* idx, const int32_t* n_sel,
                                                 const float* sink, float scale,
                                                 const void* w_o, void* attn, float* out,
                                                 int R, int H, int N, int k_max, int d_out,
                                                 void* stream);

/*
 * Largest number of (row, 128-key chunk) units that
 * dsa_sparse_attn_decode_noalloc() accepts: B * ceil(k_max / 128) <= 64,
 * e.g. 8 rows with k_max <= 1024.
 */
#define DSA_NOALLOC_MAX_UNITS 64

/*
 * Decode without any device allocation.  The pages have no counterpart to
 * this entry point; it exists for callers of this library that must not
 * allocate device memory: engines that reserve all device memory when they
 * start and forbid allocation afterwards, and callers on a latency-critical
 * path where cudaMalloc / cudaFree would synchronise the device.
 *
 * Same arguments, layouts and results as dsa_sparse_attn_decode() (the same
 * kernels with the same key chunking), bf16 only.  The split partials and an
 * error word live in one static device array of 8,421,632 bytes, which every
 * GPU that loads the library holds until the process exits.  The call
 * allocates nothing; the caller still passes all inputs and outputs.
 *
 * - Returns DSA_ERR_UNSUPPORTED when B * ceil(k_max / 128) exceeds
 *   DSA_NOALLOC_MAX_UNITS, or for float32 inputs; DSA_ERR_INVALID_ARG for the
 *   same bad arguments as dsa_sparse_attn_decode().
 * - The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress); make that first call before any stream capture.
 * - Every call uses the same array and it keeps the last call's contents:
 *   calls whose work overlaps on the GPU (other streams, other threads) race
 *   and corrupt each other's results.  Order them on one stream.
 * - Device errors are not reported: this entry point has its own error word
 *   in the static array, cleared at the start of every call and never read
 *   back, so none of its bits (DSA_DEVERR_IDX_RANGE, DSA_DEVERR_NSEL_RANGE,
 *   DSA_DEVERR_TIMEOUT, DSA_DEVERR_LAYOUT) reaches dsa_get_device_error().
 *   Out-of-range selections still give NaN rows.  A call whose bounded wait
 *   gave up, or that found its shared memory misaligned, leaves its outputs
 *   undefined with no signal; callers that need that signal use
 *   dsa_sparse_attn_decode().
 * - dsa_shutdown() forgets the array's looked-up address, so a call after a
 *   device reset looks it up again.
 */
DSA_API dsa_status dsa_sparse_attn_decode_noalloc(const void* q, const void* kv_cache,
                                                  const int32_t* idx, const int32_t* n_sel,
                                                  const float* sink, float scale, float* out,
                                                  int B, int H, int N, int k_max,
                                                  dsa_dtype dtype, void* stream);

/*
 * Top-k selection of an indexer's scores: the step that turns a row's index
 * scores into the selection the attention calls above read (DeepSeek V4.1
 * indexer PR #2, title: the indexer's merge and finish on a threadgroup a
 * row, the same picks; the pages give no more, and the order below is this
 * library's reading).
 *   scores  [R][ld] float32; row r's candidates are positions
 *           [0, n_valid[r]).  16-byte aligned; ld a multiple of 4,
 *           1 <= ld <= 32768.
 *   n_valid [R] int32
 *   idx     [R][k_max] int32 out: the picks of row r by ascending
 *           position, then -1
 *   n_sel   [R] int32 out: min(k, n_valid[r])
 * The picks are the first min(k, n_valid[r]) candidates in this order:
 * larger score first; NaN after every number (also after -inf); -0 and +0
 * equal; equal scores by smaller position first.  They are listed by
 * ascending position (the attention reads a set).  1 <= k <= k_max,
 * k <= 2048.  idx and n_sel can be passed straight to the attention calls.
 * An n_valid[r] outside [0, ld] sets DSA_DEVERR_NVALID_RANGE, and that row
 * selects nothing (n_sel 0, idx all -1).  Asynchronous on `stream`; reads
 * no input before the work queued before it on the stream has completed.
 * DSA_ERR_INVALID_ARG for a null pointer, a misaligned scores, or bad
 * sizes; DSA_ERR_UNSUPPORTED for k > 2048 or ld > 32768.
 * Rows with ld > 8192 are selected in two steps (each 8192-position share
 * of a row, then the shares' picks) through a per-device scratch of up to
 * 256 MB, allocated on first use (a larger call processes its rows in turn)
 * and released by dsa_shutdown(); such calls whose work overlaps on the GPU
 * share that scratch and race: order them on one stream.
 */
DSA_API dsa_status dsa_topk_select(const float* scores, int ld, const int32_t* n_valid, int R,
                                   int k, int32_t* idx, int k_max, int32_t* n_sel,
                                   void* stream);

/*
 * Head-sharded tensor parallelism (TensorFold PR #1206, "What changes": the
 * 64 heads are split over the ranks, 16 a rank at world 4; heads added to
 * fill the last rank get zero sinks; the output groups are gathered before
 * the output projections).  A rank runs the attention calls above over its
 * own heads (H = heads_per_rank); the calls below plan the split, cut a
 * rank's heads out of full arrays, and lay the gathered outputs back out.
 * The gathering itself is the caller's collective (an all-gather of every
 * rank's out [R][heads_per_rank][512], rank after rank).
 *
 * Plan for H heads over `world` ranks: heads_per_rank = ceil(H / world),
 * padded_heads = heads_per_rank * world; rank w owns heads
 * [first_head, first_head + heads_per_rank), of which the first real_heads
 * are < H and the rest are padding.  Host only; no device is touched.
 * DSA_ERR_INVALID_ARG for a null plan, H < 1, world < 1 or rank outside
 * [0, world); DSA_ERR_UNSUPPORTED when heads_per_rank > 64.
 */
typedef struct {
    int heads_per_rank;
    int padded_heads;
    int first_head;
    int real_heads;
} dsa_head_shard_plan;

DSA_API dsa_status dsa_head_shard(int H, int world, int rank, dsa_head_shard_plan* plan);

/*
 * A rank's inputs from the full ones: q_local [R][heads_per_rank][512] and
 * sink_local [heads_per_rank] take heads first_head.. of q [R][H][512] and
 * sink [H]; a padding head gets q = 0 and sink = 0.  Values are copied bit
 * for bit.  q and q_local (dtype: float32 or bf16) 16-byte aligned, device
 * pointers; asynchronous on `stream`.  Errors as dsa_head_shard, plus
 * DSA_ERR_INVALID_ARG for null or misaligned pointers or R < 0.
 */
DSA_API dsa_status dsa_shard_heads(const void* q, const float* sink, void* q_local, float* sink_local,
                                   int R, int H, int world, int rank, dsa_dtype dtype, void* stream);

/*
 * The gathered outputs laid out as one call's: gathered
 * [world][R][heads_per_rank][512] (rank after rank, as an all-gather of the
 * ranks' out arrays leaves them) into out [R][H][512]; head h comes from
 * rank h / heads_per_rank and padding heads are dropped.  Bit for bit.
 * dtype is the outputs' (DSA_F32 or DSA_BF16); both pointers 16-byte
 * aligned device pointers that do not overlap; asynchronous on `stream`.
 * Errors as dsa_shard_heads.
 */
DSA_API dsa_status dsa_unshard_heads(const void* gathered, void* out, int R, int H, int world,
                                     dsa_dtype dtype, void* stream);

/*
 * Self-test of the bounded waits (the pages have no counterpart): queues on
 * `stream` one small kernel whose only wait is on a barrier that nothing
 * completes.  After the library's wait limit (about 2 seconds) the wait gives
 * up, sets DSA_DEVERR_TIMEOUT in the device error word and the kernel
 * returns; the context stays usable.  Every wait in the attention and
 * selection kernels is bounded the same way, so a fault on the GPU's side
 * shows up as an error bit, never as a hang.
 */
DSA_API dsa_status dsa_selftest_wait_limit(void* stream);

/*
 * Synchronises `stream`, stores the current device's error word in *code
 * and clears it.  *code is 0 when no launch since the last read found a
 * problem.  DSA_ERR_INVALID_ARG if code is NULL; DSA_ERR_CUDA if the
 * synchronisation or the copy fails.
 */
DSA_API dsa_status dsa_get_device_error(void* stream, uint32_t* code);

/* Static, human-readable name of a status code. */
DSA_API const char* dsa_status_string(dsa_status status);

/*
 * Releases the per-device error word and scratch of every device the
 * library touched.  Call only when no launch of this library is pending.
 */
DSA_API dsa_status dsa_shutdown(void);

#ifdef __cplusplus
}
#endif
#endif /* DSA_H */
