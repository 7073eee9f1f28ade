/*
 * sdm.h - C ABI of the GB300 (sm_103a) sparse delta-memory (SDM) decode-state library.
 *
 * Three operations, each one kernel launch on the caller's stream:
 *   sdm_decode_step  one write-then-read token for every stream (sdm_decode_step_ex: with flags)
 *   sdm_decode_seq   T tokens for every stream in one persistent launch (sdm_decode_seq_ex: with
 *                    flags, e.g. the stream-major [n_streams, T, .] layout of a prompt)
 *   sdm_gather       per-token weighted sums of bank rows (one or two operands), optional stash
 *                    (sdm_gather_kpos: with a compact snapshot instead; sdm_gather_plan_*: a
 *                    checked launch, replayed per slab of an index tensor; _launch_ex: with
 *                    flags)
 *
 * Common rules
 *   - Every pointer argument except `stream` (and the host records and arrays named as such) is a
 *     DEVICE pointer the caller owns; the library keeps no pointer after the call returns (apart
 *     from the work it enqueued, and from a gather plan record, which the caller owns and which
 *     holds the pointers it was made with) and frees nothing.
 *   - Calls allocate no memory, synchronise nothing and only enqueue work on `stream` (NULL = the
 *     legacy default stream), so they may be captured in a CUDA graph.
 *   - Return value: 0 = launched (or nothing to do); < 0 = argument error (an SDM_E* code below,
 *     nothing launched); > 0 = the cudaError_t of a failed launch (the error state is consumed).
 *   - Index ranges are the caller's contract: decode slots must lie in the bank, every stream's
 *     slots must be private to it and its W write slots distinct (none of this is checked, as in
 *     the reference). A float32 bank of 64 or more columns is taken to hold fewer than 2^32 rows
 *     (it would exceed 1 TiB otherwise): its streaming kernel keeps slots as 32-bit row indices. The gather knows the bank's row count and skips out-of-range rows, raising
 *     SDM_DEV_BAD_INDEX in the device status word (sdm_device_status).
 *   - Launches use programmatic stream serialization: a kernel may be scheduled while the previous
 *     kernel on the stream is still finishing, but it reads and writes no memory before that kernel
 *     has completed (griddepcontrol.wait), so stream order is kept. The one exception is opt-in:
 *     with SDM_INPUTS_READY an _ex call may read its inputs (never the bank, never its outputs)
 *     and warm L2 before that wait, on the caller's promise that those inputs are already final.
 *   - bfloat16 data is raw 16-bit patterns (the high half of an IEEE float32).
 *   - Results are deterministic: every sum is accumulated in a fixed order independent of the GPU.
 *
 * Reference: the "sparse-delta-memory 2.0.0" wheel, files sparse_delta_memory/decode.py
 * (sdm_decode_step, _decode_launch, _sdm_decode_kernel) and sparse_delta_memory/cuda/gather_cuda.py
 * (module docstring, token_gather).
 */
#ifndef SDM_H
#define SDM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle; layout-compatible with cudaStream_t / CUstream. */
typedef struct CUstream_st* sdm_stream_t;

/* bank / weight element types */
#define SDM_BF16 0
#define SDM_F32 1
/* index element types */
#define SDM_I32 0
#define SDM_I64 1

/* argument errors (negative return values; nothing was launched) */
#define SDM_OK 0
#define SDM_ENULL (-1)      /* a required pointer is NULL */
#define SDM_EDTYPE (-2)     /* bank or weight dtype is not SDM_BF16 / SDM_F32 */
#define SDM_EIDX (-3)       /* index dtype is not SDM_I32 / SDM_I64 */
#define SDM_EHD (-4)        /* head_dim < 1 or > 65536 */
#define SDM_EWIDTH (-5)     /* W, R or a gather width outside 1..256 */
#define SDM_EGATES (-6)     /* G is neither 1 nor W */
#define SDM_ECOUNT (-7)     /* negative count, n_slots < 1 or >= 2^31, or more units than one launch holds */
#define SDM_ECHUNK (-8)     /* chunk < 1, tokens not a multiple of chunk, or valid outside 0..chunk */
#define SDM_EALIGN (-9)     /* a pointer is not aligned to its element size */
#define SDM_EOVERLAP (-10)  /* a gather output or the stash overlaps the bank */
#define SDM_ENOPS (-11)     /* gather operand count is not 1 or 2 */
#define SDM_EPLAN (-12)     /* not an initialised gather or decode plan (wrong tag or record size) */
#define SDM_EROW (-13)      /* row0 outside 0..row0_max, row0_max + tokens beyond the index rows, or a plan step outside 0..T-1 */
#define SDM_EDEVICE (-14)   /* the current device is not the one the plan was made on */
#define SDM_EFLAGS (-15)    /* unknown bits in the flags of an _ex entry point */

/* bits of the device status word */
#define SDM_DEV_TIMEOUT 1u   /* reserved: a kernel gave up a bounded wait (no current kernel waits) */
#define SDM_DEV_BAD_INDEX 2u /* the gather met a row index outside [0, n_slots) and skipped it */

/*
 * sdm_decode_step - advance every stream by one token: write, then read.
 *
 * Defined by sdm_decode_step (decode.py): per stream s, with d_w = exp(g[s, G == 1 ? 0 : w]),
 *     retrieved      = sum_w k_val[s,w] * d_w * bank[k_idx[s,w]]
 *     delta_v        = beta[s] * (v[s] - retrieved)
 *     bank[k_idx[w]] = d_w * bank[k_idx[w]] + k_val[s,w] * delta_v        (all w)
 *     out[s]         = sum_r q_val[s,r] * bank[q_idx[s,r]]                (after the write)
 * k_val, v and q_val are rounded to the bank dtype (round to nearest even) before use; beta and
 * g are used in float32; d_w is the float32 nearest to e^g; all arithmetic is float32 and the
 * new rows and the readings are rounded to the bank dtype.
 *
 *   bank      [n_slots, hd] bank dtype, row-major, updated in place
 *   k_idx     [n_streams, W] idx dtype: write slots (distinct within a stream)
 *   k_val     [n_streams, W] float32: write weights
 *   v         [n_streams, hd] float32: values
 *   beta      [n_streams] float32: write strengths
 *   g         [n_streams, G] float32: log-decay per token (G == 1) or per write (G == W)
 *   q_idx     [n_streams, R] idx dtype: read slots (repeats allowed)
 *   q_val     [n_streams, R] float32: read weights
 *   out       [n_streams, hd] bank dtype: readings
 *   n_streams >= 0 (0: nothing launched); hd >= 1; 1 <= W, R <= 256; G in {1, W}
 *   bank_dtype SDM_BF16 | SDM_F32; idx_dtype SDM_I32 | SDM_I64 (both index arrays)
 */
int sdm_decode_step(void* bank, const void* k_idx, const float* k_val, const float* v, const float* beta,
                    const float* g, const void* q_idx, const float* q_val, void* out, int64_t n_streams, int hd,
                    int W, int R, int G, int bank_dtype, int idx_dtype, sdm_stream_t stream);

/*
 * sdm_decode_step_ex - sdm_decode_step with flags; flags == 0 is sdm_decode_step.
 *
 * SDM_INPUTS_READY promises that every input but the bank (k_idx, k_val, v, beta, g, q_idx,
 * q_val) was complete before the kernel enqueued just ahead of this launch on the stream began.
 * The launch may then read them, derive the token's weights and gates and warm L2 with the
 * token's bank rows before it waits for that kernel (the launches of this library chain by
 * programmatic dependent launch); it reads and writes the bank, and writes `out`, only after the
 * wait. Results are the same bits as without the flag. Use it for steps whose inputs are staged
 * ahead (e.g. one CUDA graph of many steps over inputs filled before the replay); without the
 * promise the flag may read stale inputs. Unknown bits return SDM_EFLAGS.
 */
#define SDM_INPUTS_READY 1u
int sdm_decode_step_ex(void* bank, const void* k_idx, const float* k_val, const float* v, const float* beta,
                       const float* g, const void* q_idx, const float* q_val, void* out, int64_t n_streams, int hd,
                       int W, int R, int G, int bank_dtype, int idx_dtype, unsigned flags, sdm_stream_t stream);

/*
 * sdm_decode_seq - T tokens for every stream in one launch, equal to T sdm_decode_step calls.
 *
 * One block owns one (stream, column slice) for all T tokens; the reads of token t and the
 * retrieve of token t+1 are ordered after token t's writes by a block barrier, which is valid
 * because no other block touches those slots and columns (the barrier argument of
 * _sdm_decode_kernel in decode.py).
 *
 * Every per-token array gains a leading time axis (time-major): k_idx, k_val [T, n_streams, W];
 * v [T, n_streams, hd]; beta [T, n_streams]; g [T, n_streams, G]; q_idx, q_val [T, n_streams, R];
 * out [T, n_streams, hd]. T >= 0 (0: nothing launched). Other arguments as sdm_decode_step.
 */
int sdm_decode_seq(void* bank, const void* k_idx, const float* k_val, const float* v, const float* beta,
                   const float* g, const void* q_idx, const float* q_val, void* out, int64_t n_streams, int hd,
                   int W, int R, int G, int T, int bank_dtype, int idx_dtype, sdm_stream_t stream);

/*
 * sdm_decode_seq_ex - sdm_decode_seq with flags; flags == 0 is sdm_decode_seq.
 *
 * SDM_STREAM_MAJOR: every per-token array is in the layer's own stream-major layout, each
 * stream's T tokens contiguous: k_idx, k_val [n_streams, T, W]; v [n_streams, T, hd]; beta
 * [n_streams, T]; g [n_streams, T, G]; q_idx, q_val [n_streams, T, R]; and the readings go to
 * out [n_streams, T, hd]. This is the [P, T, .] layout of a prompt that forward_steps
 * (forward.py) stages to time-major with stage_time_major before its steps and whose readings it
 * takes back with unstage_time_major; here the kernel reads and writes that layout by stride, so
 * neither staging copy is made. Results are the bits of sdm_decode_seq on the staged arrays.
 * SDM_INPUTS_READY: as for sdm_decode_step_ex (token 0's inputs are read before the wait).
 * Unknown bits return SDM_EFLAGS. Other arguments as sdm_decode_seq.
 */
#define SDM_STREAM_MAJOR 2u
int sdm_decode_seq_ex(void* bank, const void* k_idx, const float* k_val, const float* v, const float* beta,
                      const float* g, const void* q_idx, const float* q_val, void* out, int64_t n_streams, int hd,
                      int W, int R, int G, int T, int bank_dtype, int idx_dtype, unsigned flags, sdm_stream_t stream);

/*
 * Decode-step plan: T single-token steps over time-major inputs, checked once (the decode-side
 * counterpart of the gather launch plan below, for a loop that launches one token at a time, e.g.
 * while serving; the pages drive their decode step from such a loop, forward.py, and check each
 * launch in decode.py's sdm_decode_step). sdm_decode_plan_init checks the arguments of sdm_decode_seq(..., T, ...) once
 * and records the launch of one token; sdm_decode_plan_launch(t) then launches exactly
 * sdm_decode_step on the rows of token t (k_idx + t * n_streams * W, ..., out + t * n_streams * hd),
 * and sdm_decode_plan_walk launches tokens t0 .. t0 + n - 1 in order from one call. The record is
 * caller-owned, valid on the device current at init, in this process, until the library is
 * unloaded; it keeps the pointers given at init (their memory must stay allocated). Every step
 * returns 0, an SDM_E* code (nothing launched) or the cudaError_t of a failed launch.
 */
#define SDM_DECODE_PLAN_BYTES 512
typedef struct sdm_decode_plan {
    uint64_t opaque[SDM_DECODE_PLAN_BYTES / 8];
} sdm_decode_plan;

/*
 * sdm_decode_plan_init - check a time-major T-token decode once and record a one-token launch in
 * *plan (nothing is launched). Arguments as sdm_decode_seq; T >= 0. Returns 0, an SDM_E* code
 * (the record untouched) or a cudaError_t from the device queries and settings.
 */
int sdm_decode_plan_init(sdm_decode_plan* plan, void* bank, const void* k_idx, const float* k_val, const float* v,
                         const float* beta, const float* g, const void* q_idx, const float* q_val, void* out,
                         int64_t n_streams, int hd, int W, int R, int G, int T, int bank_dtype, int idx_dtype);

/*
 * sdm_decode_plan_launch - step t of a plan (0 <= t < T, else SDM_EROW); flags 0 or
 * SDM_INPUTS_READY (as for sdm_decode_step_ex). Checks, in order: the flags (SDM_EFLAGS), the
 * record (SDM_EPLAN), t (SDM_EROW), the current device (SDM_EDEVICE).
 */
int sdm_decode_plan_launch(const sdm_decode_plan* plan, int t, unsigned flags, sdm_stream_t stream);

/*
 * sdm_decode_plan_walk - steps t0, t0 + 1, ..., t0 + n - 1 of a plan, enqueued in order from one
 * call (n >= 0, else SDM_ECOUNT; every step inside 0..T-1, else SDM_EROW). All checks come before
 * the first launch; a positive return is the cudaError_t of the first failed launch (the steps
 * before it were launched, none after it).
 */
int sdm_decode_plan_walk(const sdm_decode_plan* plan, int t0, int n, unsigned flags, sdm_stream_t stream);

/*
 * sdm_gather - token gather (gather_cuda.py, module docstring and token_gather).
 *
 * For every token t in [0, tokens) and operand o in [0, n_ops):
 *     out[o][t, :] = sum_n w[o][t, n] * bank[idx[o][t, n], :]    (float32, ascending n, fmaf)
 *     stash[t, n, :] = bank[idx[0][t, n], :]                      (raw rows of operand 0)
 * Token t is padding when t % chunk >= valid_t, where valid_t = chunk_valid[t / chunk] if
 * chunk_valid is not NULL, else `valid`. Padding tokens read nothing and get zero outputs and
 * all-zero stash rows. The bank must not be written while the gather runs.
 *
 *   bank       [n_slots, hd] bank dtype (read only); 1 <= n_slots < 2^31
 *   n_ops      1 or 2; idx[1], w[1], out[1], width[1] are ignored when n_ops == 1
 *   idx[o]     [tokens, width[o]] idx dtype (same dtype for both operands)
 *   w[o]       [tokens, width[o]] w dtype: SDM_BF16 or SDM_F32 (same for both operands)
 *   out[o]     [tokens, hd] float32
 *   width[o]   1..256
 *   stash      [tokens, width[0], hd] bank dtype, or NULL for no stash
 *   tokens     >= 0, a multiple of chunk; chunk >= 1; 0 <= valid <= chunk (ignored when
 *              chunk_valid is given)
 *   chunk_valid [tokens / chunk] int32 per-chunk valid counts in 0..chunk, or NULL
 * The arrays idx, w, out and width are HOST arrays of two entries holding device pointers.
 * Outputs and the stash must not overlap the bank.
 */
int sdm_gather(const void* bank, int64_t n_slots, int hd, int bank_dtype, int n_ops, const void* const idx[2],
               const void* const w[2], float* const out[2], const int width[2], int idx_dtype, int w_dtype,
               void* stash, int64_t tokens, int chunk, int valid, const int32_t* chunk_valid, sdm_stream_t stream);

/*
 * sdm_gather_kpos - token gather with a compact snapshot of operand 0 instead of the stash
 * (gather_cuda.py, the compact-snapshot form of the kernel: `kpos`, `crow`).
 *
 * Outputs as sdm_gather. Operand 0's rows go to a snapshot of chunk * width[0] rows per chunk:
 * for every live token t and entry n with kpos[t, n] >= 0,
 *     compact[t / chunk, kpos[t, n], :] = bank[idx[0][t, n], :]
 * (kpos names the entry's first position among the chunk's sorted rows, so each distinct row is
 * stored once per chunk). Entries with kpos = -1 and padding tokens store nothing, and no other
 * snapshot row is written. An entry whose kpos is >= chunk * width[0] or whose row index is outside
 * [0, n_slots) stores nothing and raises SDM_DEV_BAD_INDEX.
 *
 *   compact    [tokens / chunk, chunk * width[0], hd] bank dtype (device), must not overlap the bank
 *   kpos       [tokens, width[0]] int32 (device)
 * Other arguments as sdm_gather (there is no stash argument).
 */
int sdm_gather_kpos(const void* bank, int64_t n_slots, int hd, int bank_dtype, int n_ops, const void* const idx[2],
                    const void* const w[2], float* const out[2], const int width[2], int idx_dtype, int w_dtype,
                    void* compact, const int32_t* kpos, int64_t tokens, int chunk, int valid,
                    const int32_t* chunk_valid, sdm_stream_t stream);

/*
 * Gather launch plan (gather_cuda.py, token_gather_dc_plan / token_gather_dc_step): the checks
 * and the launch geometry of a no-stash gather, done once; each step then only checks row0 and
 * valid and relaunches the same kernel. Meant for a loop over the slabs of one index tensor:
 * launch k reads index and weight rows [row0, row0 + tokens) and writes out[o][0 .. tokens).
 *
 * The plan is a caller-owned record (any memory the caller likes, usually a host stack or struct
 * field); the library writes it in sdm_gather_plan_init and only reads it afterwards. It holds the
 * device pointers it was given: they must stay valid (and the arrays unresized) while the plan is
 * used. It is valid on the device that was current at init, in this process, until the library is
 * unloaded. Copying the record copies the plan.
 */
#define SDM_GATHER_PLAN_BYTES 512
typedef struct sdm_gather_plan {
    uint64_t opaque[SDM_GATHER_PLAN_BYTES / 8];
} sdm_gather_plan;

/*
 * sdm_gather_plan_init - check a no-stash sdm_gather once, at the largest row0 it will be used
 * with, and record its launch in *plan. Nothing is launched.
 *
 *   plan       host pointer to the record to fill (written only when 0 is returned)
 *   idx[o], w[o] [rows, width[o]]: the whole index / weight arrays of operand o (device)
 *   out[o]     [tokens, hd] float32, written by every launch (device)
 *   rows       index rows the arrays hold; row0_max >= 0 with row0_max + tokens <= rows
 *   tokens, chunk  tokens per launch (>= 0, a multiple of chunk), chunk >= 1
 * Other arguments as sdm_gather. Returns 0, an SDM_E* code, or a cudaError_t from the device
 * queries and settings (current device, multiprocessor count, the kernel's shared-memory limit,
 * occupancy).
 */
int sdm_gather_plan_init(sdm_gather_plan* plan, const void* bank, int64_t n_slots, int hd, int bank_dtype, int n_ops,
                         const void* const idx[2], const void* const w[2], float* const out[2], const int width[2],
                         int idx_dtype, int w_dtype, int64_t rows, int64_t row0_max, int64_t tokens, int chunk);

/*
 * sdm_gather_plan_launch - one step of a plan: the planned gather over index rows
 * [row0, row0 + tokens) with `valid` live tokens per chunk (the tokens at t % chunk >= valid are
 * padding, as in sdm_gather). Checks, in order: the record (SDM_EPLAN), 0 <= row0 <= row0_max
 * (SDM_EROW), 0 <= valid <= chunk (SDM_ECHUNK), the current device (SDM_EDEVICE); then launches
 * on `stream` exactly what sdm_gather would launch for the same rows. Returns 0, an SDM_E* code
 * (nothing launched) or the cudaError_t of a failed launch.
 */
int sdm_gather_plan_launch(const sdm_gather_plan* plan, int64_t row0, int valid, sdm_stream_t stream);

/*
 * sdm_gather_plan_launch_ex - sdm_gather_plan_launch with flags; flags == 0 is
 * sdm_gather_plan_launch. SDM_INPUTS_READY promises that the launch's index and weight rows
 * [row0, row0 + tokens) were complete before the kernel enqueued just ahead of it on the stream
 * began: the launch may then read them and warm L2 with the rows they name before it waits for
 * that kernel (which may still be writing the bank). The bank is read, and the outputs written,
 * only after the wait; results are the same bits as without the flag. Unknown bits return
 * SDM_EFLAGS before any other check.
 */
int sdm_gather_plan_launch_ex(const sdm_gather_plan* plan, int64_t row0, int valid, unsigned flags,
                              sdm_stream_t stream);

/*
 * sdm_gather_plan_walk - n steps of a plan from one call: the native step loop over a walk of
 * slabs (sparse-delta-memory 2.0.0, cuda/gather_cuda.py: `token_gather_dc_step` driven from a
 * native loop), without a host-language call per slab.
 *
 *   row0[i]    host array of n slab offsets (each 0 <= row0[i] <= row0_max)
 *   valid[i]   host array of n live-token counts per chunk (0..chunk), or NULL: chunk for every slab
 *   n          slabs, >= 0
 *   flags      0 or SDM_INPUTS_READY (applies to every slab; see sdm_gather_plan_launch_ex)
 * Slab i is exactly sdm_gather_plan_launch_ex(plan, row0[i], valid[i], flags, stream), enqueued in
 * order on `stream`. Every argument is checked before the first launch: an SDM_E* code means
 * nothing was launched. A positive return is the cudaError_t of the first failed launch; the
 * slabs before it were launched, none after it.
 */
int sdm_gather_plan_walk(const sdm_gather_plan* plan, const int64_t* row0, const int32_t* valid, int n,
                         unsigned flags, sdm_stream_t stream);

/* A static string naming a return code of the calls above. */
const char* sdm_status_string(int status);

/*
 * sdm_device_status - read (and, if clear != 0, reset) the device status word of the current
 * device: an OR of SDM_DEV_* bits raised by kernels since the last reset. Synchronises the whole
 * device first (cudaDeviceSynchronize), so that the kernels of every stream, non-blocking streams
 * included, have finished before the word is read or cleared; not for use inside graph capture.
 * Returns 0 or a cudaError_t (then *status is 0); *status receives the word.
 */
int sdm_device_status(unsigned int* status, int clear);

/* Library version, major * 10000 + minor * 100 + patch. */
int sdm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SDM_H */
