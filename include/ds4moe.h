/*
 * ds4moe.h -- C ABI of libds4moe: the routed mixture-of-experts FFN of one
 * DeepSeek-V4-Flash-shaped layer on one GB300 GPU (sm_103a).
 *
 * What the layer computes (by page title and section):
 *   - "DeepSeek V4 Flash -- DFlash Integration", Model Architecture: hidden
 *     4096; 256 routed experts, top-6, plus 1 shared; expert FFN 2048; the
 *     first 3 layers route by a token-ID -> expert table, the others by
 *     "top-k over learned router + optional bias"; Execution Modes
 *     (--ds4-expert-top-k): the kept experts' weights are renormalised.
 *   - "Baekpica/ds4 dfm Edition" README, two-bank batching notes: the router
 *     returns selected expert IDs and normalized weights; the expert path is
 *     gate/up, weighted SwiGLU, expert down, plus the shared expert.
 *   - DwarfStar README, Model Weights: routed experts 2-bit, shared experts
 *     and router kept at higher precision (Q8_0, "SExpQ8").
 *   - ds4-rocm fork README, __launch_bounds__ list: activations are
 *     pre-quantised to int8 for the Q8_0 matmuls ("_preq" kernels).
 *
 * Every float operation follows one fixed binary32 order (the canonical
 * arithmetic spec): the library's results are bit-identical to a scalar
 * CPU evaluation of the same spec, for every token count and every code path.
 *
 * Conventions for every entry point:
 *   - Pointers are CUDA device pointers unless the name says host.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   - Argument and shape errors are detected on the host before anything is
 *     enqueued; the call then returns an error status and changes nothing.
 *   - ds4moe_route / ds4moe_forward enqueue work only: no allocation, no
 *     host synchronisation, so they may be captured in a CUDA graph.
 *   - Data errors found on the device (a hash token id outside [0, vocab),
 *     a non-finite activation) never trap: the device sets a flag that
 *     ds4moe_get_device_error reports; an out-of-range token contributes
 *     nothing to y.
 *   - One handle must not be used on two streams at once; distinct handles
 *     are independent.
 */
#ifndef DS4MOE_H
#define DS4MOE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DS4MOE_ABI_VERSION 1

typedef enum {
  DS4MOE_OK = 0,
  DS4MOE_ERR_INVALID_ARG = 1, /* bad pointer, shape, format or token count */
  DS4MOE_ERR_UNSUPPORTED = 2, /* valid request the library does not handle */
  DS4MOE_ERR_OOM = 3,         /* device allocation failed                  */
  DS4MOE_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed      */
  DS4MOE_ERR_DEVICE = 5       /* the device error flag was set             */
} ds4moe_status;

/* Weight formats (canonical byte layouts; all little endian).
 *   DS4MOE_F32  : row-major binary32 (router only).
 *   DS4MOE_Q8_0 : blocks of 32 weights, 34 bytes: fp16 d, int8 q[32];
 *                 w_i = d * q_i.
 *   DS4MOE_Q2S  : superblocks of 256 weights, 84 bytes:
 *                 uint8 sm[16] | uint8 qs[64] | fp16 d | fp16 dmin;
 *                 group g = i/16, sc = sm[g] & 15, mn = sm[g] >> 4,
 *                 q_i = (qs[i/4] >> 2*(i%4)) & 3,
 *                 w_i = d*sc*q_i - dmin*mn   (2.625 bits per weight).
 *   DS4MOE_Q4S  : superblocks of 256 weights, 148 bytes (routed experts of
 *                 the 4-bit layers; this library's own layout -- the DwarfStar
 *                 README, Model Weights, names a "q2 with the last 6 layers
 *                 q4" variant but not its bytes):
 *                 uint8 sm[16] | uint8 qs[128] | fp16 d | fp16 dmin;
 *                 group g = i/16, sc = sm[g] & 15, mn = sm[g] >> 4,
 *                 q_i = (qs[i/2] >> 4*(i%2)) & 15,
 *                 w_i = d*sc*q_i - dmin*mn   (4.625 bits per weight).
 * A matrix [R][K] is R rows of K/32 (Q8_0) or K/256 (Q2S, Q4S) blocks, rows
 * contiguous; expert tensors stack their E matrices contiguously. */
typedef enum { DS4MOE_F32 = 0, DS4MOE_Q8_0 = 1, DS4MOE_Q2S = 2, DS4MOE_Q4S = 3 } ds4moe_fmt;

typedef enum { DS4MOE_ROUTE_LEARNED = 0, DS4MOE_ROUTE_HASH = 1 } ds4moe_route_kind;

/* Device error flag bits (ds4moe_get_device_error). */
#define DS4MOE_DEVERR_TOKEN_ID 1u   /* hash token id outside [0, vocab)     */
#define DS4MOE_DEVERR_NONFINITE 2u  /* non-finite activation quantised      */
#define DS4MOE_DEVERR_TIMEOUT 4u    /* a bounded on-chip wait gave up       */
#define DS4MOE_DEVERR_INTERNAL 8u   /* an internal consistency check failed */

typedef struct {
  uint32_t abi_version; /* = DS4MOE_ABI_VERSION */
  int32_t hidden;       /* H: multiple of 256 (4096 for DeepSeek-V4-Flash)          */
  int32_t n_experts;    /* E routed experts, 1..1024 (256)                          */
  int32_t top_k;        /* k, 1..min(E, 16) (6)                                     */
  int32_t ffn;          /* F: multiple of 64; of 256 with Q2S/Q4S matrices (2048)   */
  int32_t n_shared;     /* 0 or 1 shared expert, always added with weight 1         */
  int32_t route;        /* ds4moe_route_kind                                        */
  int32_t vocab;        /* hash routing: table rows (129280); ignored otherwise     */
  int32_t router_fmt;   /* DS4MOE_F32 or DS4MOE_Q8_0 (learned routing)              */
  int32_t routed_fmt;   /* DS4MOE_Q8_0, DS4MOE_Q2S or DS4MOE_Q4S                    */
  int32_t shared_fmt;   /* DS4MOE_Q8_0, DS4MOE_Q2S or DS4MOE_Q4S                    */
  float route_scale;    /* multiplies the renormalised routed weights (1.0)         */
  int32_t max_tokens;   /* largest n_tok of any later call, 1..1048576. A call of   */
                        /* fewer than 65 tokens runs on the decode path in chunks  */
                        /* of at most 64 tokens; a larger one (when hidden and ffn */
                        /* are multiples of 128) on the prefill path in chunks of  */
                        /* at most 4096 tokens. Scratch is sized at create for     */
                        /* Ts = max(min(max_tokens, 64), min(max_tokens, 4096))    */
                        /* tokens: about 560 MB at 4096 tokens and the DS4 shape   */
} ds4moe_layer_desc;

/* Canonical weight buffers, DEVICE memory, read only during ds4moe_create
 * (the library keeps its own re-laid-out copy; the caller may free these
 * when create returns). Unused pointers may be NULL. */
typedef struct {
  const void *router_w;       /* [E][H] router_fmt                (learned)   */
  const float *router_bias;   /* [E] selection bias               (learned)   */
  const int32_t *hash_table;  /* [vocab][k] expert ids in [0, E)  (hash)      */
  const void *gate, *up;      /* [E][F][H] routed_fmt                         */
  const void *down;           /* [E][H][F] routed_fmt                         */
  const void *sh_gate, *sh_up;/* [F][H] shared_fmt                (n_shared)  */
  const void *sh_down;        /* [H][F] shared_fmt                (n_shared)  */
} ds4moe_weights;

typedef struct ds4moe_layer ds4moe_layer; /* opaque handle */

/* Validate `desc`, allocate the handle's device memory on the current device
 * (weights in the library's layout plus scratch for one chunk of tokens),
 * re-lay out the weights, and synchronise. On success *out owns all of it;
 * on error *out is NULL and nothing stays allocated.
 * Errors: INVALID_ARG (desc, missing or non-device pointer), UNSUPPORTED
 * (a shape whose kernels do not fit one SM, e.g. more than ~700 experts),
 * OOM, CUDA. */
ds4moe_status ds4moe_create(const ds4moe_layer_desc *desc, const ds4moe_weights *w,
                            ds4moe_layer **out);

/* Release everything the handle owns (synchronises the device). NULL is a no-op. */
void ds4moe_destroy(ds4moe_layer *h);

/* Routing only (steps: int8 quantisation of x, router GEMV, sigmoid,
 * bias-for-selection top-k, renormalisation; or the hash-table lookup).
 * Passages: "DeepSeek V4 Flash -- DFlash Integration", Model Architecture
 * (routed experts chosen by top-k over a learned router plus an optional
 * bias; the first layers route by a token-ID table) and Execution Modes
 * (--ds4-expert-top-k: the kept experts' weights are renormalised).
 *   x        [n_tok][H] fp32 (learned routing; may be NULL for hash)
 *   token_ids[n_tok] int32 (hash routing; may be NULL for learned)
 *   ids_out  [n_tok][k] int32: expert ids in descending key order
 *            (hash: table order); -1 for an out-of-range token id
 *   w_out    [n_tok][k] fp32: renormalised weights * route_scale (0 for -1)
 * n_tok in 0..max_tokens. Enqueued on `stream`. */
ds4moe_status ds4moe_route(ds4moe_layer *h, const float *x, const int32_t *token_ids, int32_t n_tok,
                           int32_t *ids_out, float *w_out, void *stream);

/* Routing without a handle and without any device allocation.
 * No counterpart in the pages: they describe no allocation-free entry point.
 * It exists for callers that cannot call cudaMalloc: plug-ins and embedders
 * whose host application owns all device memory (for example a serving engine
 * that reserves the GPU's memory up front and accounts for every byte, so an
 * allocation behind its back fails or breaks its budget), and code paths that
 * cannot afford cudaMalloc's implicit device-wide synchronisation.
 *
 * Computes exactly what ds4moe_route computes (same ids, same weight bits)
 * from the caller's canonical buffers, read on every call:
 *   desc: hidden, n_experts, top_k, route, vocab, router_fmt and route_scale
 *         are used (same rules as ds4moe_create); the other fields are ignored.
 *   w:    router_w + router_bias (learned) or hash_table (hash), device memory;
 *         other members are ignored.
 *   x, token_ids, ids_out, w_out: as for ds4moe_route.
 *   err_flags: device uint32, may be NULL; DS4MOE_DEVERR_* bits are OR-ed in
 *         (a hash-table entry outside [0, n_experts) gives id -1, weight 0
 *         and DS4MOE_DEVERR_INTERNAL).
 * Scratch: one fixed device array of DS4MOE_NOALLOC_SCRATCH_BYTES (512 KiB)
 * per device, built into the library. Learned routing needs
 * n_tok * 32 * E_pad bytes of it (E_pad = n_experts rounded up to 32): at most
 * 64 tokens per call for 256 experts. A larger n_tok returns
 * DS4MOE_ERR_UNSUPPORTED and enqueues nothing. Hash routing uses no scratch.
 * Nothing in the array has to start at zero; a call reads only what it wrote.
 * Every call on a device shares the one array, so calls whose work can
 * overlap on the GPU (issued on different streams without an order between
 * them, or from several host threads) race and give wrong results: issue
 * them on one stream, or order them.
 * The first call on each device, with that device current, looks up the
 * array's address (cudaGetSymbolAddress) and sets a kernel attribute; make
 * that first call before any stream capture.
 * Errors: INVALID_ARG (desc, pointers, n_tok < 0), UNSUPPORTED (scratch too
 * small for n_tok), CUDA. */
#define DS4MOE_NOALLOC_SCRATCH_BYTES (512u * 1024u)
ds4moe_status ds4moe_route_noalloc(const ds4moe_layer_desc *desc, const ds4moe_weights *w, const float *x,
                                   const int32_t *token_ids, int32_t n_tok, int32_t *ids_out, float *w_out,
                                   uint32_t *err_flags, void *stream);

/* The whole layer: y[t] += MoE(x[t]) for t < n_tok, i.e.
 * Passages: "DeepSeek V4 Flash -- DFlash Integration", Model Architecture
 * (256 routed experts top-6 plus 1 shared, expert FFN 2048) and Forward Pass
 * (the MoE FFN adds its output to the residual stream); "Baekpica/ds4 dfm
 * Edition" README, two-bank batching notes (router -> top-k -> gate/up ->
 * weighted SwiGLU -> expert down, plus the shared expert).
 *   y[t] += sum_j w_j * down_j(hq_j) + shared(x[t])
 * with hq_j the int8-requantised silu(gate_j x) * (up_j x).
 *   x         [n_tok][H] fp32, read only
 *   token_ids [n_tok] int32, required for hash routing, else may be NULL
 *   y         [n_tok][H] fp32, read and written (must not alias x)
 * n_tok in 0..max_tokens. Enqueued on `stream`; no host synchronisation.
 * Calls of fewer than 65 tokens take the decode path (router, gate/up and
 * down kernels, chunks of at most 64 tokens; units of eight tokens take
 * their int8 block dots from the tensor cores); larger calls the prefill
 * path (tensor-core grouped GEMMs, chunks of at most 4096 tokens; when hidden
 * and ffn are multiples of 128, else the decode path). All give the same
 * bits. */
ds4moe_status ds4moe_forward(ds4moe_layer *h, const float *x, int32_t n_tok, const int32_t *token_ids,
                             float *y, void *stream);

/* One layer of a stack: the RMSNorm with unit gain of ds4moe_rmsnorm (same
 * arithmetic, same bits) folded into the forward,
 *   y[t] += MoE(x[t] / sqrt(mean(x[t]^2) + eps)),
 * for a residual stream that passes RMSNorm, then the MoE FFN added to it
 * ("DeepSeek V4 Flash -- DFlash Integration", Forward Pass). From two tokens
 * on (and on the prefill path) the router kernel normalises the rows as it
 * quantises them, so no normalised copy is written and no extra kernel runs;
 * a one-token decode call runs the RMSNorm kernel into a row buffer of the
 * handle first (faster there). Bit-identical to ds4moe_rmsnorm into a
 * buffer followed by ds4moe_forward on it.
 *   x  [n_tok][H] fp32, read only, 16-byte aligned
 *   y  [n_tok][H] fp32, read and written; may be x itself (y += on the
 *      residual in place: every read of x completes before any write of y),
 *      else must not overlap it
 * Other arguments, paths, errors and stream behaviour as ds4moe_forward;
 * DS4MOE_ERR_INVALID_ARG also for a NaN eps, an unaligned x or a partial
 * overlap of x and y. */
ds4moe_status ds4moe_forward_rmsnorm(ds4moe_layer *h, const float *x, int32_t n_tok, const int32_t *token_ids,
                                     float eps, float *y, void *stream);

/* ds4moe_forward on HOST buffers (pinned or pageable): y_host += MoE(x_host),
 * synchronising `stream` before it returns. Decode-sized calls (n_tok up to
 * min(max_tokens, 64)) on pinned buffers: the kernels read x and token_ids
 * and update y in them directly over the CPU-GPU link. Decode-sized calls on
 * pageable buffers copy them into mapped pinned buffers owned by the handle
 * and replay one CUDA graph per token count (captured on the first call of
 * that count; kept until ds4moe_destroy). Larger calls copy x, the token
 * ids and y to device staging buffers chunk by chunk (Ts tokens at a time,
 * see max_tokens), run the layer on each chunk and copy y back.
 * Memory: the first call allocates, and keeps until ds4moe_destroy, device
 * staging of 2 * Ts * hidden * 4 + Ts * 4 bytes (about 128 MB at Ts = 4096,
 * hidden 4096) and, for pageable callers, 2 * min(max_tokens, 64) * hidden * 4
 * + min(max_tokens, 64) * 4 bytes of mapped pinned host memory. Not reentrant
 * on one handle. Same arguments otherwise. */
ds4moe_status ds4moe_forward_host(ds4moe_layer *h, const float *x_host, int32_t n_tok,
                                  const int32_t *token_ids_host, float *y_host, void *stream);

/* RMSNorm with unit gain between stacked layers:
 *   out[t] = x[t] / sqrt(mean(x[t]^2) + eps)   (x, out [n_tok][hidden] fp32;
 * out may equal x). hidden must be a multiple of 32. (DFlash Integration page,
 * Forward Pass, step 5: RMSNorm before the output projection.) */
ds4moe_status ds4moe_rmsnorm(const float *x, float *out, int32_t n_tok, int32_t hidden, float eps,
                             void *stream);

/* Synchronise `stream`, read and clear the handle's device error flag.
 * *flags_out (may be NULL) receives the DS4MOE_DEVERR_* bits.
 * When DS4MOE_DEVERR_TIMEOUT is among them, a kernel gave up a bounded wait
 * and left some cross-block completion counters unfinished: this call also
 * zeroes them (and synchronises the device), so the next call starts from a
 * clean state. Outputs of calls made between the timeout and this call are
 * undefined.
 * Returns DS4MOE_ERR_DEVICE when any bit was set, else DS4MOE_OK. */
ds4moe_status ds4moe_get_device_error(ds4moe_layer *h, void *stream, uint32_t *flags_out);

/* Read-only device view of the handle's scratch after the last forward call,
 * for inspecting intermediate results. With C = Ts (see max_tokens) and
 * NS = k + n_shared, `which`:
 *   0 xq  int8  [C][H]        activation codes (CAS step 1)
 *   1 dx  fp32  [C][H/32]     activation scales
 *   2 gs  int16 [C][H/16]     16-group sums of xq
 *   3 ids int32 [C][k]        routed expert ids
 *   4 w   fp32  [C][k]        renormalised weights
 *   5 hq  int8  [C*NS][F]     SwiGLU codes, row t*NS+slot (slot k = shared)
 *   6 dh  fp32  [C*NS][F/32]  SwiGLU scales
 *   7 a   fp32  [C*NS][H]     per-slot down-projection outputs
 * Rows refer to the tokens of the last chunk of that call (64 tokens at most
 * on the decode path, 4096 on the prefill path); other rows are undefined.
 * Errors: INVALID_ARG for an unknown `which`. */
ds4moe_status ds4moe_debug_scratch(ds4moe_layer *h, int32_t which, const void **ptr_out, uint64_t *bytes_out);

/* Per-stage timing with CUDA events recorded on the call's stream.
 * ds4moe_profile_enable(h, 1) makes every later ds4moe_forward record an
 * event before each stage and after the last one; ds4moe_profile_collect
 * waits for the last forward's events and adds the stage durations to the
 * handle's totals; ds4moe_profile_read copies the totals (milliseconds,
 * summed over collected calls) for the stages
 *   0 quantise x, 1 route (router GEMV + top-k, or hash), 2 bucket,
 *   3 gate/up, 4 down, 5 combine
 * into ms_out[0..n) and the number of collected calls into *calls.
 * ds4moe_profile_enable(h, 0) stops recording and zeroes the totals.
 * Profiling adds event records to the stream; it is off by default. */
#define DS4MOE_N_STAGES 6
ds4moe_status ds4moe_profile_enable(ds4moe_layer *h, int32_t on);
ds4moe_status ds4moe_profile_collect(ds4moe_layer *h);
ds4moe_status ds4moe_profile_read(const ds4moe_layer *h, double *ms_out, int32_t n, int64_t *calls);

/* ---------------------------------------------------------------------------
 * Dense Q8_0 product beside the MoE: y = W x for the output head (129280 x
 * 4096, "OutQ8") and the attention projections, on activations pre-quantised
 * to int8 per 32-block.
 * Passages: ds4-rocm fork README, Performance optimizations (the
 * matmul_q8_0_preq_* kernels: Q8_0 matmuls on pre-quantised activations, the
 * largest share of decode time beside the MoE); DwarfStar README, Model
 * Weights (the OutQ8 model name).
 * Arithmetic (canonical spec): x quantised as for the MoE (CAS step 1); each
 * output is the CAS row sum of its Q8_0 block terms (d * dx) * I over
 * S = min(8, n_in/32) contiguous segments, as for an expert row.
 *
 * ds4moe_dense_create: w_q8 is the canonical [n_out][n_in] Q8_0 matrix (rows
 *   of n_in/32 blocks of 34 bytes) in DEVICE memory, read only during the call
 *   (re-laid out into a handle-owned copy; rows padded to a multiple of 32).
 *   n_out 1..2^24; n_in a multiple of 32, up to 65536, with n_in/32 a multiple
 *   of min(8, n_in/32); max_tokens 1..65536 sizes the activation scratch
 *   and the segment-sum scratch of split rows (min(8, n_in/32) x
 *   min(max_tokens, 8) x n_out floats). Synchronises. Errors: INVALID_ARG,
 *   UNSUPPORTED (n_in too wide for a block's shared memory), OOM, CUDA; on
 *   error *out is NULL.
 * ds4moe_dense_forward: y[t][n] = sum_k W[n][k] x[t][k] for t < n_tok
 *   (x [n_tok][n_in] fp32, y [n_tok][n_out] fp32, overwritten; device
 *   pointers), enqueued on `stream` (two launches, three for split rows; no
 *   allocation, no host synchronisation). Built for decode-sized n_tok: the
 *   matrix is streamed once per pass of up to 8 tokens (fewer for very wide
 *   n_in); from two tokens on the integer block dots run on the tensor
 *   cores (the int8 codes as fp16 with f32 accumulation: every partial sum
 *   is an integer below 2^24, so the dots are exact and the bits the same);
 *   a call of one pass may split rows over several warps by whole
 *   segments, whose sums a third launch adds in segment order (the same bits
 *   as unsplit). Calls on one handle must not run concurrently (shared
 *   scratch).
 *   Errors: INVALID_ARG (pointers, n_tok outside 0..max_tokens), CUDA.
 * ds4moe_dense_get_device_error: as ds4moe_get_device_error, for the dense
 *   handle's flag (DS4MOE_DEVERR_NONFINITE, DS4MOE_DEVERR_TIMEOUT).
 * ds4moe_dense_destroy: releases everything (synchronises); NULL is a no-op. */
typedef struct ds4moe_dense ds4moe_dense;
ds4moe_status ds4moe_dense_create(int32_t n_out, int32_t n_in, int32_t max_tokens, const void *w_q8,
                                  ds4moe_dense **out);
ds4moe_status ds4moe_dense_forward(ds4moe_dense *h, const float *x, int32_t n_tok, float *y, void *stream);
ds4moe_status ds4moe_dense_get_device_error(ds4moe_dense *h, void *stream, uint32_t *flags_out);
void ds4moe_dense_destroy(ds4moe_dense *h);
uint64_t ds4moe_dense_device_bytes(const ds4moe_dense *h);
uint64_t ds4moe_dense_launch_count(const ds4moe_dense *h);
/* ds4moe_dense_debug_config: overrides the dense kernel's launch geometry for
 *   later calls (a tuning and test hook; the results are the same bits under
 *   every setting): ks = K steps per ring stage (a divisor of n_in/32/S, at
 *   most 8), nst = ring stages per warp (2..6, within shared memory), ns =
 *   units per 32-row item (a divisor of S), tc = the block-dot step: 1 the
 *   dp4a step only, 2 the tensor-core step for every call (where eight
 *   tokens' fp16 codes fit a pass; the automatic choice takes it from two tokens
 *   on). 0 keeps the automatic choice of that value. A call whose tokens do
 *   not fit one pass of the segment-sum scratch runs unsplit (ns = 1)
 *   whatever ns says; a (ks, nst) that does not fit a call's shared memory
 *   falls back to the automatic ring.
 *   Errors: INVALID_ARG (NULL, a value outside its range). */
ds4moe_status ds4moe_dense_debug_config(ds4moe_dense *h, int32_t ks, int32_t nst, int32_t ns, int32_t tc);

/* Test hooks for failure detection (no counterpart in the pages; they make
 * failures happen on the host side or through a short wait bound, never by
 * faulting the GPU).
 * ds4moe_debug_set_wait_limit: bound, in SM cycles, of the hand-off waits of
 *   the decode path's expert kernels (a warp waiting for another warp of its
 *   block, or for the router's count of quantised x); 0 restores the default
 *   (about 2^31 cycles). A wait that runs out raises DS4MOE_DEVERR_TIMEOUT
 *   and its block leaves; waits for the block's own copies keep the default
 *   bound, so no copy is left in flight. Errors: INVALID_ARG (NULL, < 0).
 * ds4moe_debug_fail_alloc: the n-th device allocation the library makes
 *   from now on (in ds4moe_create, or the first ds4moe_forward_host) fails
 *   as if the device were out of memory; 0 turns it off. Process-wide.
 *   Errors: INVALID_ARG (n < 0). */
ds4moe_status ds4moe_debug_set_wait_limit(ds4moe_layer *h, int64_t cycles);
ds4moe_status ds4moe_debug_fail_alloc(int32_t n);

/* Number of kernels this handle has launched since create. */
uint64_t ds4moe_launch_count(const ds4moe_layer *h);

/* Bytes of device memory the handle owns (weights + scratch). */
uint64_t ds4moe_device_bytes(const ds4moe_layer *h);

/* Human-readable status name (static storage). */
const char *ds4moe_status_string(ds4moe_status s);

/* = DS4MOE_ABI_VERSION of the loaded library. */
uint32_t ds4moe_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DS4MOE_H */
