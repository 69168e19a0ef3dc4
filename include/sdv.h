/*
 * sdv.h -- C ABI of libsdv, the GB300 (sm_103a) kernels of the verify forward
 * of greedy speculative decoding.
 *
 * The operations and where they are defined:
 *
 *  - per-block-32 absmax symmetric int8 / int4 weight quantisation:
 *    "Riding Apple's pipelined GPU engine -- 3.5x over a hand-rolled loop, zero
 *    custom kernels", section "Quantization on the GPU delegate" (int8 linear
 *    per-block-32 is the ship configuration; q4_0 is per-block-32 absmax
 *    symmetric int4; big-vocabulary heads use plain absmax, never clipping);
 *  - the verify forward over a static window of S = K+1 rows:
 *    "Spec-decode on GDN hybrids (Qwen3.5/3.6 family) -- static-S verify
 *    design", section "Verify graph = STATIC S=K+1 + chunked GDN scan", and
 *    "Stream C -- Speculative decoding: feasibility verdict + implementation
 *    plan", section "TL;DR" (a K-token verify forward costs about one decode
 *    step: it is bound by reading the weights once);
 *  - the batched on-GPU argmax [S, vocab] -> [S] and the greedy accept rule:
 *    "Stream C ...", section "The delta -- new ENGINE work for greedy n-gram
 *    spec-decode", and "Spec-decode on GDN hybrids ...", section "Hybrid state
 *    discipline" (a0 is committed first; the row after the last accepted draft
 *    becomes the next a0; pad drafts are never accepted);
 *  - only the sampled ids cross back to the host: "Riding Apple's pipelined GPU
 *    engine", section "Why hand-rolled per-token loops lose ~3x";
 *  - the fused SwiGLU MLP: "Flagship dramatic-speedup plan -- the full stackable
 *    tuning set", section "Axis 4 -- kernel micro-opts";
 *  - gathered routed experts (top-8 of 256): same page, section "Baseline byte
 *    model".
 *
 * Conventions for every entry point:
 *  - Tensor pointers are DEVICE pointers owned by the caller; the library never
 *    allocates, frees or keeps state between calls.  Row-major everywhere.
 *  - fp16 values (activations, scales, h) are passed as IEEE binary16 bit
 *    patterns (uint16_t).
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  Results are valid once the stream has been synchronised.
 *  - Arguments are validated on the host before any launch; an invalid argument
 *    returns an error and launches nothing.  Errors are returned, never thrown,
 *    and the library never exits the process.
 *  - Weight code and scale pointers, activation pointers and workspaces must be
 *    16-byte aligned (weights are read by the Tensor Memory Accelerator).
 *  - Workspaces ("ws") are caller-owned device scratch of at least
 *    sdv_workspace_bytes(...) bytes, ZERO-FILLED before their first use
 *    (sdv_workspace_init does it).  Every completed call leaves the workspace's
 *    counters back at zero, so one workspace serves any number of calls issued
 *    in stream order.  Calls that overlap on the GPU must not share a workspace.
 */
#ifndef SDV_H
#define SDV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SDV_API __attribute__((visibility("default")))
#else
#define SDV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the runtime's stream handle), declared without CUDA headers. */
typedef struct CUstream_st* sdv_stream_t;

typedef enum {
  SDV_OK = 0,
  SDV_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, n_valid out of range */
  SDV_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels handle (e.g. S > 32) */
  SDV_ERR_CUDA = 3,        /* a CUDA runtime error while launching */
  SDV_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up (see sdv_last_device_status) */
  SDV_ERR_WORKSPACE = 5    /* workspace null, misaligned or smaller than required */
} sdv_status;

typedef enum { SDV_Q8 = 8, SDV_Q4 = 4, SDV_F4 = 2 } sdv_qtype;

/* Operation ids for sdv_workspace_bytes. */
typedef enum {
  SDV_OP_QLINEAR = 1,
  SDV_OP_QLINEAR_SWIGLU = 2,
  SDV_OP_VERIFY_HEAD = 3,
  SDV_OP_MOE = 4,
  SDV_OP_VERIFY_SAMPLE = 5
} sdv_op;

/*
 * A per-block-32 quantised weight W[n, k] (n output rows, reduction length k,
 * k % 32 == 0).  Block b of row r covers W[r, 32b .. 32b+31] and has one fp16
 * scale s[r, b]; the weight is q * s with q in [-127, 127] (Q8) or [-7, 7] (Q4),
 * or an FP4 value (F4).
 *   Q8: codes = int8  [n][k]    (one two's-complement byte per weight)
 *   Q4: codes = uint8 [n][k/2]  (two's-complement nibbles; byte i of a row holds
 *                                 weight 2i in bits 0-3 and weight 2i+1 in bits 4-7)
 *   F4: codes = uint8 [n][k/2]  (E2M1 nibbles as in the OCP Microscaling spec:
 *                                 sign bit 3, magnitude index 0..7 for 0, 0.5, 1,
 *                                 1.5, 2, 3, 4, 6; nibble order as Q4).  The
 *                                 pages' "FP4 (E2M1)" 4-bit lever ("Flagship
 *                                 dramatic-speedup plan", Axis 1, lever 1c).
 *                                 Computed on the tensor-core path only:
 *                                 SDV_ERR_UNSUPPORTED where its plan does not fit
 *                                 and no row chunking applies.
 *   scales = fp16 [n][k/32]
 */
typedef struct {
  int32_t qtype;          /* SDV_Q8, SDV_Q4 or SDV_F4 */
  int32_t n;              /* output rows, >= 1 */
  int32_t k;              /* reduction length, >= 32, multiple of 32 */
  const void* codes;      /* device, 16-byte aligned */
  const uint16_t* scales; /* device, 16-byte aligned */
} sdv_qweight;

/*
 * Quantise fp32 w[n][k] per block of 32 along k:  s32 = max|w| / Q (IEEE fp32
 * division), s = fp16(s32) rounded to nearest even, q = clamp(rint(w / s), -Q, Q)
 * (IEEE fp32 division, ties to even); s == 0 gives q = 0.  Q = 127 (SDV_Q8) or
 * 7 (SDV_Q4).  SDV_F4: s32 = max|w| / 6 and the code of r = w / s is the nearest
 * E2M1 magnitude, ties to the even mantissa bit, saturating at 6, with the sign
 * bit set for r < 0 unless the magnitude is 0.  Writes `codes` in the
 * sdv_qweight layout of `qtype` and `scales` fp16 [n][k/32].  No workspace.
 */
SDV_API sdv_status sdv_quantize_block32(const float* w, int32_t n, int32_t k, int32_t qtype,
                                void* codes, uint16_t* scales, sdv_stream_t stream);

/*
 * Dequantised skinny GEMM:  y[s][r] = sum_h x[s][h] * q[r][h] * s[r][h/32]
 * for s < S, r < w->n; fp16 activations, fp32 accumulation, fp32 output.
 *   x: fp16 [S][w->k];  y: fp32 [S][w->n];  1 <= S <= 32.
 */
SDV_API sdv_status sdv_qlinear(const sdv_qweight* w, const uint16_t* x, int32_t S, float* y,
                       void* ws, size_t ws_bytes, sdv_stream_t stream);

/*
 * Fused SwiGLU gate/up projection: h[s][r] = fp16( SiLU(g) * u ) with
 * g = (x G^T)[s][r], u = (x U^T)[s][r] accumulated in fp32 and
 * SiLU(t) = t / (1 + exp(-t)); the result is rounded once to fp16 (nearest even).
 * gate and up must have equal n, k and qtype.   x: fp16 [S][k];  h: fp16 [S][n].
 */
SDV_API sdv_status sdv_qlinear_swiglu(const sdv_qweight* gate, const sdv_qweight* up,
                              const uint16_t* x, int32_t S, uint16_t* h,
                              void* ws, size_t ws_bytes, sdv_stream_t stream);

/*
 * The verify head over one window [a0, d_1 .. d_{S-1}]:
 *   logits[s][v] = sum_h x[s][h] * q[v][h] * s[v][h/32]        (fp32 accumulate)
 *   argmax[s]    = the lowest v with logits[s][v] == max_v' logits[s][v']
 *   accepted     = the largest j <= n_valid with drafts[i] == argmax[i] for all i < j
 *   next_a0      = argmax[accepted]   (the correction on a miss, the bonus token
 *                                       when all n_valid drafts were accepted)
 * head: the quantised lm_head, n = vocabulary size, k = hidden size.
 * x: fp16 [S][k] hidden states of the window rows (row 0 = the row of a0).
 * drafts: int32 [S-1], drafts[i] = the token at window position i+1; entries at
 *   i >= n_valid are pad and never accepted.  May be NULL when n_valid == 0.
 * n_valid: 0 <= n_valid <= S-1.
 * logits_or_null: fp32 [S][n] written when non-NULL (parity/debug; the hot path
 *   passes NULL and the full logits never leave the chip).
 * argmax: int32 [S];  accepted, next_a0: int32 [1] each.
 * One kernel launch: a persistent dequant GEMM whose epilogue reduces each
 * CTA's vocabulary slab to per-row (max, index) partials in `ws`; the last CTA
 * to finish reduces the partials and runs the accept.  When the window rows of
 * a long reduction do not fit one tensor-core launch's shared memory next to
 * its ring (e.g. k = 2560 at S >= 17), each CTA takes part of the reduction: one
 * pass over the head writes fp32 partial logits into `ws` (the workspace size
 * sdv_workspace_bytes gives for such a shape includes them), and a second
 * launch sums them in split order, takes the argmax and runs the accept.  With
 * a workspace too small for the partials (at least the size for a one-row head)
 * the rows are verified in chunks instead, each streaming the head once, and a
 * single-warp launch runs the accept.
 */
SDV_API sdv_status sdv_verify_head(const sdv_qweight* head, const uint16_t* x, int32_t S,
                           const int32_t* drafts, int32_t n_valid, float* logits_or_null,
                           int32_t* argmax, int32_t* accepted, int32_t* next_a0,
                           void* ws, size_t ws_bytes, sdv_stream_t stream);

/*
 * The sampling (temperature > 0) verify of one window: speculative sampling
 * (Leviathan, Kalman & Matias, ICML 2023) with a drafter that proposes each
 * token deterministically, the lossless temperature > 0 variant that "Stream C --
 * Speculative decoding: feasibility verdict + implementation plan" defers
 * (section "Deferred / harder": probabilities and a residual resample).
 *   p_i(v)   = softmax over v of logits[i][v] / temperature   (logits as in
 *              sdv_verify_head)
 *   samples[i] = argmax_v ( logits[i][v] / temperature + g_i(v) )   (Gumbel-max
 *              draw from p_i; ties to the lower v)
 *   accepted = the first i < n_valid with NOT (u_i < p_i(drafts[i])), else n_valid
 *   next_token = at a rejection in row i: argmax over v != drafts[i] of
 *              logits[i][v] / temperature + g_i(v) (a draw from the residual
 *              distribution); when every draft is kept: samples[n_valid]
 * Random numbers: SplitMix64 (Steele, Lea & Flood 2014) keyed by
 *   key = mix(seed + (counter + 1) * 0x9E3779B97F4A7C15); output
 *   w(c) = mix(key + (c + 1) * 0x9E3779B97F4A7C15) carries element 2c in its low
 *   and 2c + 1 in its high 32 bits h, u = (2 * (h >> 9) + 1) * 2^-24;
 *   g_i(v) = -log(-log(u)) with e = 32 * v + i; u_i with e = 32 * n + i.
 *   A caller advances `counter` once per call.
 * Arguments as for sdv_verify_head; temperature: finite and > 0 (else
 * SDV_ERR_INVALID_ARG); samples: int32 [S]; next_token: int32 [1]; the workspace
 * is sdv_workspace_bytes(SDV_OP_VERIFY_SAMPLE, n, k, S, 0, 0) bytes.  Runs on the
 * tcgen05 path only: SDV_ERR_UNSUPPORTED where its plan does not fit (window rows
 * x reduction length beyond shared memory, e.g. an int8 head with k = 2560 at S >= 17).
 * One kernel launch; fp32 logits, so a draw or an accept whose margin is below
 * the logits' rounding may differ from an fp64 evaluation.
 */
SDV_API sdv_status sdv_verify_sample(const sdv_qweight* head, const uint16_t* x, int32_t S,
                             const int32_t* drafts, int32_t n_valid, float temperature,
                             uint64_t seed, uint64_t counter, float* logits_or_null,
                             int32_t* samples, int32_t* accepted, int32_t* next_token,
                             void* ws, size_t ws_bytes, sdv_stream_t stream);

/*
 * sdv_verify_head without a workspace, for callers that cannot allocate device
 * memory: code that only receives a stream and tensors from a host framework
 * which owns all device memory and forbids side allocations, or that runs in a
 * latency-critical loop where cudaMalloc (which may synchronise the device) is
 * not allowed.  The pages have no counterpart of this entry point.
 * Same arguments, outputs, definition and argument errors as sdv_verify_head
 * minus ws/ws_bytes; every argument is checked before anything is launched.
 * Its scratch (status word, last-CTA ticket, per-CTA argmax partials) is a
 * fixed 65,792-byte device array inside the library, resident on every GPU that
 * loads the library until the process exits.  Limit: the scratch the call needs
 * (256 + 8 * S * number-of-SMs bytes) must fit, else SDV_ERR_WORKSPACE; on a
 * 152-SM GB300 every S <= 32 fits.
 * Set-up: the first call in a CUDA context looks up the array's device address
 * (cudaGetSymbolAddress) with that device current.  Under lazy module loading
 * (CUDA_MODULE_LOADING=LAZY, the default) that lookup may load this library's
 * module, and the driver then places the array in device memory; make that
 * first call at set-up, before any stream capture.  A new context (e.g. after
 * cudaDeviceReset) is detected by its id and the address looked up again.
 * Every call shares the one array and it keeps the last call's contents: each
 * call clears the ticket (which must start at zero) on `stream` first, so calls
 * that overlap on the GPU (other streams, other host threads) race and must be
 * serialised by the caller.  The status word is not cleared by a call: a bounded
 * device wait that gave up stays recorded until sdv_noalloc_device_status reads
 * it (sdv_last_device_status, which takes a workspace, does not apply).
 * The library itself allocates nothing here: no cudaMalloc, cudaFree or
 * allocating library routine.
 */
SDV_API sdv_status sdv_verify_head_noalloc(const sdv_qweight* head, const uint16_t* x, int32_t S,
                                   const int32_t* drafts, int32_t n_valid,
                                   float* logits_or_null, int32_t* argmax, int32_t* accepted,
                                   int32_t* next_a0, sdv_stream_t stream);

/*
 * Tree accept over the S rows of a tree-shaped window (the tree variant of the
 * verify that "Stream C -- Speculative decoding: feasibility verdict +
 * implementation plan" defers, section "Deferred / harder"): node 0 is the root
 * (the row of a0); node i > 0 carries the draft tokens[i] and hangs below
 * parent[i], which must lie in [0, i) -- any other value marks an absent (pad)
 * node, never accepted.  argmax[i] (device int32 [S], e.g. from
 * sdv_verify_head over the node rows) is the target's prediction after the path
 * root -> i.  Node i is accepted iff its parent is and tokens[i] ==
 * argmax[parent[i]].  The commit is the path to the deepest accepted node (the
 * lowest index among equally deep ones):
 *   accepted = its depth (accepted drafts), path[0 .. accepted-1] = the node
 *   indices from the root's child down (entries past it untouched),
 *   next_a0 = argmax[that node].
 * A chain (parent[i] = i-1 for the real drafts, -1 for pads) gives the greedy
 * accept.  tokens, parent: device int32 [S] (entry 0 ignored); path: device
 * int32 [S-1]; they may be NULL when S == 1.  One single-warp launch.
 */
SDV_API sdv_status sdv_tree_accept(const int32_t* argmax, int32_t S, const int32_t* tokens,
                           const int32_t* parent, int32_t* path, int32_t* accepted,
                           int32_t* next_a0, sdv_stream_t stream);

/*
 * Host-side n-gram drafter ("Stream C -- Speculative decoding: feasibility
 * verdict + implementation plan", section "The delta": a pure host hashtable over
 * the prompt + generated stream, the last m tokens mapping to their most recent
 * continuation).  All pointers are HOST pointers; nothing touches the GPU.
 *   sdv_ngram_create(m, &d): a drafter of order m (1 <= m <= 64).
 *   sdv_ngram_append(d, tokens, count): extend the stream.
 *   sdv_ngram_propose(d, k, drafts, &count): look up the stream's last m tokens;
 *     if an earlier occurrence with a continuation exists, copy up to k tokens
 *     from the latest one's continuation into drafts (int32 [k]) and set count,
 *     else count = 0.  Proposals are read past the stream's last token, so a
 *     loop appends its anchor token a0 before asking.
 *   sdv_ngram_destroy(d): free it (NULL is accepted).
 * Errors: SDV_ERR_INVALID_ARG for null or out-of-range arguments,
 * SDV_ERR_UNSUPPORTED when a host allocation fails.  Not thread-safe per drafter.
 */
typedef struct sdv_ngram sdv_ngram;
SDV_API sdv_status sdv_ngram_create(int32_t m, sdv_ngram** out);
SDV_API sdv_status sdv_ngram_destroy(sdv_ngram* d);
SDV_API sdv_status sdv_ngram_append(sdv_ngram* d, const int32_t* tokens, int32_t count);
SDV_API sdv_status sdv_ngram_propose(const sdv_ngram* d, int32_t k, int32_t* drafts, int32_t* count);

/*
 * The greedy accept rule alone, on a given argmax[S] (device, int32), with the
 * same definition and outputs as sdv_verify_head.  No workspace.
 */
SDV_API sdv_status sdv_greedy_accept(const int32_t* argmax, int32_t S, const int32_t* drafts,
                             int32_t n_valid, int32_t* accepted, int32_t* next_a0,
                             sdv_stream_t stream);

/*
 * Gathered-expert SwiGLU MoE over the window rows:
 *   route:   per row s, the top_k experts by router_logits[s][e] (ties to the
 *            lower id), weights w = softmax over the top_k selected logits;
 *   experts: for each selected (s, e): h = SiLU(x[s] G_e^T) * (x[s] U_e^T),
 *            y = h D_e^T;
 *   combine: out[s] = sum_j w[s][j] * y(s, e_j).
 * gate, up: stacked [E*I][H] (expert e owns rows e*I .. e*I+I-1);
 * down: stacked [E*H][I] (expert e owns rows e*H .. e*H+H-1); all the same qtype.
 * x: fp16 [S][H]; router_logits: fp32 [S][E]; out: fp32 [S][H].
 * topk_ids_or_null (int32 [S][top_k]) and topk_w_or_null (fp32 [S][top_k]) are
 * written, in selection order, when non-NULL.
 */
SDV_API sdv_status sdv_moe_gather_qmm(const sdv_qweight* gate, const sdv_qweight* up,
                              const sdv_qweight* down, int32_t E, int32_t I, int32_t H,
                              int32_t top_k, const uint16_t* x, const float* router_logits,
                              int32_t S, float* out, int32_t* topk_ids_or_null,
                              float* topk_w_or_null, void* ws, size_t ws_bytes,
                              sdv_stream_t stream);

/*
 * The MoE routing and grouping steps alone (the first launch of
 * sdv_moe_gather_qmm), for inspection and parity tests:
 *   ids, weights: int32 / fp32 [S][top_k], per row the top_k experts by
 *     router_logits (larger first, ties to the lower id) and their softmax over
 *     the selection;
 *   offsets: int32 [E+1], pair_rows: int32 [S*top_k]: the (row, expert)
 *     selections counting-sorted by expert, rows ascending within an expert;
 *     expert e's rows are pair_rows[offsets[e] .. offsets[e+1]-1];
 *   n_hit: int32 [1], hit: int32 [E]: the distinct selected experts, ascending,
 *     in hit[0 .. n_hit-1].
 * 1 <= S <= 32, top_k <= min(E, 32), E <= 1024.  All pointers are device memory.
 */
SDV_API sdv_status sdv_moe_route(const float* router_logits, int32_t S, int32_t E, int32_t top_k,
                         int32_t* ids, float* weights, int32_t* offsets, int32_t* pair_rows,
                         int32_t* n_hit, int32_t* hit, sdv_stream_t stream);

/*
 * Workspace bytes an operation needs on the current device.
 * `op` is an sdv_op; n, k are the weight's (for SDV_OP_MOE: n = I, k = H);
 * S the window rows; E, top_k for SDV_OP_MOE (ignored otherwise).
 * Returns 0 for invalid arguments (S outside [1, 32], n < 1, k not a positive
 * multiple of 32, an unknown op); the operation itself reports them.
 */
SDV_API size_t sdv_workspace_bytes(int32_t op, int32_t n, int32_t k, int32_t S, int32_t E,
                           int32_t top_k);

/* Zero-fill a workspace (cudaMemsetAsync on `stream`). */
SDV_API sdv_status sdv_workspace_init(void* ws, size_t ws_bytes, sdv_stream_t stream);

/*
 * Synchronise `stream`, then read and clear the device status word a kernel
 * leaves in `ws`: SDV_OK, or SDV_ERR_TIMEOUT if a bounded device-side wait gave
 * up (the outputs of that call are then undefined; later calls on the same
 * workspace are unaffected).  Any other flag (the tensor-memory allocation was
 * not where the kernel expects it) reads as SDV_ERR_CUDA.  The status word
 * collects the flags of every call since the last read.
 * (The boundary's "bounded-wait / debug-assert flags" read: "Stream C --
 * Speculative decoding: feasibility verdict + implementation plan", section
 * "The delta": only ids and a status cross back to the host.)
 */
SDV_API sdv_status sdv_last_device_status(void* ws, sdv_stream_t stream);

/* The same as sdv_last_device_status (the name earlier versions exported). */
SDV_API sdv_status sdv_device_status(void* ws, sdv_stream_t stream);

/*
 * The status read of sdv_verify_head_noalloc's fixed scratch on the current
 * device: synchronise `stream`, then read and clear its status word, with the
 * meaning of sdv_last_device_status.  The pages have no counterpart.
 */
SDV_API sdv_status sdv_noalloc_device_status(sdv_stream_t stream);

/*
 * Select the implementation of the weight-streaming GEMM behind sdv_qlinear and
 * sdv_verify_head (process-wide; for measurement and tests):
 *   0 = automatic: the tcgen05 path (tensor-memory accumulators, 128-row tiles)
 *       whenever its shared-memory plan fits, else the mma.sync path;
 *   1 = the mma.sync path (m16n8k16 tensor-core MMA from registers);
 *   2 = the tcgen05 path only (SDV_ERR_UNSUPPORTED where its plan does not fit);
 *   3 = the CUDA-core GEMV (fp32 FMAs, no tensor cores) for windows of one or
 *       two rows -- sdv_qlinear and sdv_verify_head with S <= 2 -- else as 0.
 * Returns the previous selection, or -1 for an invalid value (nothing changes).
 */
SDV_API int32_t sdv_set_gemm_path(int32_t path);

/*
 * Test hook of the timeout path (process-wide; every later launch of the
 * tcgen05 path uses it until it is reset with (-1, 0)).  withhold_stage >= 0:
 * in every CTA the weight copy of that stage of the CTA's stage sequence is
 * never issued, so the converters waiting for it give up after the wait limit
 * -- a wait on a barrier that nothing completes, with no copy in flight behind
 * it; the kernel then drains what it issued, writes undefined outputs and sets
 * the status word (sdv_last_device_status / sdv_noalloc_device_status return
 * SDV_ERR_TIMEOUT); later calls are unaffected.  wait_limit_ns: the limit of
 * every bounded device wait (0 = the built-in 2 s; else at least 100000).
 * -1 and 0 switch both off.  Returns SDV_ERR_INVALID_ARG for other values.
 * For the library's own tests; no production caller needs it.
 */
SDV_API sdv_status sdv_debug_fault(int32_t withhold_stage, uint64_t wait_limit_ns);

/*
 * Number of kernels this library has launched in this process (every device
 * and stream, counted when the launch is issued); the difference of two reads
 * brackets a region.  For measurement; the pages have no counterpart.
 */
SDV_API uint64_t sdv_launch_count(void);

/* A static, human-readable name of a status code. */
SDV_API const char* sdv_status_string(sdv_status status);

/* Library version (major * 10000 + minor * 100 + patch). */
SDV_API int32_t sdv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SDV_H */
