/*
 * csa.h -- certified sparse decode attention on GB300 (sm_103a), C ABI.
 *
 * The operation is the decode-attention step of "Certified Sparse Attention
 * via Perturbed Retrieval" (arXiv 2610.24991): picx.dev summary,
 * "Methodology / Problem Setup" (scores s_i = q.k_i / sqrt(d), c* = max s_i,
 * w_i = exp(s_i - c*), o = sum w_i v_i / sum w_i) and "Algorithm Components"
 * 1-4 (window of the last 64 tokens read exactly; perturbations
 * E_i = -ln u_i, u_i built from 53 hashed bits; threshold sample
 * S(tau) = {i in pool : s_i - c* + E_i >= log tau}; Horvitz-Thompson
 * estimates on the grid tau_j = 2^(-j/r); Chernoff / Hilbert-space Bernstein
 * certificate beta; each head ends at its lowest certified level; one
 * 4-bit scan per GQA group bounding every score), and the readsearch.ai
 * abstract page (the perturbations are drawn anew for each decode step).
 *
 * Conventions for every entry point:
 *  - Pointers named as device memory are device pointers owned by the
 *    caller; the library allocates no device memory at all.  Scratch space
 *    is the caller's `workspace` buffer (size from csa_workspace_size /
 *    csa_dense_workspace_size), except for csa_dense_decode_static, which
 *    uses a fixed array compiled into the library.
 *  - Host arrays (len, step_seed) are read before the call returns.
 *  - Work is enqueued on `stream` (a cudaStream_t, NULL = legacy default
 *    stream); outputs are valid once the stream has synchronised.  The call
 *    never synchronises the stream, so a decode step can be captured into a
 *    CUDA graph (the host arrays are copied into kernel arguments).
 *  - Argument errors return CSA_ERR_INVALID_ARG / CSA_ERR_UNSUPPORTED before
 *    anything is enqueued.  Launch failures return CSA_ERR_CUDA.  Errors
 *    found on the device (non-finite inputs, an exhausted buffer) are
 *    recorded in a status word inside the workspace; csa_check reads it.
 *  - Nothing throws across the ABI.
 *
 * Memory layouts (row-major, contiguous):
 *   q      [B][Hq][d]                      element type `dtype`
 *   K, V   [B][Hkv][n_max][d]              element type `dtype`
 *   K4     [B][Hkv][nblk_max * 64][d/2]    uint8, two 4-bit codes per byte,
 *                                          even channel in the low nibble
 *   bounds [B][Hkv][nblk_max][2][d]        float: per block and channel the
 *                                          minimum m_c, then the step Delta_c
 *   vmax   [B][Hkv][nblk_max]              float: per-block bound on ||v_i||
 *   vnorm2 [B][Hkv][n_max]                 float: ||v_i||^2 of each token, the
 *                                          sequential float32 sum of v_c^2
 *   o      [B][Hq][d] float;  beta, level, keys_read: [B][Hq]
 * with nblk_max = ceil(n_max / 64).  Query head h uses KV head h / (Hq/Hkv).
 */
#ifndef CSA_H_
#define CSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CSA_OK = 0,
  CSA_ERR_INVALID_ARG = 1,   /* null pointer, bad size or parameter          */
  CSA_ERR_UNSUPPORTED = 2,   /* valid but not built: d, G or B out of range  */
  CSA_ERR_CUDA = 3,          /* a CUDA call or launch failed                  */
  CSA_ERR_NONFINITE = 4,     /* NaN/Inf met in q, K or the statistics         */
  CSA_ERR_TIMEOUT = 5,       /* reserved: a bounded device wait gave up       */
  CSA_ERR_WORKSPACE = 6      /* workspace missing or too small               */
} csa_status;

typedef enum { CSA_BF16 = 0, CSA_F32 = 1 } csa_dtype;

/* Error measure that stops a head (picx.dev "Problem Setup"):
 *  VALUE  ||o_hat - o|| <= eps * M,  M^2 = sum_i a_i ||v_i||^2  (default)
 *  OUTPUT ||o_hat - o|| <= eps * ||o||
 *  DENOM  |D_hat - D|   <= eps * D
 *  CLT    UNCERTIFIED comparison rule (picx.dev "Theoretical Contributions",
 *         which compares the certificate with CLT-style stop rules): stops at
 *         the first level with z sqrt(tau G_hat) / D_hat <= eps M_hat, z the
 *         two-sided normal quantile at delta, M_hat the plug-in value scale;
 *         the returned beta is that normal-approximation estimate, not a
 *         bound.                                                             */
typedef enum {
  CSA_MEASURE_VALUE = 0, CSA_MEASURE_OUTPUT = 1, CSA_MEASURE_DENOM = 2,
  CSA_MEASURE_CLT = 3
} csa_measure;

typedef struct {
  int B;          /* sequences, 1..128                                       */
  int Hq;         /* query heads, 1..1024                                    */
  int Hkv;        /* KV heads, 1..1024; G = Hq / Hkv in {1, 2, 4, 8}         */
  int d;          /* head dimension, 64 or 128                               */
  int64_t n_max;  /* token capacity of K, V, K4 per (sequence, KV head)      */
  csa_dtype dtype;/* element type of q, K, V                                 */
} csa_shape;

typedef struct {
  float eps;      /* target error, > 0                                      */
  float delta;    /* failure probability per (sequence, query head), (0,1)  */
  int r;          /* grid resolution tau_j = 2^(-j/r), 1..4                  */
  int measure;    /* csa_measure                                             */
  int J_override; /* -1: last level J = ceil(r log2 |pool|); else J (<= 255) */
  int sub_batches;/* scheduling only, results do not depend on it: 0 = two
                   * when B >= 2, else one; 1..4 = that many sub-batches of
                   * consecutive sequences, each an independent chain of
                   * launches on a library-owned stream, forked from and
                   * joined back onto the caller's stream                   */
  int perturb;    /* 0: one perturbation draw per (sequence, KV head, key),
                   * shared by the group's query heads (default); 1: one draw
                   * per query head (stream 2^20 + g G + h of the keying)   */
  int qcode;      /* query code of the 4-bit bounds: 0 = int8 (QM = 127) with
                   * the residual summed per channel (default); 1 = two s8
                   * digits (QM = 127 * 257) with the closed-form residual
                   * 15 d alpha (1/2 + 2^-6): narrower bounds, fewer
                   * candidates; results do not depend on it               */
  int refine8;    /* 8-bit refinement tier (picx.dev "Algorithm Components"
                   * 4: an 8-bit stage before the exact 16-bit reads); needs
                   * csa_decode_step_refined and bf16 caches.  0 = off;
                   * 1 = every group; 2 = groups whose first gather range
                   * reaches level r (the near-uniform groups, which stop
                   * near level 0, stay on the 4-bit bounds).  Results do
                   * not depend on it; keys_read counts the refined levels */
  int dots;       /* the scan's exact integer dot products: 0 = tensor cores
                   * (mma.sync u8 x s8, default); 1 = CUDA-core dp4a (the
                   * comparison the choice rests on; int8 query codes only).
                   * Results are identical                                  */
} csa_params;

/* Optional per-(sequence, query head) diagnostics. */
typedef struct {
  int32_t level;            /* stop level j*, J+1 after the exact fallback  */
  int32_t keys_read;        /* 64 + |exact-max set U candidates jbar <= j*| */
  int32_t values_read;      /* 64 + |S(tau_j*)|                             */
  int32_t n_candidates;     /* pool keys with bound level jbar <= J         */
  int32_t n_near_threshold; /* keys within 1e-5 nats of a threshold at j*   */
  int32_t J;                /* last grid level of this sequence             */
  int32_t rounds;           /* gather rounds the head needed (1..3)         */
  int32_t group_keys_read;  /* 64 + |union over the head's GQA group of the */
                            /* pool rows counted in keys_read| (one bf16 K  */
                            /* row load serves the whole group)             */
  int32_t group_values_read;/* the same union for values_read              */
  int32_t rows8;            /* refinement tier: 8-bit rows of the head's    */
                            /* candidates outside its exact-max set with    */
                            /* jbar <= j* (0 without the tier)              */
} csa_head_stats;

/* Bytes of workspace csa_decode_step needs for this shape and parameters.
 * Returns 0 when the arguments are invalid. */
size_t csa_workspace_size(const csa_shape* shape, const csa_params* params);

/* 4-bit key quantiser and value-norm metadata (picx.dev "Algorithm
 * Components" 4: 4-bit per-block per-channel codes as in KIVI).
 * Rebuilds every 64-token block that holds a token at position
 * >= from_token and < len[b]: codes, (m_c, Delta_c), vmax and the
 * blocks' vnorm2 entries.  In decode, from_token = the position of the
 * token just appended (one block).
 *   K, V   device, layout above;  len host [B], 0 <= len[b] <= n_max
 *   K4, bounds, vmax, vnorm2: device outputs, layout above.
 * Positions >= len[b] inside a rebuilt block get code 0 and vnorm2 0. */
csa_status csa_quantize_keys(const csa_shape* shape, const void* K,
                             const void* V, const int64_t* len,
                             int64_t from_token, uint8_t* K4, float* bounds,
                             float* vmax, float* vnorm2, void* stream);

/* One certified sparse decode-attention step for every (sequence, query
 * head).  Inputs: q, K, V, K4, bounds, vmax, vnorm2 (device, layout above;
 * K4, bounds, vmax and vnorm2 must describe the first len[b] tokens, see
 * csa_quantize_keys), len host [B] (1 <= len[b] <= n_max), step_seed host
 * [B] (fresh every step; the caller mixes in the layer).  Outputs (device):
 *   o          [B][Hq][d]  o_hat at the stop level (exact o after fallback)
 *   beta       [B][Hq]     certified bound on ||o_hat - o|| (0 after the
 *                          exact fallback or when len <= 64; under
 *                          CSA_MEASURE_CLT the uncertified estimate)
 *   level      [B][Hq]     stop level j*; J+1 after the exact fallback
 *   keys_read  [B][Hq]     see csa_head_stats
 *   stats      [B][Hq]     optional (NULL to skip)
 * workspace: device buffer of at least csa_workspace_size bytes, 256-byte
 * aligned; its contents on entry do not matter.  params->refine8 must be 0
 * here (the tier's 8-bit inputs come through csa_decode_step_refined).
 * With sub-batches (csa_params.sub_batches) the call forks onto the
 * library's streams of the current device and joins back onto `stream`
 * before returning control of the outputs; enqueueing is serialised by a
 * host lock, so concurrent callers are safe but queue behind one another.
 * Everything is asynchronous on `stream` and capturable into a CUDA graph
 * (the fork and join are event waits). */
csa_status csa_decode_step(const csa_shape* shape, const csa_params* params,
                           const void* q, const void* K, const void* V,
                           const uint8_t* K4, const float* bounds,
                           const float* vmax, const float* vnorm2,
                           const int64_t* len,
                           const uint64_t* step_seed, float* o, float* beta,
                           int32_t* level, int32_t* keys_read,
                           csa_head_stats* stats, void* workspace,
                           size_t workspace_bytes, void* stream);

/* 8-bit codes of the same blocks, for the refinement tier (picx.dev
 * "Algorithm Components" 4).  Per block and channel: the same minimum m_c as
 * csa_quantize_keys, Delta8_c = fl((max - min) / 255) (0 -> 1), code =
 * clamp(rint(fl(fl(k - m_c) / Delta8_c)), 0, 255), one byte per code.
 * Rebuilds every block that holds a token at position >= from_token and
 * < len[b].
 *   K8      device [B][Hkv][nblk_max * 64][d] uint8
 *   delta8  device [B][Hkv][nblk_max][d] float
 * Positions >= len[b] inside a rebuilt block get code 0. */
csa_status csa_quantize_keys8(const csa_shape* shape, const void* K,
                              const int64_t* len, int64_t from_token,
                              uint8_t* K8, float* delta8, void* stream);

/* csa_decode_step with the 8-bit refinement tier (params->refine8 = 1 or 2,
 * bf16 caches): before each gather round's exact rescoring, the candidates
 * the round would read also get the upper bound from their 8-bit codes
 * (K8, delta8 from csa_quantize_keys8, same blocks; query codes of 12 bits
 * per (block, head)), and a key whose level from the tighter of the two
 * bounds lies past the round's range is not read in that round.  The
 * refined level never exceeds the exact one, so o, beta, level and
 * values_read are those of csa_decode_step; keys_read counts the refined
 * levels.  Other arguments, results and errors as csa_decode_step. */
csa_status csa_decode_step_refined(const csa_shape* shape,
                                   const csa_params* params, const void* q,
                                   const void* K, const void* V,
                                   const uint8_t* K4, const float* bounds,
                                   const float* vmax, const float* vnorm2,
                                   const uint8_t* K8, const float* delta8,
                                   const int64_t* len,
                                   const uint64_t* step_seed, float* o,
                                   float* beta, int32_t* level,
                                   int32_t* keys_read, csa_head_stats* stats,
                                   void* workspace, size_t workspace_bytes,
                                   void* stream);

/* The same step with the lengths and seeds in device memory, for whole-token
 * decode captured once into a CUDA graph and replayed every token (the
 * readsearch.ai abstract: the perturbations are drawn anew at every decode
 * step, so a replayed step must read the new seeds; picx.dev "CPU Speed":
 * whole decode steps over all layers are what is timed).
 *   len        device [B] int64, 1 <= len[b] <= n_max (a value outside is
 *              clamped and reported by csa_check as CSA_ERR_INVALID_ARG)
 *   step_seed  device [B] uint64
 *   requantize_last  1: before scanning, rebuild the 64-token block that
 *              holds token len[b] - 1 of every sequence (codes, bounds,
 *              vmax, vnorm2 from K and V: what csa_quantize_keys with
 *              from_token = len[b] - 1 does), inside the step's first
 *              kernel; for the token just appended.  0: the caller keeps
 *              K4, bounds, vmax and vnorm2 current.  With 1, K4, bounds,
 *              vmax and vnorm2 are written.
 * Both arrays are read by the step's first kernel, in stream order, so a
 * kernel or copy earlier on `stream` (or in the same graph) may write them.
 * Grids are sized from n_max rather than the longest live sequence.  The
 * refinement tier is not available here (params->refine8 must be 0).  Other
 * arguments, results and errors as csa_decode_step. */
csa_status csa_decode_step_device(const csa_shape* shape, const csa_params* params,
                                  const void* q, const void* K, const void* V,
                                  uint8_t* K4, float* bounds, float* vmax,
                                  float* vnorm2, const int64_t* len,
                                  const uint64_t* step_seed,
                                  int requantize_last, float* o, float* beta,
                                  int32_t* level, int32_t* keys_read,
                                  csa_head_stats* stats, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* Bytes of workspace csa_dense_decode needs (a status word, then the
 * split-K partials). */
size_t csa_dense_workspace_size(const csa_shape* shape);

/* Dense decode attention (the same-build comparator, and the exact formula
 * of picx.dev "Problem Setup"): o = softmax(q K^T / sqrt d) V over the first
 * len[b] tokens, float32 accumulation.  q, K, V device; len host [B];
 * o device [B][Hq][d] float. */
csa_status csa_dense_decode(const csa_shape* shape, const void* q,
                            const void* K, const void* V, const int64_t* len,
                            float* o, void* workspace, size_t workspace_bytes,
                            void* stream);

/* Dense decode attention with no workspace argument and no allocation by
 * anyone.  The paper has no counterpart to this entry point: it is a
 * deployment variant of csa_dense_decode for callers that cannot allocate
 * device memory where they call it -- a plain C host program that links only
 * this library and owns no device allocator, or a callback that runs while
 * another component holds the device memory and its allocator.
 *
 * Same operation, arguments, layouts and results as csa_dense_decode (the
 * same two kernels run); the split-K partials live in a file-scope device
 * array of CSA_DENSE_STATIC_SCRATCH_BYTES (16 MiB) per device instead.
 *  - The shape needs csa_dense_workspace_size(shape) bytes of scratch; a
 *    shape that needs more than CSA_DENSE_STATIC_SCRATCH_BYTES returns
 *    CSA_ERR_WORKSPACE before anything is enqueued (16 MiB holds, e.g.,
 *    B = 4, Hq = 32, d = 128 up to n_max = 258,048).
 *  - The array's contents on entry do not matter: every partial the combine
 *    step reads is written earlier in the same call.
 *  - All calls on one device share the array.  Calls whose work overlaps in
 *    time (different streams, or several host threads) race on it and give
 *    wrong results; serialise them (one stream, or events between streams).
 *  - The array's device address is looked up (cudaGetSymbolAddress, with
 *    the device current) on every call made outside a stream capture, and
 *    cached with the device's current CUDA context; the first call on a
 *    device also loads the library's device code there.  A call made while
 *    `stream` is being captured uses that cached address instead, so make
 *    at least one call outside a capture first (again after a device reset,
 *    which ends the context and the array with it); without one the call
 *    returns CSA_ERR_CUDA.  A failed lookup returns CSA_ERR_CUDA.
 * Other errors as csa_dense_decode. */
#define CSA_DENSE_STATIC_SCRATCH_BYTES (16u << 20)
csa_status csa_dense_decode_static(const csa_shape* shape, const void* q,
                                   const void* K, const void* V,
                                   const int64_t* len, float* o, void* stream);

/* Where csa_decode_step keeps its intermediate arrays inside the workspace
 * (byte offsets), for diagnostics and parity tests.  Valid after the step's
 * stream has synchronised, until the workspace is reused.
 *   ubar     float [B][Hkv][n_max][G]   4-bit upper bounds of every key
 *   cmax     uint32 [B][Hq][4]          c*_lo, c*_hi, cb, c32 as ordered
 *            integers (u >= 2^31: float bits u - 2^31; else bits ~u)
 *   s32      float [B][Hkv][n_max-64][G] float32 score of each candidate
 *            pool key for each head; after a step called with `stats`,
 *            -inf where the key is not a candidate of the head or was not
 *            rescored (without `stats` the other entries are left stale)
 *   jr_hist  uint32 [B][Hq][J+2]        first level at which the key's bf16
 *            row is needed (exact-max set: level 0); keys never needed
 *            (level J+1) are not counted, that entry stays 0
 *   bcnt     uint32 [B][Hkv][J1]        entries appended to each level bucket
 *            over the step's gather rounds (one per key, level and round at
 *            which the key changes a head's sums; each entry is one
 *            value-row load of the gather)
 *   J1       largest J + 1 (row stride of jr_hist is J1 + 1)
 * With sub-batches the arrays above are those of sub-batch 0 (its first
 * sub_B sequences); sub-batch c's are sub_stride * c bytes further.  (While
 * phase timing is enabled the step runs unsplit: its arrays are then where
 * the map for sub_batches = 1 puts them.)
 *   total        workspace bytes (csa_workspace_size)
 *   sub_batches  sub-batches the step runs as
 *   sub_stride   bytes between sub-batch regions
 *   sub_B        sequences per sub-batch (the last may hold fewer) */
typedef struct {
  size_t ubar, cmax, s32, jr_hist, bcnt, total;
  int32_t J1, sub_batches;
  size_t sub_stride;
  int32_t sub_B, reserved;
} csa_workspace_map;

csa_status csa_workspace_layout(const csa_shape* shape,
                                const csa_params* params,
                                csa_workspace_map* out);

/* Phase timing (tracing).  When enabled, csa_decode_step records a CUDA
 * event at every phase boundary on its stream; csa_profile_read waits for
 * the recorded events and returns the accumulated milliseconds per phase
 * since the previous read (then resets).  Up to 64 steps are buffered;
 * older ones are dropped.  `launches` counts the library's kernel launches
 * (profiling on or off) since the previous read.  Not thread-safe.
 * Phases: 0 workspace clear, 1 scan, 2 exact max, 3 candidates (with the
 * value-free level histograms), 4 rescoring of candidate K rows (per
 * round), 5 predictor + window, 6 level buckets, 7 gather plan, 8 V gather,
 * 9 certificate, 10 exact fallback, 11 diagnostics, 12 8-bit refinement. */
#define CSA_NPHASE 13
typedef struct {
  float ms[CSA_NPHASE];
  int32_t steps;
  int64_t launches;
} csa_phase_times;

csa_status csa_profile_enable(int on);
csa_status csa_profile_read(csa_phase_times* out);

/* Synchronises `stream`, then returns the device status word recorded in
 * `workspace` by the last csa_decode_step, csa_decode_step_device or
 * csa_dense_decode that used it: CSA_OK, CSA_ERR_NONFINITE,
 * CSA_ERR_WORKSPACE, CSA_ERR_TIMEOUT (a bounded wait of the dense kernel
 * gave up) or CSA_ERR_INVALID_ARG (a device length out of range); or
 * CSA_ERR_CUDA if the stream reports an error. */
csa_status csa_check(void* workspace, void* stream);

/* Static English description of a status code. */
const char* csa_status_string(csa_status s);

#ifdef __cplusplus
}
#endif

#endif /* CSA_H_ */
