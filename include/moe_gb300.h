/*
 * moe_gb300.h -- C ABI of the GB300 (sm_103a) MoE routing-layer library.
 *
 * One mixture-of-experts layer under batch-level routing control:
 *
 *   y(x) = sum_{j in Top-k(G(x))} G(x)_j * E_j(x)
 *       ("MACS: Modality-Aware Capacity Scaling for Efficient Multimodal MoE
 *        Inference", sec. 3.1, Eq. (1))
 *
 * computed as   moe_route        router GEMM + fp32 softmax + top-R ranking,
 *                                optionally fused with the SERE batch reroute
 *               moe_reroute_sere the SERE reroute on its own
 *               moe_route_dispatch
 *                                decode batches: moe_route (optionally with
 *                                SERE) and the uncapped dispatch in one launch
 *               moe_dispatch_capacity
 *                                expert-sorted permutation, optionally under a
 *                                weighted capacity with overflow reroute / drop
 *               moe_ffn_grouped  grouped SwiGLU expert FFN, combine fused in
 *               moe_combine      weighted combine of per-row expert outputs
 *               moe_token_weights
 *                                entropy-weighted token load for the capacity
 *                                dispatch, and the effective visual ratio
 *               moe_similarity_calibrate
 *                                the SERE similarity matrix from the experts'
 *                                outputs on calibration tokens
 *
 * Conventions for every entry point
 *  - Pointers named "host" are host memory; every other pointer is device
 *    memory (cudaMalloc / PyTorch CUDA tensors).  The caller owns all memory;
 *    the library allocates nothing, frees nothing and never synchronises.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls are asynchronous on that stream; launch configurations
 *    depend only on the scalar arguments, so a sequence of calls can be
 *    captured into a CUDA graph.
 *  - Arguments are checked on the host before anything is launched.  A bad
 *    argument returns a negative moe_status_t and launches nothing.
 *  - Errors that depend on the data (non-finite logits, an out-of-range id,
 *    an internal wait that timed out) are written asynchronously into the
 *    optional device-side status word `st` (first error wins; clear it to
 *    zero before use).  Outputs of a call that set an error are unspecified.
 *  - Matrices are row-major and densely packed unless a leading dimension
 *    (`ld`) is given.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int moe_status_t;
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1)   /* a pointer, size, alignment or option is invalid */
#define MOE_ERR_UNSUPPORTED (-2)   /* valid but outside what the kernels support (see limits) */
#define MOE_ERR_CUDA (-3)          /* a CUDA launch or driver call failed */
#define MOE_ERR_WORKSPACE (-4)     /* workspace missing or smaller than moe_workspace_size() */

/* Device-side status word, written by kernels. */
typedef struct moe_dev_status {
    int32_t code;    /* MOE_DEV_* */
    int32_t detail;  /* code-specific: token index, expert id, or wait site */
} moe_dev_status;
#define MOE_DEV_OK 0
#define MOE_DEV_NONFINITE 1        /* a router logit was NaN or infinite (detail = token) */
#define MOE_DEV_TIMEOUT 2          /* a bounded on-chip wait gave up (detail = wait site) */
#define MOE_DEV_BAD_INDEX 3        /* an expert id or row index was out of range (detail = value) */

#define MOE_DTYPE_F32 0
#define MOE_DTYPE_BF16 1

/* Compile-time limits of the library. */
#define MOE_MAX_EXPERTS 256        /* N */
#define MOE_MAX_RANKS 16           /* R (and k <= R) */

/* ---------------------------------------------------------------- */
/* moe_route                                                          */
/* ---------------------------------------------------------------- */
#define MOE_ROUTE_FROM_LOGITS 1u   /* `logits` is an input; x and w_router are not read */
#define MOE_ROUTE_RENORM_TOPK 2u   /* divide the first k gates by their fp32 sum */

/* SERE parameters ("SERE" expert rerouting, Xiaohongshu multi-image QA
 * inference article, sec. 4.1-4.2). */
typedef struct moe_sere_params {
    int k_primary;            /* K': ranks [0, K') are primaries, 1 <= K' <= k */
    float rho;                /* a secondary moves only if sim > rho (strict) */
    const float* sim;         /* [N][N] fp32 expert similarity, row = source expert */
    const uint8_t* protect;   /* [N] 0/1, nonzero = this source never moves; NULL = none */
    uint32_t* union_bitmap;   /* out [ceil(N/32)]: bit p set iff expert p is in the
                                 primary union P; may be NULL */
    int32_t* stats;           /* out [8]: union before, |P|, union after, moved, merged,
                                 kept-protected, kept-dissimilar, 0; may be NULL */
} moe_sere_params;

/*
 * Router scores, softmax gate and ranking.  "MACS" sec. 3.1, Eq. (1): the
 * router G(x) scores all N experts; the layer keeps the top-k and weights
 * each by its gate.
 *
 *   x          [T][H]  token activations, x_dtype BF16 or F32 (16-byte aligned)
 *   w_router   [N][H]  fp32 router weight
 *   logits     [T][N]  fp32; written (router GEMM, fp32 accumulation), or read
 *                      with MOE_ROUTE_FROM_LOGITS
 *   ids        [T][R]  int32 out: expert ids by logit descending, ties to the lower id
 *   gates      [T][R]  fp32 out: softmax gate of each ranked expert (over all N),
 *                      computed in a fixed fp32 order so that results are
 *                      reproducible bit for bit
 *   k                  the number of experts a token uses (k <= R); used by
 *                      MOE_ROUTE_RENORM_TOPK and by SERE
 *   sere               NULL, or SERE parameters: then R must equal k and the
 *                      reroute runs inside the same kernel as the ranking
 *                      (one CTA, T <= 4096), rewriting ids/gates in place:
 *                      moved slots take the target id, merged slots become
 *                      (-1, 0.0f) with the gate added to the slot that holds
 *                      the target.
 * Limits: 1 <= N <= 256, 1 <= k <= R <= min(16, N), T >= 0, H >= 1
 * (H % 8 == 0 for BF16 x, H % 4 == 0 for F32 x).
 */
moe_status_t moe_route(const void* x, int x_dtype, const float* w_router, int T, int H, int N, int R,
                       int k, uint32_t flags, float* logits, int32_t* ids, float* gates,
                       const moe_sere_params* sere, moe_dev_status* st, void* stream);

/*
 * Decode routing and dispatch in one launch: the results of moe_route with
 * R = k (and `sere`, if given) followed by the uncapped
 * moe_dispatch_capacity, bit for bit, for batches of up to 256 tokens.
 * "SERE" article sec. 4.2: the reroute feeds the fused MoE with no host round
 * trip; at decode sizes the ranking, reroute and permutation touch a few KB,
 * so they run in the last CTA of the router launch instead of in launches of
 * their own.
 *
 *   x, x_dtype, w_router, T, H, N, k, logits, ids, gates, sere
 *              as for moe_route with R = k (logits is a required output;
 *              flags: MOE_ROUTE_RENORM_TOPK only)
 *   counts, offsets, row_token, row_gate, active
 *              as for moe_dispatch_capacity with capacity_factor <= 0 and
 *              ld = k: rows ordered by (expert, token)
 *   workspace  moe_workspace_size(MOE_OP_ROUTE_DISPATCH, ...) bytes, 256-byte
 *              aligned, ZERO-FILLED before its first use (it holds a counter
 *              that every call leaves at zero); two calls must not use one
 *              workspace concurrently
 * Limits: 0 <= T <= 256, T * k <= 2048, 1 <= k <= min(16, N), N <= 256;
 * H % 8 == 0 for BF16 x, H % 4 == 0 for F32 x.
 */
moe_status_t moe_route_dispatch(const void* x, int x_dtype, const float* w_router, int T, int H, int N, int k,
                                uint32_t flags, float* logits, int32_t* ids, float* gates,
                                const moe_sere_params* sere, int32_t* counts, int32_t* offsets,
                                int32_t* row_token, float* row_gate, int32_t* active, void* workspace,
                                size_t ws_bytes, moe_dev_status* st, void* stream);

/*
 * One decode MoE layer in one call: moe_route_dispatch, then the grouped
 * SwiGLU FFN with the weighted combine fused in (y = sum_j G(x)_j E_j(x),
 * "MACS" sec. 3.1 Eq. (1); with `sere`, the "SERE" article's batch reroute,
 * sec. 4.1-4.2).  As soon as ranking ends, while the routing launch still
 * reroutes and permutes, the FFN starts streaming the weights of a published
 * set of experts: without SERE the union of the ranked experts; with SERE
 * its primary union P (sec. 4.1: primaries are never rerouted), or the whole
 * union before the reroute when that union's phase-1 units fit one wave of
 * the SMs, or two waves while P's would fill at most a third of one and the
 * other experts' more than one (an expert that then moves costs only its
 * phase 1).  The other experts and the down projections wait for the final
 * routing.  Results equal moe_route_dispatch followed by moe_ffn_grouped
 * with MOE_FFN_FUSE_COMBINE (up to the fp32 summation order of y).
 *
 *   x, w_router, sere, logits, ids, gates, counts, offsets, row_token,
 *   row_gate, active: as moe_route_dispatch (x is BF16, [T][H])
 *   w_gate, w_up [N][I][H], w_down [N][H][I]  bf16 expert weights
 *   y          [T][H] fp32 out: zeroed first when ffn_flags has
 *              MOE_FFN_ZERO_Y, else the layer output is added into it
 *   route_flags  MOE_ROUTE_RENORM_TOPK or 0
 *   ffn_flags    MOE_FFN_ZERO_Y or 0 (the combine is always fused)
 *   route_ws   moe_workspace_size(MOE_OP_ROUTE_DISPATCH, ...) bytes
 *   ffn_ws     moe_workspace_size(MOE_OP_FFN, T, H, I, N, k, k, 0, BF16) bytes
 *              both 256-byte aligned and ZERO-FILLED before their first use
 *              (every call leaves their counters at zero); a pair of
 *              workspaces serves one call at a time.
 * Limits: 1 <= T <= 64, T * k <= 2048, N <= 256, 1 <= k <= min(16, N),
 * H % 128 == 0, I % 128 == 0, pointers 16-byte aligned.  Errors: argument
 * errors return before anything is launched; data-dependent errors and
 * bounded waits that ran out go to st.
 */
moe_status_t moe_decode_layer(const void* x, const float* w_router, const void* w_gate, const void* w_up,
                              const void* w_down, int T, int H, int I, int N, int k, uint32_t route_flags,
                              uint32_t ffn_flags, const moe_sere_params* sere, float* logits, int32_t* ids,
                              float* gates, int32_t* counts, int32_t* offsets, int32_t* row_token,
                              float* row_gate, int32_t* active, float* y, void* route_ws, size_t route_ws_bytes,
                              void* ffn_ws, size_t ffn_ws_bytes, moe_dev_status* st, void* stream);

/*
 * SERE batch reroute on given routing ("SERE" article, sec. 4.1: the union P
 * of every token's top-K' primary experts is the shared candidate set; every
 * secondary outside P whose source is not protected (sec. 4.2) moves to its
 * most similar member of P when that similarity exceeds rho; ties to the
 * lower id; a token that already holds the target gets the gate added).
 *
 *   ids, gates [T][ld] in/out (the first k columns are used); same rewrite
 *   rules as moe_route with `sere`.  One CTA; T <= 4096.
 */
moe_status_t moe_reroute_sere(int32_t* ids, float* gates, int ld, int T, int N, int k,
                              const moe_sere_params* sere, moe_dev_status* st, void* stream);

/* ---------------------------------------------------------------- */
/* moe_dispatch_capacity                                              */
/* ---------------------------------------------------------------- */
#define MOE_SLOT_KEPT 0
#define MOE_SLOT_REROUTED 1
#define MOE_SLOT_DROPPED 2

/*
 * Expert-sorted permutation, optionally under a weighted capacity.
 *
 * Uncapped (capacity_factor <= 0): every slot with id >= 0 among the first k
 * columns of ids becomes one row.  Capped ("MACS" sec. 3.1 Eq. (3) and
 * sec. 3.2 Eq. (6)): token weights w are taken in fixed point
 * w_q = rint(w * 2^24); S = sum w_q; C = floor(((double)S * k) *
 * capacity_factor / N).  Each expert admits its (token, slot) pairs in
 * (gate desc, token asc) order while the cumulative w_q stays <= C.  Then, in
 * rounds i = 0 .. R-k-1, every token with an overflowed slot offers its
 * lowest-rank overflowed slot (with that slot's gate) to its rank-(k+i)
 * expert, which admits offers in the same order while load + cumulative
 * w_q <= C.  Slots left over are dropped (the "MACS" Fig. 1 overflow path:
 * reroute locally, else drop).
 *
 *   ids, gates   [T][ld]  ranked routing (ld >= R when capped, >= k otherwise)
 *   token_w      [T] fp32 >= 0, or NULL (all 1); capped mode only (e.g. the
 *                      entropy weights of moe_token_weights)
 *   modality_bias [N] int8, or NULL: per-expert capacity ("MACS" sec. 3.3:
 *                      m_j = +1 visual, -1 text, 0 shared expert).  The page
 *                      stops before its scaling formula; this library reads it
 *                      as C_j = floor(c * (1 + m_j * (R_v - 1/2))) with
 *                      c = ((double)S * k) * capacity_factor / N unfloored, so
 *                      m_j = 0 or R_v = 1/2 keep the static C.  Capped mode only.
 *   r_v          [1] fp32 device scalar in [0, 1] (the effective visual ratio of
 *                      moe_token_weights); required with modality_bias.  A bias
 *                      outside {-1, 0, 1} or a ratio outside [0, 1] is reported
 *                      in st and that expert keeps the static C.
 *   counts       [N]      out: rows per expert
 *   offsets      [N+1]    out: exclusive prefix of counts
 *   row_token    [T*k]    out: token of each row, rows ordered by (expert, token)
 *   row_gate     [T*k]    out: gate of each row
 *   active       [N+1]    out: active[0] = experts with rows, active[1..] their ids ascending
 *   out_ids, out_gates [T][k] out (may be NULL): final expert and gate per slot,
 *                      (-1, 0.0f) for empty or dropped slots
 *   slot_row     [T][k]   out (may be NULL): row index of each slot, -1 if none
 *   slot_status  [T][k]   out (may be NULL): MOE_SLOT_*; capped mode only
 *   load_q       [N]      out (may be NULL): final weighted load in 2^-24 units
 *   cap_q        [1]      out (may be NULL): the static C in 2^-24 units
 *   workspace    device scratch of moe_workspace_size(MOE_OP_DISPATCH, ...) bytes
 * Limits: N <= 256, k <= R <= min(16, N); capped mode T <= 16384.
 */
moe_status_t moe_dispatch_capacity(const int32_t* ids, const float* gates, int ld, int T, int N, int k,
                                   int R, const float* token_w, float capacity_factor,
                                   const int8_t* modality_bias, const float* r_v, int32_t* counts,
                                   int32_t* offsets, int32_t* row_token, float* row_gate, int32_t* active,
                                   int32_t* out_ids, float* out_gates, int32_t* slot_row,
                                   uint8_t* slot_status, int64_t* load_q, int64_t* cap_q, void* workspace,
                                   size_t ws_bytes, moe_dev_status* st, void* stream);

/*
 * moe_dispatch_capacity_static -- the same dispatch as moe_dispatch_capacity,
 * for callers that cannot allocate device memory.  The paper has no
 * counterpart; this is an interface of this library only.
 *
 * Who needs it: code that is not allowed to call cudaMalloc or to hold a
 * workspace of its own, for example a plugin inside a serving engine that
 * hands out all device memory from its own pool, or code running while a
 * stream is captured into a CUDA graph under a capture mode that forbids
 * allocation calls.  Such a caller still passes its inputs and outputs; only
 * the scratch memory moves into the library.
 *
 * Scratch: one file-scope device array of MOE_STATIC_DISPATCH_SCRATCH_BYTES
 * (4.5 MiB), present on every GPU that loads the library until the process
 * exits.  It is enough for every size with T <= MOE_STATIC_DISPATCH_MAX_T
 * (2048 tokens) and the limits of moe_dispatch_capacity; larger T returns
 * MOE_ERR_UNSUPPORTED and launches nothing.  No call allocates or frees.
 * The first call on a device looks up the array's device address (with that
 * device current) and caches it; make that first call before any stream
 * capture.  Every call on a device shares the one array: calls whose work
 * overlaps on the GPU (two streams, or two host threads) race and give wrong
 * results, so serialise them.  Each call clears the parts of the array that
 * must start at zero, so leftovers of the previous call do no harm.
 *
 * Arguments, outputs and errors are those of moe_dispatch_capacity without
 * `workspace` and `ws_bytes`.
 */
#define MOE_STATIC_DISPATCH_MAX_T 2048
#define MOE_STATIC_DISPATCH_SCRATCH_BYTES (4608u * 1024u)
moe_status_t moe_dispatch_capacity_static(const int32_t* ids, const float* gates, int ld, int T, int N, int k,
                                          int R, const float* token_w, float capacity_factor,
                                          const int8_t* modality_bias, const float* r_v, int32_t* counts,
                                          int32_t* offsets, int32_t* row_token, float* row_gate,
                                          int32_t* active, int32_t* out_ids, float* out_gates,
                                          int32_t* slot_row, uint8_t* slot_status, int64_t* load_q,
                                          int64_t* cap_q, moe_dev_status* st, void* stream);

/* ---------------------------------------------------------------- */
/* moe_ffn_grouped                                                    */
/* ---------------------------------------------------------------- */
#define MOE_FFN_FUSE_COMBINE 1u    /* out is y[T][H] fp32: y[t] += gate * E_e(x_t) per row */
#define MOE_FFN_ZERO_Y 2u          /* with FUSE_COMBINE: zero y first */

/*
 * Grouped SwiGLU expert FFN ("MACS" sec. 3.1 Eq. (1), E_j(x) =
 * W_down_j (silu(W_gate_j x) * (W_up_j x))) over the rows of
 * moe_dispatch_capacity, only for active experts.
 *
 *   x       [T][H]     activations, dtype BF16 or F32 (same dtype as the weights)
 *   w_gate  [N][I][H], w_up [N][I][H], w_down [N][H][I]  expert weights
 *   offsets [N+1], row_token [T*k], row_gate [T*k], active [N+1]  from dispatch
 *   out     FUSE_COMBINE: y [T][H] fp32 (accumulated into); otherwise
 *           rows_out [T*k][H] fp32, row r = E_e(x_token(r)) without the gate
 *   workspace  device scratch of moe_workspace_size(MOE_OP_FFN, ...) bytes,
 *           256-byte aligned.  BF16 needs it: a work counter, one counter
 *           per (expert, token chunk), three more counters and the bf16
 *           SwiGLU activations of every row (T*k*I*2 bytes plus a few KiB);
 *           F32 needs none.  ZERO-FILL it once before its first use: the
 *           counters must start at zero, and every call (including one that
 *           reports an error in st) leaves them at zero again, so nothing
 *           needs clearing between calls.  Two calls in flight at once must
 *           not share a workspace.
 *   flags   MOE_FFN_ZERO_Y: y is zeroed inside the same launch (in chunks,
 *           all of them before any row is added into it).
 * BF16 runs on the tensor cores (tcgen05, TMA-fed) with fp32 accumulation;
 * the SwiGLU activation is rounded to bf16 before the down projection.
 * F32 runs a CUDA-core kernel in fp32.
 * Limits BF16: H % 128 == 0, I % 128 == 0, all pointers 16-byte aligned;
 * rows_out mode needs FUSE_COMBINE off and is accumulated, so zero it first.
 * Limits F32: (H + I) * 4 <= 227 KiB (a row's x and activations are held
 * in shared memory); larger sizes return MOE_ERR_UNSUPPORTED.
 */
moe_status_t moe_ffn_grouped(const void* x, int dtype, const void* w_gate, const void* w_up,
                             const void* w_down, int T, int H, int I, int N, int k, const int32_t* offsets,
                             const int32_t* row_token, const float* row_gate, const int32_t* active,
                             uint32_t flags, float* out, void* workspace, size_t ws_bytes,
                             moe_dev_status* st, void* stream);

/*
 * Expert similarity from calibration tokens (SERE article sec. 4.2: the
 * similarity matrix is prepared offline as the Frobenius similarity of the
 * experts' outputs on calibration data):
 *
 *   sim[i][j] = <E_i(X), E_j(X)>_F / (||E_i(X)||_F ||E_j(X)||_F)
 *
 * with E_e(X) the [n][H] SwiGLU outputs of expert e on the calibration
 * tokens X.  The diagonal is 1; a pair with an expert whose output is all
 * zero gets 0.  Every expert's output on every token comes from the grouped
 * tcgen05 FFN; they are rounded to bf16 and the Gram matrix E E^T runs on the
 * tensor cores split over the SMs, summed and normalised in double.  The
 * result feeds moe_sere_params.sim (the matrix is exactly symmetric).
 *
 *   x          [n][H] bf16 calibration tokens
 *   w_gate, w_up, w_down   bf16 expert weights as in moe_ffn_grouped
 *   sim        [N][N] fp32 out
 *   workspace  moe_workspace_size(MOE_OP_CALIBRATE, n, H, I, N, 1, 1, 0,
 *              MOE_DTYPE_BF16) bytes, 256-byte aligned
 * Limits: 2 <= N <= 128, H % 128 == 0, I % 128 == 0, n * N and n * H below 2^31.
 */
moe_status_t moe_similarity_calibrate(const void* x, int n, const void* w_gate, const void* w_up,
                                      const void* w_down, int H, int I, int N, float* sim, void* workspace,
                                      size_t ws_bytes, moe_dev_status* st, void* stream);

/*
 * Entropy-weighted token load ("MACS" sec. 3.2 Eqs. (4)-(5) and sec. 3.3
 * Eq. (7)): the per-token load weights that moe_dispatch_capacity takes as
 * token_w, and the batch's effective visual ratio.
 *
 *   x          [T][H] token features z (the layer's input rows), BF16 or F32,
 *              16-byte aligned, H % 8 == 0
 *   is_visual  [T] uint8, nonzero = visual token, 0 = text token
 *   delta      sensitivity of the entropy-to-weight map (finite)
 *   eps        added to the standard deviation (> 0)
 *   entropy    [T] fp32 out: Shannon entropy (natural log) of Softmax(z), every token
 *   token_w    [T] fp32 out: sigmoid(-delta * (H - mu) / (sigma + eps)) for
 *              visual tokens, where mu and sigma are the mean and population
 *              standard deviation of the visual tokens' entropies in this
 *              batch; 1 for text tokens
 *   r_v        [1] fp32 out (may be NULL): sum of visual weights / sum of all
 *              weights (0 when T == 0)
 *   workspace  moe_workspace_size(MOE_OP_TOKEN_WEIGHTS, T, ...) bytes (24 bytes
 *              per 8 tokens + 16 per 256 tokens + 16), 256-byte aligned; no
 *              initial contents needed
 * Entropies and weights are computed in fp32 (one warp per token for the
 * entropy, exponentials in base 2); the statistics (count, sum and sum of
 * squares of the visual entropies) and the two weight sums of R_v are added
 * up as 64-bit fixed-point integers (entropy in 2^-32, its square in 2^-24,
 * weights in 2^-32 units), so results do not depend on summation order and
 * are reproducible bit for bit; the population variance is formed from them
 * exactly in 128-bit integers, then mean, standard deviation and R_v in
 * fp32.  T is at most 2^24 (MOE_ERR_UNSUPPORTED beyond), which keeps those
 * sums in range.  Two calls must not share a workspace concurrently (it
 * holds a completion counter).
 * A token whose entropy comes out non-finite sets MOE_DEV_NONFINITE (detail =
 * token) in st: any non-finite feature does so, and so can a row with
 * features of magnitude 2^126 or more (its base-2 exponents overflow fp32).
 */
moe_status_t moe_token_weights(const void* x, int x_dtype, int T, int H, const uint8_t* is_visual, float delta,
                               float eps, float* entropy, float* token_w, float* r_v, void* workspace,
                               size_t ws_bytes, moe_dev_status* st, void* stream);

/*
 * Weighted combine ("MACS" Eq. (1)): y[t] = sum_r gate[t][r] * rows_out[slot_row[t][r]]
 * over the slots r < k with slot_row >= 0, in slot order (deterministic).
 *   rows_out [M][H] fp32, slot_row [T][k], slot_gate [T][k], y [T][H] fp32 out.
 */
moe_status_t moe_combine(const float* rows_out, const int32_t* slot_row, const float* slot_gate, int T,
                         int H, int k, float* y, void* stream);

/*
 * Residual rounding between stacked layers: y[i] = bf16(x[i]), round to
 * nearest, ties to even, for i < n.  In a stack of layers the FFN adds
 * sum_j G_j E_j(x) ("MACS" Eq. (1)) into the fp32 residual (moe_ffn_grouped
 * with MOE_FFN_FUSE_COMBINE and without MOE_FFN_ZERO_Y), and the next
 * layer's routing and FFN read bf16 tokens; this is that rounding, as a
 * launch that overlaps its neighbours (programmatic dependent launch).
 *   x [n] fp32 in, y [n] bf16 out (device, 16-byte aligned, caller-owned);
 *   n a multiple of 8.  Bad sizes or alignment return MOE_ERR_INVALID_ARG
 *   with no launch; n = 0 is a no-op.
 */
moe_status_t moe_residual_to_bf16(const float* x, void* y, long long n, void* stream);

/* ---------------------------------------------------------------- */
/* Workspace sizes and status strings                                 */
/* ---------------------------------------------------------------- */
#define MOE_OP_DISPATCH 1
#define MOE_OP_FFN 2
#define MOE_OP_CALIBRATE 3   /* moe_similarity_calibrate: T = calibration tokens n */
#define MOE_OP_TOKEN_WEIGHTS 4   /* moe_token_weights: depends on T only */
#define MOE_OP_ROUTE_DISPATCH 5  /* moe_route_dispatch: a fixed 512 bytes */

/* Bytes of device workspace that `op` needs for these sizes (0 if none).
 * capped != 0 asks for the capacity-mode size of MOE_OP_DISPATCH; dtype
 * selects the FFN kernel.  Returns 0 for invalid arguments. */
size_t moe_workspace_size(int op, int T, int H, int I, int N, int k, int R, int capped, int dtype);

/* Static string for a status code (host or device MOE_DEV_* codes are
 * told apart by the `device` flag). */
const char* moe_status_string(int code, int device);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
