/*
 * attnres.h -- C ABI of libattnres: Block Attention Residuals (Block AttnRes)
 * depth aggregation on NVIDIA GB300 (sm_103a).
 *
 * What the operations compute (sources cited by page title and section):
 *
 *  - [Deep-dive 2] "Kimi K3 deep-dive series (2): AttnRes and Stable
 *    LatentMoE", §2: for one token and layer l with sources H (S rows of d)
 *    and a learned pseudo-query w_l,
 *        a_l = softmax_s( w_l . RMSNorm(H_s) ),     r_l = sum_s a_l[s] H_s,
 *    RMSNorm without a gain, no temperature, values are the raw sources.
 *    [Atlas] "LLM Atlas · Kimi K3", §07 Attention Residuals, states the same
 *    weights alpha_{i->l} and h_l = sum_i alpha_{i->l} v_i.
 *  - [Parts 6] "Kimi K3 model structure (6): inputs and parts", odd facts:
 *    RMSNorm eps = 1e-5 model-wide.  Here rms(h) = sqrt(mean_c h_c^2 + eps).
 *  - [Tutorial] Kimi K3 chaptered tutorial (kimi.papertok.ai), ch. 4.3,
 *    Eq. 10: layers are split into blocks of B layers; a completed block is
 *    kept as the SUM of its layers' outputs b_n; layer i of block n reads
 *    [b_0 .. b_{n-1}] if i = 1 and [b_0 .. b_{n-1}, partial] if i >= 2,
 *    where b_0 is the embedding h_0 and the partial sum holds the outputs of
 *    layers 1..i-1 of block n.  The final output layer aggregates all block
 *    representations.  Ch. 4.5: K3 uses B = 12 over 93 layers (the 8th block
 *    has 9 layers), so at most 9 sources.  Ch. 4.6: block representations
 *    are produced once at the block boundary and then stay resident.
 *
 * Conventions for every call:
 *  - Tensors are row-major [T, d] (token-major, channel contiguous) in device
 *    memory of the CURRENT device (cudaGetDevice), on which every call
 *    launches; `sources` / `block_reps` are HOST arrays of DEVICE pointers.
 *  - The caller owns and allocates every buffer.  The library makes no
 *    device allocation and keeps no device-side global state, with one
 *    exception: the fixed scratch array built into it for
 *    attnres_aggregate_backward_noalloc (see there).
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL = the legacy default stream) and never synchronise the device.
 *  - Argument errors are detected on the host before any launch and return
 *    a negative attnres_status; nothing is written then.  A failed launch
 *    returns ATTNRES_ECUDA; attnres_last_error() gives the CUDA message
 *    (per host thread).
 *  - dev_err (nullable): a device int32 the kernels OR error bits into
 *    (ATTNRES_DEVERR_*); they never clear it.  Every spin-wait inside the
 *    kernels has a time limit; when one runs out the kernel sets the bit,
 *    writes NaN to the affected outputs, drains its own copies and returns.
 *  - Any pointer alignment and any d >= 1 is accepted; rows that start on a
 *    16-byte boundary with 16-byte-multiple row length take the bulk-copy
 *    (TMA) path, others a plain-load kernel (still on the GPU).
 *  - Environment, read once per process: ATTNRES_NO_PDL=1 launches without
 *    programmatic dependent launch; ATTNRES_SPLIT=1 lets a launch of at most
 *    9 sources over few tokens (T times the cluster size within the SM
 *    count) share each token across a thread-block cluster of 2, 4 or 8
 *    CTAs.  Results agree with the default path to the order of fp32 sums.
 */
#ifndef ATTNRES_H
#define ATTNRES_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTNRES_OK = 0,
  ATTNRES_EINVAL = -1, /* null pointer, non-positive size, bad eps */
  ATTNRES_EDTYPE = -2, /* dtype code not one of attnres_dtype */
  ATTNRES_ERANGE = -4, /* S > ATTNRES_MAX_SOURCES, too many blocks, T*d overflow */
  ATTNRES_ECUDA = -5,  /* a CUDA runtime call or launch failed */
  ATTNRES_ESTATE = -6  /* stack call out of order (see attnres_state) */
} attnres_status;

typedef enum { ATTNRES_F32 = 0, ATTNRES_BF16 = 1 } attnres_dtype;

/* bits ORed into *dev_err by the kernels */
#define ATTNRES_DEVERR_WAIT_TIMEOUT 0x1 /* a bounded wait on a copy gave up */

#define ATTNRES_MAX_SOURCES 128
#define ATTNRES_MAX_BLOCKS (ATTNRES_MAX_SOURCES - 1)
#define ATTNRES_DEFAULT_EPS 1e-5f

/* ------------------------------------------------------------------------
 * attnres_aggregate -- one layer of depth-wise attention ([Deep-dive 2] §2).
 *
 *   for every token t in [0, T):
 *     z[s]  = (sum_c w_l[c] * src_s[t,c]) / sqrt(mean_c src_s[t,c]^2 + eps)
 *     a[t,:] = softmax_s(z)                         (fp32)
 *     r[t,c] = sum_s a[t,s] * src_s[t,c]            (fp32 accumulate)
 *
 * sources     host array of S device pointers, each [T, d] of src_dtype
 *             (a [S, T, d] slab: sources[s] = base + s*T*d elements)
 * S           1 .. ATTNRES_MAX_SOURCES
 * T, d        T >= 0 (T = 0 launches nothing and accepts NULL buffers), d >= 1
 * src_dtype   ATTNRES_F32 or ATTNRES_BF16
 * w_l         device [d] fp32 pseudo-query
 * eps         > 0 or 0 (1e-5 in K3)
 * out_r       device [T, d] of out_dtype; bf16 is rounded to nearest even
 * out_weights device [T, S] fp32, or NULL to skip
 * Each source row is read from device memory once.  out_r and out_weights
 * may not share a byte with a source or with each other (ATTNRES_EINVAL);
 * sources may repeat.  Returns ATTNRES_OK or a negative attnres_status.
 * ---------------------------------------------------------------------- */
int attnres_aggregate(const void* const* sources, int S, int64_t T, int d, int src_dtype,
                      const float* w_l, float eps, void* out_r, int out_dtype,
                      float* out_weights, int* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * attnres_aggregate_fold -- one layer whose last source is a partial sum
 * formed in the same launch ([Tutorial] ch. 4.3: the partial sum of a block
 * is the sum of its layer outputs so far), i.e. attnres_layer_step without
 * a state:
 *
 *   p[t,c] = round(prev[t,c] + F[t,c])   (or round(F[t,c]) when prev is
 *            NULL; fp32 add, rounded to dtype), stored to dst;
 *   then attnres_aggregate over [sources[0..n_stored-1], p] (p as read back
 *   from dst's rounding, so the weights see exactly the stored bits).
 *
 * sources     host array of n_stored (0..127) device pointers [T, d] of
 *             dtype (NULL when n_stored = 0)
 * prev        device [T, d] or NULL; F: device [T, d]; dst: device [T, d]
 *             (may be prev itself, updated in place, but no other row)
 * dtype       of every row and of out_r
 * w_l, eps, out_r, out_weights ([T, n_stored + 1] fp32 or NULL), dev_err,
 *             stream: as attnres_aggregate.
 * flags       0, or ATTNRES_STATE_EARLY_LOADS: the stored rows and prev of
 *             the first token are loaded before the kernel launched just
 *             before this call has finished, only F after it -- under the
 *             conditions given at that flag (here: that kernel writes
 *             nothing this call reads except F).
 * Results equal attnres_fold followed by attnres_aggregate bit for bit,
 * with one launch and one row fewer per token.  Outputs may not share
 * memory with any row (ATTNRES_EINVAL).
 * ---------------------------------------------------------------------- */
int attnres_aggregate_fold(const void* const* sources, int n_stored, const void* prev, const void* F, void* dst,
                           int64_t T, int d, int dtype, const float* w_l, float eps, void* out_r,
                           float* out_weights, int flags, int* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * attnres_aggregate_host -- attnres_aggregate on sources, query and outputs
 * that live in HOST memory.  The pages have no counterpart: this is the
 * library's way in for data that starts on the CPU.
 *
 * The tokens are cut into chunks of chunk_tokens (the last may be shorter).
 * Chunk c goes to staging slot c mod nslots of `workspace`: its S source
 * rows are copied in, aggregated as soon as they have arrived, and its r
 * (and weights) copied out while later chunks are still coming in, so the
 * host link carries both directions at once.  Results are those of
 * attnres_aggregate on the same data (each token is computed alone).
 *
 * sources_host host array of S HOST pointers, each [T, d] of src_dtype.
 *             Page-locked memory (cudaHostAlloc, cudaHostRegister) lets the
 *             copies run at the link's rate, asynchronously; pageable memory
 *             works, but the driver then stages each copy and the call
 *             returns only once the sources have been read.
 * w_host      host [d] fp32 pseudo-query
 * r_host      host [T, d] of out_dtype; weights_host host [T, S] fp32 or NULL
 * chunk_tokens >= 1 (values above T act as T)
 * workspace   device buffer owned by the caller, 256-byte aligned, of
 *             workspace_bytes >= attnres_aggregate_host_workspace_size(...,
 *             1); the call uses as many slots as fit, at most 8 and at most
 *             the number of chunks (2 to 3 slots let copies and compute
 *             overlap).  Its contents on entry do not matter.
 * stream      work already on `stream` comes first; work issued on `stream`
 *             after the call waits until r_host / weights_host hold the
 *             results, so synchronise `stream` before reading them or
 *             writing the inputs again.  The copies run on two streams that
 *             the call creates and destroys (CUDA defers their release until
 *             their work is done).  A stream being captured into a graph
 *             is refused (ATTNRES_EINVAL).  If a CUDA call fails part way
 *             (ATTNRES_ECUDA), the copies already queued are still joined
 *             into `stream` before the call returns.
 * Other arguments, bounds and errors as attnres_aggregate; nothing is
 * copied or launched when an argument is rejected.
 * ---------------------------------------------------------------------- */
int attnres_aggregate_host(const void* const* sources_host, int S, int64_t T, int d,
                           int src_dtype, const float* w_host, float eps, void* r_host,
                           int out_dtype, float* weights_host, int64_t chunk_tokens,
                           void* workspace, int64_t workspace_bytes, int* dev_err,
                           void* stream);

/* Bytes of workspace attnres_aggregate_host needs for `slots` staging slots
 * of chunk_tokens tokens (the query, then per slot the [S, chunk_tokens, d]
 * sources, r and, if with_weights, the weights, each part 256-byte
 * aligned); slots 1..8.  Host only.  Negative attnres_status on bad
 * arguments. */
int64_t attnres_aggregate_host_workspace_size(int S, int64_t chunk_tokens, int d, int src_dtype,
                                              int out_dtype, int with_weights, int slots);

/* ------------------------------------------------------------------------
 * attnres_aggregate_backward -- gradients of attnres_aggregate.  In training
 * AttnRes runs under activation checkpointing ([Tutorial] ch. 4.6): nothing
 * is kept from the forward; the logits and weights are recomputed here from
 * the sources.  Per token, with rho_s = rms(h_s), z_s = w.h_s / rho_s,
 * a = softmax(z) and dr the gradient of the loss with respect to r:
 *   g_s = dr.h_s,  gbar = sum_s a_s g_s,  dz_s = a_s (g_s - gbar),
 *   alpha_s = dz_s / rho_s,  beta_s = alpha_s z_s / (d rho_s)
 *   grad_sources[s][t,:]  =  (or +=)  a_s dr + alpha_s w - beta_s h_s
 *   grad_w[c]             =  sum_t sum_s alpha_s h_s[t,c]
 *
 * sources, S, T, d, w_l, eps  as in attnres_aggregate; dtype is that of the
 *             sources, of grad_r and of grad_sources
 * grad_r      device [T, d] of dtype
 * grad_sources host array of S device pointers [T, d] of dtype, none of them
 *             sharing memory with a source, with grad_r or with each other
 *             (ATTNRES_EINVAL); overwritten (accumulate = 0)
 *             or added to (accumulate = 1: a source read by several layers
 *             collects the gradient of each)
 * grad_w      device [d] fp32, overwritten (fp32 sums in a fixed order:
 *             bit-reproducible)
 * workspace   device scratch, 4-byte aligned, at least
 *             attnres_aggregate_backward_workspace_size(T, d) bytes, owned
 *             by the caller; its contents on entry do not matter
 * Reads (S + 1) rows and writes S rows per token (S more read with
 * accumulate).  T = 0 only zeroes grad_w.
 * ---------------------------------------------------------------------- */
int attnres_aggregate_backward(const void* const* sources, int S, int64_t T, int d, int dtype,
                               const float* w_l, float eps, const void* grad_r,
                               void* const* grad_sources, int accumulate, float* grad_w,
                               void* workspace, int64_t workspace_bytes, int* dev_err,
                               void* stream);

/* Bytes of workspace attnres_aggregate_backward needs for T tokens of d
 * channels on the current device (one fp32 row of d per CTA it runs, at most
 * one CTA per SM).  Negative attnres_status on error. */
int64_t attnres_aggregate_backward_workspace_size(int64_t T, int d);

/* ------------------------------------------------------------------------
 * attnres_aggregate_backward_noalloc -- attnres_aggregate_backward without
 * a caller workspace, for callers that cannot allocate device memory (code
 * that runs under a fixed device-memory budget or must not call cudaMalloc
 * once it is running, e.g. inside a serving or replay loop).  The pages
 * have no counterpart: this is a library convenience.
 *
 * The workspace is a scratch array built into the library (1,310,720 fp32
 * values, 5 MiB, held by every GPU that loads the library until the process
 * exits).  Calls needing more (CTAs x d fp32 values, CTAs = min(T, SMs); on
 * a 152-SM GB300 any T with d <= 8192 fits) return ATTNRES_ERANGE with a
 * message naming the sizes; use attnres_aggregate_backward then.  Nothing
 * is allocated and no allocating library routine is called.
 *
 * The first call on a device looks up the array's device address (one
 * cudaGetSymbolAddress, with that device current) and caches it, keyed by
 * the device and its current context: make that first call before any
 * stream capture, and again after the device's context was torn down and
 * recreated (cudaDeviceReset), when the address is looked up anew.  All calls share the array and it
 * keeps the previous call's contents (every value a call reads it has
 * written first, so nothing needs clearing); calls whose kernels overlap on
 * a GPU (other streams or host threads) race on it and must be serialised.
 * Arguments, results and errors otherwise as attnres_aggregate_backward.
 * ---------------------------------------------------------------------- */
int attnres_aggregate_backward_noalloc(const void* const* sources, int S, int64_t T, int d,
                                       int dtype, const float* w_l, float eps,
                                       const void* grad_r, void* const* grad_sources,
                                       int accumulate, float* grad_w, int* dev_err,
                                       void* stream);

/* ------------------------------------------------------------------------
 * Stack state: the resident depth sources of one batch of T tokens.
 * ([Tutorial] ch. 4.3-4.6: b_0 = embedding, b_1 .. b_N completed block sums
 * kept resident, one running partial sum of the current block.)
 *
 * The caller allocates the buffers (each [T, d] of `dtype`) and fills the
 * struct with attnres_state_init; the library only updates `folded`.
 * `folded` = number of layer outputs v_1 .. v_folded already folded into the
 * partial sum / block representations.  Layer outputs must be folded in
 * order: attnres_block_step(p) needs folded == p-1; attnres_layer_step(l)
 * needs folded == l-2 when it is given v_{l-1} to fold, folded == l-1
 * when not; attnres_layer_sources(l) needs folded == l-1.  Anything else
 * returns ATTNRES_ESTATE.
 * ---------------------------------------------------------------------- */
typedef struct attnres_state {
  const void* h0;                          /* device [T, d]: b_0, the embedding */
  void* block_reps[ATTNRES_MAX_BLOCKS];    /* block_reps[k-1] = b_k, k = 1..N */
  void* partial;                           /* device [T, d]: running partial sum */
  int64_t T;
  int d;
  int dtype;                               /* attnres_dtype of every buffer */
  int num_layers;                          /* L */
  int block_size;                          /* B */
  float eps;
  int folded;                              /* progress, maintained by the library */
  int flags;                               /* ATTNRES_STATE_*, set by the caller after init */
} attnres_state;

/* attnres_state.flags bit: a layer step that folds F_prev (the fused step)
 * may load the first token's stored rows -- h0, the block sums, the
 * partial sum -- before the kernel launched just before it on the stream
 * has finished (programmatic dependent launch), so that their DRAM latency
 * overlaps that kernel; only F_prev waits for it.  attnres_intrablock_step
 * with F_prev does the same with the partial sum and r_inter.  Set it only
 * when, before every such step, (a) the kernel launched just before it on
 * the stream writes none of the rows the step reads other than F_prev (in
 * a stack that kernel is the layer body; a step issued directly after
 * another step of the same state breaks this), and (b) that kernel is
 * launched without programmatic dependent launch, or signals its
 * dependents only after it has waited for its own prerequisites, as every
 * kernel of this library does: then everything launched before it has
 * completed when the step starts.  The stack drivers of the Python package
 * set it; results are the same bits either way. */
#define ATTNRES_STATE_EARLY_LOADS 0x1

/* Fill *st.  n_block_reps must be >= ceil(L/B) (ATTNRES_ERANGE if
 * ceil(L/B) > ATTNRES_MAX_BLOCKS).  The buffers may not share memory with
 * each other (ATTNRES_EINVAL; *st is not written then).
 * Host only; sets folded = 0 and flags = 0. */
int attnres_state_init(attnres_state* st, const void* h0, void* const* block_reps,
                       int n_block_reps, void* partial, int64_t T, int d, int dtype,
                       int num_layers, int block_size, float eps);

/* Rewind to layer 1 (folded = 0).  Host only; buffers are left as they are. */
int attnres_state_reset(attnres_state* st);

/* attnres_state_resume -- take up a stack after layer `folded` (0..L), for
 * a pipeline stage that starts at layer folded + 1 ([Tutorial] ch. 4.6:
 * cache-based pipeline communication sends a later stage only the blocks
 * completed since it last received, plus the open partial sum).  Host only:
 * sets st->folded and touches no buffer.  The caller has already placed in
 * the state's buffers what layer folded + 1 reads: h0, b_1 .. b_c
 * (c = completed blocks after layer `folded`) and, when layer `folded`
 * does not end its block, the partial sum of v_{first..folded} of the open
 * block; the sender forms them with attnres_block_step(folded) after its
 * last layer.  The next call is attnres_layer_step(folded + 1) with
 * F_prev = NULL (or attnres_layer_sources(folded + 1)).  ATTNRES_EINVAL for
 * folded outside 0..L; other errors as attnres_state_reset. */
int attnres_state_resume(attnres_state* st, int folded);

/* Number of sources layer `layer_idx` (1..L, or L+1 for the final output
 * aggregation) reads: n + [i >= 2] for layer i of block n, ceil(L/B) + 1 for
 * L+1 ([Tutorial] ch. 4.3 Eq. 10; [Atlas] §28 workbench: ceil(L/S) +
 * embedding).  Host only, pure.  Negative status on bad arguments. */
int attnres_num_sources(int layer_idx, int block_size, int num_layers);

/* Host only: the device pointers of layer `layer_idx`'s sources in order
 * [h_0, b_1 .. b_{n-1}, partial (if non-empty)] into out_ptrs (capacity
 * ATTNRES_MAX_SOURCES), their count into *out_S.  Needs folded ==
 * layer_idx - 1.  With attnres_block_step this gives the unfused path:
 * block_step(p) then aggregate(layer_sources(p+1)). */
int attnres_layer_sources(const attnres_state* st, int layer_idx, const void** out_ptrs,
                          int* out_S);

/* ------------------------------------------------------------------------
 * attnres_block_step -- fold layer `layer_idx`'s output v = F_out into the
 * block bookkeeping ([Tutorial] ch. 4.3, 4.6):
 *   new = (partial non-empty) ? partial + v : v      (fp32 add, one rounding)
 *   if layer_idx ends its block (layer_idx % B == 0 or layer_idx == L):
 *        b_n = new, partial becomes empty
 *   else partial = new
 * F_out: device [T, d] of st->dtype, sharing no memory with the state's
 * rows (ATTNRES_EINVAL).  Needs folded == layer_idx - 1; advances folded.
 * One elementwise launch.
 * ---------------------------------------------------------------------- */
int attnres_block_step(attnres_state* st, const void* F_out, int layer_idx, int* dev_err,
                       void* stream);

/* ------------------------------------------------------------------------
 * attnres_layer_step -- the fused hot path of one layer: fold F_prev =
 * v_{l-1} (exactly as attnres_block_step(l-1) would, same rounding, written
 * to the partial sum or to b_n) and aggregate layer l over its sources,
 * using the freshly formed partial / b_n as the last source without reading
 * it back.  One launch.
 *   layer_idx  1..L+1 (L+1 = the final output aggregation over [h_0, b_1..b_N])
 *   F_prev     device [T, d] of st->dtype; NULL when v_{l-1} is already
 *              folded (layer 1, or a state resumed with attnres_state_resume
 *              at folded == l-1): then layer l is aggregated over the
 *              state's sources as they are
 *   w_l        device [d] fp32 pseudo-query of this layer
 *   out_r      device [T, d] of st->dtype; it and out_weights may not share
 *              memory with the state's rows or F_prev (ATTNRES_EINVAL)
 *   out_weights device [T, S_l] fp32 or NULL
 * Needs folded == layer_idx - 2 with F_prev, layer_idx - 1 without;
 * leaves folded at layer_idx - 1.  Bit-identical to block_step(l-1) +
 * aggregate(layer_sources(l)).
 * ---------------------------------------------------------------------- */
int attnres_layer_step(attnres_state* st, const void* F_prev, const float* w_l, int layer_idx,
                       void* out_r, float* out_weights, int* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * Two-phase schedule of inference ([Tutorial] ch. 4.4 and 4.6): the cached
 * sources [h_0, b_1 .. b_{n-1}] do not change inside block n, so one
 * batched inter-block pass reads each of them once and aggregates them for
 * every layer query of the block; each layer then folds in its own partial
 * sum with an online-softmax merge.  Same results as attnres_layer_step up
 * to fp32 rounding.  Both calls need rows of a 16-byte multiple with at
 * most 2 x 448 16-byte vectors (d <= 7168 bf16 / 3584 fp32) and 16-byte
 * aligned buffers (ATTNRES_ERANGE / ATTNRES_EINVAL otherwise).
 *
 * attnres_interblock -- phase 1 for one block.
 *   sources    host array of n (1..9) device pointers [T, d] of dtype
 *   w_queries  host array of Q (1..16) device pointers [d] fp32 (the
 *              block's layer queries in order), each 16-byte aligned
 *   out_r      device [Q, T, d] fp32: per query, the softmax-weighted sum
 *              over the n sources (normalised)
 *   out_lse    device [Q, T] fp32: log sum_s exp(z_qs) of those logits
 *   out_weights device [Q, T, n] fp32 (softmax over the n sources) or NULL
 *   out_r0     device [T, d] of dtype, 16-byte aligned, or NULL: query 0's
 *              row rounded to dtype -- the output of the block's first
 *              layer, the same bits attnres_intrablock_step writes for it
 *              (which the caller may then skip: it folds nothing there)
 *   out_weights0 device [T, n] fp32 or NULL: query 0's weights, the first
 *              layer's (the same bits attnres_intrablock_step writes)
 *   workspace  NULL, or device scratch of at least
 *              attnres_interblock_workspace_size(n, T, d, dtype, Q) bytes,
 *              256-byte aligned, owned by the caller, sharing no memory
 *              with an input or output (its contents on entry do not
 *              matter).  With it (bf16 sources, d a multiple of 64) the
 *              Q x n logits of all tokens are taken on the tensor cores
 *              (tcgen05.mma): the queries split into three bf16 terms
 *              (hi + mid + lo, fp32 accumulation), tiles of tokens x
 *              sources loaded by TMA, the channels split across CTAs; the
 *              softmax and the weighted sums then read the sources again.
 *              Without it (or when the size is 0) every step runs on the
 *              CUDA cores in one pass.  Results agree to fp32 rounding.
 *   workspace_bytes  its size
 *   Every source row is read once for all Q queries (twice with the
 *   workspace: once for the logits, once for the weighted sums).  No output
 *   may share memory with a source or with another output (ATTNRES_EINVAL).
 * ---------------------------------------------------------------------- */
int attnres_interblock(const void* const* sources, int n, int64_t T, int d, int dtype,
                       const float* const* w_queries, int Q, float eps, float* out_r,
                       float* out_lse, float* out_weights, void* out_r0, float* out_weights0,
                       void* workspace, int64_t workspace_bytes, int* dev_err, void* stream);

/* Bytes of workspace attnres_interblock's tensor-core logits need for n
 * sources of T tokens and d channels and Q queries on the current device
 * (the partial dot products of every channel split); 0 when that path does
 * not apply (fp32 sources, d not a multiple of 64).  Negative
 * attnres_status on bad arguments. */
int64_t attnres_interblock_workspace_size(int n, int64_t T, int d, int dtype, int Q);

/* attnres_intrablock_step -- phase 2 for layer l (1..L) of block n:
 *   first layer of its block (i = 1): F_prev NULL and the previous block
 *     already closed (attnres_block_step); r = r_inter.
 *   later layers (i >= 2): F_prev = v_{l-1} is folded into the partial sum
 *     exactly as attnres_layer_step folds it, p = the new partial sum,
 *     z_p = w_l . RMSNorm(p), m = max(lse, z_p) and
 *       r = (e^{lse-m} r_inter + e^{z_p-m} p) / (e^{lse-m} + e^{z_p-m}).
 *   r_inter, lse_inter, a_inter: this layer's rows of attnres_interblock's
 *     outputs ([T, d], [T], [T, n] or NULL).
 *   out_r: device [T, d] of st->dtype; out_weights: [T, S_l] fp32 or NULL
 *     (the cached sources' weights scaled into the merged softmax, then the
 *     partial sum's).
 * Needs folded == l-1 (i = 1) or l-2 (i >= 2); advances folded like
 * attnres_layer_step.  The final aggregation (L+1) uses attnres_layer_step.
 * Later layers with bf16 rows of d = 7168 stream their rows (previous
 * partial, F_prev, r_inter) through the persistent TMA ring; its waits are
 * bounded, and one that runs out sets ATTNRES_DEVERR_WAIT_TIMEOUT in
 * dev_err and leaves NaN in that token's outputs. */
int attnres_intrablock_step(attnres_state* st, const void* F_prev, const float* w_l,
                            int layer_idx, const float* r_inter, const float* lse_inter,
                            const float* a_inter, void* out_r, float* out_weights,
                            int* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * attnres_synthetic_layer -- the stand-in layer body used to drive a stack
 * forward without trained weights (not part of the method):
 *   out[t,c] = tanh(x[t,c] * g[c]) * s[c], fp32 math, rounded to `dtype`.
 * x, out: device [T, d] of dtype (may alias); g, s: device [d] fp32.
 * ---------------------------------------------------------------------- */
int attnres_synthetic_layer(const void* x, const float* g, const float* s, void* out, int64_t T,
                            int d, int dtype, void* stream);

/* ------------------------------------------------------------------------
 * attnres_synthetic_layer_backward -- gradient of attnres_synthetic_layer
 * (the stand-in body, not part of the method), for a stack backward:
 *   grad_x[t,c] = (grad_out_a + grad_out_b)[t,c] * (1 - tanh(x g)^2) * g[c] * s[c]
 * x: the layer's input [T, d] of dtype; grad_out_a: [T, d] of dtype, the
 * gradient of the loss with respect to the layer's output; grad_out_b: a
 * second such term added to it, or NULL; grad_x: [T, d] of dtype (may alias
 * either gradient input); g, s: [d] fp32.  fp32 math, rounded to dtype.
 * T = 0 launches nothing and accepts NULL buffers.
 * ---------------------------------------------------------------------- */
int attnres_synthetic_layer_backward(const void* x, const float* g, const float* s, const void* grad_out_a,
                                     const void* grad_out_b, void* grad_x, int64_t T, int d, int dtype,
                                     void* stream);

/* ------------------------------------------------------------------------
 * attnres_fold -- the block bookkeeping of [Tutorial] ch. 4.3 (Eq. 10) on
 * plain buffers, without a state: dst = prev + F (fp32 sum, one rounding to
 * dtype), or dst = F when prev is NULL (a block's first layer output opens
 * its partial sum).  prev, F, dst: device [T, d] of dtype; elementwise, so
 * dst may alias prev or F.  Used where the partial sums of a block are kept
 * per layer (the recomputed forward of a stack backward).
 * ---------------------------------------------------------------------- */
int attnres_fold(const void* prev, const void* F, void* dst, int64_t T, int d, int dtype, void* stream);

/* ------------------------------------------------------------------------
 * attnres_debug_wait_test -- a diagnostic with no counterpart in the pages:
 * makes the bounded waits of the ring kernels launched afterwards from this
 * process run out on a healthy GPU, so that their timeout path can be tested
 * without a fault.
 *   wait_limit_ns  limit of every main-loop wait (a ring slot's landing or
 *                  release); 0 = the default, 2 s.  The drain at a kernel's
 *                  exit always waits up to 2 s for the copies it issued.
 *   withhold_row   0..7: every CTA's producer arms that row of its first
 *                  token but issues no copy for it, so the consumers' wait
 *                  on it runs out after wait_limit_ns; -1 = none.
 * Expected effect: ATTNRES_DEVERR_WAIT_TIMEOUT in dev_err, NaN outputs for
 * the abandoned token, the kernel returns (no slot is refilled under a copy
 * in flight; its copies are drained), the context stays usable.  Outputs of
 * kernels launched in this mode are not meaningful.  (0, -1) restores
 * normal operation.  Process-wide; not for use while other threads launch.
 * Returns ATTNRES_OK, or ATTNRES_EINVAL for withhold_row outside -1..7.
 * ---------------------------------------------------------------------- */
int attnres_debug_wait_test(uint64_t wait_limit_ns, int withhold_row);

/* Human-readable name of a status code (static string). */
const char* attnres_status_string(int status);

/* Detail of the last error returned on this host thread ("" if none). */
const char* attnres_last_error(void);

/* ABI version: (major << 16) | minor. */
int attnres_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTNRES_H */
