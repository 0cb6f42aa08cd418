/*
 * glacore.h -- C ABI of the chunk-parallel gated linear attention library
 * (GLA and Mamba-2 SSD, forward and backward) for NVIDIA GB300 (sm_103a).
 *
 * The operation (FLAT blog, trainstation-project.github.io/blog/flat,
 * section "Linear Attention / Forward Recurrence" and its architecture
 * table; JLA product page, karlex.ai/jla, for segment_ids and states):
 *
 *     S_t = diag(exp(g_t)) S_{t-1} + k_t v_t^T,     o_t = scale * S_t^T q_t
 *
 * with S a K x V state per (document, head).  GLA: g is a log-decay per key
 * channel, g[B,T,H,K].  Mamba-2 SSD: one scalar log-decay per head,
 * g[B,T,H].  A document starts at t = 0 of every batch row and wherever
 * segment_ids[b,t] != segment_ids[b,t-1]; the state restarts there from the
 * document's initial state (or zero).  Documents are numbered 0..n_seqs-1
 * in row-major order of their first token.  The first token of a document
 * decays the initial state: S_{t0} = diag(exp(g_{t0})) h0 + k v^T.
 *
 * Backward (FLAT blog, "Backward Recurrence" and "Backward Kernels"): the
 * state gradient runs backwards in time; the gate gradient is the suffix
 * sum over the document of q (.) dq - k (.) dk plus the final-state term
 * (S_T (.) dht) 1_V.  States are recomputed inside the backward call; the
 * forward stores nothing for it.
 *
 * Conventions (all entry points):
 *  - Every data pointer is a DEVICE pointer owned by the caller.  The
 *    library allocates no memory, never synchronises the stream (except
 *    glacore_get_device_error, which says so) and
 *    enqueues all work on `stream` (NULL = legacy default stream).
 *  - Layouts are row-major; q, k and v may have a token stride (below), all
 *    other tensors are contiguous.  Offsets are computed in 64-bit.
 *      q, k        [B, T, Hqk, K]   (dtype)
 *      v, o, do    [B, T, H, V]     (dtype)
 *      g, dg       GLA: [B, T, H, K] fp32;  SSD: [B, T, H] fp32  (g <= 0)
 *      segment_ids [B, T] int32 or NULL (then every row is one document)
 *      states      [n_seqs, H, K, V] fp32 (initial_state, final_state,
 *                  dht, dh0)
 *      dq, dk      [B, T, Hqk, K] (dtype); summed over the H/Hqk heads that
 *                  share q and k.  dv [B, T, H, V] (dtype).
 *  - Every output is fully overwritten (no read-modify-write of outputs).
 *  - Host-side validation runs before any launch; on failure nothing is
 *    enqueued and an error status is returned.
 *  - Inconsistencies that only the device can see (the number of documents
 *    in segment_ids differs from n_seqs; a decay outside the kernels'
 *    range) set a device error word instead of trapping; read it with
 *    glacore_get_device_error.
 *  - Decay range.  Inside a chunk the kernels evaluate exp(G_t - G_s) as
 *    exp(G_t) * exp(-G_s), with G the prefix sum of g from the chunk start
 *    (FLAT blog, "Gated Linear Attention": decay ratios as exponentiated
 *    chunk-local prefix sums).  That product stays inside the fp32 / bf16
 *    exponent range while the summed log-decay of every chunk, in every
 *    key channel, is at least -80.  A call that meets a chunk below that
 *    sets GLACORE_ERR_RANGE and its outputs are not valid.  The CUDA-core
 *    kernels (chunk_size 16) have the same bound per 16 tokens, so they
 *    cover decays four times stronger: up to an average log-decay of -5
 *    per token, against -1.25 on the tensor-core path.
 *  - Pointers passed to the tensor-core path must be 16-byte aligned.
 *  - Calls on different streams may run concurrently provided they use
 *    different workspace buffers.
 */
#ifndef GLACORE_H
#define GLACORE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st *glacore_stream_t;

typedef enum {
  GLACORE_OK = 0,
  GLACORE_ERR_INVALID_ARG = 1, /* bad size, NULL required pointer, misalignment */
  GLACORE_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. chunk_size) */
  GLACORE_ERR_CUDA = 3,        /* a CUDA runtime call failed */
  GLACORE_ERR_TIMEOUT = 4,     /* a bounded device wait ran out */
  GLACORE_ERR_WORKSPACE = 5,   /* workspace NULL or smaller than *_workspace_size */
  GLACORE_ERR_DOCS = 6,        /* device: document count != n_seqs */
  GLACORE_ERR_RANGE = 7        /* device: a chunk's decay is outside the kernels' range (below) */
} glacore_status;

typedef enum { GLACORE_F32 = 0, GLACORE_BF16 = 1 } glacore_dtype;

/* One problem description, shared by the forward and backward entries.
 *   B, T        batch rows and tokens per row (T >= 0; B >= 1)
 *   H           value heads; Hqk heads of q/k (H % Hqk == 0; see head sharing below)
 *   K, V        key and value head dims (1..256)
 *   dtype       element type of q, k, v, o, do, dq, dk, dv
 *   chunk_size  chunk length of the chunk-parallel form: 0, 16, 32 or 64
 *               (any other value: GLACORE_ERR_UNSUPPORTED).  The tensor-core
 *               kernels (bf16; GLA with K = V = 128; SSD with K = 128 and V
 *               of 64 or 128) run chunks
 *               of 64 and take chunk_size 0 or 64.  Every other problem, and
 *               any problem given chunk_size 16 or 32, runs the CUDA-core
 *               kernels with chunks of chunk_size tokens (0: 16); those take
 *               32 and 64 only where their shared memory fits (64: K = V =
 *               64 or smaller; 32: K * V up to about 8192), and
 *               GLACORE_ERR_UNSUPPORTED otherwise.  Results do not depend
 *               on it beyond rounding.
 *   scale       output scale (GLA usually K^-1/2; Mamba-2: 1)
 *   n_seqs      number of documents: B when segment_ids is NULL
 *   initial_state  [n_seqs,H,K,V] fp32 or NULL (zero)
 *   workspace   device scratch of at least *_workspace_size(problem) bytes
 *               (may be NULL when that size is 0); 256-byte aligned
 *   q_stride, k_stride, v_stride
 *               elements between consecutive tokens (rows of [B*T]) of q,
 *               k and v; 0 means contiguous (Hqk*K, Hqk*K, H*V).  Within a
 *               token the heads stay contiguous ([heads, D]).  This lets q,
 *               k and v be read in place from one fused projection
 *               [B, T, 2*Hqk*K + H*V] (FLAT blog, "Forward Kernels / Data
 *               movement" and "Full Linear Attention Layer": no layout copies
 *               between the projection and the kernels).  A stride must be
 *               at least the contiguous one; on the tensor-core path it must
 *               be a multiple of 8 elements (16 bytes), as must the three
 *               base addresses.
 * Head sharing (FLAT blog, "Gated Linear Attention": queries, keys, values
 * and the gate may use different head counts): Hqk q/k heads serve H value
 * heads (H % Hqk == 0, value head h reads q/k head h / (H / Hqk)); the gate
 * and the state are per value head; dq and dk are summed over the heads
 * that share them. */
typedef struct glacore_problem {
  int64_t B, T, H, Hqk, K, V;
  int32_t dtype;
  int32_t chunk_size;
  float scale;
  int32_t reserved0; /* must be 0 */
  const void *q, *k, *v;
  const float *g;
  const int32_t *segment_ids;
  int64_t n_seqs;
  const float *initial_state;
  void *workspace;
  size_t workspace_bytes;
  int64_t q_stride, k_stride, v_stride;
} glacore_problem;

/* Scratch bytes needed by the matching call (0 if none).  Returns 0 and
 * does nothing else for an invalid problem (the call itself reports it). */
size_t gla_fwd_workspace_size(const glacore_problem *p);
size_t gla_bwd_workspace_size(const glacore_problem *p);
size_t ssd_fwd_workspace_size(const glacore_problem *p);
size_t ssd_bwd_workspace_size(const glacore_problem *p);

/* GLA forward (per-key-channel gate, g [B,T,H,K]).
 *   o            [B,T,H,V] dtype, written
 *   final_state  [n_seqs,H,K,V] fp32, written, or NULL (not returned)
 * FLAT blog, "Pallas Kernels for Linear Attention / Forward Kernels" (fused
 * block-recurrent forward: intra-chunk masked product plus the readout of
 * the carried state, state kept on chip across chunks). */
glacore_status gla_fwd(const glacore_problem *p, void *o, float *final_state,
                       glacore_stream_t stream);

/* GLA backward.
 *   do_   [B,T,H,V] dtype: dL/do
 *   dht   [n_seqs,H,K,V] fp32: dL/dfinal_state, or NULL (zero)
 *   dq, dk [B,T,Hqk,K], dv [B,T,H,V] (dtype), dg like g (fp32): written
 *   dh0   [n_seqs,H,K,V] fp32: dL/dinitial_state, written; may be NULL
 * FLAT blog, "Backward Recurrence" and "Backward Kernels" (a state pass
 * that reruns the forward recurrence, then a gradient pass over the chunks
 * in reverse carrying the state gradient; gate gradient as a suffix sum). */
glacore_status gla_bwd(const glacore_problem *p, const void *do_,
                       const float *dht, void *dq, void *dk, void *dv,
                       float *dg, float *dh0, glacore_stream_t stream);

/* Mamba-2 SSD: the same two calls with one scalar log-decay per head
 * (g and dg are [B,T,H]); q = C, k = B, v = x; q/k may be shared by
 * H/Hqk heads.  FLAT blog, section "Mamba-2" (scalar data-dependent gate
 * evaluated in log space). */
glacore_status ssd_fwd(const glacore_problem *p, void *o, float *final_state,
                       glacore_stream_t stream);
glacore_status ssd_bwd(const glacore_problem *p, const void *do_,
                       const float *dht, void *dq, void *dk, void *dv,
                       float *dg, float *dh0, glacore_stream_t stream);

/* gla_bwd without a workspace, for callers that cannot allocate device
 * memory when they call the backward (for example a host framework that
 * owns all device memory and gives its plugins no allocator, or a training
 * loop that forbids allocation after start-up).  The pages have no
 * counterpart to this entry point.
 * Same arguments and results as gla_bwd; p->workspace and
 * p->workspace_bytes are ignored.  The scratch is one fixed device array of
 * GLACORE_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds
 * until the process exits; a problem whose gla_bwd_workspace_size exceeds
 * it is rejected with GLACORE_ERR_WORKSPACE before any launch.  The first
 * call on each device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  All
 * calls share the array and it keeps the last call's contents: calls whose
 * work overlaps on the GPU (other streams, other host threads) race, so the
 * caller must serialise them.  It makes no cudaMalloc, cudaFree or other
 * allocating call. */
#define GLACORE_NOALLOC_SCRATCH_BYTES ((size_t)48 << 20)
glacore_status gla_bwd_noalloc(const glacore_problem *p, const void *do_,
                               const float *dht, void *dq, void *dk, void *dv,
                               float *dg, float *dh0, glacore_stream_t stream);

/* ---- sequence split across devices (context parallelism) ---------------
 * JLA product page ("our split is exact", unlike starting each piece from
 * zero); FLAT blog, "Future work" (sharding the sequence across chips).  The
 * recurrence is linear in the state, so a sequence cut into R consecutive
 * pieces (one per device, each holding all heads of its tokens) runs
 * exactly as a whole:
 *   1. every piece: gla_fwd_state -> its local end state L (from a zero
 *      initial state) and total decay D = exp(sum of g over the piece);
 *   2. gather L and D of all pieces ([R, ...], piece order) on every device;
 *      glacore_state_scan(reverse = 0, seed = the sequence's initial state)
 *      gives the state entering piece r;
 *   3. gla_fwd with that initial state gives the piece's o (and, on the last
 *      piece, the sequence's final state).
 * Backward: gla_bwd_state -> the piece's local state gradient at its start
 * (from a zero gradient at its end) and total decay; gather;
 * glacore_state_scan(reverse = 1, seed = dht of the sequence) gives the
 * state gradient leaving piece r; gla_bwd with the entering state as
 * initial_state and that gradient as dht gives the piece's dq, dk, dv, dg
 * exactly (dh0 of the first piece is the sequence's).
 * The two state entries run the tensor-core kernels (GLA, bf16, K = V = 128)
 * without segment_ids (GLACORE_ERR_UNSUPPORTED otherwise); they take no
 * workspace.
 *   L   [n_seqs, H, K, V] fp32, D [n_seqs, H, K] fp32, written
 *   do_ [B, T, H, V] (dtype) */
glacore_status gla_fwd_state(const glacore_problem *p, float *L, float *D,
                             glacore_stream_t stream);
glacore_status gla_bwd_state(const glacore_problem *p, const void *do_,
                             float *L, float *D, glacore_stream_t stream);
/* out = the fold for piece r of R: with s = seed (or 0),
 *   reverse = 0:  s <- diag(D[q]) s + L[q]  for q = 0 .. r-1
 *   reverse = 1:  s <- diag(D[q]) s + L[q]  for q = R-1 down to r+1
 * over every one of `mats` K x V fp32 matrices (L [R, mats, K, V],
 * D [R, mats, K], seed and out [mats, K, V], device pointers). */
glacore_status glacore_state_scan(const float *L, const float *D, int64_t R,
                                  int64_t mats, int64_t K, int64_t V,
                                  const float *seed, int64_t r, int32_t reverse,
                                  float *out, glacore_stream_t stream);

/* ---- operations around the recurrence ----------------------------------
 * Per-head RMSNorm times a swish output gate, on the recurrence's output
 * (FLAT blog, "Full Linear Attention Layer": the layer's per-head RMSNorm
 * multiplied by a swish output gate; FLA documentation, "Norm Layers with
 * Gating").  Over every row of V values (one token and head):
 *     y = o * rsqrt(mean(o^2) + eps) * w * z * sigmoid(z)
 *   o, z, y     [rows, V] (dtype; rows = B * T * H for o [B,T,H,V]),
 *               16-byte aligned
 *   w           [V] fp32 (one weight per channel, shared by the heads)
 *   V           8, 16, 32, 64, 128 or 256;  eps >= 0
 * Backward: do_, dz [rows, V] (dtype) and dw [V] fp32 written.  dw is
 * reduced deterministically through the workspace (at least
 * norm_gate_bwd_workspace_size bytes, 256-byte aligned). */
glacore_status norm_gate_fwd(const void *o, const void *z, const float *w,
                             int64_t rows, int64_t V, int32_t dtype, float eps,
                             void *y, glacore_stream_t stream);
size_t norm_gate_bwd_workspace_size(int64_t rows, int64_t V);
glacore_status norm_gate_bwd(const void *o, const void *z, const float *w,
                             const void *dy, int64_t rows, int64_t V,
                             int32_t dtype, float eps, void *do_, void *dz,
                             float *dw, void *workspace, size_t workspace_bytes,
                             glacore_stream_t stream);

/* Depthwise causal short convolution with bias and optional SiLU, the step
 * before the recurrence (FLAT blog, "Depthwise Causal Short Convolution"):
 * tap k of Kc reads the input Kc-1-k tokens back inside the token's
 * document (inputs before a row start or a segment id change read as 0),
 *     z_t = b + sum_k w[k] (.) x_{t-(Kc-1-k)},   y_t = SiLU(z_t) or z_t
 *   x, y        [B, T, D] (dtype), 16-byte aligned; D a multiple of 8
 *               (a fused q/k/v projection is one x of D = 3 H K)
 *   w           [Kc, D] fp32;  b [D] fp32 or NULL (no bias);  Kc in 1..4
 *   segment_ids [B, T] int32 or NULL (every row one document)
 *   activation  1: SiLU, 0: none
 * Backward: dx [B,T,D] (dtype), dw [Kc,D] and db [D] fp32 written (db is
 * the bias gradient even when b is NULL).  dw and db are reduced
 * deterministically through the workspace (at least
 * short_conv_bwd_workspace_size bytes, 256-byte aligned). */
glacore_status short_conv_fwd(const void *x, const float *w, const float *b,
                              const int32_t *segment_ids, int64_t B, int64_t T,
                              int64_t D, int32_t Kc, int32_t dtype,
                              int32_t activation, void *y,
                              glacore_stream_t stream);
size_t short_conv_bwd_workspace_size(int64_t B, int64_t T, int64_t D,
                                     int32_t Kc);
glacore_status short_conv_bwd(const void *x, const float *w, const float *b,
                              const int32_t *segment_ids, const void *dy,
                              int64_t B, int64_t T, int64_t D, int32_t Kc,
                              int32_t dtype, int32_t activation, void *dx,
                              float *dw, float *db, void *workspace,
                              size_t workspace_bytes, glacore_stream_t stream);

/* Counts the documents in segment_ids [B,T] (device pointer) and writes
 * the count, as int64, to *n_docs (DEVICE pointer, 8-byte aligned).
 * Asynchronous on `stream`; the caller reads the count after the stream
 * reaches it.  Used to size final_state / dh0 before a call. */
glacore_status glacore_count_docs(const int32_t *segment_ids, int64_t B,
                                  int64_t T, int64_t *n_docs,
                                  glacore_stream_t stream);

/* Reads and clears the library's device error word (set by kernels for
 * GLACORE_ERR_DOCS, GLACORE_ERR_RANGE or GLACORE_ERR_TIMEOUT).  Synchronises `stream`.
 * Returns GLACORE_OK if no device error was recorded. */
glacore_status glacore_get_device_error(glacore_stream_t stream);

/* Self-test of the bounded device waits.  Launches one CTA that waits on
 * a shared-memory mbarrier nothing ever arrives on, with a limit of
 * `cycles` SM clock cycles (1 .. 2^40), through the same bounded wait the
 * kernels use; when the limit runs out it records GLACORE_ERR_TIMEOUT in
 * the device error word and returns.  No copy, tensor-core work or tensor
 * memory is in flight.  Asynchronous on `stream`; read the result with
 * glacore_get_device_error.  The pages have no counterpart: it exists so
 * that the timeout path of every kernel can be shown to end. */
glacore_status glacore_selftest_wait(int64_t cycles, glacore_stream_t stream);

/* The CUDA runtime's description of the error behind this host thread's
 * last GLACORE_ERR_CUDA ("no CUDA error" if there was none; static). */
const char *glacore_last_cuda_error(void);

/* Static English description of a status code. */
const char *glacore_status_string(glacore_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
int glacore_version(void);

/* Measurement hook.  After this call, every kernel launch made by the next
 * gla_ / ssd_ entry call on this host thread is followed by a record of the
 * next event of `events` (cudaEvent_t[n_events], created by the caller) on
 * the call's stream, so the caller can time each kernel with
 * cudaEventElapsedTime.  Each entry call restarts at events[0].  Pass NULL
 * to switch it off.  glacore_timing_count() returns how many events the
 * last call recorded and glacore_timing_label(i) names the kernel launched
 * just before events[i] (static string). */
void glacore_set_timing_events(void *events, int n_events);
int glacore_timing_count(void);
const char *glacore_timing_label(int i);

#ifdef __cplusplus
}
#endif

#endif /* GLACORE_H */
