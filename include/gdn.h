/*
 * gdn.h -- C ABI of the GB300 (sm_103a) chunked Gated DeltaNet training path.
 *
 * The operation (one value head h, one document, state reset to zero at the
 * document start, q/k head j = h / (HV/H)):
 *
 *     S_t = a_t S_{t-1} + beta_t k^_t (v_t - a_t S_{t-1}^T k^_t)^T,   a_t = exp(g_t)
 *     o_t = scale * S_t^T q^_t
 *
 * with q^, k^ the L2-normalised q, k (x / sqrt(x.x + 1e-6)) when l2norm != 0,
 * else q, k as given; S is a dk x dv matrix kept in FP32.  This is the gated
 * delta rule that the flashinfer Cake GDN training pages run: "packed GDN
 * layers" over variable-length documents with head dim 128, BF16 q/k/v and
 * output gradient, FP32 g and beta, grouped heads (H query/key heads, HV value
 * heads), optional in-kernel q/k L2 norm, chunk states every 64 tokens
 * ("feat(cake_gdn_kcp): ... Cake GDN chunked autograd backend - #8172" page,
 * its #8181 section; "#8542" page, the opening description and the save-set
 * table).  The backward returns the gradients of sum(o * dO) with respect to
 * q, k, v, g and beta.
 *
 * Conventions (all entry points):
 *   - Sizes: dk = dv = 128, HV % H == 0, T = cu_seqlens[N], chunk = 64.
 *   - Layouts, all contiguous and token-major:
 *       q, k, dq, dk      [T][H][128]   BF16
 *       v, dO, o, dv      [T][HV][128]  BF16
 *       g, beta, dg, dbeta [T][HV]      FP32
 *       cu_seqlens        [N+1]         int32, 0 = cu[0] <= cu[1] <= ... <= cu[N] = T
 *     Device pointers must be 16-byte aligned.
 *   - cu_seqlens is passed twice: the host copy drives planning (chunk counts,
 *     segment plan, buffer sizes) and the device copy drives the kernels.  The
 *     two must hold the same values.
 *   - Ownership: the caller allocates and owns every buffer (inputs, outputs,
 *     `saved`, `workspace`).  The library allocates no device memory at run
 *     time and launches everything asynchronously on `stream` in stream order;
 *     it never synchronises the host except in gdn_device_status().  Calls on
 *     different streams must use different workspaces.  The library keeps no
 *     per-call state outside the caller's buffers, except two process-wide
 *     items: the optional launch counters and timing events of
 *     gdn_profile_enable() / gdn_profile_read(), and the fixed device array of
 *     gdn_fwd_noalloc(), which every GPU that loads the library reserves
 *     (GDN_FWD_NOALLOC_SCRATCH_BYTES) whether or not that entry point is
 *     called.
 *   - Errors are returned, never thrown.  Host-side checks (null pointers,
 *     sizes, cu_seqlens, alignment, buffer sizes) return before any launch.
 *     Conditions only the device can see (a saved buffer whose header does
 *     not match the call, a bounded wait that ran out) are written to an
 *     error word in the workspace; later kernels of the same call then skip
 *     their work, and gdn_device_status() reports the word.
 *   - Results are bitwise reproducible run to run for a fixed problem and plan
 *     (every reduction has a fixed order).
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t */

typedef struct {
    int64_t T;        /* total packed tokens (= cu_seqlens[N]) */
    int32_t N;        /* number of documents (>= 1; empty documents allowed) */
    int32_t H;        /* query/key heads */
    int32_t HV;       /* value heads, a multiple of H */
    int32_t dk;       /* must be 128 */
    int32_t dv;       /* must be 128 */
    float scale;      /* output scale (typically dk^-0.5) */
    int32_t l2norm;   /* non-zero: L2-normalise q and k inside the kernels */
    int32_t segments; /* 0: the planner chooses the segment split;
                         > 0: split the longest document into `segments`
                         segments (see gdn_plan_segment_chunks()) */
    int32_t saved_form; /* what the forward keeps for the backward:
                           GDN_SAVED_FULL (0): the state tape plus the per-chunk
                             UT blocks and V_new (the backward recomputes nothing);
                           GDN_SAVED_REPLAY (1): the state tape only; the backward
                             runs the UT / WY preparation again and recomputes
                             V_new = U - W S from the saved states (the pages'
                             replay form, "#8542" page, save-set table).
                           Both give the same bits; see gdn_saved_bytes(). */
} gdn_problem;

#define GDN_SAVED_FULL 0
#define GDN_SAVED_REPLAY 1

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,        /* null pointer, bad size, bad cu_seqlens, misalignment */
    GDN_ERR_UNSUPPORTED = 2,        /* dk or dv != 128, HV % H != 0 */
    GDN_ERR_WORKSPACE_TOO_SMALL = 3,/* ws_bytes below the gdn_saved_bytes() figure */
    GDN_ERR_SAVED_MISMATCH = 4,     /* device-side: `saved` was not written by a forward of this problem */
    GDN_ERR_CUDA = 5,               /* a CUDA runtime call or launch failed */
    GDN_ERR_TIMEOUT = 6,            /* device-side: a bounded wait ran out */
    GDN_ERR_DEVICE = 7,             /* device-side: any other kernel-detected fault */
    GDN_ERR_GATE_RANGE = 8          /* device-side (KDA entry points): a key channel's decay within one
                                       16-token block is steeper than 2^-96 (see gdn_kda_fwd) */
} gdn_status;

/*
 * Byte sizes of the caller-owned buffers for this problem.
 *   saved_bytes      the set gdn_fwd() writes for gdn_bwd(): a 4 KiB header,
 *                    the BF16 state entering every 64-token chunk of every
 *                    value head (32 KiB per chunk and value head; the pages'
 *                    "h tape" of states every 64 tokens), and, where a
 *                    document is split into P > 1 segments, the FP32 segment
 *                    transfer plane M_seg ((P-1) x HV x 64 KiB per document)
 *                    that the backward's merges read ("#8542" page: the full
 *                    saved set keeps M_seg at P > 1).  In the full form
 *                    (prob->saved_form == GDN_SAVED_FULL) it also keeps the
 *                    per-chunk UT blocks (T = (I + A)^-1 with its scaled forms
 *                    and the gated Aqk rows, 33 KiB per chunk and value head)
 *                    and the BF16 V_new^T = (U - W S)^T of every chunk (16 KiB
 *                    per chunk and value head; the pages' v_new rows); the
 *                    replay form (GDN_SAVED_REPLAY) keeps neither and the
 *                    backward recomputes them.
 *   workspace_bytes  scratch for one gdn_fwd / gdn_bwd / gdn_ckpt_fwd_bwd call
 *                    (in the replay form it also holds the recomputed blocks).
 * Returns GDN_ERR_INVALID_ARG / GDN_ERR_UNSUPPORTED on a bad problem.
 */
gdn_status gdn_saved_bytes(const gdn_problem *prob, const int32_t *cu_seqlens_host,
                           size_t *saved_bytes, size_t *workspace_bytes);

/*
 * Forward.  Writes o.  If `saved` is non-null it also writes the saved set
 * (header + state tape [+ M_seg]) that gdn_bwd() consumes; with saved == NULL
 * no state is stored (the forward of a checkpointed step).
 */
gdn_status gdn_fwd(const gdn_problem *prob, const void *q, const void *k, const void *v,
                   const float *g, const float *beta, const int32_t *cu_seqlens_dev,
                   const int32_t *cu_seqlens_host, void *o, void *saved, void *workspace,
                   size_t ws_bytes, struct CUstream_st *stream);

/*
 * Backward.  Given dO and the saved set of a gdn_fwd() of the same problem and
 * inputs, writes dq, dk, dv (BF16) and dg, dbeta (FP32).  Every output element
 * is written (no accumulation into the caller's buffers).  A saved set whose
 * header does not match the problem sets GDN_ERR_SAVED_MISMATCH on the device
 * (see gdn_device_status) and leaves the gradients unwritten.
 */
gdn_status gdn_bwd(const gdn_problem *prob, const void *q, const void *k, const void *v,
                   const float *g, const float *beta, const int32_t *cu_seqlens_dev,
                   const int32_t *cu_seqlens_host, const void *dO, const void *saved,
                   void *dq, void *dk, void *dv, float *dg, float *dbeta, void *workspace,
                   size_t ws_bytes, struct CUstream_st *stream);

/*
 * Activation-checkpointed step: a forward that keeps no states and writes o,
 * then a forward that writes the saved set into `saved_scratch` (saved_bytes
 * large), then the backward.  This is the pages' "ckpt" operation, two
 * forwards plus one backward.  With o == NULL the first forward, which would
 * produce nothing, is skipped.
 */
gdn_status gdn_ckpt_fwd_bwd(const gdn_problem *prob, const void *q, const void *k,
                            const void *v, const float *g, const float *beta,
                            const int32_t *cu_seqlens_dev, const int32_t *cu_seqlens_host,
                            const void *dO, void *o, void *dq, void *dk, void *dv, float *dg,
                            float *dbeta, void *saved_scratch, void *workspace,
                            size_t ws_bytes, struct CUstream_st *stream);

/*
 * Per-document boundary states.  These are gdn_fwd / gdn_bwd for documents
 * that do not start from a zero state or whose last state is wanted: the
 * state passed between the pieces of a document split across calls (or
 * across devices): the pages' incoming boundary states S_in, kept in FP32
 * ("#8542" page, the save-set table's S_in row).
 * Every state is FP32 S in [N][HV][dk][dv] layout (document, value head,
 * k index, v index), 16-byte aligned, caller-owned.
 *
 * gdn_fwd_states: as gdn_fwd, with
 *   s_in   the state each document starts from (NULL: zero);
 *   s_out  written with the state after each document's last token (NULL:
 *          not written).  An empty document passes s_in through.
 *   o, saved and s_out may each be NULL, but not all three.
 * A saved set written here already holds the effect of s_in (the state
 * entering every chunk), so the backward needs no s_in.
 *
 * gdn_bwd_states: as gdn_bwd, with
 *   ds_out the gradient of the loss with respect to s_out (NULL: zero);
 *   ds_in  written with the gradient with respect to s_in (NULL: not
 *          written).  An empty document passes ds_out through.
 * The gradients dq, dk, dv, dg, dbeta then include the terms of ds_out.
 */
gdn_status gdn_fwd_states(const gdn_problem *prob, const void *q, const void *k, const void *v,
                          const float *g, const float *beta, const int32_t *cu_seqlens_dev,
                          const int32_t *cu_seqlens_host, const float *s_in, void *o, float *s_out,
                          void *saved, void *workspace, size_t ws_bytes, struct CUstream_st *stream);
gdn_status gdn_bwd_states(const gdn_problem *prob, const void *q, const void *k, const void *v,
                          const float *g, const float *beta, const int32_t *cu_seqlens_dev,
                          const int32_t *cu_seqlens_host, const void *dO, const float *ds_out,
                          const void *saved, void *dq, void *dk, void *dv, float *dg, float *dbeta,
                          float *ds_in, void *workspace, size_t ws_bytes, struct CUstream_st *stream);

/*
 * The short causal convolution + SiLU in front of the GDN layer, over the
 * packed q/k/v channels (C = (2 H + HV) x 128 = 10,240 at (16, 48)), restarting
 * at every document ("#8542" page: the B23 shape description and the family's
 * conv1d + SiLU training backend; its save-set table keeps at most three
 * history rows, a four-tap kernel).  Per channel c, with W taps:
 *     z[t, c] = b[c] + sum_{i<W} w[c, i] x[t - (W-1) + i, c]   (x = 0 before t's document)
 *     y[t, c] = z / (1 + exp(-z))
 * Layouts: x, y, dy, dx [T][C] BF16 (token-major, contiguous); w, dw [C][W]
 * FP32; b, db [C] FP32 (b may be NULL: no bias; db may be NULL: not
 * written).  C must be a multiple of 8, 1 <= W <= 4 (else
 * GDN_ERR_INVALID_ARG / GDN_ERR_UNSUPPORTED).  Pointers 16-byte aligned.
 * Accumulation is FP32 in a fixed order; dw and db are sums of per-range
 * partials added in range order (bitwise reproducible).  The caller owns
 * every buffer; the backward needs `workspace` of gdn_conv1d_workspace_bytes,
 * which opens with the device status word that gdn_device_status reads (a
 * bounded wait on a row copy that never completes sets GDN_ERR_TIMEOUT there).
 */
typedef struct {
    int64_t T;   /* total packed tokens (= cu_seqlens[N]) */
    int32_t N;   /* documents */
    int32_t C;   /* channels */
    int32_t W;   /* taps */
} gdn_conv_problem;
gdn_status gdn_conv1d_workspace_bytes(const gdn_conv_problem *prob, const int32_t *cu_seqlens_host,
                                      size_t *workspace_bytes);
gdn_status gdn_conv1d_fwd(const gdn_conv_problem *prob, const void *x, const float *w, const float *b,
                          const int32_t *cu_seqlens_dev, const int32_t *cu_seqlens_host, void *y,
                          struct CUstream_st *stream);
gdn_status gdn_conv1d_bwd(const gdn_conv_problem *prob, const void *x, const float *w, const float *b,
                          const int32_t *cu_seqlens_dev, const int32_t *cu_seqlens_host, const void *dy,
                          void *dx, float *dw, float *db, void *workspace, size_t ws_bytes,
                          struct CUstream_st *stream);

/*
 * The per-channel-decay form (KDA): the same recurrence with one decay per key channel,
 *
 *     S_t = Diag(a_t) S_{t-1} + beta_t k^_t (v_t - (Diag(a_t) S_{t-1})^T k^_t)^T,   a_t = exp(g_t) in R^dk
 *     o_t = scale * S_t^T q^_t
 *
 * ("perf(cake_kda) ... #7097" page: the packed KDA training family beside the GDN one; the pages
 * print no formula, and this is the GDN rule above with its scalar decay replaced by a per-channel
 * one).  Conventions as for the GDN entry points, except:
 *   - g and dg are [T][HV][128] FP32: the log decay of each key channel (g <= 0 for a decay);
 *   - the saved set holds the header, the BF16 state entering every chunk (32 KiB per chunk and
 *     value head), M_seg where a document is split, and the BF16 V_new^T of every chunk (16 KiB
 *     per chunk and value head).  With prob->saved_form == GDN_SAVED_FULL (the default) it also
 *     keeps the forward's per-chunk blocks of decay products and UT tiles (82,944 B per chunk and
 *     value head: Kd, -W^T, T'', T, Aqk, M^T, Q~, the scalars), which the backward reads; with
 *     GDN_SAVED_REPLAY the backward recomputes them (the pages' replay of w, u and the A
 *     matrices).  Both give the same gradients, bit for bit;
 *   - a chunk in which some key channel decays by more than 2^-96 within one 16-token block (a
 *     log decay below -66.5 over 16 tokens) is refused on the device: the error word is set to
 *     GDN_ERR_GATE_RANGE and the outputs are left unwritten.  Below that bound every chunk is
 *     computed (the kernels factor the decays per 16-token block, and the factors must stay in
 *     BF16's exponent range).
 * gdn_kda_saved_bytes: the sizes of `saved` and of the workspace (forward and backward).
 * gdn_kda_fwd: writes o (required) and, if `saved` is non-null, the saved set.
 * gdn_kda_bwd: given dO and the saved set of a gdn_kda_fwd of the same problem and inputs, writes
 *   dq, dk, dv (BF16), dg [T][HV][128] and dbeta [T][HV] (FP32).
 */
gdn_status gdn_kda_saved_bytes(const gdn_problem *prob, const int32_t *cu_seqlens_host,
                               size_t *saved_bytes, size_t *workspace_bytes);
gdn_status gdn_kda_fwd(const gdn_problem *prob, const void *q, const void *k, const void *v,
                       const float *g, const float *beta, const int32_t *cu_seqlens_dev,
                       const int32_t *cu_seqlens_host, void *o, void *saved, void *workspace,
                       size_t ws_bytes, struct CUstream_st *stream);
gdn_status gdn_kda_bwd(const gdn_problem *prob, const void *q, const void *k, const void *v,
                       const float *g, const float *beta, const int32_t *cu_seqlens_dev,
                       const int32_t *cu_seqlens_host, const void *dO, const void *saved, void *dq,
                       void *dk, void *dv, float *dg, float *dbeta, void *workspace, size_t ws_bytes,
                       struct CUstream_st *stream);

/* Static description of a status code. */
const char *gdn_status_string(gdn_status s);

/*
 * Synchronises `stream`, then returns the device-side error word of the last
 * call that used `workspace` (GDN_OK if none), or GDN_ERR_CUDA if the stream
 * reports a CUDA error.
 */
gdn_status gdn_device_status(void *workspace, struct CUstream_st *stream);

/*
 * Introspection for tests and tools: byte offsets, into the workspace, of the
 * chunk tables every call builds from cu_seqlens (int32 arrays:
 * offsets[0] -> chunk_offsets[N+1], the index of each document's first chunk;
 * offsets[1] -> chunk_doc[NC]; offsets[2] -> chunk_tok0[NC], first token of
 * each chunk; offsets[3] -> chunk_len[NC], 1..64 tokens), and NC.
 */
gdn_status gdn_chunk_table_offsets(const gdn_problem *prob, const int32_t *cu_seqlens_host,
                                   size_t offsets[4], int32_t *num_chunks);

/*
 * Introspection for tests and tools: byte offsets, into the workspace, of the
 * intermediate tapes a gdn_bwd() call leaves there (each [NC][HV] blocks):
 *   offsets[0] UT blocks, 33,792 B each (T' at 0, T'' at 8 KiB, Aqk at 16 KiB,
 *              T at 24 KiB: BF16 64 x 64 tiles in the kernels' swizzled tile
 *              layout; then 1 KiB of per-token scalars)      (replay form; else 0)
 *   offsets[1] V_new^T tiles, 16 KiB each (BF16 128 x 64)   (replay form; else 0)
 *   offsets[2] dS' tiles, 32 KiB each (BF16 128 x 128 dS'^T: the gradient of
 *              the state leaving each chunk)
 *   offsets[3] dV_new^T tiles, 16 KiB each (BF16 128 x 64)
 */
gdn_status gdn_backward_tape_offsets(const gdn_problem *prob, const int32_t *cu_seqlens_host,
                                     size_t offsets[4]);

/*
 * Forward for callers that cannot allocate device memory.  The pages have no
 * counterpart to this entry point; it exists for hosts that give a library
 * only its inputs and outputs (plugin-style runtimes without a workspace
 * query, or latency-bound paths that may not call cudaMalloc because it
 * synchronises the device).
 *
 * It computes exactly what gdn_fwd(prob, ..., o, saved = NULL, ...) computes,
 * with the workspace taken from a fixed array of GDN_FWD_NOALLOC_SCRATCH_BYTES
 * (64 MiB) that the library keeps in device memory on every GPU where it is
 * loaded, until the process exits.  Inputs and `o` are the caller's, as for
 * gdn_fwd; no saved set is written (use gdn_fwd for training).
 *   - A problem whose forward workspace exceeds 64 MiB is refused with
 *     GDN_ERR_WORKSPACE_TOO_SMALL before any launch (at HV = 48 that is about
 *     40 chunks of 64 tokens; see gdn_saved_bytes for the general size).
 *   - The first call on a device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress); make that first call
 *     before any stream capture.
 *   - Every call shares the one array and the array keeps the last call's
 *     contents; the forward rewrites everything it reads.  Calls that overlap
 *     on the GPU (different streams, or different host threads) race on the
 *     array and must be serialised by the caller.
 *   - Device-side conditions (a device copy of cu_seqlens that disagrees with
 *     the host copy, a bounded wait that ran out) are recorded in the array,
 *     which the caller cannot address, so this entry point reports only
 *     host-side statuses; after such a condition the kernels skip their work
 *     and `o` is left undefined (whatever it held before the call).  A caller
 *     that needs the device-side status uses gdn_fwd with its own workspace
 *     and gdn_device_status.
 * No cudaMalloc, cudaFree or allocating library routine is called.
 */
#define GDN_FWD_NOALLOC_SCRATCH_BYTES (64u << 20)
gdn_status gdn_fwd_noalloc(const gdn_problem *prob, const void *q, const void *k, const void *v,
                           const float *g, const float *beta, const int32_t *cu_seqlens_dev,
                           const int32_t *cu_seqlens_host, void *o, struct CUstream_st *stream);

/*
 * Optional per-kernel timing, for benchmarks and tools.  The library counts
 * every kernel it launches; while profiling is enabled it also records a CUDA
 * event pair on the launching stream around each launch.  gdn_profile_read()
 * synchronises on the recorded events, fills up to max_entries records (one
 * per kernel that launched since the last read: its name, the number of
 * launches, how many of them were timed, and their summed device time in ms),
 * resets the counters and returns the number of kernels with launches.  The
 * bookkeeping is process-wide and thread-safe.
 */
typedef struct {
    const char *name;
    long long launches;
    long long timed_launches;
    double total_ms;
} gdn_kernel_stat;
void gdn_profile_enable(int on);
int gdn_profile_read(gdn_kernel_stat *out, int max_entries);

/*
 * The segment length (in 64-token chunks) the planner uses for this problem:
 * documents longer than this are split into ceil(chunks / seg) segments whose
 * transfer operators are composed by a merge kernel (the intra-GPU segment
 * split).  With prob->segments > 0 the answer is ceil(max_doc_chunks /
 * prob->segments), i.e. the longest document gets `segments` segments.
 * Returns 0 on an invalid problem.
 */
int32_t gdn_plan_segment_chunks(const gdn_problem *prob, const int32_t *cu_seqlens_host);

/*
 * Tensor-pipe probe, for the roofline's own BF16 peak: the benchmark reports
 * tensor-core fractions against the vendor's dense figure and against the rate
 * this probe measures with the library's own tcgen05 code.  Launches one CTA per SM of
 * the current device on `stream`; each issues iters x 4 BF16 tcgen05 products
 * of M = 128, N = 256, K = 16 (FP32 accumulation in TMEM) on operand tiles
 * that stay in shared memory, so no memory traffic competes with the tensor
 * cores.  *flops receives the products' FLOP count (2 M N K each); the caller
 * times the launch with events on `stream` and reads *dev_err (a device int,
 * zero on entry) afterwards: nonzero means a bounded wait ran out.
 * iters: 1 .. 2^20.  Returns GDN_ERR_INVALID_ARG outside that range or for a
 * null pointer, GDN_ERR_CUDA if the launch fails; nothing is allocated.
 */
gdn_status gdn_tensor_probe(int32_t iters, int32_t *dev_err, double *flops, struct CUstream_st *stream);

#ifdef __cplusplus
}
#endif
#endif /* GDN_H_ */
