/*
 * ssd.h -- C ABI of libssd: the Mamba-2 selective state-space (SSD) layer's
 * chunked scan, forward and backward, on one NVIDIA GB300 (sm_103a).
 *
 * The operation (page "llm-mamba-200" (gigipick.blogspot.com), sections 1-2:
 * a selective linear recurrence whose steps combine associatively; the
 * equations are lost from the page text and are taken in their Mamba-2 form
 * with one scalar decay per head):
 *
 *   dt_eff[t,h] = softplus(dt[t,h] + dt_bias[h])
 *   h_t         = exp(dt_eff[t,h] * A[h]) * h_{t-1} + dt_eff[t,h] * x_t (outer) B_t
 *   y_t         = h_t . C_t + D[h] * x_t
 *
 * per batch row and head, with h_{-1} = initial_states (or 0).  When seq_idx
 * is given, a token whose id differs from the previous token's starts a new
 * sequence with a zero state; initial_states feeds only the first one.
 * final_states is the state after the last token.
 *
 * It is evaluated by chunks of chunk_size tokens (page "llm-mamba-200",
 * section 3: carry-out state of one chunk is the carry-in of the next), with
 * the cross-chunk state passing, forward and backward, done as an associative
 * scan (page "B200 Helion Mamba-2" (aitrends.kr/articles/109906), section
 * "Helion based B200 kernel redesign").
 *
 * Shapes (b = batch, L = seqlen, H = nheads, P = headdim, N = dstate,
 * G = ngroups; head h reads group floor(h*G/H), i.e. G contiguous blocks of
 * H/G heads).  Every tensor is dense row-major, device memory:
 *
 *   x, y, dy, dx            (b, L, H, P)   dtype
 *   dt, ddt                 (b, L, H)      dtype
 *   B, C, dB, dC            (b, L, G, N)   dtype
 *   dt_bias, A, D and grads (H)            fp32
 *   initial_states, final_states, dfinal_states, dinitial_states
 *                           (b, H, P, N)   fp32
 *   seq_idx                 (b, L)         int32, nondecreasing along each row
 *
 * where dtype is SSD_F32 (fp32) or SSD_BF16 (bf16; fp32 accumulation inside).
 * Every pointer must be 16-byte aligned.
 *
 * Ownership: the caller allocates every buffer, the workspace included, and
 * keeps them alive until the stream work completes.  The library never
 * allocates, never synchronises (except the two status readers and
 * ssd_profile_stop) and keeps no mutable global state other than a
 * per-device cache of device attributes, the optional timing records and
 * the one exception below: the fixed device array behind ssd_fwd_noalloc
 * (SSD_NOALLOC_SCRATCH_BYTES on every GPU that loads the library) with a
 * per-device cache of its address, shared by all ssd_fwd_noalloc calls --
 * calls of it that overlap on the GPU race on that array (see there).
 * Calls enqueue work on the given stream and return before it completes.
 *
 * Errors: every entry point validates its arguments before enqueuing
 * anything and returns an ssd_status; nothing is thrown across the ABI.
 * Errors detected on the device (a bounded wait that expired) are recorded
 * in a status word at the start of the workspace; read it with
 * ssd_read_device_status (ssd_fwd_noalloc_read_device_status for
 * ssd_fwd_noalloc, whose workspace is the library's own array).
 */
#ifndef SSD_H_
#define SSD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ssd_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  SSD_OK = 0,
  SSD_ERR_INVALID_ARGUMENT = 1, /* null required pointer, bad dims, misaligned pointer */
  SSD_ERR_UNSUPPORTED = 2,      /* shape/dtype outside the compiled set, or not an sm_103 device */
  SSD_ERR_WORKSPACE_TOO_SMALL = 3,
  SSD_ERR_CUDA = 4,             /* a CUDA runtime error while enqueuing */
  SSD_ERR_TIMEOUT = 5,          /* a device-side bounded wait expired (read via the status word) */
  SSD_ERR_NO_KEPT_STATES = 6    /* ssd_bwd with SSD_KEEP_FWD_STATES found no forward intermediates of
                                   this problem in the workspace (read via the status word) */
} ssd_status;

typedef enum { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype;

enum {
  SSD_HAS_INIT = 1,      /* initial_states is given */
  SSD_HAS_SEQ_IDX = 2,   /* seq_idx is given */
  SSD_HAS_DFINAL = 4,    /* ssd_bwd: dfinal_states (upstream gradient of final_states) is given */
  SSD_WANT_DINIT = 8,    /* ssd_bwd: write dinitial_states */
  /* Keep the forward's intermediates for the backward (the usual training
   * step: forward, then backward on the same inputs).  ssd_fwd with this
   * flag leaves in its workspace what the backward would otherwise
   * recompute -- dt_eff, the chunk-local cumsums of dt_eff * A, the per-chunk
   * decays and the carry-in state of every chunk (in the problem's dtype) --
   * and stamps the workspace with the problem's signature; ssd_fwd without it
   * clears the stamp.  A forward on the separate kernels also keeps the fp32
   * carry-in states (its scan writes them over the fp32 chunk states) and
   * says so in the stamp.  ssd_bwd with this flag, given that same
   * workspace, takes them from there instead of recomputing them: where it
   * runs its single-pass state chains, from either forward; where it runs
   * the separate kernels, from a forward on the separate kernels (if the
   * same problem's forward takes the single-pass kernel, that backward
   * recomputes as usual and ignores the flag).  The inputs must be the ones
   * that forward saw: the stamp covers the problem's shape, not its values.
   * A workspace without the stamp this backward needs makes it report
   * SSD_ERR_NO_KEPT_STATES in the device status word (its results are then
   * garbage).  Forward results do not depend on the flag; backward results
   * agree with the recomputing backward to rounding (bit for bit on the
   * separate kernels, which keep exactly what they would recompute). */
  SSD_KEEP_FWD_STATES = 16,
  /* Testing only: the first scan tile of the first state chain never
   * publishes its prefix, so the tiles after it exhaust their bounded wait
   * (0.1 s with this flag, 2 s otherwise) and the call ends with
   * SSD_ERR_TIMEOUT in the device status word instead of hanging.  Results
   * of such a call are garbage. */
  SSD_TEST_DROP_SCAN_PUBLISH = 1 << 16,
  /* Path selection (comparisons and tests; results agree to rounding).  By
   * default the library takes its single-pass kernels -- in ssd_fwd one
   * persistent CTA per (batch row, head) that keeps the carry on chip, in
   * ssd_bwd one such CTA per chain for the forward and the reverse state
   * chains (bf16, headdim 64, d_state 64 or 128) -- when there are at least
   * about three chains per four SMs, and otherwise its separate kernels
   * (chunk cumsum, chunk states, state-passing scan, chunk output).
   * SSD_PATH_MULTI_KERNEL forces the separate kernels; SSD_PATH_SINGLE_PASS
   * forces the single-pass kernels wherever their shape set allows. */
  SSD_PATH_MULTI_KERNEL = 1 << 17,
  SSD_PATH_SINGLE_PASS = 1 << 18,
  /* Testing only: the persistent token-gradient kernel runs on at most two
   * CTAs, so that a small problem walks several work units per CTA.  Results
   * are the same bits as without the flag. */
  SSD_TEST_FEW_CTAS = 1 << 19,
  /* Comparison: the separate kernels' forward state-passing scan takes each
   * segment's local scan across the lanes of a warp (Hillis-Steele steps of
   * warp shuffles, lane k holding chunk k) instead of sequentially inside
   * each thread; the join of the segments is the same.  Results agree to
   * rounding. */
  SSD_SCAN_WARP_SHUFFLE = 1 << 20
};

typedef struct {
  int64_t batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size;
  int32_t dtype; /* ssd_dtype */
  int32_t flags; /* SSD_HAS_* / SSD_WANT_* */
} ssd_problem;

/* Limits of the compiled kernels (checked by every entry point):
 *   1 <= chunk_size <= 256, chunk_size % 16 == 0
 *   headdim in {16, 32, 64, 128}; dstate in {16, 32, 64, 128};
 *   headdim * dstate <= 8192
 *   nheads % ngroups == 0; batch, seqlen >= 1                              */

/* Bytes of device workspace ssd_fwd / ssd_bwd need for this problem
 * (a pure function of the problem; 0 if the problem is invalid). */
size_t ssd_fwd_workspace_bytes(const ssd_problem* prob);
size_t ssd_bwd_workspace_bytes(const ssd_problem* prob);

/* Forward.  Writes y and (if non-NULL) final_states.  initial_states must be
 * non-NULL iff SSD_HAS_INIT, seq_idx iff SSD_HAS_SEQ_IDX.  Enqueues on
 * `stream` and returns without waiting. */
int ssd_fwd(const ssd_problem* prob, const void* x, const void* dt, const float* dt_bias,
            const float* A, const void* B, const void* C, const float* D,
            const float* initial_states, const int32_t* seq_idx, void* y, float* final_states,
            void* workspace, size_t workspace_bytes, ssd_stream_t stream);

/* Backward (reverse mode of ssd_fwd for the upstream gradients dy and,
 * if SSD_HAS_DFINAL, dfinal_states).  The forward intermediates are
 * recomputed inside (the call is stateless).  Gradients are overwritten, not
 * accumulated: dx, ddt, dB, dC in dtype; ddt_bias, dA, dD (H) fp32;
 * dinitial_states (fp32) iff SSD_WANT_DINIT.  All reductions (dA, dD,
 * ddt_bias over tokens, dB and dC over the heads of a group) are taken in a
 * fixed order: results are bitwise reproducible run to run. */
int ssd_bwd(const ssd_problem* prob, const void* x, const void* dt, const float* dt_bias,
            const float* A, const void* B, const void* C, const float* D,
            const float* initial_states, const int32_t* seq_idx, const void* dy,
            const float* dfinal_states, void* dx, void* ddt, float* ddt_bias, float* dA,
            void* dB, void* dC, float* dD, float* dinitial_states, void* workspace,
            size_t workspace_bytes, ssd_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* ssd_status_string(int status);

/* Synchronises `stream`, then reads the device status word of the last call
 * that used `workspace` (SSD_OK, SSD_ERR_TIMEOUT or SSD_ERR_NO_KEPT_STATES;
 * a timeout is reported first).  Returns SSD_ERR_CUDA if the
 * synchronisation or the copy fails. */
int ssd_read_device_status(const void* workspace, ssd_stream_t stream);

/* Allocation-free forward.  The pages have no counterpart: this is a
 * library convenience for callers that cannot allocate device memory where
 * they call the layer -- a plain C host with no handle on the framework's
 * caching allocator, or a latency-critical loop where an allocation (and
 * the synchronisation cudaMalloc implies) is not allowed.  Same arguments
 * and results as ssd_fwd, minus the workspace: the workspace is a
 * library-owned device array of SSD_NOALLOC_SCRATCH_BYTES (32 MiB) that
 * every GPU loading libssd holds until the process exits.  Problems whose
 * ssd_fwd_workspace_bytes exceeds it are rejected with
 * SSD_ERR_WORKSPACE_TOO_SMALL.  The call allocates nothing.  Its first call
 * on a device looks up the array's device address (cudaGetSymbolAddress,
 * with that device current) and caches it; make that first call before any
 * stream capture.  All calls share the one array and it keeps the last
 * call's contents (each call re-zeroes what must start at zero): calls that
 * can overlap on the GPU -- on different streams or from different host
 * threads -- race on it.  Its device status word is read with
 * ssd_fwd_noalloc_read_device_status. */
#define SSD_NOALLOC_SCRATCH_BYTES (32u << 20)
int ssd_fwd_noalloc(const ssd_problem* prob, const void* x, const void* dt, const float* dt_bias,
                    const float* A, const void* B, const void* C, const float* D,
                    const float* initial_states, const int32_t* seq_idx, void* y,
                    float* final_states, ssd_stream_t stream);

/* Status of the last ssd_fwd_noalloc call on the current device: the
 * counterpart of ssd_read_device_status for the library-owned array, whose
 * address callers never see.  Synchronises `stream`, then returns SSD_OK or
 * SSD_ERR_TIMEOUT (a device-side bounded wait of that call expired; its
 * results are then garbage), or SSD_ERR_CUDA if the synchronisation or the
 * copy fails.  No counterpart on the pages either. */
int ssd_fwd_noalloc_read_device_status(ssd_stream_t stream);

/* ---------------------------------------------------------------------------
 * Context parallelism: the sequence split into contiguous shards (one per
 * rank, or run one after another on one GPU), each shard run through
 * ssd_fwd / ssd_bwd as a problem of its own, the shards joined by two
 * exclusive folds.  Page "B200 Helion Mamba-2" (aitrends.kr/articles/109906)
 * names context parallelism as the module's integration goal without a
 * method; it follows from the recurrence: a shard maps the state h entering
 * it to dec * h + final(0) (dec = product of its per-token decays
 * exp(dt_eff * A), 0 when a sequence starts after its first token; final(0)
 * = its final state from a zero start), and its dinitial_states is affine
 * in the gradient g at its final state, dinit(g) = dec * g + dinit(0).
 *
 * Forward: every shard runs from a zero state (its final_states = local),
 * ssd_shard_decay gives dec and the segment ids of its first and last
 * tokens; after the exchange of (dec, local, ids) of all shards,
 * ssd_shard_fold (reverse = 0, boundary = initial_states or NULL) gives the
 * state entering every shard (out) and the layer's final state (total);
 * every shard runs again from its entering state.  Backward: every shard's
 * dinitial_states with no upstream final gradient (local), exchanged,
 * folded with reverse = 1 (boundary = dfinal_states or NULL) gives every
 * shard its upstream dfinal_states (out); each shard then runs its backward;
 * dA, dD and ddt_bias are sums over the shards.  A shard whose first token
 * starts a new sequence enters from zero and sends no gradient back. */

/* dec (b, H) fp32 of one shard (prob: the shard as a problem; only batch,
 * seqlen, nheads, dtype and SSD_HAS_SEQ_IDX are read) and, if first_ids /
 * last_ids (b) int32 are non-NULL (both or neither), the segment ids of the
 * shard's first and last tokens (0 without seq_idx).  dt (b, Ls, H) dtype;
 * dt_bias, A (H) fp32; seq_idx (b, Ls) iff SSD_HAS_SEQ_IDX. */
int ssd_shard_decay(const ssd_problem* prob, const void* dt, const float* dt_bias, const float* A,
                    const int32_t* seq_idx, float* decay, int32_t* first_ids, int32_t* last_ids,
                    ssd_stream_t stream);

/* The exclusive fold over nshards shards, in order (reverse = 0) or from
 * the right (reverse = 1).  decay (R, b, H) fp32; local, out (R, b, H, P, N)
 * fp32; first_ids, last_ids (R, b) int32 or both NULL (no sequence starts on
 * shard boundaries); boundary (b, H, P, N) fp32 or NULL (zero); total
 * (b, H, P, N) fp32 or NULL.  Forward: h = boundary; for r: h = 0 if shard
 * r > 0 starts a new sequence; out[r] = h; h = decay[r] h + local[r];
 * total = h.  Reverse: g = boundary; for r = R-1 .. 0: out[r] = g;
 * g = decay[r] g + local[r]; g = 0 if shard r > 0 starts a new sequence;
 * total = g.  Device pointers, 16-byte aligned; enqueue only. */
int ssd_shard_fold(int64_t nshards, int64_t batch, int64_t nheads, int64_t headdim, int64_t dstate,
                   const float* decay, const float* local, const int32_t* first_ids,
                   const int32_t* last_ids, const float* boundary, float* out, float* total,
                   int reverse, ssd_stream_t stream);

/* ---------------------------------------------------------------------------
 * Gated RMSNorm of the Mamba-2 block: the normalisation the block applies to
 * the scan's output y, gated by the block's z branch.  Page "B200 Helion
 * Mamba-2" (aitrends.kr/articles/109906) measures its backward
 * (`_layer_norm_bwd`, a memory-bound row reduction) at batch 2, seqlen 8192,
 * bf16, without writing out the operation; it is read as
 *
 *   g[r,j]    = y[r,j] * silu(z[r,j])        (g = y without SSD_NORM_HAS_Z)
 *   rstd[r,k] = 1 / sqrt(mean_{j in group k} g[r,j]^2 + eps)
 *   out[r,j]  = g[r,j] * rstd[r,k] * weight[j]
 *
 * over rows r (tokens) and groups k of group_size contiguous columns (in the
 * Mamba-2 block: dim = nheads * headdim, group_size = dim / ngroups).  The
 * backward gives dy, dz and dweight = sum over rows of dout * g * rstd; that
 * sum is folded across thread blocks in a fixed order (page "Cake RMSNorm",
 * blog.secrett2633.cloud, flashinfer PR 6997, section "Fixed-order tree fold
 * reduction"), so dweight is bitwise reproducible run to run on one device.
 *
 * Layouts (dense row-major, device memory, 16-byte aligned):
 *   y, z, out, dout, dy, dz   (rows, dim)   dtype
 *   weight, dweight           (dim)         fp32
 *   rstd                      (rows, dim / group_size) fp32
 * Limits: dim % group_size == 0; group_size a multiple of 8 (bf16) or 4
 * (fp32) and at most 4096 (bf16) or 2048 (fp32); eps >= 0.
 * Ownership, errors and stream semantics as above.  The calls have no
 * device-side waits and use no status word. */
enum { SSD_NORM_HAS_Z = 1 /* z (the gate) is given */ };

typedef struct {
  int64_t rows, dim, group_size;
  float eps;
  int32_t dtype; /* ssd_dtype of y, z, out, dout, dy, dz */
  int32_t flags; /* SSD_NORM_HAS_Z */
} ssd_norm_problem;

/* Forward: writes out and, if non-NULL, rstd.  z must be non-NULL iff
 * SSD_NORM_HAS_Z. */
int ssd_gated_rmsnorm_fwd(const ssd_norm_problem* prob, const void* y, const void* z,
                          const float* weight, void* out, float* rstd, ssd_stream_t stream);

/* Bytes of device workspace ssd_gated_rmsnorm_bwd needs (the per-block
 * dweight partials; a pure function of the problem, 0 if it is invalid). */
size_t ssd_gated_rmsnorm_bwd_workspace_bytes(const ssd_norm_problem* prob);

/* Backward for the upstream gradient dout (rstd is recomputed from y and z).
 * Overwrites dy, dz (non-NULL iff SSD_NORM_HAS_Z) and dweight. */
int ssd_gated_rmsnorm_bwd(const ssd_norm_problem* prob, const void* y, const void* z,
                          const float* weight, const void* dout, void* dy, void* dz,
                          float* dweight, void* workspace, size_t workspace_bytes,
                          ssd_stream_t stream);

/* Library build/version string, e.g. "libssd 0.1 sm_103a". */
const char* ssd_version(void);

/* Per-kernel timing, a measurement aid.  ssd_profile_start (re)starts
 * recording on the current device: from then on every kernel launched by
 * ssd_fwd/ssd_bwd is bracketed by two CUDA events recorded on the call's
 * stream.  ssd_profile_stop ends recording and waits for the recorded events
 * (it synchronises), folding them into per-kernel totals that
 * ssd_profile_count/ssd_profile_get report (name is a static string).  The
 * event pool holds 32768 launches; ssd_profile_stop returns
 * SSD_ERR_WORKSPACE_TOO_SMALL if launches beyond it went unrecorded.  Use
 * from one host thread. */
int ssd_profile_start(void);
int ssd_profile_stop(void);
int ssd_profile_count(void);
int ssd_profile_get(int index, const char** name, int* launches, double* total_ms);

#ifdef __cplusplus
}
#endif
#endif /* SSD_H_ */
