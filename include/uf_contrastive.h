/*
 * uf_contrastive.h -- C ABI of a GB300 (sm_103a) library for the batched Matryoshka
 * contrastive loss, forward and backward, on one GPU.
 *
 * What it computes.  Two bf16 embedding matrices A (Na x D) and B (Nb x D), row-major
 * with row stride D, are scored all-against-all at nested prefixes p_1 < ... < p_n of
 * the embedding (the Matryoshka ladder {64, 128, 256, 512, 1024}: UForm README,
 * "Matryoshka" paragraph; blog "Scaling-Up Contrastive Learning over NVLink
 * Multicast", section "One Set or Two").  For each prefix p every row is
 * L2-normalised on its first p dimensions, cos_ij = <a_i[:p], b_j[:p]> / (|a_i[:p]| |b_j[:p]|),
 * and one of three losses is applied:
 *   UF_LOSS_CLIP_SYMMETRIC  s = scale * cos; L_p = 1/2 (mean_i CE_row(i) + mean_j CE_col(j)),
 *                           positives on the diagonal (Na == Nb).  The blog, section
 *                           "One Set or Two": CLIP turns each row of cosines into a
 *                           softmax over the batch; the symmetric form adds the columns.
 *   UF_LOSS_SIGLIP          x = scale * cos + bias; L_p = -(1/N) sum_ij log sigmoid(z_ij x_ij),
 *                           z = +1 on the diagonal, -1 elsewhere (Na == Nb).  The blog's
 *                           SigLIP equation, same section.
 *   UF_LOSS_INFONCE_ROWS    L_p = mean_{i<Na} CE over all Nb keys of row i, the positive
 *                           of query i being key i (Nb >= Na).
 * The gradients returned are those of sum_p w_p L_p (w_p = 1 unless given).
 * Precision policy (UForm README, "Training is BF16"): operands bf16, products and
 * every accumulation fp32, gradients fp32.  The forward never stores the Na x Nb logits.
 * The backward does store Na x Nb data in the caller's workspace: for every prefix, the
 * bf16 per-cell weights rho_i sigma_j dL/dcos_ij (a chunk of A's rows by B's rows at a
 * time when the workspace is smaller than uf_contrastive_workspace_size), which tensor-core
 * GEMMs then contract with the embeddings.
 *
 * Conventions (UForm Swift binding page, sections "Errors" and "Design": one C verb per
 * operation named <lib>_<noun>_<verb>, an enum status with a name function; section
 * "Arenas": the caller owns every output and the scratch, and nothing is allocated on
 * the call path).  All entry points are thread-safe; a call only enqueues work on the
 * caller's stream and returns without synchronising, so it can be captured in a CUDA
 * graph.  Calls on different streams are independent as long as each has its own
 * workspace and outputs.  The kernels of a call are launched with programmatic dependent
 * launch (each waits for the grid before it on the stream before it touches memory): a
 * caller's kernel that follows a call on the same stream and is itself launched with the
 * programmatic stream serialization attribute must wait for its predecessor
 * (cudaGridDependencySynchronize) before it reads the outputs; an ordinary launch, a copy
 * or an event needs nothing.
 *
 * Buffers.  No buffer a call writes may overlap another such buffer or any input.  The written
 * buffers are the loss, the terms, the gradients, the scalar gradients, *device_status and the
 * workspace; the inputs are A, B, the device-held scalars and the label lists.  A call that
 * breaks this returns UF_INVALID_ARGUMENT and enqueues nothing.  The inputs may overlap one
 * another (A == B is a valid request).
 */
#ifndef UF_CONTRASTIVE_H_
#define UF_CONTRASTIVE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define UF_API __attribute__((visibility("default")))
#else
#define UF_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  UF_DEVICE_TIMEOUT is only ever written to *device_status by a kernel
 * whose bounded wait ran out; the host-side call itself never returns it.  A kernel also
 * writes UF_INVALID_ARGUMENT there when a logit scale or bias that it reads from device
 * memory (uf_contrastive_fwd_bwd_ex) is out of range. */
typedef enum uf_status {
  UF_OK = 0,
  UF_INVALID_ARGUMENT = 1,    /* null pointer, bad size, misaligned pointer, bad prefix ladder */
  UF_UNSUPPORTED = 2,         /* valid request the library does not implement (e.g. scale > 256) */
  UF_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < uf_contrastive_workspace_min(...) */
  UF_CUDA_ERROR = 4,          /* a CUDA runtime call or kernel launch failed */
  UF_DEVICE_TIMEOUT = 5       /* a kernel gave up a bounded wait (read from *device_status) */
} uf_status_t;

typedef enum uf_loss_kind {
  UF_LOSS_CLIP_SYMMETRIC = 0,
  UF_LOSS_SIGLIP = 1,
  UF_LOSS_INFONCE_ROWS = 2
} uf_loss_kind_t;

/* Static spelling of a status ("ok", "invalid-argument", ...); "unknown" otherwise. */
UF_API const char* uf_status_name(int status);

/* Version of this library as major*10000 + minor*100 + patch. */
UF_API int uf_contrastive_version(void);

/*
 * Load every kernel of the library on `device` and set their shared-memory limits.
 * Idempotent.  Calling it once per device before the first uf_contrastive_fwd_bwd (and
 * before any stream capture) keeps lazy module loading off the hot path; the blog's
 * section "Across the Box" describes the host blocking on lazy loading inside a step.
 * Returns UF_CUDA_ERROR when the device is absent or is not sm_103.
 */
UF_API uf_status_t uf_contrastive_init(int device);

/*
 * Recommended bytes of device scratch for uf_contrastive_fwd_bwd with these arguments (a
 * pure function of the arguments; 0 when they are invalid).  want_grads != 0 sizes the
 * workspace for the backward as well.  The backward keeps the bf16 weights of every
 * prefix for a chunk of rows of A by rows of B in the workspace (n_prefix x R x C x 2
 * bytes); the recommended size holds every weight in one chunk unless that exceeds 48 GiB,
 * in which case the weights are cut into about square chunks.  For CLIP and ROWS with long
 * contractions (more than about 4864 rows at D = 1024) and a second-widest prefix that is a
 * multiple of 512, it also holds the sums that let the two widest prefixes share one weight
 * array (4 (Na/128) Nb + (4 s + 1) Na + Nb floats, s the weight pass's column split; 0.54 GB
 * at N = 65536), which the backward then uses.  Any workspace of at least
 * uf_contrastive_workspace_min() bytes works: a smaller one only means more chunks (dA then
 * adds over the chunks of B's rows, dB over the chunks of A's rows, in a fixed order).
 */
UF_API size_t uf_contrastive_workspace_size(int64_t Na, int64_t Nb, int D, const int* prefixes, int n_prefix,
                                     int kind, int want_grads);

/* The smallest workspace that uf_contrastive_fwd_bwd accepts for these arguments (the
 * smallest chunk of weights: 128 rows of A by 256 rows of B, or by all of B when it has no
 * more); 0 when they are invalid. */
UF_API size_t uf_contrastive_workspace_min(int64_t Na, int64_t Nb, int D, const int* prefixes, int n_prefix,
                                    int kind, int want_grads);

/*
 * Forward and (optionally) backward of the Matryoshka contrastive loss.
 *
 *   A, B            device, bf16, row-major Na x D and Nb x D, 16-byte aligned.
 *   Na, Nb, D       rows and width.  D is a multiple of 64 and <= 4096; Na, Nb >= 1.
 *                   CLIP needs Na == Nb; ROWS and SigLIP need Nb >= Na: row i < Na of A is
 *                   paired with row i of B, and the rows of B past Na are extra negatives
 *                   (explicit hard negatives) for every row of A.
 *   prefixes        host, n_prefix strictly increasing multiples of 64, last <= D.
 *   n_prefix        1..8.
 *   kind            a uf_loss_kind_t.
 *   logit_scale     CLIP/ROWS: tau in s = tau * cos, 0 < tau <= 256 (larger tau returns
 *                   UF_UNSUPPORTED).  Up to tau = 40 the softmax sums use the fixed shift
 *                   s - tau (every term stays a normal float); above it they take each
 *                   row's and column's largest logit as its shift, found by one more pass
 *                   over the scores.  SigLIP: t in x = t cos + b, |t| + |b| <= 80.
 *   bias            SigLIP b; ignored otherwise.
 *   prefix_weights  host, n_prefix weights w_p of the gradient, or NULL for all 1.
 *   loss_per_prefix device fp32 [n_prefix]: the unweighted L_p.
 *   row_terms       device fp32 [n_prefix][Na] or NULL: per-row terms whose mean is the
 *                   row half of L_p (CLIP: LSE_j s_ij - s_ii; ROWS: the same; SigLIP:
 *                   sum_j softplus(-z_ij x_ij), so L_p = mean_i row_terms).
 *   col_terms       device fp32 [n_prefix][Nb] or NULL: CLIP only (LSE_i s_ij - s_jj);
 *                   written as 0 for the other kinds.
 *   dA, dB          device fp32 Na x D / Nb x D, 16-byte aligned, or both NULL for a
 *                   forward-only call.  Columns at or past the last prefix are written 0.
 *   workspace       device scratch of workspace_bytes >= uf_contrastive_workspace_min(),
 *                   256-byte aligned (uf_contrastive_workspace_size() bytes recommended).
 *                   Owned by the caller; one call at a time per workspace.
 *   device_status   device int or NULL.  Kernels that give up a bounded wait store
 *                   UF_DEVICE_TIMEOUT there (it is never cleared by the library).
 *   stream          a cudaStream_t (0 = legacy default stream).
 * Zero-norm prefixes use 1/max(|x|, 1e-30) as their inverse norm.
 * Argument errors are found on the host before anything is enqueued; the outputs are then
 * untouched.  Launch failures return UF_CUDA_ERROR; outputs are then unspecified.
 */
UF_API uf_status_t uf_contrastive_fwd_bwd(const void* A, const void* B, int64_t Na, int64_t Nb, int D,
                                   const int* prefixes, int n_prefix, int kind, float logit_scale, float bias,
                                   const float* prefix_weights, float* loss_per_prefix, float* row_terms,
                                   float* col_terms, float* dA, float* dB, void* workspace,
                                   size_t workspace_bytes, int* device_status, void* stream);

/*
 * uf_contrastive_fwd_bwd for a loss whose two scalar parameters are learned (blog post
 * "Scaling-Up Contrastive Learning over NVLink Multicast", section "One Set or Two":
 * SigLIP's learned temperature t and bias b; CLIP's logit scale likewise).  It can read
 * them from device memory and differentiates the weighted loss sum_p w_p L_p in them:
 *   logit_scale_dev device fp32 scalar or NULL.  When given, the kernels read the logit
 *                   scale there when they run (logit_scale is ignored), so a CUDA graph
 *                   captured once follows a scale that the optimizer updates in place.
 *                   CLIP/ROWS then always take the max-shifted statistics (the host cannot
 *                   pick the fixed shift for a value it does not see).  A value outside
 *                   the range logit_scale allows makes the first kernel store
 *                   UF_INVALID_ARGUMENT in *device_status; the outputs are then undefined.
 *   bias_dev        device fp32 scalar or NULL: the same for bias (SigLIP).
 *   pos_offsets,    SigLIP only (else UF_UNSUPPORTED): the positive pairs as CSR lists on the
 *   pos_ids         device, in place of the diagonal (blog, section "Scaling-Up": each entry
 *                   can carry several positives and explicit hard negatives).  Row i of A
 *                   has the positives B[pos_ids[q]] for pos_offsets[i] <= q < pos_offsets[i+1];
 *                   every other cell is a negative (z = -1).  pos_offsets: int64 [Na + 1],
 *                   8-byte aligned, pos_offsets[0] = 0, nondecreasing; pos_ids: int32, each
 *                   row's ids strictly increasing in [0, Nb).  A row may have no positive.
 *                   Entries that break these rules are skipped and make the kernels store
 *                   UF_INVALID_ARGUMENT in *device_status (the ids array must still hold
 *                   pos_offsets[Na] entries).  Both NULL: the diagonal (i, i), i < Na.
 *                   The row terms then hold sum_j softplus(-z_ij x_ij) for the labels.
 *   d_logit_scale   device fp32 scalar or NULL: dL/d(logit_scale) (tau for CLIP / ROWS,
 *                   t for SigLIP), computed as (1 / logit_scale) sum_ij dL/dcos_ij cos_ij
 *                   from the backward's row scalars; SigLIP with logit_scale == 0 returns
 *                   UF_UNSUPPORTED when it is requested.
 *   d_bias          device fp32 scalar or NULL: dL/db for SigLIP, from the per-row sums of
 *                   sigmoid(x_ij) over the negatives and the positives' sigmoid(-x_ii);
 *                   written 0 for CLIP and ROWS.
 * d_logit_scale and d_bias need the backward (dA and dB non-NULL), else
 * UF_INVALID_ARGUMENT.  Every other argument means what it means in
 * uf_contrastive_fwd_bwd, which is this call with the six new pointers NULL.
 */
UF_API uf_status_t uf_contrastive_fwd_bwd_ex(const void* A, const void* B, int64_t Na, int64_t Nb, int D,
                                      const int* prefixes, int n_prefix, int kind, float logit_scale,
                                      float bias, const float* logit_scale_dev, const float* bias_dev,
                                      const int64_t* pos_offsets, const int* pos_ids,
                                      const float* prefix_weights, float* loss_per_prefix,
                                      float* row_terms, float* col_terms, float* dA, float* dB,
                                      float* d_logit_scale, float* d_bias, void* workspace,
                                      size_t workspace_bytes, int* device_status, void* stream);

/*
 * One-set SigLIP: the set X scored against itself (blog post "Scaling-Up Contrastive
 * Learning over NVLink Multicast", section "One Set or Two": one set, the same labels and
 * weights for mirrored cells, so the owner of a row differentiates both of its cells; an
 * image and its caption are two rows of the set marked as a positive pair):
 *   L_p = -(1/N) sum_i sum_{j != i} log sigmoid(z_ij (t cos_ij + b)),
 * cos_ij between rows i and j of X on the prefix, z_ij = +1 for the listed pairs, -1 else.
 *   X               device bf16 N x D, 16-byte aligned.
 *   pos_offsets,    required: the positive pairs as device CSR lists (format as in
 *   pos_ids         uf_contrastive_fwd_bwd_ex).  They must be symmetric (j listed in row i
 *                   exactly when i is listed in row j) and name no self-pair; entries that
 *                   break this are skipped and reported as UF_INVALID_ARGUMENT in
 *                   *device_status.
 *   row_terms       device fp32 [n_prefix][N] or NULL: sum_{j != i} softplus(-z_ij x_ij).
 *   dX              device fp32 N x D or NULL (forward only): the gradient of
 *                   sum_p w_p L_p through both cells of every pair.
 *   workspace       at least uf_contrastive_workspace_min(N, N, D, prefixes, n_prefix,
 *                   UF_LOSS_SIGLIP, dX != NULL) bytes (uf_contrastive_workspace_size
 *                   recommended), 256-byte aligned.
 * Every other argument as in uf_contrastive_fwd_bwd_ex.  The symmetric weights make the
 * gradient one contraction: the B side of the two-set backward is skipped.
 */
UF_API uf_status_t uf_contrastive_oneset_fwd_bwd(const void* X, int64_t N, int D, const int* prefixes,
                                          int n_prefix, float logit_scale, float bias,
                                          const float* logit_scale_dev, const float* bias_dev,
                                          const int64_t* pos_offsets, const int* pos_ids,
                                          const float* prefix_weights, float* loss_per_prefix,
                                          float* row_terms, float* dX, float* d_logit_scale, float* d_bias,
                                          void* workspace, size_t workspace_bytes, int* device_status,
                                          void* stream);

/*
 * uf_contrastive_fwd_bwd without a workspace argument, for callers that cannot allocate
 * device memory: hosts that reserve all of their memory at start-up and forbid
 * allocation afterwards, plugins whose host application owns every device buffer, or
 * processes whose allocator is a fixed pool.  (The pages describe no such entry point;
 * it exists for these callers only.)
 *
 * The scratch is one device array of UF_STATIC_WORKSPACE_BYTES inside the library, which
 * every GPU that loads the library keeps until the process exits.  The caller still
 * passes inputs and outputs, with the same meaning and rules as uf_contrastive_fwd_bwd.
 *   - A request whose uf_contrastive_workspace_min() exceeds UF_STATIC_WORKSPACE_BYTES
 *     returns UF_WORKSPACE_TOO_SMALL before anything is enqueued (at D = 1024 with the
 *     five-prefix ladder and Na = Nb = N, with gradients: CLIP fits up to N = 14208,
 *     SigLIP up to N = 19456); inside that bound the backward cuts the weights into as many
 *     chunks (rows of A by rows of B) as the array needs.
 *   - The first call on a device looks up the array's device address (with that device
 *     current), and so does the first call after the device's context was replaced
 *     (cudaDeviceReset); make such a call before any stream capture.
 *   - All calls on a device share the one array, and it keeps whatever the last call left
 *     there (nothing in it needs clearing: every element is written before it is read).
 *     Calls whose GPU work overlaps -- on different streams, or from different threads --
 *     race on it and give wrong results; serialise them.
 *   - It calls no allocator: no cudaMalloc, no cudaFree, no allocating library routine.
 */
#define UF_STATIC_WORKSPACE_BYTES (96u << 20)
UF_API uf_status_t uf_contrastive_fwd_bwd_static(const void* A, const void* B, int64_t Na, int64_t Nb, int D,
                                                  const int* prefixes, int n_prefix, int kind, float logit_scale,
                                                  float bias, const float* prefix_weights, float* loss_per_prefix,
                                                  float* row_terms, float* col_terms, float* dA, float* dB,
                                                  int* device_status, void* stream);

/*
 * Self-test of the failure path: every pipeline kernel waits on its barriers with a bound
 * (4 s) and, when one runs out, stores UF_DEVICE_TIMEOUT in *device_status and ends, so the
 * CUDA context stays usable.  This enqueues one kernel that takes the same bounded wait on a
 * barrier that nothing completes, with a limit of limit_ms (1..10000) milliseconds: after it,
 * *device_status (a device int, 4-byte aligned) holds UF_DEVICE_TIMEOUT.  Nothing faults,
 * traps or hangs.  Returns UF_INVALID_ARGUMENT for a NULL or misaligned status or a limit out
 * of range, UF_CUDA_ERROR when the launch fails.
 */
UF_API uf_status_t uf_contrastive_selftest_wait(int* device_status, int limit_ms, void* stream);

/*
 * Optional per-kernel timing, for benchmarks and profiling (not part of the loss).
 * While enabled, every uf_contrastive_fwd_bwd records a pair of CUDA events on its
 * stream around each group of internal kernel launches and keeps the pairs in a host
 * list (this list grows, so do not enable it under stream capture or on a hot path that
 * must not allocate).  uf_contrastive_profile_read() waits for the recorded events,
 * folds them into per-kernel totals and returns them.  Kernel groups:
 */
typedef enum uf_kernel_group {
  UF_KERNEL_PREP = 0,       /* per-prefix inverse norms and positives' cosines (1 launch) */
  UF_KERNEL_TRANSPOSE = 1,  /* bf16 transposes for the gradient operand (1 launch) */
  UF_KERNEL_FWD_TILE = 2,   /* fused tcgen05 forward: row sums of every prefix */
  UF_KERNEL_STATS = 3,      /* loss statistics and per-prefix loss (1 launch; 2 on the max-shifted path) */
  UF_KERNEL_BWD_TILE = 4,   /* tcgen05 backward weight pass: score recompute, bf16 weights to HBM */
  UF_KERNEL_NORM_BWD = 5,   /* projection term and positive-pair correction */
  UF_KERNEL_GEMM = 6,       /* tcgen05 gradient contraction over the bf16 weights */
  UF_KERNEL_GROUPS = 7
} uf_kernel_group_t;

/* enable != 0: start timing (clears the totals); 0: stop.  Process-wide. */
UF_API uf_status_t uf_contrastive_profile(int enable);
/* Totals of one group since the last enable: summed milliseconds, timed event pairs,
 * and kernel launches.  Synchronises with the recorded events. */
UF_API uf_status_t uf_contrastive_profile_read(int group, double* total_ms, int64_t* pairs, int64_t* launches);
/* Static name of a group ("bwd_tile", ...), or "unknown". */
UF_API const char* uf_contrastive_profile_name(int group);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* UF_CONTRASTIVE_H_ */
