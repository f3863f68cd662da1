// launch.h -- host-side launchers of the kernels (internal to the library).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "common.cuh"

namespace ufc {

// SM count of the current device (grid caps of the grid-stride kernels).
int current_sm_count();

// Launches kernel k with programmatic stream serialization, so that it may be scheduled while
// the kernel before it on the stream drains (every kernel here calls griddep_enter() before it
// touches global memory), and, with cluster > 1, in clusters of that many CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       unsigned cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (cluster > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, k, static_cast<Args&&>(args)...);
}

// Load every auxiliary kernel now (aux_kernels.cu).
cudaError_t aux_kernels_setup();

// Forward statistics with 128 x 256 score tiles (fwd_kernel.cu): row sums of every
// prefix over the negatives, and (CLIP) 128-row partial column sums.  Modes:
//   kFwdSum      sums of 2^(x - L), x = tau log2(e) cos (the fixed shift L = tau log2(e))
//   kFwdMax      maxima of x over the row / the 128 rows of the column (padding excluded,
//                the positive included): the shifts of the max-shifted path
//   kFwdShifted  sums of 2^(x - u_i) per row and 2^(x - v_j) per column, u and v the
//                maxima of a kFwdMax pass (log2 units)
enum FwdMode : int { kFwdSum = 0, kFwdMax = 1, kFwdShifted = 2 };
struct FwdParams {
  int64_t nx, ny;
  int n_prefix;
  int prefix_end[kMaxPrefix];
  int n_col_tiles;          // ceil(ny / 256)
  int tiles_per_split;
  int mode;                 // FwdMode (SigLIP: kFwdSum only)
  Scalars sc;
  const float* rinv_x;
  const float* rinv_y;
  const float* shift_x;     // kFwdShifted: u [n][nx]
  const float* shift_y;     // kFwdShifted, CLIP: v [n][ny]
  int no_diag;              // SigLIP with a label matrix: the diagonal is not special (every cell a negative)
  float* rowacc;            // [split * 4 + column quarter][n][nx]
  float* colacc;            // [row block][n][ny] (CLIP only)
  int* status;
};
constexpr int kFwdCols = 256;
cudaError_t fwd_kernel_setup();
cudaError_t launch_fwd(int kind, const CUtensorMap& tm_x, const CUtensorMap& tm_y, const FwdParams& p, dim3 grid,
                       cudaStream_t stream);

// Backward weights (wgt_kernel.cu): m^k_ij = rho_i sigma_j dL/dcos^k_ij as bf16 into a
// [prefix][row][column] array (row stride in elements fixed by tm_w), plus (SigLIP) the
// row loss sums.  One launch covers rows [row0, row0 + rows) of X against rows
// [col0, col0 + cols) of Y; grid = (ceil(rows / 128), splits of the 256-column tiles).
// tm_x: [128 x 64] boxes of X; tm_y: [128 x 64] boxes of Y (each CTA of a pair stages half of
// the 256-row tile); tm_w: [32 x 64] boxes of the weight array viewed as
// [n * w_rows_per_prefix rows][ny columns].  Launched as CTA pairs (clusters of 2 along x).
struct WgtParams {
  int64_t nx, ny;                 // full sizes of X and Y
  int64_t row0, rows;             // this launch's rows of X
  int64_t col0, cols;             // this launch's rows of Y (columns of the weights; the array holds
                                  // column col0 + c at its column c)
  int add_rows;                   // SigLIP: add the row sums into rowacc / rowsig (a later column range)
  int n_col_tiles;                // ceil(cols / 256)
  int n_prefix;
  int prefix_end[kMaxPrefix];
  int tiles_per_split;
  Scalars sc;
  int shifted;                    // CLIP/ROWS: the max-shifted statistics (alpha_x, beta_y in log2 form)
  const float* rinv_x;            // [n][nx]
  const float* alpha_x;           // [n][nx] rho_i alpha_i (CLIP/ROWS) or NULL; shifted: log2(rho_i alpha_i / w_k) - u_i
  const float* rinv_y;            // [n][ny]
  const float* beta_y;            // [n][ny] sigma_j beta_j (CLIP) or NULL; shifted: log2(sigma_j beta_j / w_k) - v_j
  float m_scale[kMaxPrefix];      // SigLIP: w_k / N (times t in the kernel); shifted CLIP/ROWS: w_k
  int no_diag;                    // SigLIP with a label matrix: weights for every cell as a negative
  int64_t w_rows_per_prefix;      // rows between prefixes in the weight array (multiple of 128)
  float* rowacc;                  // SigLIP: [split * 4 + quarter][n][nx] loss sums (log2 units), or NULL
  float* rowsig;                  // SigLIP, with rowacc: the same slots, sums of sigmoid(x_ij) over the
                                  // negatives (the bias gradient), or NULL
  // merge: the two widest prefixes share one array on the dimensions below p_{n-2} (a multiple
  // of 512).  At prefix n-1 the block that prefix n-2 stored becomes bf16(W^{n-1} + W^{n-2})
  // (W = the stored bf16 weights) by a bulk reduce-add through tm_w; C = sum_j W^{n-1}_ij
  // d^{n-1}_ij (d the raw dot) is summed per row into r5_row[split * 4 + quarter][nx] and per
  // 32-row block and column into r5_col[row block * 4 + quadrant][ny].
  int merge;
  float* r5_row;
  float* r5_col;
  int* status;
};
constexpr int kWgtCols = 256;
constexpr int kWgtStoreRows = 32;
cudaError_t wgt_kernel_setup();
cudaError_t launch_wgt(int kind, const CUtensorMap& tm_x, const CUtensorMap& tm_y, const CUtensorMap& tm_w,
                       const WgtParams& p, dim3 grid, cudaStream_t stream);

// Gradient contraction (gemm_kernel.cu), for rows g = row0 + [0, m_rows) of G:
//   weights K-major (A side):  G[g, d] = sum_k [d < p_k] sum_c m^k[g - row0, c] Y[c, d]
//   weights MN-major (B side): G[g, d] = sum_k [d < p_k] sum_c m^k[c, g] Y[b_col0 + c, d]
// with c over [0, kdim), and the projection scalars crow[slice][k][g] = X[g, slice] . G^k[g, slice]
// (partial over each 256-dimension slice).  accumulate: add into G and crow instead of
// writing them.  tm_w: the weight array [n * w_rows_per_prefix rows][columns], boxes of
// [128 x 64] (K-major) or [64 x 64] (MN-major); tm_yt / tm_yt128: [32 x 64] / [128 x 64] boxes
// of Y^T ([d rows][rows of Y]).
struct GemmParams {
  int64_t m_rows;                 // rows of G computed by this launch
  int64_t row0;                   // their first row in G, X and crow
  int64_t kdim;                   // contraction length
  int64_t b_col0;                 // first column of Y^T for this launch's contraction range
  int64_t w_rows_per_prefix;
  int d;                          // row stride of G and X in elements
  int n_prefix;
  int prefix_end[kMaxPrefix];
  int accumulate;
  float* G;
  int merge;                      // 1: slice groups below p_{n-2} contract prefixes n-2 .. (array n-2 holds
                                  // the merged weights of n-2 and n-1) into G; prefix n-1 runs only above
  int split_rest;                 // 1: the prefixes below the widest run as their own units, into G2
  float* G2;                      // [m_rows][g2_ld] (split_rest): their part of G, dimensions < g2_ld
  int64_t g2_ld;                  // the second-widest prefix's end
  const uint16_t* X;              // bf16 rows of the side G belongs to
  float* crow;                    // [slice][n][crow_rows]
  int64_t crow_rows;
  int* status;
};
constexpr int kGemmBBox = 32;   // rows per TMA box of the GEMMs' B operand (Y^T)
cudaError_t gemm_kernel_setup();
cudaError_t launch_gemm(const CUtensorMap& tm_w, const CUtensorMap& tm_yt, const CUtensorMap& tm_yt128,
                        const GemmParams& p, bool weights_mn, cudaStream_t stream);
// CTA pairs of one contraction's grid, and the dA grid size (in waves of CTA pairs) below which
// both contractions go in one grid.
double gemm_grid_pairs(const GemmParams& p);
constexpr double kGemmOneGridWaves = 4.0;
// Both contractions of one weight chunk (dA with K-major weights, dB with MN-major ones) as one
// grid, so the dB CTAs fill the dA contraction's last wave.
cudaError_t launch_gemm_both(const CUtensorMap& tk_w, const CUtensorMap& tk_yt, const CUtensorMap& tk_yt128,
                             const GemmParams& pk, const CUtensorMap& tn_w, const CUtensorMap& tn_yt,
                             const CUtensorMap& tn_yt128, const GemmParams& pn, cudaStream_t stream);

// Per-row inverse norms of every prefix for A and B, plus the positives' cosines
// cos_ii for i < min(Na, Nb).  Layouts [n][rows].
struct PrepParams {
  int kind;
  Scalars sc;              // device scalars are range-checked here (status = kStatusBadScalar)
  int* status;
  const uint16_t* A;
  const uint16_t* B;
  int64_t na, nb, nmin;
  int d, n_prefix;
  int prefix_end[kMaxPrefix];
  float* rinv_a;
  float* rinv_b;
  float* pos_cos;
  unsigned* stats_done;    // the statistics pass's block counter, zeroed here
};
cudaError_t launch_prep(const PrepParams& p, cudaStream_t stream);

// X[z] (rows[z] x d, bf16) -> Xt[z] (d x ld[z], bf16): Xt[c][r] = X[r][c] for r < rows, 0 up to
// ld (rows rounded up to 64), for z < count (one or two matrices, one launch).
struct TransposeParams {
  const uint16_t* X[2];
  uint16_t* Xt[2];
  int64_t rows[2], ld[2];
  int d, count;
};
cudaError_t launch_transpose(const TransposeParams& p, cudaStream_t stream);

// Loss statistics after the forward (CLIP / ROWS) or the A-side backward (SigLIP).
struct StatsParams {
  int kind;
  int64_t na, nb;
  int n_prefix;
  int prefix_end[kMaxPrefix];
  Scalars sc;
  float weight[kMaxPrefix];
  const float* rinv_a;
  const float* rinv_b;
  const float* pos_cos;
  const float* shift_a;    // NULL: the fixed shift tau; else the rows' shifts u [n][na] (log2 units)
  const float* shift_b;    // CLIP, with shift_a: the columns' shifts v [n][nb]
  int diag_pos;            // 1: the diagonal cells (i, i), i < min(na, nb), are the positives
  const float* pos_term;   // SigLIP with a label matrix: [n][na] the positives' share of the row terms, or NULL
  const float* rowacc_a;   // [slots_a][n][na]
  int slots_a;
  const float* rowacc_b;   // [slots_b][n][nb] (CLIP)
  int slots_b;
  float* zr;               // [n][na]  row sums over the negatives, relative to the row's shift (CLIP/ROWS)
  float* zc;               // [n][nb]
  float* fa;               // [n][na]  rho_i alpha_i (backward factor); shifted: log2(rho_i alpha_i / w_k) - u_i
  float* fb;               // [n][nb]  sigma_j beta_j; shifted: log2(sigma_j beta_j / w_k) - v_j
  float* terms_a;          // [n][na]  row terms
  float* terms_b;          // [n][nb]  column terms (CLIP; 0 otherwise)
  float* loss;             // [n]
  double* part;            // [kStatsBlocks][kMaxPrefix] per-block sums of the terms
  unsigned* done;          // blocks finished; 0 before the launch (the prep pass zeroes it), 0 after
};
// The statistics pass: kStatsThreads threads a block, at most kStatsBlocks blocks (a constant,
// so that the workspace does not depend on the device).
constexpr int kStatsThreads = 256;
constexpr int kStatsBlocks = 1216;
static_assert(kStatsThreads / 32 >= kMaxPrefix, "the statistics pass sums one prefix per warp");
cudaError_t launch_stats(const StatsParams& p, cudaStream_t stream);

// dX = G (+ G2) - r_c * X + q_c * Y (diagonal rows), 0 past the last prefix.
struct NormBwdParams {
  int kind;
  int64_t nx, ny, nmin, n_total;  // n_total: batch size used by the loss normaliser
  int d, n_prefix;
  int prefix_end[kMaxPrefix];
  Scalars sc;
  float weight[kMaxPrefix];
  const uint16_t* X;
  const uint16_t* Y;
  const float* rinv_x;
  const float* rinv_y;
  const float* pos_cos;
  const float* z_x;        // CLIP/ROWS sums of X's rows over negatives (ROWS: the queries')
  const float* z_y;        // CLIP: of Y's rows
  const float* shift_x;    // NULL: the fixed shift; else the shifts of z_x's rows (log2 units)
  const float* shift_y;    // likewise for z_y
  int x_is_query;          // ROWS: 1 when X holds the queries
  const float* crow;       // [slots][n][nx]
  int crow_slots;
  const float* G;          // [nx][d]
  const float* G2;         // NULL, or [nx][g2_ld]: added to G below dimension g2_ld
  int64_t g2_ld;
  const float* r5;         // NULL, or (merged widest prefixes) [nx]: prefix n-1's C off the diagonal; its
                           // slots in crow then hold only the dimensions above p_{n-2}, and prefix
                           // n-2's slots the merged weights' x . G
  float* dX;               // [nx][d]
  float* csum;             // NULL or [nx]: sum over prefixes of the full row scalar C_k (logit-scale gradient)
  int double_out;          // one-set loss: write 2 dX (the row's gradient through both roles of every cell)
};
// sides: one or two (A's rows, then B's), run as one grid.
cudaError_t launch_norm_bwd(const NormBwdParams* sides, int n_sides, cudaStream_t stream);

// Merged widest prefixes: r5_a[i] = sum_s row[s][i] (s < row_slots), r5_b[j] = sum_q col[q][j]
// (q < col_parts), each in a fixed order.
struct R5Params {
  int64_t na, nb;
  const float* row;
  int row_slots;
  const float* col;
  int col_parts;
  float* r5_a;
  float* r5_b;
};
cudaError_t launch_r5(const R5Params& p, cudaStream_t stream);

// Gradients of the weighted loss in the logit scale and (SigLIP) the bias, from the row
// scalars: d_scale = (1 / scale) sum_i csum[i]  (sum_ij W_ij cos_ij = scale dL/dscale), and
// d_bias = sum_k (w_k / N) (sum_i sum_slots rowsig[.][k][i] - sum_i sigmoid(-x_ii)).
// One block, float64, fixed order.
struct ScaleGradParams {
  int kind;
  int64_t na, nmin;
  int n_prefix;
  Scalars sc;
  float weight[kMaxPrefix];
  const float* csum;       // [na]
  const float* rowsig;     // SigLIP: [slots][n][na]
  int sig_slots;
  const float* lcount;     // SigLIP with a label matrix: [na] positives per row (else the diagonal)
  const float* pos_cos;    // [n][nmin]
  float* d_scale;          // device scalar or NULL
  float* d_bias;           // device scalar or NULL
};
cudaError_t launch_scale_grad(const ScaleGradParams& p, cudaStream_t stream);

// The shifts of the max-shifted path from a kFwdMax forward: u[k][i] = max over the row
// slots, v[k][j] = max over the column partials of every row block (CLIP; NULL otherwise).
struct MaxReduceParams {
  int n_prefix;
  int64_t na, nb;
  const float* rowmax;     // [slots_a][n][na]
  int slots_a;
  const float* colmax;     // [blocks][n][nb] or NULL
  int blocks;
  float* u;                // [n][na]
  float* v;                // [n][nb] or NULL
};
cudaError_t launch_max_reduce(const MaxReduceParams& p, cudaStream_t stream);

// SigLIP with a label matrix given as CSR positive lists (offsets [na + 1], ids), one warp
// per row of A.  Every positive (i, j) gets its cosines recomputed per prefix (fp32 dot of
// the bf16 rows) and x = t cos + b.  Entries that break the format (a row whose offsets
// decrease, an id outside [0, nb) or not above the row's previous id) are skipped and
// set *status = kStatusBadScalar.
//   terms mode (W == NULL): pos_term[k][i] = -sum_j x^k_ij (the loss of a positive cell is
//                the negative cell's minus x), lcount[i] = valid positives of row i
//   patch mode (W != NULL): for rows [row0, row0 + rows) write the exact weight of every
//                positive cell, bf16(-sigmoid(-x) rho sigma w_k t / N), over the negative-cell
//                weight the weight pass stored at W[(k * w_rows_per_prefix + i - row0) * ldw + j]
struct LabelParams {
  const int64_t* offsets;
  const int* ids;
  const uint16_t* A;
  const uint16_t* B;
  int64_t na, nb;
  int d, n_prefix;
  int prefix_end[kMaxPrefix];
  Scalars sc;
  float weight[kMaxPrefix];
  const float* rinv_a;
  const float* rinv_b;
  float* pos_term;
  float* lcount;
  uint16_t* W;             // patch mode: the weights of rows [row0, row0 + rows), columns [col0, col0 + cols)
  int64_t row0, rows, w_rows_per_prefix, ldw;
  int64_t col0, cols;
  int oneset;              // one-set loss: a self-pair (j == i) or a pair whose mirror is missing is malformed
  int* status;
};
cudaError_t launch_labels(const LabelParams& p, cudaStream_t stream);

// One thread waits, with the pipeline kernels' bounded wait, on a barrier nothing completes.
cudaError_t launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t stream);

}  // namespace ufc
