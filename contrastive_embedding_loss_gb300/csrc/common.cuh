// common.cuh -- parameters shared by the host launcher and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace ufc {

constexpr int kMaxPrefix = 8;
constexpr int kTileRows = 128;   // rows of X per CTA = UMMA M
constexpr int kChunk = 64;       // K elements per shared-memory stage: one 128-byte swizzle row
constexpr int kSliceDims = 256;  // gradient columns one backward CTA accumulates in TMEM

enum Kind : int { KIND_CLIP = 0, KIND_SIGLIP = 1, KIND_ROWS = 2 };

constexpr int kStatusTimeout = 5;  // == UF_DEVICE_TIMEOUT

// One launch of the backward kernel.  "X" is the owner side (its rows are the CTA's
// 128 rows, thread = row), "Y" the side whose rows are walked as columns.
struct TileParams {
  int64_t nx, ny;
  int d;                          // embedding width (row stride of X and Y, in elements)
  int n_prefix;
  int prefix_end[kMaxPrefix];     // prefix ends in elements, multiples of 64
  int n_col_tiles;                // ceil(ny / 256)
  int tiles_per_split;            // column tiles per CTA along blockIdx.y
  float L;                        // CLIP/ROWS: tau*log2(e) (also the fixed shift); SigLIP: t*log2(e)
  float b2;                       // SigLIP: bias*log2(e)
  // per-prefix row factors of X, [n_prefix][nx]
  const float* rinv_x;            // rho_i = 1/|x_i[:p]|
  const float* alpha_x;           // backward CLIP/ROWS: rho_i * alpha_i (row part of W', scaled)
  // per-prefix column factors of Y, [n_prefix][ny]
  const float* rinv_y;            // sigma_j
  const float* beta_y;            // backward CLIP/ROWS: sigma_j * beta_j
  float m_scale[kMaxPrefix];      // backward SigLIP: w_k * t / N
  // outputs (slot = split*4 + column quarter)
  float* rowacc;                  // [slot][n_prefix][nx]: SigLIP loss sums over the negatives, in
                                  // log2 units (NULL: not wanted)
  float* crow;                    // [slot][n_prefix][nx]: sum_j m_ij dot_ij (off-diagonal)
  float* grad;                    // [split][nx][d]: sum_j m_ij y_j over this CTA's columns
  int* status;
};

}  // namespace ufc
