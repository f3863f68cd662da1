// aux_kernels.cu -- the HBM-streaming steps around the fused score kernel:
//   prep      per-prefix inverse norms of every row and the positives' cosines
//   transpose bf16 X (rows x d) -> X^T (d x rows), the K-major operand of the gradient MMA
//   stats     fixed-shift row/column sums -> row terms, backward factors, and the per-prefix
//             loss (fp64, fixed reduction order, by the last block to finish)
//   norm_bwd  dX = G - r_c X + q_c Y: the cosine's projection term and the diagonal
//             (positive-pair) correction, band by band.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "launch.h"
#include "ptx.cuh"

namespace ufc {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ int band_of(int e, const int* pend, int n) {
  int b = 0;
#pragma unroll
  for (int k = 0; k < kMaxPrefix; ++k) b += (k < n && pend[k] <= e) ? 1 : 0;
  return b;  // == n past the last prefix
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ------------------------------------------------------------------------------ prep
// Eight lanes per item, four items per warp; item r < max(Na, Nb) covers rows A_r and B_r
// together while r < Nmin (so the positive pair's dot products come from the same
// registers), otherwise the one row.  A lane reads every eighth 16-byte chunk of the row,
// four chunks in flight, and the eight lanes of an item meet in a 3-stage shuffle reduce.
__global__ void __launch_bounds__(256) prep_kernel(const PrepParams p) {
  griddep_enter();
  const int lane = threadIdx.x & 31;
  const int sub = lane & 7;  // the lane within its item's group of eight
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_items = p.na > p.nb ? p.na : p.nb;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int n = p.n_prefix;
  if (blockIdx.x == 0 && threadIdx.x == 0) *p.stats_done = 0u;
  if (blockIdx.x == 0 && threadIdx.x == 0 && p.status && (p.sc.scale_ptr || p.sc.bias_ptr)) {
    // scalars that only the device knows are range-checked here, where the host checks its own
    const float t = p.sc.t(), b = p.sc.b();
    const bool ok = p.kind == KIND_SIGLIP ? (isfinite(t) && isfinite(b) && fabsf(t) + fabsf(b) <= kMaxSiglipRange)
                                          : (t > 0.f && t <= kMaxLogitScale);
    if (!ok) atomicExch(p.status, kStatusBadScalar);
  }
  const int pn = p.prefix_end[n - 1];
  const int n_chunks = pn / 8;  // 16-byte chunks of a row up to the last prefix end
  for (int64_t r0 = warp_id * 4; r0 < n_items; r0 += n_warps * 4) {  // uniform over the warp
    const int64_t r = r0 + (lane >> 3);
    const bool has_a = r < p.na, has_b = r < p.nb, pair = r < p.nmin;
    float ssa[kMaxPrefix], ssb[kMaxPrefix], dab[kMaxPrefix];
#pragma unroll
    for (int k = 0; k < kMaxPrefix; ++k) ssa[k] = ssb[k] = dab[k] = 0.f;
    const uint4* ra = reinterpret_cast<const uint4*>(p.A + (has_a ? r : 0) * p.d);
    const uint4* rb = reinterpret_cast<const uint4*>(p.B + (has_b ? r : 0) * p.d);
    for (int ch0 = sub; ch0 < n_chunks; ch0 += 32) {
      uint4 va[4], vb[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {  // the loads first: four chunks of each row in flight
        const int ch = ch0 + 8 * u;
        va[u] = make_uint4(0u, 0u, 0u, 0u);
        vb[u] = make_uint4(0u, 0u, 0u, 0u);
        if (ch < n_chunks) {
          if (has_a) va[u] = __ldg(ra + ch);
          if (has_b) vb[u] = __ldg(rb + ch);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int ch = ch0 + 8 * u;
        const int b = band_of(ch * 8, p.prefix_end, n);  // == n past the end: adds nowhere
        const uint32_t wa[4] = {va[u].x, va[u].y, va[u].z, va[u].w}, wb[4] = {vb[u].x, vb[u].y, vb[u].z, vb[u].w};
        float sa = 0.f, sb = 0.f, sd = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float a0 = bf16_lo(wa[q]), a1 = bf16_hi(wa[q]);
          const float b0 = bf16_lo(wb[q]), b1 = bf16_hi(wb[q]);
          sa = fmaf(a0, a0, fmaf(a1, a1, sa));
          sb = fmaf(b0, b0, fmaf(b1, b1, sb));
          sd = fmaf(a0, b0, fmaf(a1, b1, sd));
        }
#pragma unroll
        for (int k = 0; k < kMaxPrefix; ++k)
          if (k == b) {
            ssa[k] += sa;
            ssb[k] += sb;
            dab[k] += sd;
          }
      }
    }
    float ca = 0.f, cb = 0.f, cd = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxPrefix; ++k) {
      if (k >= n) break;
      float va = ssa[k], vb = ssb[k], vd = dab[k];
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) {  // the eight lanes of this item
        va += __shfl_xor_sync(0xffffffffu, va, o);
        vb += __shfl_xor_sync(0xffffffffu, vb, o);
        vd += __shfl_xor_sync(0xffffffffu, vd, o);
      }
      ca += va;
      cb += vb;
      cd += vd;
      if (sub == 0) {
        const float rA = 1.f / fmaxf(sqrtf(ca), 1e-30f);
        const float rB = 1.f / fmaxf(sqrtf(cb), 1e-30f);
        if (has_a) p.rinv_a[k * p.na + r] = rA;
        if (has_b) p.rinv_b[k * p.nb + r] = rB;
        if (pair) p.pos_cos[k * p.nmin + r] = cd * rA * rB;
      }
    }
  }
}

cudaError_t launch_prep(const PrepParams& p, cudaStream_t stream) {
  const int64_t items = p.na > p.nb ? p.na : p.nb;
  int64_t blocks = (items * 8 + 255) / 256;  // eight lanes per item
  if (blocks > int64_t(16) * current_sm_count()) blocks = int64_t(16) * current_sm_count();
  return launch_pdl(prep_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, 1, p);
}

// ------------------------------------------------------------------------------ transpose
// 64 x 64 tiles through shared memory, 16-byte global accesses both ways: a thread loads 8
// consecutive columns of one row of X and stores 8 consecutive rows of one column (a row of
// X^T).  The tile is kept as [column][row] in 8-row chunks whose order within a column is
// XOR-swizzled with the column's 8-column group, so the scalar stores of a warp (one chunk of
// 8 columns per 8 threads) and its 16-byte loads hit distinct banks.
// One launch for up to two matrices: blockIdx.z picks one (blocks past its rows return).
__global__ void __launch_bounds__(256) transpose_kernel(const TransposeParams p) {
  griddep_enter();
  __shared__ __align__(16) uint16_t tile[64][64];
  const bool z = blockIdx.z != 0;  // (selects, not indexes: no copy of the parameters to local memory)
  const uint16_t* __restrict__ X = z ? p.X[1] : p.X[0];
  uint16_t* __restrict__ Xt = z ? p.Xt[1] : p.Xt[0];
  const int64_t rows = z ? p.rows[1] : p.rows[0], ld = z ? p.ld[1] : p.ld[0];
  const int d = p.d;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * 64;
  if (r0 >= ld) return;  // the other matrix has more rows
  const int c0 = blockIdx.y * 64;
  const int sub = threadIdx.x & 7;  // which 8-element chunk a thread moves
  const int lr = threadIdx.x >> 3;  // 0..31
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int y = lr + 32 * h;  // row within the tile
    const int64_t r = r0 + y;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    // rows past the end load zeros: the grid spans ld = rows rounded up to 64, so the
    // padding columns of X^T, which the gradient GEMM reads with zero weights, hold no NaNs
    if (r < rows) v = *reinterpret_cast<const uint4*>(X + r * d + c0 + sub * 8);
    const uint16_t* e = reinterpret_cast<const uint16_t*>(&v);
    const int phys = (((y >> 3) ^ sub) << 3) | (y & 7);  // columns sub*8 + k all lie in group `sub`
#pragma unroll
    for (int k = 0; k < 8; ++k) tile[sub * 8 + k][phys] = e[k];
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int x = lr + 32 * h;  // column within the tile: a row of X^T
    const int phys = sub ^ ((x >> 3) & 7);
    const uint4 v = *reinterpret_cast<const uint4*>(&tile[x][phys * 8]);
    *reinterpret_cast<uint4*>(Xt + static_cast<int64_t>(c0 + x) * ld + r0 + sub * 8) = v;
  }
}

cudaError_t launch_transpose(const TransposeParams& p, cudaStream_t stream) {
  int64_t ld_max = 0;
  for (int z = 0; z < p.count; ++z) ld_max = p.ld[z] > ld_max ? p.ld[z] : ld_max;
  dim3 grid(static_cast<unsigned>((ld_max + 63) / 64), static_cast<unsigned>(p.d / 64), static_cast<unsigned>(p.count));
  return launch_pdl(transpose_kernel, grid, dim3(256), 0, stream, 1, p);
}

// ------------------------------------------------------------------------------ stats
// Elementwise over (prefix, row) of A and then of B.  The forward sums cover the
// negatives only (Zneg, relative to the row's shift S: tau, or the row's largest logit on
// the max-shifted path); the positive's share is handled here:
//   CLIP/ROWS  term = -log P_ii = softplus(log Zneg + S - s_ii),  Z = Zneg + e^{s_ii - S}
//   SigLIP     term = ln2 * (sum of negatives' softplus in log2 units) + softplus(-x_ii)
// In fp32: every input is an fp32 value and each result is a few roundings from it
// (GB300's fp64 pipe would make this pass, not its memory traffic, the cost).
__device__ __forceinline__ float softplus_f(float y) { return y > 0.f ? y + log1pf(expf(-y)) : log1pf(expf(y)); }

// Sum of the slot partials acc[sl * stride] for sl < slots, in one fixed order: eight
// interleaved fp32 accumulators (eight loads in flight per thread) combined pairwise.  The
// partials are positive fp32 sums themselves, so fp32 keeps the total to a few ulps.
__device__ __forceinline__ float sum_slots(const float* acc, int slots, int64_t stride) {
  float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int sl = 0;
  for (; sl + 8 <= slots; sl += 8) {
#pragma unroll
    for (int u = 0; u < 8; ++u) s[u] += acc[static_cast<int64_t>(sl + u) * stride];
  }
  for (; sl < slots; ++sl) s[0] += acc[static_cast<int64_t>(sl) * stride];
  return ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
}

// Each block also adds its terms per prefix in fp64 (a fixed order within the block) and
// stores the sums in slot blockIdx.x of p.part; the last block to finish adds the slots in
// block order into L_k.
__global__ void __launch_bounds__(kStatsThreads) stats_kernel(const StatsParams p) {
  griddep_enter();
  constexpr float kLn2 = 0.693147180559945309f, kLog2e = 1.442695040888963407f;
  __shared__ double red[kStatsThreads / 32][kMaxPrefix];
  __shared__ bool last_block;
  // a thread's own terms in fp32 (the grid holds up to kStatsBlocks x 256 threads, so a thread
  // adds about n (Na + Nb) / 311296 terms: four at N = 65536), the block and final sums in fp64
  float tsum[kMaxPrefix];
#pragma unroll
  for (int k = 0; k < kMaxPrefix; ++k) tsum[k] = 0.f;
  // adds t to tsum[k] (k is not a compile-time index)
  auto add_term = [&](int k, float t) {
#pragma unroll
    for (int kk = 0; kk < kMaxPrefix; ++kk)
      if (kk == k) tsum[kk] += t;
  };
  const int n = p.n_prefix;
  const float tau = p.sc.t(), bias = p.sc.b();
  const float N = static_cast<float>(p.na);
  const int64_t total_a = static_cast<int64_t>(n) * p.na;
  const int64_t total = total_a + static_cast<int64_t>(n) * p.nb;
  const int64_t nmin = p.na < p.nb ? p.na : p.nb;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const bool side_a = e < total_a;
    const int64_t nrows = side_a ? p.na : p.nb;
    const int64_t ee = side_a ? e : e - total_a;
    const int k = static_cast<int>(ee / nrows);
    const int64_t i = ee % nrows;
    const float* acc = side_a ? p.rowacc_a : p.rowacc_b;
    const int slots = side_a ? p.slots_a : p.slots_b;
    const float w = p.weight[k];
    const bool has_pos = p.diag_pos && i < nmin;
    const float cos_ii = has_pos ? p.pos_cos[k * nmin + i] : 0.f;
    if (p.kind == KIND_SIGLIP) {
      if (!side_a) {
        p.terms_b[ee] = 0.f;
        continue;
      }
      const float s = sum_slots(acc + static_cast<int64_t>(k) * nrows + i, slots, static_cast<int64_t>(n) * nrows);
      // (log2 units)
      const float x_ii = fmaf(tau, cos_ii, bias);
      const float lab = p.pos_term ? p.pos_term[ee] : 0.f;  // -sum of the positives' x
      const float term = s * kLn2 + (has_pos ? softplus_f(-x_ii) : 0.f) + lab;
      p.terms_a[ee] = term;
      add_term(k, term);
      continue;
    }
    if (p.kind == KIND_ROWS && !side_a) {
      p.terms_b[ee] = 0.f;
      continue;
    }
    // sum over negatives of exp(s_ij - S), S the shift of this row (column)
    const float zneg = sum_slots(acc + static_cast<int64_t>(k) * nrows + i, slots, static_cast<int64_t>(n) * nrows);
    const float* shift = side_a ? p.shift_a : p.shift_b;
    const float ush = shift ? shift[ee] : tau * kLog2e;  // log2 units
    const float S = shift ? ush * kLn2 : tau;
    const float s_ii = tau * cos_ii;
    const float e_ii = has_pos ? expf(s_ii - S) : 0.f;
    const float z = zneg + e_ii;
    // (zneg = 0 happens on the shifted path when the positive outweighs every negative
    // beyond fp32's range: log gives -inf and softplus(-inf) = 0, the exact limit)
    const float term = has_pos ? softplus_f(logf(zneg) + S - s_ii) : logf(zneg) + S;
    const float rho = side_a ? p.rinv_a[k * p.na + i] : p.rinv_b[k * p.nb + i];
    float f;
    if (shift) {  // log2(rho alpha / w) - u: the weight pass multiplies by w and takes 2^(x + f)
      const float coef = (p.kind == KIND_CLIP) ? tau / (2.f * N) : tau / N;
      f = log2f(rho * coef / z) - ush;
    } else {
      const float coef = (p.kind == KIND_CLIP) ? w * tau / (2.f * N) : w * tau / N;
      f = rho * coef / z;
    }
    if (side_a) {
      p.zr[ee] = zneg;
      p.fa[ee] = f;
      p.terms_a[ee] = term;
    } else {
      p.zc[ee] = zneg;
      p.fb[ee] = f;
      p.terms_b[ee] = term;
    }
    add_term(k, term);
  }
  // the block's sums: warps, then the warp sums in warp order
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int k = 0; k < kMaxPrefix; ++k) {
    if (k >= n) break;
    double v = static_cast<double>(tsum[k]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[wid][k] = v;
  }
  __syncthreads();
  if (threadIdx.x < n) {
    double v = 0.0;
    for (int w = 0; w < kStatsThreads / 32; ++w) v += red[w][threadIdx.x];
    p.part[static_cast<int64_t>(blockIdx.x) * kMaxPrefix + threadIdx.x] = v;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last_block = atomicAdd(p.done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last_block) return;
  __threadfence();
  // thread t adds slots t, t + 256, ... (every load issued up front), then the block adds the
  // threads' sums as above: a fixed order for a given grid
  double v[kMaxPrefix];
#pragma unroll
  for (int k = 0; k < kMaxPrefix; ++k) v[k] = 0.0;
#pragma unroll
  for (int r = 0; r < (kStatsBlocks + kStatsThreads - 1) / kStatsThreads; ++r) {
    const unsigned b = threadIdx.x + r * kStatsThreads;
    if (b < gridDim.x)
#pragma unroll
      for (int k = 0; k < kMaxPrefix; ++k)
        if (k < n) v[k] += __ldcg(&p.part[static_cast<int64_t>(b) * kMaxPrefix + k]);
  }
  __syncthreads();  // (red is reused)
#pragma unroll
  for (int k = 0; k < kMaxPrefix; ++k) {
    if (k >= n) break;
    double x = v[k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0) red[wid][k] = x;
  }
  __syncthreads();
  if (threadIdx.x < n) {
    double x = 0.0;
    for (int w = 0; w < kStatsThreads / 32; ++w) x += red[w][threadIdx.x];
    const double denom = (p.kind == KIND_CLIP) ? 2.0 * p.na : static_cast<double>(p.na);
    p.loss[threadIdx.x] = static_cast<float>(x / denom);
  }
  if (threadIdx.x == 0) *p.done = 0u;  // ready for the next launch
}

cudaError_t launch_stats(const StatsParams& p, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(p.n_prefix) * (p.na + p.nb);
  int64_t blocks = (total + kStatsThreads - 1) / kStatsThreads;
  if (blocks > kStatsBlocks) blocks = kStatsBlocks;
  return launch_pdl(stats_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kStatsThreads), 0, stream, 1, p);
}

// ------------------------------------------------------------------------------ norm_bwd
// One warp per row of X.  Lanes k < n first form, for prefix k, the row's diagonal
// weight W_ii = W'_ii + w (the positive pair, in fp32), its full row scalar
// C_k = sum_j W_ij cos_ij, and from them the band coefficients
//   r_c = sum_{k>=c} rho_k^2 C_k,  q_c = sum_{k>=c} rho_k sigma_k W_ii,k.
// Then the warp streams the row: dX[d] = G[d] (+ G2[d]) - r_c X[d] + q_c Y[d].
// One side's rows: warp warp_id of n_warps takes rows warp_id, warp_id + n_warps, ...
// HAS_G2: G2 (the split gradient contraction's second part) is added below dimension g2_ld.
template <bool HAS_G2>
__device__ __forceinline__ void norm_bwd_body(const NormBwdParams& p, int64_t warp_id, int64_t n_warps) {
  const int lane = threadIdx.x & 31;
  const int n = p.n_prefix;
  const int pn = p.prefix_end[n - 1];
  const float t_sc = p.sc.t(), b_sc = p.sc.b();
  for (int64_t i = warp_id; i < p.nx; i += n_warps) {
    const bool diag = i < p.nmin;
    float rk = 0.f, qk = 0.f, Ck = 0.f;
    float S = 0.f;  // lane k < n: prefix k's slot sum of x . G^k, off the diagonal
    if (lane < n)
      for (int s = 0; s < p.crow_slots; ++s) S += p.crow[(static_cast<int64_t>(s) * n + lane) * p.nx + i];
    if (p.r5) {
      // merged widest prefixes: prefix n-2's slots hold x . (G^{n-2} + G^{n-1}) below p_{n-2},
      // prefix n-1's only the part above; r5 is prefix n-1's whole sum (from the weight pass)
      const float s_top = __shfl_sync(0xffffffffu, S, n - 1);
      const float r5 = p.r5[i];
      if (lane == n - 1)
        S = r5;
      else if (lane == n - 2)
        S = S + s_top - r5;
    }
    if (lane < n) {
      const int k = lane;
      const float rho = p.rinv_x[k * p.nx + i];
      float C = S;
      float Wd = 0.f;
      if (diag) {
        const float cosd = p.pos_cos[k * p.nmin + i];
        const float sig = p.rinv_y[k * p.ny + i];
        const float w = p.weight[k];
        const double N = static_cast<double>(p.n_total);
        // W_ii = W'_ii + w, written without cancellation: 1 - P_ii = Zneg / Z and
        // sigmoid(x) - 1 = -sigmoid(-x).
        if (p.kind == KIND_SIGLIP) {
          const float x = t_sc * cosd + b_sc;
          const float sg_neg = 1.f / (1.f + expf(x));
          Wd = -static_cast<float>(w * t_sc / N) * sg_neg;
        } else {
          const float tau = t_sc;
          // e^{s_ii - S} for the shift S of each normaliser (tau, or the row's / column's
          // largest logit on the max-shifted path, stored in log2 units)
          const float ln2 = 0.6931471805599453f;
          const float sx = p.shift_x ? p.shift_x[k * p.nx + i] * ln2 : tau;
          const float sy = p.shift_y ? p.shift_y[k * p.ny + i] * ln2 : tau;
          const float ex = expf(tau * cosd - sx), ey = expf(tau * cosd - sy);
          if (p.kind == KIND_CLIP) {
            const float c = static_cast<float>(w * tau / (2.0 * N));
            const float zx = p.z_x[k * p.nx + i], zy = p.z_y[k * p.ny + i];
            Wd = -c * (zx / (zx + ex) + zy / (zy + ey));
          } else {
            const float c = static_cast<float>(w * tau / N);
            const float zq = p.x_is_query ? p.z_x[k * p.nx + i] : p.z_y[k * p.ny + i];
            const float eq = p.x_is_query ? ex : ey;
            Wd = -c * (zq / (zq + eq));
          }
        }
        C += Wd * cosd;
        qk = rho * sig * Wd;
      }
      rk = rho * rho * C;
      Ck = C;
    }
    if (p.csum) {  // sum_k C_k: this row's share of sum_ij W_ij cos_ij (logit-scale gradient)
      float cs = Ck;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) cs += __shfl_xor_sync(0xffffffffu, cs, o);
      if (lane == 0) p.csum[i] = cs;
    }
    // suffix sums over prefixes: band c uses every prefix k >= c
    float rc[kMaxPrefix], qc[kMaxPrefix];
    float ar = 0.f, aq = 0.f;
#pragma unroll
    for (int k = kMaxPrefix - 1; k >= 0; --k) {
      const float r_k = __shfl_sync(0xffffffffu, rk, k);
      const float q_k = __shfl_sync(0xffffffffu, qk, k);
      if (k < n) {
        ar += r_k;
        aq += q_k;
      }
      rc[k] = ar;
      qc[k] = aq;
    }
    const uint16_t* xr = p.X + i * p.d;
    const uint16_t* yr = p.Y + (diag ? i : 0) * p.d;
    const float* gr = p.G + i * p.d;
    float* out = p.dX + i * p.d;
    const float s = p.double_out ? 2.f : 1.f;
    // the row in pieces of 4 x 128 columns: every load of a piece is issued before its first
    // use, so a row waits on memory once per piece, not once per 128 columns
    constexpr int kU = 4;
    for (int base = 0; base < p.d; base += 128 * kU) {
      float4 gv[kU], g2v[HAS_G2 ? kU : 1];
      uint2 xv[kU], yv[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int c4 = base + 128 * u + lane * 4;
        gv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        xv[u] = yv[u] = make_uint2(0u, 0u);
        if constexpr (HAS_G2) g2v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c4 < pn) {
          gv[u] = *reinterpret_cast<const float4*>(gr + c4);
          if constexpr (HAS_G2)
            if (c4 < p.g2_ld) g2v[u] = *reinterpret_cast<const float4*>(p.G2 + i * p.g2_ld + c4);
          xv[u] = *reinterpret_cast<const uint2*>(xr + c4);
          if (diag) yv[u] = *reinterpret_cast<const uint2*>(yr + c4);
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int c4 = base + 128 * u + lane * 4;
        if (c4 >= p.d) continue;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (HAS_G2)
          gv[u] = make_float4(gv[u].x + g2v[u].x, gv[u].y + g2v[u].y, gv[u].z + g2v[u].z, gv[u].w + g2v[u].w);
        if (c4 < pn) {
          const int b = band_of(c4, p.prefix_end, n);
          float r_c = 0.f, q_c = 0.f;
#pragma unroll
          for (int k = 0; k < kMaxPrefix; ++k)
            if (k == b) {
              r_c = rc[k];
              q_c = qc[k];
            }
          o.x = s * (gv[u].x - r_c * bf16_lo(xv[u].x) + q_c * bf16_lo(yv[u].x));
          o.y = s * (gv[u].y - r_c * bf16_hi(xv[u].x) + q_c * bf16_hi(yv[u].x));
          o.z = s * (gv[u].z - r_c * bf16_lo(xv[u].y) + q_c * bf16_lo(yv[u].y));
          o.w = s * (gv[u].w - r_c * bf16_hi(xv[u].y) + q_c * bf16_hi(yv[u].y));
        }
        *reinterpret_cast<float4*>(out + c4) = o;
      }
    }
  }
}

// Both sides in one grid: blocks [0, split) take side a's rows, the rest side b's.
template <bool HAS_G2>
__global__ void __launch_bounds__(256) norm_bwd_kernel(const __grid_constant__ NormBwdParams pa,
                                                       const __grid_constant__ NormBwdParams pb,
                                                       const unsigned split, const int sides) {
  griddep_enter();
  const bool first = blockIdx.x < split;
  const unsigned blk = first ? blockIdx.x : blockIdx.x - split;
  const unsigned nblk = first ? split : gridDim.x - split;
  const int64_t warp_id = (static_cast<int64_t>(blk) * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(nblk) * blockDim.x) >> 5;
  if (first)
    norm_bwd_body<HAS_G2>(pa, warp_id, n_warps);
  else if (sides == 2)
    norm_bwd_body<HAS_G2>(pb, warp_id, n_warps);
}

__global__ void __launch_bounds__(1024) scale_grad_kernel(const ScaleGradParams p) {
  griddep_enter();
  __shared__ double red[2][32];
  const int n = p.n_prefix;
  const float scale = p.sc.t(), bias = p.sc.b();
  double s = 0.0, sb = 0.0;
  if (p.csum)
    for (int64_t i = threadIdx.x; i < p.na; i += blockDim.x) s += p.csum[i];
  if (p.kind == KIND_SIGLIP && p.rowsig) {  // the sigmoid sums exist only when the bias gradient is asked for
    const double N = static_cast<double>(p.na);
    for (int k = 0; k < n; ++k) {
      const double wk = p.weight[k] / N;
      for (int64_t i = threadIdx.x; i < p.na; i += blockDim.x) {
        double neg = 0.0;  // sum over the negatives of row i of sigmoid(x_ij), fixed slot order
        for (int sl = 0; sl < p.sig_slots; ++sl) neg += p.rowsig[(static_cast<int64_t>(sl) * n + k) * p.na + i];
        double pos = 0.0;  // the positive's share: sigmoid(x_ii) - 1 = -sigmoid(-x_ii)
        if (p.lcount) {    // labelled positives were summed as negatives: -1 for each
          pos = -static_cast<double>(p.lcount[i]);
        } else if (i < p.nmin) {
          const double x = static_cast<double>(scale) * p.pos_cos[k * p.nmin + i] + bias;
          pos = -1.0 / (1.0 + exp(x));
        }
        sb += wk * (neg + pos);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, o);
    sb += __shfl_xor_sync(0xffffffffu, sb, o);
  }
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = s;
    red[1][threadIdx.x >> 5] = sb;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    double v = (threadIdx.x < (blockDim.x >> 5)) ? red[0][threadIdx.x] : 0.0;
    double vb = (threadIdx.x < (blockDim.x >> 5)) ? red[1][threadIdx.x] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      v += __shfl_xor_sync(0xffffffffu, v, o);
      vb += __shfl_xor_sync(0xffffffffu, vb, o);
    }
    if (threadIdx.x == 0) {
      // (scale = 0, possible only for SigLIP, gives 0/0: the host refuses a host t = 0, a
      // device one is the caller's to avoid)
      if (p.d_scale) *p.d_scale = static_cast<float>(v / static_cast<double>(scale));
      if (p.d_bias) *p.d_bias = static_cast<float>(p.kind == KIND_SIGLIP ? vb : 0.0);
    }
  }
}

// ------------------------------------------------------------------------------ max_reduce
__global__ void __launch_bounds__(256) max_reduce_kernel(const MaxReduceParams p) {
  griddep_enter();
  const int n = p.n_prefix;
  const int64_t total_a = static_cast<int64_t>(n) * p.na;
  const int64_t total = total_a + (p.v ? static_cast<int64_t>(n) * p.nb : 0);
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float m = -INFINITY;
    if (e < total_a) {
      for (int s = 0; s < p.slots_a; ++s) m = fmaxf(m, p.rowmax[static_cast<int64_t>(s) * total_a + e]);
      p.u[e] = m;
    } else {
      const int64_t ee = e - total_a;
      const int64_t total_b = static_cast<int64_t>(n) * p.nb;
      for (int s = 0; s < p.blocks; ++s) m = fmaxf(m, p.colmax[static_cast<int64_t>(s) * total_b + ee]);
      p.v[ee] = m;
    }
  }
}

cudaError_t launch_max_reduce(const MaxReduceParams& p, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(p.n_prefix) * (p.na + (p.v ? p.nb : 0));
  int64_t blocks = (total + 255) / 256;
  if (blocks > int64_t(8) * current_sm_count()) blocks = int64_t(8) * current_sm_count();
  return launch_pdl(max_reduce_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, 1, p);
}

// ------------------------------------------------------------------------------ labels
// SigLIP with explicit positives (see LabelParams).  The dense passes score every cell as
// a negative; a positive cell differs by the label only: its loss is softplus(-x) =
// softplus(x) - x and its gradient in x is sigmoid(x) - 1 = -sigmoid(-x).  So the loss takes
// -x per positive (terms mode) and the positive cells' weights are rewritten with their
// exact value before the gradient GEMMs read them (patch mode).
// Is i among row j's positives?  (binary search of its increasing ids, within bounds)
__device__ __forceinline__ bool has_mirror(const LabelParams& p, int j, int i, int64_t total) {
  int64_t lo = p.offsets[j], hi = p.offsets[j + 1];
  if (lo < 0 || hi > total || hi < lo) return false;
  while (lo < hi) {
    const int64_t mid = lo + (hi - lo) / 2;
    const int v = p.ids[mid];
    if (v == i) return true;
    if (v < i) lo = mid + 1;
    else hi = mid;
  }
  return false;
}

__global__ void __launch_bounds__(256) labels_kernel(const LabelParams p) {
  griddep_enter();
  const int lane = threadIdx.x & 31;
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int n = p.n_prefix;
  const bool patch = p.W != nullptr;
  const int64_t first = patch ? p.row0 : 0, last = patch ? p.row0 + p.rows : p.na;
  const float t = p.sc.t(), bias = p.sc.b();
  const int pn = p.prefix_end[n - 1];
  const int64_t total = p.offsets[p.na];  // entries of ids (the caller's promise): no read goes past it
  for (int64_t i = first + warp_id; i < last; i += n_warps) {
    const int64_t lo = p.offsets[i];
    int64_t hi = p.offsets[i + 1];
    bool bad = lo < 0 || hi < lo || hi > total;
    if (hi > total) hi = total;
    float xs[kMaxPrefix];
#pragma unroll
    for (int k = 0; k < kMaxPrefix; ++k) xs[k] = 0.f;
    int count = 0;
    const uint4* ra = reinterpret_cast<const uint4*>(p.A + i * p.d);
    int prev = -1;
    for (int64_t q = bad ? hi : lo; q < hi; ++q) {
      const int j = p.ids[q];
      if (j < 0 || j >= p.nb || j <= prev) {  // out of range, repeated or out of order: skipped
        bad = true;
        continue;
      }
      if (p.oneset && (j == i || !has_mirror(p, j, static_cast<int>(i), total))) {
        bad = true;  // one set: no self-pairs, and mirrored cells share their label
        continue;
      }
      prev = j;
      ++count;
      const uint4* rb = reinterpret_cast<const uint4*>(p.B + static_cast<int64_t>(j) * p.d);
      float dab[kMaxPrefix];
#pragma unroll
      for (int k = 0; k < kMaxPrefix; ++k) dab[k] = 0.f;
      for (int ch = lane; ch * 8 < pn; ch += 32) {
        const int b = band_of(ch * 8, p.prefix_end, n);
        const uint4 va = __ldg(ra + ch), vb = __ldg(rb + ch);
        const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
        float sd = 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) sd = fmaf(bf16_lo(wa[u]), bf16_lo(wb[u]), fmaf(bf16_hi(wa[u]), bf16_hi(wb[u]), sd));
#pragma unroll
        for (int k = 0; k < kMaxPrefix; ++k)
          if (k == b) dab[k] += sd;
      }
      float cum = 0.f;
#pragma unroll
      for (int k = 0; k < kMaxPrefix; ++k) {
        if (k >= n) break;
        cum += warp_sum(dab[k]);  // the prefix-k dot product, on every lane
        const float rho = p.rinv_a[k * p.na + i], sig = p.rinv_b[k * p.nb + j];
        const float x = t * (cum * rho * sig) + bias;
        if (!patch) {
          xs[k] += x;
        } else if (lane == 0 && j >= p.col0 && j < p.col0 + p.cols) {  // (this launch's columns)
          const float m = -(1.f / (1.f + expf(x))) * rho * sig *
                          static_cast<float>(p.weight[k] * t / static_cast<double>(p.na));
          const __nv_bfloat16 h = __float2bfloat16_rn(m);
          p.W[(static_cast<int64_t>(k) * p.w_rows_per_prefix + (i - p.row0)) * p.ldw + (j - p.col0)] =
              *reinterpret_cast<const uint16_t*>(&h);
        }
      }
    }
    if (lane == 0) {
      if (bad && p.status) atomicExch(p.status, kStatusBadScalar);
      if (!patch) {
        for (int k = 0; k < n; ++k) p.pos_term[k * p.na + i] = -xs[k];
        p.lcount[i] = static_cast<float>(count);
      }
    }
  }
}

cudaError_t launch_labels(const LabelParams& p, cudaStream_t stream) {
  const int64_t rows = p.W ? p.rows : p.na;
  int64_t blocks = (rows * 32 + 255) / 256;
  if (blocks > int64_t(16) * current_sm_count()) blocks = int64_t(16) * current_sm_count();
  if (blocks < 1) blocks = 1;
  return launch_pdl(labels_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, 1, p);
}

// ------------------------------------------------------------------------------ wait self-test
// The bounded wait of the pipeline kernels, on a barrier that nothing completes: one thread
// gives up after limit_ns and reports as they do (UF_DEVICE_TIMEOUT in *status), and the
// kernel ends, leaving the context usable.
__global__ void wait_selftest_kernel(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
    if (!mbar_wait_abortable(&bar, 0, &abort_flag, limit_ns)) {
      abort_flag = 1;
      atomicExch(status, kStatusTimeout);
    }
  }
}

cudaError_t launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_scale_grad(const ScaleGradParams& p, cudaStream_t stream) {
  return launch_pdl(scale_grad_kernel, dim3(1), dim3(1024), 0, stream, 1, p);
}

cudaError_t launch_norm_bwd(const NormBwdParams* sides, int n_sides, cudaStream_t stream) {
  // blocks in proportion to each side's rows, at most 16 per SM in all
  const int64_t cap = int64_t(16) * current_sm_count();
  int64_t blocks[2] = {0, 0};
  int64_t total = 0;
  for (int s = 0; s < n_sides; ++s) total += (sides[s].nx * 32 + 255) / 256;
  for (int s = 0; s < n_sides; ++s) {
    const int64_t want = (sides[s].nx * 32 + 255) / 256;
    blocks[s] = total > cap ? (want * cap + total - 1) / total : want;
    if (blocks[s] < 1) blocks[s] = 1;
  }
  const unsigned grid = static_cast<unsigned>(blocks[0] + blocks[1]);
  const unsigned split = static_cast<unsigned>(blocks[0]);
  if (sides[0].G2)
    return launch_pdl(norm_bwd_kernel<true>, dim3(grid), dim3(256), 0, stream, 1, sides[0], sides[n_sides - 1], split,
                      n_sides);
  return launch_pdl(norm_bwd_kernel<false>, dim3(grid), dim3(256), 0, stream, 1, sides[0], sides[n_sides - 1], split,
                    n_sides);
}

// ------------------------------------------------------------------------------ r5
// Merged widest prefixes: the weight pass's per-slot row sums and per-32-row-block column sums
// of prefix n-1's C, each added in slot order.
__global__ void __launch_bounds__(256) r5_kernel(const R5Params p) {
  griddep_enter();
  const int64_t total = p.na + p.nb;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const bool side_a = e < p.na;
    const int64_t i = side_a ? e : e - p.na;
    const int64_t rows = side_a ? p.na : p.nb;
    const float* src = side_a ? p.row : p.col;
    const int slots = side_a ? p.row_slots : p.col_parts;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // eight loads in flight
    int s = 0;
    for (; s + 8 <= slots; s += 8)
#pragma unroll
      for (int u = 0; u < 8; ++u) acc[u] += src[static_cast<int64_t>(s + u) * rows + i];
    for (; s < slots; ++s) acc[0] += src[static_cast<int64_t>(s) * rows + i];
    const float v = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
    (side_a ? p.r5_a : p.r5_b)[i] = v;
  }
}

cudaError_t launch_r5(const R5Params& p, cudaStream_t stream) {
  int64_t blocks = (p.na + p.nb + 255) / 256;
  if (blocks > int64_t(8) * current_sm_count()) blocks = int64_t(8) * current_sm_count();
  return launch_pdl(r5_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, 1, p);
}

// Force the module holding these kernels to load now (no lazy loading on the hot path).
cudaError_t aux_kernels_setup() {
  cudaFuncAttributes fa;
  cudaError_t e;
  if ((e = cudaFuncGetAttributes(&fa, prep_kernel)) != cudaSuccess) return e;
  if ((e = cudaFuncGetAttributes(&fa, transpose_kernel)) != cudaSuccess) return e;
  if ((e = cudaFuncGetAttributes(&fa, stats_kernel)) != cudaSuccess) return e;
  if ((e = cudaFuncGetAttributes(&fa, scale_grad_kernel)) != cudaSuccess) return e;
  if ((e = cudaFuncGetAttributes(&fa, max_reduce_kernel)) != cudaSuccess) return e;
  if ((e = cudaFuncGetAttributes(&fa, labels_kernel)) != cudaSuccess) return e;
  if ((e = cudaFuncGetAttributes(&fa, wait_selftest_kernel)) != cudaSuccess) return e;
  if ((e = cudaFuncGetAttributes(&fa, r5_kernel)) != cudaSuccess) return e;
  if ((e = cudaFuncGetAttributes(&fa, norm_bwd_kernel<true>)) != cudaSuccess) return e;
  return cudaFuncGetAttributes(&fa, norm_bwd_kernel<false>);
}

}  // namespace ufc
