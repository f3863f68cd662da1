// tile_kernel.cu -- the fused score kernel: TMA -> shared memory -> tcgen05.mma -> TMEM
// -> per-prefix epilogue, for the forward (row statistics) and the backward (gradient
// GEMM fed by the epilogue's bf16 weights).
//
// One CTA owns 128 rows of X (thread = row in the epilogue) and walks a range of
// 128-row tiles of Y.  For every tile the K dimension (the embedding) is walked band by
// band, a band being the dimensions between two consecutive Matryoshka prefix ends, so
// each band's partial dot products land in their own TMEM accumulator.  The epilogue
// keeps the running sum over bands in registers, so after band k it holds the prefix-k
// dot products of its 64 cells and evaluates prefix k on them.  All prefixes cost one
// pass over K (the blog's "On the Chip" section gets the same effect by subtracting
// bands with the negate-A bit of the instruction descriptor; accumulating each band on
// its own avoids the extra 1984/1024 MMA work that needs).
//
// Forward (MODE_FWD): per row and prefix, over the negatives j != i only, CLIP/ROWS:
// sum_j exp(s_ij - tau) with the fixed shift tau (|cos| <= 1 bounds every logit, so no
// running maximum is needed); SigLIP: sum_j softplus(x_ij) in log2 units.  The positive
// cell is added back in float64 by the statistics kernel, which keeps nearly converged
// rows (loss ~1e-4) free of cancellation.
//
// Backward (MODE_BWD): per cell and prefix the epilogue forms
//     m_ij = rho_i sigma_j W'_ij,   W' = dL/dcos off the diagonal,
// stores it as bf16 in a 128-byte swizzled shared-memory tile, and a second MMA issuer
// accumulates  G[:, slice] += m * Y[:, slice]  in TMEM, for the prefixes that cover the
// CTA's 256-dimension gradient slice.  Diagonal cells are left out of m (their fp32
// correction is applied by the projection kernel).  Row scalars sum_j m_ij dot_ij feed
// the projection term.
//
// Warp roles (384 threads): w0 TMA for the score operands, w1 score-MMA issuer, w2
// gradient-MMA issuer, w3 TMA for the gradient operand (transposed Y), w4..w11 epilogue
// (two warps per TMEM lane quadrant, each taking 64 of the tile's 128 columns).
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace ufc {

constexpr int kThreads = 384;
constexpr int kEpiWarp0 = 4;
constexpr int kEpiThreads = 256;
constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s: far beyond any legitimate wait

constexpr int kStageBytes = kTileRows * kChunk * 2;        // 16 KB: one operand chunk
constexpr int kYtBytes = kSliceDims * kChunk * 2;          // 32 KB: [256 dims x 64 columns]
constexpr int kMBytes = kTileRows * kChunk * 2;            // 16 KB: [128 rows x 64 columns] bf16

template <int MODE>
struct Cfg;
template <>
struct Cfg<MODE_FWD> {
  static constexpr int NS = 6;   // score operand stages
  static constexpr int NB = 4;   // TMEM score accumulators (128 columns each)
  static constexpr int NCOLF = 1;
};
template <>
struct Cfg<MODE_BWD> {
  static constexpr int NS = 3;
  static constexpr int NB = 2;   // + 256 TMEM columns of gradient slice
  static constexpr int NCOLF = 2;
};

template <int MODE>
struct Layout {
  static constexpr int NS = Cfg<MODE>::NS;
  static constexpr int off_x = 0;
  static constexpr int off_y = off_x + NS * kStageBytes;
  static constexpr int off_yt = off_y + NS * kStageBytes;
  static constexpr int off_m = off_yt + (MODE == MODE_BWD ? 2 * kYtBytes : 0);
  static constexpr int off_colf = off_m + (MODE == MODE_BWD ? 2 * kMBytes : 0);
  static constexpr int colf_bytes = 2 * kMaxPrefix * Cfg<MODE>::NCOLF * kTileCols * 4;
  static constexpr int off_rowf = off_colf + colf_bytes;
  static constexpr int rowf_bytes = kMaxPrefix * 3 * kTileRows * 4;
  static constexpr int off_bar = off_rowf + rowf_bytes;
  static constexpr int n_bars = 2 * NS + 2 * Cfg<MODE>::NB + 2 + 2 + 2 + 2 + 1 + 1;
  static constexpr int off_misc = off_bar + n_bars * 8;
  static constexpr int bytes = off_misc + 16 + 4 * kMaxPrefix;
  static constexpr int alloc_bytes = bytes + 1024;  // slack for 1024-byte alignment
};
static_assert(Layout<MODE_FWD>::alloc_bytes <= 232448, "forward shared memory");
static_assert(Layout<MODE_BWD>::alloc_bytes <= 232448, "backward shared memory");

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

struct Barriers {
  uint64_t* s_full;
  uint64_t* s_empty;
  uint64_t* acc_full;
  uint64_t* acc_empty;
  uint64_t* m_full;     // [2] per column half
  uint64_t* m_empty;    // [2]
  uint64_t* yt_full;    // [2]
  uint64_t* yt_empty;   // [2]
  uint64_t* grad_done;  // [1]
  uint64_t* drain;      // [1]
};

__device__ __forceinline__ void record_timeout(const TileParams& p, volatile int* abort_flag) {
  *abort_flag = 1;
  if (p.status) atomicExch(p.status, kStatusTimeout);
}

// Wait that also gives up as soon as another role of this CTA has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}

// ------------------------------------------------------------------------------------
// Epilogue math for one band end (prefix k) over 32 of this thread's cells.
// run[]: prefix-k dot products of row i with those 32 columns; cf1/cf2: the columns'
// factors; col0: their first column within the tile; R1..R3: the row's factors.
template <int MODE, int KIND, bool MASK, bool DIAG>
__device__ __forceinline__ void epi_cells32(const float* run, const float* cf1, const float* cf2, float R1, float R2,
                                            float R3, float L, float b2, int col0, int ncols_valid, int diag_col,
                                            float& acc_row, float& acc_c, uint32_t (&packed)[16]) {
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    float mv[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int jj = j + u;
      const float s1 = cf1[jj];
      const float t = R1 * s1;
      const bool valid = !MASK || (col0 + jj < ncols_valid);
      const bool diag = DIAG && (col0 + jj == diag_col);
      if constexpr (KIND == KIND_SIGLIP) {
        const float x2 = fmaf(t, run[jj], b2);
        const float e = ex2_approx(-fabsf(x2));
        if constexpr (MODE == MODE_FWD) {
          const float l = fmaxf(x2, 0.f) + lg2_approx(1.f + e);
          acc_row += (valid && !diag) ? l : 0.f;
          mv[u] = 0.f;
        } else {
          const float d = 1.f + e;
          const float r = rcp_approx(d);
          const float sig = x2 >= 0.f ? r : e * r;
          float m = sig * (R2 * s1);  // R2 = rho_i * w t / N; s1 = 0 on padded columns
          if (diag) m = 0.f;
          acc_c = fmaf(m, run[jj], acc_c);
          if (R3 != 0.f) {  // R3 != 0 marks the CTA that also sums the SigLIP loss
            const float l = fmaxf(x2, 0.f) + lg2_approx(d);
            acc_row += (valid && !diag) ? l : 0.f;
          }
          mv[u] = m;
        }
      } else {
        const float x = fmaf(t, run[jj], -L);
        const float e = ex2_approx(x);
        if constexpr (MODE == MODE_FWD) {
          acc_row += (valid && !diag) ? e : 0.f;
          mv[u] = 0.f;
        } else {
          // m = e * rho_i * sigma_j * (alpha_i + beta_j) = e * (R2 * s1 + R3 * s2)
          float m = e * fmaf(R2, s1, R3 * cf2[jj]);
          if (diag) m = 0.f;
          acc_c = fmaf(m, run[jj], acc_c);
          mv[u] = m;
        }
      }
    }
    if constexpr (MODE == MODE_BWD) packed[j / 2] = pack_bf16x2(mv[0], mv[1]);
  }
}

// ------------------------------------------------------------------------------------
template <int MODE, int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    tile_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_y,
                const __grid_constant__ CUtensorMap tm_yt, const TileParams p) {
  using LO = Layout<MODE>;
  constexpr int NS = Cfg<MODE>::NS;
  constexpr int NB = Cfg<MODE>::NB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sx = smem + LO::off_x;
  uint8_t* sy = smem + LO::off_y;
  uint8_t* syt = smem + LO::off_yt;
  uint8_t* sm = smem + LO::off_m;
  float* colf = reinterpret_cast<float*>(smem + LO::off_colf);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LO::off_bar);
  Barriers B;
  B.s_full = bars;
  B.s_empty = B.s_full + NS;
  B.acc_full = B.s_empty + NS;
  B.acc_empty = B.acc_full + NB;
  B.m_full = B.acc_empty + NB;
  B.m_empty = B.m_full + 2;
  B.yt_full = B.m_empty + 2;
  B.yt_empty = B.yt_full + 2;
  B.grad_done = B.yt_empty + 2;
  B.drain = B.grad_done + 1;
  float* rowf = reinterpret_cast<float*>(smem + LO::off_rowf);
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(smem + LO::off_misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + LO::off_misc + 4);
  int* pend = reinterpret_cast<int*>(smem + LO::off_misc + 16);  // prefix ends (kernel parameter copy)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kTileRows;
  const int split = blockIdx.y;
  const int slice = blockIdx.z;
  const int d0 = slice * kSliceDims;
  const int n = p.n_prefix;
  const int t_begin = split * p.tiles_per_split;
  const int t_end = min(p.n_col_tiles, t_begin + p.tiles_per_split);
  const int T = t_end - t_begin;
  int nchunk = 0, k_first = 0;  // K chunks of the widest prefix; first prefix reaching the slice
#pragma unroll
  for (int k = 0; k < kMaxPrefix; ++k) {
    if (k < n) nchunk = p.prefix_end[k] / kChunk;
    if (MODE == MODE_BWD && k < n && p.prefix_end[k] <= d0) k_first = k + 1;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&B.s_full[s], 1);
      mbar_init(&B.s_empty[s], 1);
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(&B.acc_full[b], 1);
      mbar_init(&B.acc_empty[b], kEpiThreads / 32);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(&B.m_full[h], 4);
      mbar_init(&B.m_empty[h], 1);
      mbar_init(&B.yt_full[h], 1);
      mbar_init(&B.yt_empty[h], 1);
    }
    mbar_init(B.grad_done, 1);
    mbar_init(B.drain, 1);
    *abort_flag = 0;
#pragma unroll
    for (int k = 0; k < kMaxPrefix; ++k) pend[k] = p.prefix_end[k];
    fence_mbar_init();
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_y);
    if constexpr (MODE == MODE_BWD) tma_prefetch_desc(&tm_yt);
  }
  if (warp == 1) {
    tmem_alloc(tmem_base_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_slot;
  const uint32_t tmem_grad = tmem + NB * kTileCols;  // backward: 256 gradient columns

  if constexpr (MODE == MODE_BWD) {
    // zero the gradient accumulator: every later MMA accumulates onto it
    if (warp >= kEpiWarp0) {
      const int q = warp & 3, h = (warp - kEpiWarp0) >> 2;
      const uint32_t base = tmem_grad + (static_cast<uint32_t>(q * 32) << 16) + h * 128;
#pragma unroll
      for (int c = 0; c < 128; c += 32) tmem_st32_zero(base + c);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  if (T > 0 && warp == 0 && lane == 0) {
    // ---------------------------------------------------------- score operand producer
    uint32_t it = 0;
    bool ok = true;
    for (int t = 0; t < T && ok; ++t) {
      const int j0 = (t_begin + t) * kTileCols;
      for (int c = 0; c < nchunk; ++c, ++it) {
        const uint32_t s = it % NS, ph = (it / NS) & 1;
        if (!wait_or_abort(&B.s_empty[s], ph ^ 1, abort_flag)) {
          record_timeout(p, abort_flag);
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&B.s_full[s], 2 * kStageBytes);
        tma_load_2d(sx + s * kStageBytes, &tm_x, &B.s_full[s], c * kChunk, static_cast<int>(i0));
        tma_load_2d(sy + s * kStageBytes, &tm_y, &B.s_full[s], c * kChunk, j0);
      }
    }
    // drain: let every copy this thread issued land before the CTA can exit
    for (uint32_t k = 0; k < NS && k < it; ++k) {
      const uint32_t q = it - 1 - k;
      mbar_wait(&B.s_full[q % NS], (q / NS) & 1, kWaitLimitNs);
    }
  } else if (T > 0 && warp == 1 && lane == 0) {
    // ---------------------------------------------------------- score MMA issuer
    const uint32_t idesc = idesc_bf16_f32(kTileRows, kTileCols);
    uint32_t it = 0, ait = 0;
    bool ok = true;
    for (int t = 0; t < T && ok; ++t) {
      int c = 0;
      for (int b = 0; b < n && ok; ++b, ++ait) {
        const uint32_t ab = ait % NB, aph = (ait / NB) & 1;
        if (!wait_or_abort(&B.acc_empty[ab], aph ^ 1, abort_flag)) {
          record_timeout(p, abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + ab * kTileCols;
        const int c_end = pend[b] / kChunk;
        const int c_first = c;
        for (; c < c_end; ++c, ++it) {
          const uint32_t s = it % NS, ph = (it / NS) & 1;
          if (!wait_or_abort(&B.s_full[s], ph, abort_flag)) {
            record_timeout(p, abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ax = smem_u32(sx + s * kStageBytes), ay = smem_u32(sy + s * kStageBytes);
#pragma unroll
          for (int kk = 0; kk < kChunk / 16; ++kk) {
            umma_bf16(d_tmem, sdesc_kmajor_sw128(ax + kk * 32), sdesc_kmajor_sw128(ay + kk * 32), idesc,
                      (c != c_first || kk != 0) ? 1u : 0u);
          }
          umma_commit(&B.s_empty[s]);
        }
        if (ok) umma_commit(&B.acc_full[ab]);
      }
    }
    // drain: wait until every MMA this thread issued has finished
    umma_commit(B.drain);
    mbar_wait(B.drain, 0, kWaitLimitNs);
  } else if (MODE == MODE_BWD && T > 0 && warp == 2 && lane == 0) {
    // ---------------------------------------------------------- gradient MMA issuer
    uint32_t cnt = 0;
    bool ok = true;
    for (int t = 0; t < T && ok; ++t) {
      for (int k = k_first; k < n && ok; ++k, ++cnt) {
        const int nk = min(pend[k], d0 + kSliceDims) - d0;  // multiple of 64, <= 256
        const uint32_t idesc = idesc_bf16_f32(kTileRows, static_cast<uint32_t>(nk));
        for (int h = 0; h < 2; ++h) {
          if (!wait_or_abort(&B.m_full[h], cnt & 1, abort_flag) ||
              (k == k_first && !wait_or_abort(&B.yt_full[h], t & 1, abort_flag))) {
            record_timeout(p, abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t am = smem_u32(sm + h * kMBytes), ayt = smem_u32(syt + h * kYtBytes);
#pragma unroll
          for (int kk = 0; kk < kChunk / 16; ++kk)
            umma_bf16(tmem_grad, sdesc_kmajor_sw128(am + kk * 32), sdesc_kmajor_sw128(ayt + kk * 32), idesc, 1u);
          umma_commit(&B.m_empty[h]);
          if (k == n - 1) umma_commit(&B.yt_empty[h]);
        }
      }
    }
    umma_commit(B.grad_done);
    mbar_wait(B.grad_done, 0, kWaitLimitNs);
  } else if (MODE == MODE_BWD && T > 0 && warp == 3 && lane == 0) {
    // ---------------------------------------------------------- gradient operand producer
    bool ok = true;
    for (int t = 0; t < T && ok; ++t) {
      const int j0 = (t_begin + t) * kTileCols;
      for (int h = 0; h < 2; ++h) {
        if (!wait_or_abort(&B.yt_empty[h], (t & 1) ^ 1, abort_flag)) {
          record_timeout(p, abort_flag);
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&B.yt_full[h], kYtBytes);
        tma_load_2d(syt + h * kYtBytes, &tm_yt, &B.yt_full[h], j0 + h * kChunk, d0);
      }
    }
    if (T > 0) {
      const int tl = T - 1;
      for (int h = 0; h < 2; ++h) mbar_wait(&B.yt_full[h], tl & 1, kWaitLimitNs);
    }
  } else if (warp >= kEpiWarp0) {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;                   // TMEM lane quadrant
    const int h = (warp - kEpiWarp0) >> 2;    // column half of the tile
    const int r = q * 32 + lane;              // row within the tile
    const int64_t gi = i0 + r;
    const bool row_ok = gi < p.nx;
    const int etid = threadIdx.x - kEpiWarp0 * 32;
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    constexpr int NCF = Cfg<MODE>::NCOLF;
    constexpr int CF_STRIDE = kMaxPrefix * NCF * kTileCols;  // floats per column-factor buffer

    // Row factors of this CTA's rows, once: R1 = L rho, and for the backward
    // CLIP/ROWS: R2 = rho alpha (prescaled), R3 = rho; SigLIP: R2 = rho w t / N, R3 = loss flag.
    if (h == 0) {
#pragma unroll
      for (int k = 0; k < kMaxPrefix; ++k) {
        if (k >= n) break;
        const float rho = row_ok ? p.rinv_x[k * p.nx + gi] : 0.f;
        float R2 = 0.f, R3 = 0.f;
        if constexpr (MODE == MODE_BWD) {
          if constexpr (KIND == KIND_SIGLIP) {
            R2 = rho * p.m_scale[k];
            R3 = (slice == 0 && p.rowacc) ? 1.f : 0.f;
          } else {
            R2 = (row_ok && p.alpha_x) ? p.alpha_x[k * p.nx + gi] : 0.f;
            R3 = rho;
          }
        }
        rowf[(k * 3 + 0) * kTileRows + r] = p.L * rho;
        rowf[(k * 3 + 1) * kTileRows + r] = R2;
        rowf[(k * 3 + 2) * kTileRows + r] = R3;
      }
    }
    // Column factors of tile t land in colf[t & 1] by cp.async, one tile ahead.
    auto prefetch_colf = [&](int t) {
      const int64_t j0 = static_cast<int64_t>(t_begin + t) * kTileCols;
      float* cf = colf + (t & 1) * CF_STRIDE;
      for (int e = etid; e < n * kTileCols; e += kEpiThreads) {
        const int k = e / kTileCols, c = e % kTileCols;
        const int64_t gj = j0 + c;
        const bool v = gj < p.ny;
        const int64_t idx = v ? k * p.ny + gj : 0;
        cp_async4(cf + (k * NCF + 0) * kTileCols + c, p.rinv_y + idx, v ? 4u : 0u);
        if constexpr (NCF > 1) {
          const bool vb = v && p.beta_y;
          cp_async4(cf + (k * NCF + 1) * kTileCols + c, vb ? p.beta_y + idx : p.rinv_y, vb ? 4u : 0u);
        }
      }
    };
    if (T > 0) prefetch_colf(0);
    cp_async_commit();

    float acc_row[kMaxPrefix], acc_c[kMaxPrefix];
#pragma unroll
    for (int k = 0; k < kMaxPrefix; ++k) acc_row[k] = acc_c[k] = 0.f;
    uint32_t ait = 0, mcnt = 0;
    bool ok = true;
    // every epilogue warp runs all T iterations (an aborted warp skips the work but still
    // meets the named barriers, so the others cannot hang on them)
    for (int t = 0; t < T; ++t) {
      const int64_t j0 = static_cast<int64_t>(t_begin + t) * kTileCols;
      named_bar_sync(1, kEpiThreads);  // everyone is done with tile t-1: colf[(t+1) & 1] is free
      if (t + 1 < T) prefetch_colf(t + 1);
      cp_async_commit();
      cp_async_wait<1>();               // this thread's copies for tile t have landed
      named_bar_sync(1, kEpiThreads);  // ... and everyone else's
      if (!ok) continue;
      const float* cf = colf + (t & 1) * CF_STRIDE;
      const int64_t left = p.ny - j0;
      const int ncols_valid = left < kTileCols ? static_cast<int>(left) : kTileCols;
      const bool masked = ncols_valid < kTileCols;
      const bool diag_tile = j0 == i0;  // the tile holds the positive pairs (i, i)
      const int diag_col = r - h * 64;  // column (within my 64) of the diagonal cell
      float run[64];
      for (int b = 0; b < n && ok; ++b, ++ait) {
        const uint32_t ab = ait % NB, aph = (ait / NB) & 1;
        if (!wait_or_abort(&B.acc_full[ab], aph, abort_flag)) {
          record_timeout(p, abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        {
          float v[64];
          tmem_ld64(tmem + lane_addr + ab * kTileCols + h * 64, v);
#pragma unroll
          for (int j = 0; j < 64; ++j) run[j] = (b == 0) ? v[j] : run[j] + v[j];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.acc_empty[ab]);

        if (MODE == MODE_BWD && b < k_first) continue;  // prefix does not reach this slice
        const int k = b;
        const float R1 = rowf[(k * 3 + 0) * kTileRows + r];
        const float R2 = rowf[(k * 3 + 1) * kTileRows + r];
        const float R3 = rowf[(k * 3 + 2) * kTileRows + r];
        const float* c1 = cf + (k * NCF + 0) * kTileCols + h * 64;
        const float* c2 = cf + (k * NCF + (NCF > 1 ? 1 : 0)) * kTileCols + h * 64;
        uint8_t* mt = sm + h * kMBytes + (r >> 3) * 1024 + (r & 7) * 128;
        if constexpr (MODE == MODE_BWD) {
          // the gradient MMA must have consumed the previous weights of this half
          if (!wait_or_abort(&B.m_empty[h], (mcnt & 1) ^ 1, abort_flag)) {
            record_timeout(p, abort_flag);
            ok = false;
            break;
          }
        }
        float ar = 0.f, ac = 0.f;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t packed[16];
          const int col0 = h * 64 + hh * 32;
          const float* rr = run + hh * 32;
          if (masked) {
            if (diag_tile)
              epi_cells32<MODE, KIND, true, true>(rr, c1 + hh * 32, c2 + hh * 32, R1, R2, R3, p.L, p.b2, col0 - h * 64,
                                                  ncols_valid - h * 64, diag_col, ar, ac, packed);
            else
              epi_cells32<MODE, KIND, true, false>(rr, c1 + hh * 32, c2 + hh * 32, R1, R2, R3, p.L, p.b2, col0 - h * 64,
                                                   ncols_valid - h * 64, diag_col, ar, ac, packed);
          } else {
            if (diag_tile)
              epi_cells32<MODE, KIND, false, true>(rr, c1 + hh * 32, c2 + hh * 32, R1, R2, R3, p.L, p.b2, col0 - h * 64,
                                                   ncols_valid - h * 64, diag_col, ar, ac, packed);
            else
              epi_cells32<MODE, KIND, false, false>(rr, c1 + hh * 32, c2 + hh * 32, R1, R2, R3, p.L, p.b2,
                                                    col0 - h * 64, ncols_valid - h * 64, diag_col, ar, ac, packed);
          }
          if constexpr (MODE == MODE_BWD) {
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
              const int chunk = hh * 4 + qd;  // 16-byte chunk of the 128-byte swizzled row
              *reinterpret_cast<uint4*>(mt + ((chunk ^ (r & 7)) << 4)) =
                  make_uint4(packed[4 * qd], packed[4 * qd + 1], packed[4 * qd + 2], packed[4 * qd + 3]);
            }
          }
        }
#pragma unroll
        for (int kk = 0; kk < kMaxPrefix; ++kk)
          if (kk == k) {
            acc_row[kk] += ar;
            acc_c[kk] += ac;
          }
        if constexpr (MODE == MODE_BWD) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&B.m_full[h]);
          ++mcnt;
        }
      }
    }
    cp_async_wait<0>();
    // ---- outputs
    if (row_ok && ok) {
      const int slot = split * 2 + h;
      if (p.rowacc && (MODE == MODE_FWD || (KIND == KIND_SIGLIP && slice == 0))) {
        for (int k = 0; k < n; ++k) p.rowacc[(static_cast<int64_t>(slot) * n + k) * p.nx + gi] = acc_row[k];
      }
      if (MODE == MODE_BWD && slice == 0) {
        for (int k = 0; k < n; ++k) p.crow[(static_cast<int64_t>(slot) * n + k) * p.nx + gi] = acc_c[k];
      }
    }
    if constexpr (MODE == MODE_BWD) {
      if (T > 0 && ok && wait_or_abort(B.grad_done, 0, abort_flag)) {
        tc_fence_after();
        float* g = p.grad + (static_cast<int64_t>(split) * p.nx + gi) * p.d;
        for (int c = 0; c < 128; c += 32) {
          float v[32];
          tmem_ld32(tmem_grad + lane_addr + h * 128 + c, v);
          const int dcol = d0 + h * 128 + c;
          if (row_ok && dcol < p.d) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(g + dcol + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
          }
        }
      } else if (T > 0 && ok) {
        record_timeout(p, abort_flag);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------------------------ host
template <int MODE, int KIND>
static cudaError_t setup_one() {
  return cudaFuncSetAttribute(tile_kernel<MODE, KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Layout<MODE>::alloc_bytes);
}

cudaError_t tile_kernel_setup() {
  cudaError_t e;
  if ((e = setup_one<MODE_FWD, KIND_CLIP>()) != cudaSuccess) return e;
  if ((e = setup_one<MODE_FWD, KIND_SIGLIP>()) != cudaSuccess) return e;
  if ((e = setup_one<MODE_FWD, KIND_ROWS>()) != cudaSuccess) return e;
  if ((e = setup_one<MODE_BWD, KIND_CLIP>()) != cudaSuccess) return e;
  if ((e = setup_one<MODE_BWD, KIND_SIGLIP>()) != cudaSuccess) return e;
  if ((e = setup_one<MODE_BWD, KIND_ROWS>()) != cudaSuccess) return e;
  return cudaSuccess;
}

template <int MODE, int KIND>
static cudaError_t launch_one(const CUtensorMap& tm_x, const CUtensorMap& tm_y, const CUtensorMap& tm_yt,
                              const TileParams& p, dim3 grid, cudaStream_t stream) {
  tile_kernel<MODE, KIND><<<grid, kThreads, Layout<MODE>::alloc_bytes, stream>>>(tm_x, tm_y, tm_yt, p);
  return cudaGetLastError();
}

cudaError_t launch_tile(int mode, int kind, const CUtensorMap& tm_x, const CUtensorMap& tm_y,
                        const CUtensorMap& tm_yt, const TileParams& p, dim3 grid, cudaStream_t stream) {
  if (mode == MODE_FWD) {
    if (kind == KIND_CLIP) return launch_one<MODE_FWD, KIND_CLIP>(tm_x, tm_y, tm_yt, p, grid, stream);
    if (kind == KIND_SIGLIP) return launch_one<MODE_FWD, KIND_SIGLIP>(tm_x, tm_y, tm_yt, p, grid, stream);
    return launch_one<MODE_FWD, KIND_ROWS>(tm_x, tm_y, tm_yt, p, grid, stream);
  }
  if (kind == KIND_CLIP) return launch_one<MODE_BWD, KIND_CLIP>(tm_x, tm_y, tm_yt, p, grid, stream);
  if (kind == KIND_SIGLIP) return launch_one<MODE_BWD, KIND_SIGLIP>(tm_x, tm_y, tm_yt, p, grid, stream);
  return launch_one<MODE_BWD, KIND_ROWS>(tm_x, tm_y, tm_yt, p, grid, stream);
}

}  // namespace ufc
