// bwd_kernel.cu -- backward of the Matryoshka contrastive loss with 128 x 256 score tiles.
//
// A CTA owns 128 rows of X, one 256-dimension slice [d0, d0 + 256) of their gradient, and a
// range of 256-row tiles of Y.  Per tile:
//   * the score MMA (128 x 256 x 16 tcgen05 steps, full tensor rate) walks K band by band
//     into one TMEM accumulator; after band k the epilogue reads the prefix-k snapshot and
//     releases the accumulator for band k + 1;
//   * for every prefix k that reaches the slice, the epilogue forms the bf16 weights
//       m_ij = rho_i sigma_j W'_ij   (W' = dL/dcos off the diagonal)
//     one 64-column chunk per column quarter, and the gradient MMA issuer accumulates
//       G[:, d0 : d0 + nk] += m^k_chunk * Y[chunk, d0 : d0 + nk]      (nk = min(p_k, d0+256) - d0)
//     in the other 256 TMEM columns, the transposed Y chunk streamed by TMA per (prefix, chunk);
//   * the row scalar sum_j m_ij dot_ij of every prefix feeds the projection term, and the CTAs
//     of the first slice also sum the SigLIP loss.
// Diagonal cells are left out of m; their fp32 correction is applied by the projection kernel.
// The gradient slice needs all K of the scores, so each of the ceil(p_n / 256) slices
// recomputes them: the gradient of 128 rows over 1024 dimensions would need 512 KB of
// TMEM, and one SM has 256 KB.
//
// Warps (640 threads): 0 score-operand TMA, 1 score MMA, 2 gradient MMA, 3 transposed-Y TMA,
// 4..19 epilogue (warp w reads TMEM lanes 32 (w % 4).. and one 64-column quarter).
#include <cuda_bf16.h>

#include "launch.h"
#include "ptx.cuh"

namespace ufc {
namespace bwd {

constexpr int kCols = kBwdCols;
constexpr int kThreads = 640;
constexpr int kEpiWarp0 = 4;
constexpr int kEpiWarps = 16;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kNS = 2;                              // score operand stages
constexpr int kXBytes = kTileRows * kChunk * 2;     // 16 KB
constexpr int kYBytes = kCols * kChunk * 2;         // 32 KB
constexpr int kMBytes = kTileRows * kChunk * 2;     // 16 KB: one 64-column chunk of weights
constexpr int kNM = 2;                              // weight-chunk slots
constexpr int kYtBytes = kSliceDims * kChunk * 2;   // 32 KB: [256 dims x 64 columns]
constexpr int kNYt = 2;                             // transposed-Y slots
constexpr int kYtBox = kBwdYtBox;                   // dims per transposed-Y TMA box
constexpr uint64_t kWaitLimitNs = 4000000000ull;

constexpr int kColfBytes = kMaxPrefix * 2 * kCols * 4;  // [prefix][sigma, sigma*beta][256 columns]

constexpr int off_x = 0;
constexpr int off_y = off_x + kNS * kXBytes;
constexpr int off_m = off_y + kNS * kYBytes;
constexpr int off_yt = off_m + kNM * kMBytes;
constexpr int off_colf = off_yt + kNYt * kYtBytes;  // two buffers: tile t and tile t + 1
constexpr int off_bar = off_colf + 2 * kColfBytes;
constexpr int n_bars = 2 * kNS + 2 + kNM + 4 + 2 * kNYt + 2;
constexpr int off_pend = off_bar + n_bars * 8;      // int[kMaxPrefix]: prefix ends
constexpr int off_misc = off_pend + 4 * kMaxPrefix;
constexpr int smem_bytes = off_misc + 16 + 1024;
static_assert(smem_bytes <= 232448, "backward shared memory");

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
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

__device__ __forceinline__ void fail(const TileParams& p, volatile int* abort_flag) {
  *abort_flag = 1;
  if (p.status) atomicExch(p.status, kStatusTimeout);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 8 cells of one snapshot: their weights as four packed bf16 pairs, the row scalar and
// the SigLIP loss.  c1, c2: shared addresses of the 8 columns' factors.
template <int KIND, bool CHECK>
__device__ __forceinline__ uint4 bwd_cells8(const float* dot, uint32_t c1, uint32_t c2, float R1, float R2, float R3,
                                           float L, float b2, int col0, int ncols, int dcol, bool row_ok,
                                           float& acc_c, float& acc_l) {
  const float4 s1a = ld_shared_v4f(c1), s1b = ld_shared_v4f(c1 + 16);
  const float s1v[8] = {s1a.x, s1a.y, s1a.z, s1a.w, s1b.x, s1b.y, s1b.z, s1b.w};
  float s2v[8];
  if constexpr (KIND != KIND_SIGLIP) {
    const float4 s2a = ld_shared_v4f(c2), s2b = ld_shared_v4f(c2 + 16);
    s2v[0] = s2a.x; s2v[1] = s2a.y; s2v[2] = s2a.z; s2v[3] = s2a.w;
    s2v[4] = s2b.x; s2v[5] = s2b.y; s2v[6] = s2b.z; s2v[7] = s2b.w;
  }
  uint32_t packed[4];
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    float mv[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int jj = j + u;
      const float s1 = s1v[jj];
      const float t = R1 * s1;
      float m;
      bool keep = true;
      if constexpr (CHECK) {
        const int col = col0 + jj;
        keep = row_ok && col < ncols && col != dcol;
      }
      if constexpr (KIND == KIND_SIGLIP) {
        const float x2 = fmaf(t, dot[jj], b2);
        const float e = ex2_approx(-fabsf(x2));
        const float d = 1.f + e;
        const float r = rcp_approx(d);
        const float sig = x2 >= 0.f ? r : e * r;
        m = sig * (R2 * s1);
        if (R3 != 0.f) {  // the slice that also sums the SigLIP loss
          const float l = fmaxf(x2, 0.f) + lg2_approx(d);
          acc_l += keep ? l : 0.f;
        }
      } else {
        const float e = ex2_approx(fmaf(t, dot[jj], -L));
        m = e * fmaf(R2, s1, R3 * s2v[jj]);
      }
      if constexpr (CHECK) m = keep ? m : 0.f;
      acc_c = fmaf(m, dot[jj], acc_c);
      mv[u] = m;
    }
    packed[j / 2] = pack_bf16x2(mv[0], mv[1]);
  }
  return make_uint4(packed[0], packed[1], packed[2], packed[3]);
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_y,
               const __grid_constant__ CUtensorMap tm_yt, const TileParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sx = smem + off_x;
  uint8_t* sy = smem + off_y;
  uint8_t* sm = smem + off_m;
  uint8_t* syt = smem + off_yt;
  int* pend = reinterpret_cast<int*>(smem + off_pend);
  uint64_t* s_full = reinterpret_cast<uint64_t*>(smem + off_bar);
  uint64_t* s_empty = s_full + kNS;
  uint64_t* acc_full = s_empty + kNS;   // [1]
  uint64_t* acc_empty = acc_full + 1;   // [1]
  uint64_t* m_full = acc_empty + 1;   // [kNM] per slot
  uint64_t* m_done = m_full + kNM;    // [4] per column quarter: its chunk was consumed
  uint64_t* yt_full = m_done + 4;
  uint64_t* yt_empty = yt_full + kNYt;
  uint64_t* grad_done = yt_empty + kNYt;
  uint64_t* drain = grad_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + off_misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + off_misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kTileRows;
  const int split = blockIdx.y;
  const int slice = blockIdx.z;
  const int d0 = slice * kSliceDims;
  const int n = p.n_prefix;
  const int t_begin = split * p.tiles_per_split;
  const int T = min(p.n_col_tiles, t_begin + p.tiles_per_split) - t_begin;
  int k_first = 0;  // first prefix whose weights reach this slice
#pragma unroll
  for (int k = 0; k < kMaxPrefix; ++k)
    if (k < n && p.prefix_end[k] <= d0) k_first = k + 1;
  const int n_act = n - k_first;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kEpiWarps);
    for (int s = 0; s < kNM; ++s) mbar_init(&m_full[s], 4);  // the four warps of one column quarter
    for (int s = 0; s < 4; ++s) mbar_init(&m_done[s], 1);
    for (int s = 0; s < kNYt; ++s) {
      mbar_init(&yt_full[s], 1);
      mbar_init(&yt_empty[s], 1);
    }
    mbar_init(grad_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
#pragma unroll
    for (int k = 0; k < kMaxPrefix; ++k) pend[k] = p.prefix_end[k];
    fence_mbar_init();
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_y);
    tma_prefetch_desc(&tm_yt);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;         // columns 0..255: scores
  const uint32_t tmem_grad = tmem + kCols;  // columns 256..511: gradient slice
  if (warp >= kEpiWarp0) {  // zero the gradient accumulator: every later MMA accumulates onto it
    const int q = warp & 3, cq = (warp - kEpiWarp0) >> 2;
    const uint32_t base = tmem_grad + (static_cast<uint32_t>(q * 32) << 16) + cq * 64;
    tmem_st32_zero(base);
    tmem_st32_zero(base + 32);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (T > 0 && warp == 0 && lane == 0) {
    // ------------------------------------------------------------- score operand producer
    const int nchunk = pend[n - 1] / kChunk;
    uint32_t it = 0;
    bool ok = true;
    for (int t = 0; t < T && ok; ++t) {
      const int j0 = (t_begin + t) * kCols;
      for (int c = 0; c < nchunk; ++c, ++it) {
        const uint32_t st = it % kNS, ph = (it / kNS) & 1;
        if (!wait_bounded(&s_empty[st], ph ^ 1, abort_flag)) {
          fail(p, abort_flag);
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&s_full[st], kXBytes + kYBytes);
        tma_load_2d(sx + st * kXBytes, &tm_x, &s_full[st], c * kChunk, static_cast<int>(i0));
        tma_load_2d(sy + st * kYBytes, &tm_y, &s_full[st], c * kChunk, j0);
      }
    }
    for (uint32_t k = 0; k < kNS && k < it; ++k) {
      const uint32_t q = it - 1 - k;
      mbar_wait(&s_full[q % kNS], (q / kNS) & 1, kWaitLimitNs);
    }
  } else if (T > 0 && warp == 1 && lane == 0) {
    // ------------------------------------------------------------- score MMA issuer
    const uint32_t idesc = idesc_bf16_f32(kTileRows, kCols);
    uint32_t it = 0, snap = 0;
    bool ok = true;
    for (int t = 0; t < T && ok; ++t) {
      int c = 0;
      // snapshots are taken only at the ends of the prefixes that reach this slice
      for (int b = k_first; b < n && ok; ++b, ++snap) {
        // the epilogue must have read the previous snapshot out of the accumulator
        if (snap > 0 && !wait_bounded(acc_empty, (snap - 1) & 1, abort_flag)) {
          fail(p, abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        for (; c < pend[b] / kChunk; ++c, ++it) {
          const uint32_t st = it % kNS, ph = (it / kNS) & 1;
          if (!wait_bounded(&s_full[st], ph, abort_flag)) {
            fail(p, abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ax = smem_u32(sx + st * kXBytes), ay = smem_u32(sy + st * kYBytes);
#pragma unroll
          for (int kk = 0; kk < kChunk / 16; ++kk)  // a tile's first step starts fresh, bands accumulate
            umma_bf16(tmem, sdesc_kmajor_sw128(ax + kk * 32), sdesc_kmajor_sw128(ay + kk * 32), idesc,
                      (c != 0 || kk != 0) ? 1u : 0u);
          umma_commit(&s_empty[st]);
        }
        if (ok) umma_commit(acc_full);
      }
    }
    umma_commit(drain);
    mbar_wait(drain, 0, kWaitLimitNs);
  } else if (T > 0 && warp == 2 && lane == 0) {
    // ------------------------------------------------------------- gradient MMA issuer
    uint32_t seq = 0;  // (tile, prefix, quarter) chunk sequence shared with the epilogue and Y^T producer
    bool ok = true;
    for (int t = 0; t < T && ok; ++t) {
      for (int k = k_first; k < n && ok; ++k) {
        const int nk = min(pend[k], d0 + kSliceDims) - d0;
        const uint32_t idesc = idesc_bf16_f32(kTileRows, static_cast<uint32_t>(nk));
        for (int cq = 0; cq < 4; ++cq, ++seq) {
          const uint32_t ms = seq % kNM, mph = (seq / kNM) & 1;
          const uint32_t ys = seq % kNYt, yph = (seq / kNYt) & 1;
          if (!wait_bounded(&m_full[ms], mph, abort_flag) || !wait_bounded(&yt_full[ys], yph, abort_flag)) {
            fail(p, abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t am = smem_u32(sm + ms * kMBytes), ayt = smem_u32(syt + ys * kYtBytes);
#pragma unroll
          for (int kk = 0; kk < kChunk / 16; ++kk)
            umma_bf16(tmem_grad, sdesc_kmajor_sw128(am + kk * 32), sdesc_kmajor_sw128(ayt + kk * 32), idesc, 1u);
          umma_commit(&m_done[cq]);
          umma_commit(&yt_empty[ys]);
        }
      }
    }
    umma_commit(grad_done);
    mbar_wait(grad_done, 0, kWaitLimitNs);
  } else if (T > 0 && warp == 3 && lane == 0) {
    // ------------------------------------------------------------- transposed-Y producer
    uint32_t seq = 0;
    bool ok = true;
    for (int t = 0; t < T && ok; ++t) {
      const int j0 = (t_begin + t) * kCols;
      for (int k = k_first; k < n && ok; ++k) {
        const int nk = min(pend[k], d0 + kSliceDims) - d0;
        for (int cq = 0; cq < 4; ++cq, ++seq) {
          const uint32_t ys = seq % kNYt, yph = (seq / kNYt) & 1;
          if (!wait_bounded(&yt_empty[ys], yph ^ 1, abort_flag)) {
            fail(p, abort_flag);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&yt_full[ys], nk * kChunk * 2);
          for (int r0 = 0; r0 < nk; r0 += kYtBox)
            tma_load_2d(syt + ys * kYtBytes + r0 * kChunk * 2, &tm_yt, &yt_full[ys], j0 + cq * kChunk, d0 + r0);
        }
      }
    }
    for (uint32_t k = 0; k < kNYt && k < seq; ++k) {
      const uint32_t q = seq - 1 - k;
      mbar_wait(&yt_full[q % kNYt], (q / kNYt) & 1, kWaitLimitNs);
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------- epilogue
    const int q = warp & 3;                    // TMEM lane quadrant
    const int cq = (warp - kEpiWarp0) >> 2;    // column quarter
    const int r = q * 32 + lane;
    const int64_t gi = i0 + r;
    const bool row_ok = gi < p.nx;
    const int etid = threadIdx.x - kEpiWarp0 * 32;
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t colf_s = smem_u32(smem + off_colf);
    const uint32_t m_row = smem_u32(sm) + (r >> 3) * 1024 + (r & 7) * 128;  // row r of a weight chunk
    const uint32_t swz = r & 7;
    // column factors of tile t land in buffer t & 1 by cp.async, one tile ahead
    auto prefetch_colf = [&](int t) {
      const int64_t j0 = static_cast<int64_t>(t_begin + t) * kCols;
      const uint32_t dst = colf_s + (t & 1) * kColfBytes;
      for (int e = etid; e < n_act * 2 * kCols; e += kEpiThreads) {
        const int ka = e / (2 * kCols), f = (e / kCols) & 1, c = e % kCols;
        const int64_t gj = j0 + c;
        const float* src = f == 0 ? p.rinv_y : p.beta_y;
        const bool v = src != nullptr && gj < p.ny;
        cp_async4_u32(dst + e * 4, v ? src + static_cast<int64_t>(k_first + ka) * p.ny + gj : p.rinv_y, v ? 4u : 0u);
      }
    };
    // raw row factors (rho_i, and rho_i alpha_i for CLIP/ROWS) of the next prefix to
    // process, loaded one prefix ahead
    float n_rho = 0.f, n_alpha = 0.f;
    auto load_row = [&](int k) {
      n_rho = row_ok ? p.rinv_x[static_cast<int64_t>(k) * p.nx + gi] : 0.f;
      if constexpr (KIND != KIND_SIGLIP)
        n_alpha = (row_ok && p.alpha_x) ? p.alpha_x[static_cast<int64_t>(k) * p.nx + gi] : 0.f;
    };
    if (T > 0) {
      prefetch_colf(0);
      load_row(k_first);
    }
    cp_async_commit();
    // row scalars (and SigLIP loss sums) go to this thread's own slot, written by the
    // first tile and accumulated in place by the later ones; only the first slice keeps them
    const bool keep_rows = slice == 0 && row_ok;
    const int64_t slot_off = static_cast<int64_t>(split * 4 + cq) * n * p.nx + gi;
    const float siglip_loss = (KIND == KIND_SIGLIP && slice == 0 && p.rowacc) ? 1.f : 0.f;
    uint32_t snap = 0, seq = 0;
    bool ok = true;
    // every epilogue warp runs all T iterations (an aborted warp skips the work but still
    // meets the named barriers, so the others cannot hang on them)
    for (int t = 0; t < T; ++t) {
      named_bar_sync(1, kEpiThreads);  // everyone is done with tile t - 1: buffer (t + 1) & 1 is free
      if (t + 1 < T) prefetch_colf(t + 1);
      cp_async_commit();
      cp_async_wait<1>();              // this thread's copies for tile t have landed
      named_bar_sync(1, kEpiThreads);  // ... and everyone else's
      const uint32_t cf = colf_s + (t & 1) * kColfBytes + cq * 64 * 4;
      const int64_t j0 = static_cast<int64_t>(t_begin + t) * kCols;
      const int64_t left = p.ny - j0;
      const int ncols = left < kCols ? static_cast<int>(left) : kCols;
      const int64_t dtile = i0 - j0;
      const bool check = ncols < kCols || (dtile > -kTileRows && dtile < kCols) || (i0 + kTileRows > p.nx);
      const int diag_col = static_cast<int>(dtile) + r;  // tile column of row r's positive
      for (int b = k_first; b < n; ++b, ++snap) {
        if (!ok) continue;
        if (!wait_bounded(acc_full, snap & 1, abort_flag)) {
          fail(p, abort_flag);
          ok = false;
          continue;
        }
        tc_fence_after();
        float v[64];
        tmem_ld64(tmem + lane_addr + cq * 64, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);
        const int k = b, ka = b - k_first;
        const float rho = n_rho;
        float R2, R3;
        if constexpr (KIND == KIND_SIGLIP) {
          float ms = 0.f;
#pragma unroll
          for (int kk = 0; kk < kMaxPrefix; ++kk)
            if (kk == k) ms = p.m_scale[kk];
          R2 = rho * ms;  // rho_i w_k t / N
          R3 = siglip_loss;
        } else {
          R2 = n_alpha;   // rho_i alpha_i
          R3 = rho;
        }
        const float R1 = p.L * rho;
        load_row(b + 1 < n ? b + 1 : k_first);
        const uint32_t c1 = cf + (ka * 2 + 0) * kCols * 4;
        const uint32_t c2 = cf + (ka * 2 + 1) * kCols * 4;
        // Quarters q and q + 2 take turns in slot q % 2: quarter q's v-th chunk follows
        // quarter q + 2's (v-1)-th, which follows quarter q's (v-1)-th.  Each group waits for
        // the chunk just before its own in the slot, on that group's own barrier, so no wait
        // can be two phases off.
        const uint32_t ms = cq & 1, turn = seq >> 2;
        const bool first_user = cq < 2;
        if ((!first_user || turn > 0) &&
            !wait_bounded(&m_done[first_user ? cq + 2 : cq - 2], first_user ? (turn - 1) & 1 : turn & 1, abort_flag)) {
          fail(p, abort_flag);
          ok = false;
          continue;
        }
        const uint32_t mt = m_row + ms * kMBytes;
        float ac = 0.f, al = 0.f;
        // eight 16-byte chunks of the 128-byte swizzled row r
        if (check) {
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            st_shared_v4(mt + ((ch ^ swz) << 4),
                         bwd_cells8<KIND, true>(v + ch * 8, c1 + ch * 32, c2 + ch * 32, R1, R2, R3, p.L, p.b2,
                                                cq * 64 + ch * 8, ncols, diag_col, row_ok, ac, al));
        } else {
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            st_shared_v4(mt + ((ch ^ swz) << 4), bwd_cells8<KIND, false>(v + ch * 8, c1 + ch * 32, c2 + ch * 32, R1,
                                                                         R2, R3, p.L, p.b2, 0, 0, 0, true, ac, al));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&m_full[ms]);
        if (keep_rows) {
          float* pc = p.crow + slot_off + static_cast<int64_t>(k) * p.nx;
          if (t == 0) *pc = ac;
          else atomicAdd(pc, ac);
          if (KIND == KIND_SIGLIP && p.rowacc) {
            float* pl = p.rowacc + slot_off + static_cast<int64_t>(k) * p.nx;
            if (t == 0) *pl = al;
            else atomicAdd(pl, al);
          }
        }
        seq += 4;
      }
    }
    cp_async_wait<0>();
    // ---- output: the gradient slice
    if (T > 0 && ok && wait_bounded(grad_done, 0, abort_flag)) {
      tc_fence_after();
      float* g = p.grad + (static_cast<int64_t>(split) * p.nx + gi) * p.d;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float v[32];
        tmem_ld32(tmem_grad + lane_addr + cq * 64 + h * 32, v);
        const int dcol = d0 + cq * 64 + h * 32;
        if (row_ok && dcol < p.d) {
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(g + dcol + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
      }
    } else if (T > 0 && ok) {
      fail(p, abort_flag);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int KIND>
static cudaError_t setup_one() {
  return cudaFuncSetAttribute(bwd_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
}

}  // namespace bwd

cudaError_t bwd_kernel_setup() {
  cudaError_t e;
  if ((e = bwd::setup_one<KIND_CLIP>()) != cudaSuccess) return e;
  if ((e = bwd::setup_one<KIND_SIGLIP>()) != cudaSuccess) return e;
  return bwd::setup_one<KIND_ROWS>();
}

cudaError_t launch_bwd(int kind, const CUtensorMap& tm_x, const CUtensorMap& tm_y, const CUtensorMap& tm_yt,
                       const TileParams& p, dim3 grid, cudaStream_t stream) {
  if (kind == KIND_CLIP)
    bwd::bwd_kernel<KIND_CLIP><<<grid, bwd::kThreads, bwd::smem_bytes, stream>>>(tm_x, tm_y, tm_yt, p);
  else if (kind == KIND_SIGLIP)
    bwd::bwd_kernel<KIND_SIGLIP><<<grid, bwd::kThreads, bwd::smem_bytes, stream>>>(tm_x, tm_y, tm_yt, p);
  else
    bwd::bwd_kernel<KIND_ROWS><<<grid, bwd::kThreads, bwd::smem_bytes, stream>>>(tm_x, tm_y, tm_yt, p);
  return cudaGetLastError();
}

}  // namespace ufc
