// gemm_kernel.cu -- the gradient contraction of the Matryoshka loss as a dense tcgen05 GEMM
// over the bf16 weights m^k written by the weight kernel, for both sides of the pair:
//
//     A side:  G[i, d] = sum_k [d < p_k] sum_j m^k[i, j] B[j, d]      (weights K-major)
//     B side:  G[j, d] = sum_k [d < p_k] sum_i m^k[i, j] A[i, d]      (weights MN-major)
//
// (prefix-expanded: prefix k contributes to its first p_k dimensions).  Two CTAs on two SMs
// form a pair (a cluster of 2, cta_group::2): together they own 256 rows of G (128 each) and
// two adjacent 256-dimension slices, one 256-column TMEM accumulator each.  For each prefix
// reaching the slices, from the widest down, they stream 64-long K chunks of m^k (A operand:
// each CTA its own 128 rows, staged once for both slices) and of the other side's transposed
// embeddings restricted to each slice (B operand, K-major, N = the prefix's width within the
// slice, each CTA holding half of the rows); the leader CTA issues one 256 x N x 16 MMA per
// slice.  The prefixes accumulate into the same accumulators, so after prefix k they hold
// sum_{k' >= k} G^k'; the epilogue reads each such snapshot for the projection scalars of the
// norm backward (r^k = x_row . G^k_row, this slice's part, is the difference of x . snapshot
// between prefix k and the one before it, taken over prefix k's width) and writes G once, at
// the end.  Two slices per pair halve the re-reads of each weight tile that one slice per pair
// had (the widest prefixes reach every slice).  The weights come from HBM and the other
// operand mostly from L2: each has its own TMA ring and producer.
//
// Warps (224 threads per CTA): lane 0 of warp 0 loads the weights, lane 0 of warp 6 the
// other operand, lane 0 of warp 1 (leader CTA only) issues the MMAs, warps 2..5 are the
// epilogue (warp w reads TMEM lanes 32 (w % 4) .. + 31).
#include "launch.h"
#include "ptx.cuh"

namespace ufc {
namespace gemm {

constexpr int kThreads = 224;
constexpr int kN = 256;                          // gradient slice width = TMEM columns per accumulator
constexpr int kNA = 5;                           // weight stages
constexpr int kNB = 4;                           // stages of the other operand
constexpr int kABytes = kTileRows * kChunk * 2;  // 16 KB: this CTA's 128 rows of G x 64 of K
constexpr int kBHalf = kN / 2 * kChunk * 2;      // 16 KB: this CTA's half of up to 256 dims x 64 of K
constexpr int kBBytes = 2 * kBHalf;              // both slices of the CTA
constexpr int kBox = kGemmBBox;                  // rows per B-operand TMA box
constexpr uint64_t kWaitLimitNs = 4000000000ull;

constexpr int off_a = 0;
constexpr int off_b = off_a + kNA * kABytes;
constexpr int off_bar = off_b + kNB * kBBytes;
constexpr int n_bars = 2 * kNA + 2 * kNB + 4;
constexpr int off_misc = off_bar + n_bars * 8;
constexpr int smem_bytes = off_misc + 16 + 1024;
static_assert(smem_bytes <= 232448, "gemm shared memory");

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return mbar_wait_abortable(bar, parity, abort_flag, kWaitLimitNs);
}

__device__ __forceinline__ void fail(const GemmParams& p, volatile int* abort_flag) {
  *abort_flag = 1;
  if (p.status) atomicExch(p.status, kStatusTimeout);
}

__device__ __forceinline__ int prefix_end_of(const GemmParams& p, int k) {
  int pk = 0;
#pragma unroll
  for (int kk = 0; kk < kMaxPrefix; ++kk)
    if (kk == k) pk = p.prefix_end[kk];
  return pk;
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// One CTA of the contraction; vblock is its index in the contraction's own grid.
// AMN: the weights are the MN-major A operand (B side: rows of G are columns of m^k).
template <bool AMN>
__device__ __forceinline__ void gemm_body(const CUtensorMap& tm_w, const CUtensorMap& tm_yt,
                                          const CUtensorMap& tm_yt128, const GemmParams& p, uint32_t vblock) {
  griddep_enter();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sa = smem + off_a;
  uint8_t* sb = smem + off_b;
  uint64_t* a_full = reinterpret_cast<uint64_t*>(smem + off_bar);
  uint64_t* a_empty = a_full + kNA;
  uint64_t* b_full = a_empty + kNA;
  uint64_t* b_empty = b_full + kNB;
  uint64_t* acc_full = b_empty + kNB;  // [2]
  uint64_t* acc_empty = acc_full + 2;  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + off_misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + off_misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // 0: the leader, which issues the pair's MMAs
  // Grid: [unit type][row-block pair][rank].  A CTA pair owns 256 rows of G and the two
  // adjacent 256-dimension slices s0 = 2 grp and s1 = 2 grp + 1 of its group (one 256-column
  // TMEM accumulator each), so every weight tile is staged once for both.  A unit takes the
  // prefixes from `top` down to the narrowest one reaching s0.  With p.split_rest, a group
  // reached by two or more prefixes runs as two units: the widest prefix alone (into G) and
  // the others (into G2, which the norm backward adds); those "rest" units come first in the
  // launch, the heavier ones.  Otherwise one unit per group, the heavy first group first.
  int n_slices = 0;
#pragma unroll
  for (int kk = 0; kk < kMaxPrefix; ++kk)
    if (kk < p.n_prefix) n_slices = (p.prefix_end[kk] + kN - 1) / kN;
  const int n = p.n_prefix;
  // groups 0 .. n_rest_groups - 1 are reached by two or more prefixes (the second widest's end
  // lies past their first dimension).  With p.merge (and no split) each of those groups runs one
  // unit from prefix n-2 down: array n-2 holds the merged weights of prefixes n-2 and n-1 below
  // p_{n-2} (a multiple of 512), and prefix n-1 runs only in the groups above.
  const bool merge = p.merge && !p.split_rest && n >= 2;
  const int n_rest_groups =
      ((p.split_rest || merge) && n >= 2) ? (prefix_end_of(p, n - 2) + 2 * kN - 1) / (2 * kN) : 0;
  const int64_t pairs = (p.m_rows + 2 * kTileRows - 1) / (2 * kTileRows);
  const int64_t cta = vblock >> 1;
  const int type = static_cast<int>(cta / pairs);
  // unit types: split: [the rest units of groups 0 .. n_rest_groups - 1][one unit per group];
  // merge: [one unit per group]; neither: [one unit per group] (n_rest_groups = 0)
  const bool rest_unit = type < n_rest_groups;  // its prefixes start at n-2
  const int grp = (merge || rest_unit) ? type : type - n_rest_groups;
  const int64_t pair_i = cta % pairs;
  const int64_t m0 = (pair_i * 2 + rank) * kTileRows;  // first row of G in this launch
  const int d0 = grp * 2 * kN;                          // first dimension of slice s0
  int k_first = 0;  // prefixes k_first .. n-1 reach slice s0
#pragma unroll
  for (int k = 0; k < kMaxPrefix; ++k)
    if (k < n && p.prefix_end[k] <= d0) k_first = k + 1;
  // this unit's prefixes: top, then top-1 .. k_first (none after top for a split group's
  // widest-prefix unit)
  const int top = rest_unit ? n - 2 : n - 1;
  const bool split_group = grp < n_rest_groups;
  const int n_steps = (!rest_unit && split_group) ? 1 : top + 1 - k_first;
  float* const gout = (rest_unit && !merge) ? p.G2 : p.G;
  const int64_t gld = (rest_unit && !merge) ? p.g2_ld : p.d;
  // prefix k's width within slice s (0: it does not reach the slice)
  auto width = [&](int k, int sl) {
    const int w = prefix_end_of(p, k) - (d0 + sl * kN);
    return w < 0 ? 0 : (w > kN ? kN : w);
  };
  const int nkc = static_cast<int>((p.kdim + kChunk - 1) / kChunk);  // K chunks per prefix
  // Order of the prefixes: the unit's widest first (it writes every column the unit writes, so
  // it starts the accumulators afresh), then the narrower ones from a start that rotates with
  // the pair.  A narrow prefix reads as many weight bytes per K chunk as a wide one for a
  // fraction of the MMA work, so the pairs of one wave should not all reach the narrow ones
  // together.
  const int n_after = n_steps - 1;  // prefixes after the unit's widest
  const int rot = n_after > 0 ? static_cast<int>(pair_i % n_after) : 0;
  auto prefix_at = [&](int step) {  // step 0: top; then top-1 .. k_first, rotated
    if (step == 0) return top;
    int j = step - 1 + rot;
    if (j >= n_after) j -= n_after;
    return top - 1 - j;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNA; ++s) {
      mbar_init(&a_full[s], 1);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < kNB; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    mbar_init(&acc_full[0], 1);
    mbar_init(&acc_empty[0], 8);  // the four epilogue warps of each CTA of the pair (leader's copy)
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_yt);
  }
  if (warp == 0) {
    tmem_alloc_pair(tmem_slot, 2 * kN);  // the same columns in both SMs of the pair
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if ((warp == 0 || warp == 6) && lane == 0) {
    // ------------------------------------------------------------- TMA producers
    // warp 0: the weights (A operand); warp 6: the other side's transposed rows (B operand)
    // for both slices.  Both CTAs load their own parts into their own shared memory;
    // completion is counted on the leader's barrier, which the leader arms for both.
    const bool wa = warp == 0;
    const int ns = wa ? kNA : kNB;
    uint64_t* fullb = wa ? a_full : b_full;
    uint64_t* emptyb = wa ? a_empty : b_empty;
    uint32_t it = 0;
    bool ok = true;
    for (int step = 0; step < n_steps && ok; ++step) {
      const int k = prefix_at(step);
      const int h0 = width(k, 0) / 2, h1 = width(k, 1) / 2;  // B rows of each slice held by each CTA
      const int64_t wrow = static_cast<int64_t>(k) * p.w_rows_per_prefix;
      for (int c = 0; c < nkc; ++c, ++it) {
        const uint32_t st = it % ns, ph = (it / ns) & 1;
        if (!wait_bounded(&emptyb[st], ph ^ 1, abort_flag)) {
          fail(p, abort_flag);
          ok = false;
          break;
        }
        const uint32_t bar = mapa_shared(smem_u32(&fullb[st]), 0);
        if (rank == 0) mbar_arrive_expect_tx(&fullb[st], 2 * (wa ? kABytes : (h0 + h1) * kChunk * 2));
        if (wa) {
          if constexpr (AMN) {
            // [64 K rows x 64 M columns] twice: M blocks 0..63 and 64..127 of this CTA's rows
            for (int h = 0; h < 2; ++h)
              tma_load_2d_pair(sa + st * kABytes + h * (kABytes / 2), &tm_w, bar, static_cast<int>(m0 + h * 64),
                               static_cast<int>(wrow + c * kChunk));
          } else {
            tma_load_2d_pair(sa + st * kABytes, &tm_w, bar, c * kChunk, static_cast<int>(wrow + m0));
          }
        } else {
          for (int sl = 0; sl < 2; ++sl) {
            const int half = sl ? h1 : h0;
            const int dim0 = d0 + sl * kN + static_cast<int>(rank) * half;
            uint8_t* dst = sb + st * kBBytes + sl * kBHalf;
            // one 128-row box when the half is full (one TMA instruction: the producer's
            // issue rate limits this loop), else 32-row boxes
            if (half == kN / 2)
              tma_load_2d_pair(dst, &tm_yt128, bar, static_cast<int>(p.b_col0 + c * kChunk), dim0);
            else
              for (int r0 = 0; r0 < half; r0 += kBox)
                tma_load_2d_pair(dst + r0 * kChunk * 2, &tm_yt, bar, static_cast<int>(p.b_col0 + c * kChunk),
                                 dim0 + r0);
          }
        }
      }
    }
    if (rank == 0) {
      for (uint32_t q = 0; q < static_cast<uint32_t>(ns) && q < it; ++q) {  // let the last copies land
        const uint32_t u = it - 1 - q;
        mbar_wait(&fullb[u % ns], (u / ns) & 1, kWaitLimitNs);
      }
    } else {
      // the follower's copies are counted on the leader's barriers: wait until the MMAs that
      // read them (hence the copies) are done, i.e. the last stages are released
      for (uint32_t q = 0; q < static_cast<uint32_t>(ns) && q < it; ++q) {
        const uint32_t u = it - 1 - q;
        mbar_wait(&emptyb[u % ns], (u / ns) & 1, kWaitLimitNs);
      }
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ------------------------------------------------------------- MMA issuer (leader)
    // The prefixes accumulate, widest first, into one accumulator per slice: after prefix k
    // it holds sum_{k' >= k} G^k' (prefix k' writes its first width(k', s) columns).
    uint32_t it = 0, pi = 0;
    bool ok = true;
    for (int step = 0; step < n_steps && ok; ++step, ++pi) {
      const int k = prefix_at(step);
      const int w0 = width(k, 0), w1 = width(k, 1);
      // the epilogue must have read the previous prefix's snapshot before this one adds to it
      if (pi >= 1 && !wait_bounded(&acc_empty[0], (pi - 1) & 1, abort_flag)) {
        fail(p, abort_flag);
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t id0 = AMN ? idesc_bf16_f32_amn(2 * kTileRows, static_cast<uint32_t>(w0))
                               : idesc_bf16_f32(2 * kTileRows, static_cast<uint32_t>(w0));
      const uint32_t id1 = AMN ? idesc_bf16_f32_amn(2 * kTileRows, static_cast<uint32_t>(w1))
                               : idesc_bf16_f32(2 * kTileRows, static_cast<uint32_t>(w1));
      for (int c = 0; c < nkc; ++c, ++it) {
        const uint32_t sta = it % kNA, pha = (it / kNA) & 1;
        const uint32_t stb = it % kNB, phb = (it / kNB) & 1;
        if (!wait_bounded(&a_full[sta], pha, abort_flag) || !wait_bounded(&b_full[stb], phb, abort_flag)) {
          fail(p, abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t as = smem_u32(sa + sta * kABytes), bs = smem_u32(sb + stb * kBBytes);
#pragma unroll
        for (int kk = 0; kk < kChunk / 16; ++kk) {
          // K = 16 per MMA: MN-major A advances 16 K rows (two 1024-byte atoms), K-major 32 bytes
          const uint64_t adesc = AMN ? sdesc_mnmajor_sw128(as + kk * 2048, kABytes / 2, 1024)
                                     : sdesc_kmajor_sw128(as + kk * 32);
          const uint32_t acc = (pi != 0 || c != 0 || kk != 0) ? 1u : 0u;  // the widest prefix starts fresh
          umma_bf16_pair(tmem, adesc, sdesc_kmajor_sw128(bs + kk * 32), id0, acc);
          if (w1 > 0) umma_bf16_pair(tmem + kN, adesc, sdesc_kmajor_sw128(bs + kBHalf + kk * 32), id1, acc);
        }
        umma_commit_pair(&a_empty[sta]);  // releases the stages in both CTAs
        umma_commit_pair(&b_empty[stb]);
      }
      if (ok) umma_commit_pair(&acc_full[0]);
    }
  } else if (warp >= 2 && warp < 6) {
    // ------------------------------------------------------------- epilogue
    // After each prefix k: d_s(c) = x . S_k over the first c columns of slice s at every
    // 64-column boundary c; r^k (this slice's part) = d_s(w_k) - (the previous snapshot's
    // d_s(w_k)), as S_k - S_{k+1} = G^k over the first w_k columns.  After the last prefix,
    // the accumulators are G: written once (added over weight chunks when accumulating).
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int64_t gl = m0 + r;              // row within this launch
    const int64_t g = p.row0 + gl;          // row of G / X / crow
    const bool row_ok = gl < p.m_rows;
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const int wmax[2] = {width(top, 0), width(top, 1)};  // columns of each slice with data
    // prefixes that do not reach a slice contribute nothing to its slot (merged: nor does prefix
    // n-1 below p_{n-2}, whose weights are in the merged array)
    if (row_ok && !p.accumulate && (merge || !rest_unit))
      for (int sl = 0; sl < 2; ++sl)
        if (2 * grp + sl < n_slices)
          for (int k = 0; k < n; ++k)
            if (width(k, sl) == 0 || (merge && rest_unit && k == n - 1))
              p.crow[(static_cast<int64_t>(2 * grp + sl) * n + k) * p.crow_rows + g] = 0.f;
    float prevd[2][kN / 64], curd[2][kN / 64];
#pragma unroll
    for (int sl = 0; sl < 2; ++sl)
#pragma unroll
      for (int b = 0; b < kN / 64; ++b) prevd[sl][b] = 0.f;
    uint32_t pi = 0;
    bool ok = true;
    // x rows are read in 32-column chunks, each fetched one chunk ahead (the first before the
    // snapshot is ready): the MMA waits for this read, so it must not wait on L2 per chunk
    auto load_x = [&](int sl, int c, uint4 (&xv)[4]) {
      const uint4* src = reinterpret_cast<const uint4*>(p.X + g * p.d + d0 + sl * kN + c);
#pragma unroll
      for (int u = 0; u < 4; ++u) xv[u] = row_ok ? src[u] : make_uint4(0, 0, 0, 0);
    };
    for (int step = 0; step < n_steps; ++step, ++pi) {
      const int k = prefix_at(step);
      if (!ok) continue;
      uint4 xcur[4], xnext[4];
      load_x(0, 0, xcur);
      if (!wait_bounded(&acc_full[0], pi & 1, abort_flag)) {
        fail(p, abort_flag);
        ok = false;
        continue;
      }
      tc_fence_after();
      const bool last = step == n_steps - 1;
#pragma unroll
      for (int sl = 0; sl < 2; ++sl) {
        float run = 0.f;
        float* grow = gout + g * gld + d0 + sl * kN;
#pragma unroll
        for (int b = 0; b < kN / 64; ++b) curd[sl][b] = 0.f;
        for (int c = 0; c < wmax[sl]; c += 32) {
          // the next chunk: this slice's, else the next slice's first
          if (c + 32 < wmax[sl]) load_x(sl, c + 32, xnext);
          else if (sl == 0 && wmax[1] > 0) load_x(1, 0, xnext);
          float v[32];
          tmem_ld32(tmem + lane_addr + sl * kN + c, v);
          if (row_ok) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const uint4 xv = xcur[u];
              const int j = 8 * u;
              run = fmaf(bf16_lo(xv.x), v[j + 0], run);
              run = fmaf(bf16_hi(xv.x), v[j + 1], run);
              run = fmaf(bf16_lo(xv.y), v[j + 2], run);
              run = fmaf(bf16_hi(xv.y), v[j + 3], run);
              run = fmaf(bf16_lo(xv.z), v[j + 4], run);
              run = fmaf(bf16_hi(xv.z), v[j + 5], run);
              run = fmaf(bf16_lo(xv.w), v[j + 6], run);
              run = fmaf(bf16_hi(xv.w), v[j + 7], run);
            }
            if (last) {
#pragma unroll
              for (int j = 0; j < 32; j += 4) {
                float4 o = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                if (p.accumulate) {
                  const float4 prev = *reinterpret_cast<const float4*>(grow + c + j);
                  o.x += prev.x;
                  o.y += prev.y;
                  o.z += prev.z;
                  o.w += prev.w;
                }
                *reinterpret_cast<float4*>(grow + c + j) = o;
              }
            }
          }
#pragma unroll
          for (int b = 0; b < kN / 64; ++b)
            if (c + 32 == 64 * (b + 1)) curd[sl][b] = run;
#pragma unroll
          for (int u = 0; u < 4; ++u) xcur[u] = xnext[u];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&acc_empty[0]), 0));
      if (row_ok) {
#pragma unroll
        for (int sl = 0; sl < 2; ++sl) {
          const int w = width(k, sl);
          if (w > 0) {
            float rk = 0.f;
#pragma unroll
            for (int b = 0; b < kN / 64; ++b)
              if (w == 64 * (b + 1)) rk = curd[sl][b] - prevd[sl][b];
            float* pc = p.crow + (static_cast<int64_t>(2 * grp + sl) * n + k) * p.crow_rows + g;
            *pc = p.accumulate ? *pc + rk : rk;
          }
        }
      }
#pragma unroll
      for (int sl = 0; sl < 2; ++sl)
#pragma unroll
        for (int b = 0; b < kN / 64; ++b) prevd[sl][b] = curd[sl][b];
    }
  }

  tc_fence_before();
  cluster_sync_all();  // no MMA, copy or remote arrive of the pair is still in flight
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 2 * kN);
  }
}

template <bool AMN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_yt,
                const __grid_constant__ CUtensorMap tm_yt128, const GemmParams p) {
  gemm_body<AMN>(tm_w, tm_yt, tm_yt128, p, blockIdx.x);
}

// Both contractions of a weight chunk in one grid: the dA CTAs (K-major weights) first, then
// the dB ones (MN-major), so the second fills the first's last wave instead of waiting for
// it (split: the dA grid's size, even, so no CTA pair straddles the two).
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel_both(const __grid_constant__ CUtensorMap tk_w, const __grid_constant__ CUtensorMap tk_yt,
                     const __grid_constant__ CUtensorMap tk_yt128, const GemmParams pk,
                     const __grid_constant__ CUtensorMap tn_w, const __grid_constant__ CUtensorMap tn_yt,
                     const __grid_constant__ CUtensorMap tn_yt128, const GemmParams pn, const unsigned split) {
  if (blockIdx.x < split)
    gemm_body<false>(tk_w, tk_yt, tk_yt128, pk, blockIdx.x);
  else
    gemm_body<true>(tn_w, tn_yt, tn_yt128, pn, blockIdx.x - split);
}

template <bool AMN>
static cudaError_t setup_one() {
  return cudaFuncSetAttribute(gemm_kernel<AMN>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
}

// CTAs of one contraction: [unit type][row-block pair][rank]; the unit types are the slice
// groups (two slices each) and, with split_rest, one more per group that two or more prefixes
// reach (the same count as in gemm_body)
unsigned grid_of(const GemmParams& p) {
  const int n = p.n_prefix;
  const int pn = p.prefix_end[n - 1];
  const int64_t blocks = (p.m_rows + kTileRows - 1) / kTileRows;
  const int64_t n_slices = (pn + kN - 1) / kN;
  const int64_t groups = (n_slices + 1) / 2;
  const int64_t rest = (p.split_rest && n >= 2) ? (p.prefix_end[n - 2] + 2 * kN - 1) / (2 * kN) : 0;
  return static_cast<unsigned>((groups + rest) * ((blocks + 1) / 2) * 2);
}

}  // namespace gemm

cudaError_t gemm_kernel_setup() {
  cudaError_t e;
  if ((e = gemm::setup_one<false>()) != cudaSuccess) return e;
  if ((e = gemm::setup_one<true>()) != cudaSuccess) return e;
  return cudaFuncSetAttribute(gemm::gemm_kernel_both, cudaFuncAttributeMaxDynamicSharedMemorySize, gemm::smem_bytes);
}

double gemm_grid_pairs(const GemmParams& p) { return 0.5 * gemm::grid_of(p); }

cudaError_t launch_gemm_both(const CUtensorMap& tk_w, const CUtensorMap& tk_yt, const CUtensorMap& tk_yt128,
                             const GemmParams& pk, const CUtensorMap& tn_w, const CUtensorMap& tn_yt,
                             const CUtensorMap& tn_yt128, const GemmParams& pn, cudaStream_t stream) {
  const unsigned split = gemm::grid_of(pk);
  return launch_pdl(gemm::gemm_kernel_both, dim3(split + gemm::grid_of(pn)), dim3(gemm::kThreads), gemm::smem_bytes,
                    stream, 2, tk_w, tk_yt, tk_yt128, pk, tn_w, tn_yt, tn_yt128, pn, split);
}

cudaError_t launch_gemm(const CUtensorMap& tm_w, const CUtensorMap& tm_yt, const CUtensorMap& tm_yt128,
                        const GemmParams& p, bool weights_mn, cudaStream_t stream) {
  const dim3 grid(gemm::grid_of(p)), block(gemm::kThreads);
  if (weights_mn)
    return launch_pdl(gemm::gemm_kernel<true>, grid, block, gemm::smem_bytes, stream, 2, tm_w, tm_yt, tm_yt128, p);
  return launch_pdl(gemm::gemm_kernel<false>, grid, block, gemm::smem_bytes, stream, 2, tm_w, tm_yt, tm_yt128, p);
}

}  // namespace ufc
