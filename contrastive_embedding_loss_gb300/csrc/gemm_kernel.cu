// gemm_kernel.cu -- the gradient contraction of the Matryoshka loss as a dense tcgen05 GEMM
// over the bf16 weights m^k written by the weight kernel, for both sides of the pair:
//
//     A side:  G[i, d] = sum_k [d < p_k] sum_j m^k[i, j] B[j, d]      (weights K-major)
//     B side:  G[j, d] = sum_k [d < p_k] sum_i m^k[i, j] A[i, d]      (weights MN-major)
//
// (prefix-expanded: prefix k contributes to its first p_k dimensions).  Two CTAs on two SMs
// form a pair (a cluster of 2, cta_group::2): together they own 256 rows of G (128 each)
// and one 256-dimension slice [d0, d0 + 256).  For each prefix reaching the slice, from the
// widest down, they stream 64-long K chunks of m^k (A operand: each CTA its own 128 rows)
// and of the other side's transposed embeddings restricted to the slice (B operand, K-major,
// N = min(p_k, d0 + 256) - d0 rows, each CTA holding half of them); the leader CTA issues
// 256 x N x 16 MMAs that read both halves, so each SM loads half of the B operand a
// single-SM 128-row tile would need.  Accumulators: two per CTA in TMEM (256 columns each),
// alternating between prefixes, so the epilogue of prefix k (add G^k into G in global
// memory; r^k = x_row . G^k_row, the projection scalar of the norm backward, as this
// slice's partial) overlaps the MMAs of prefix k - 1.  The weights come from HBM and the
// other operand mostly from L2: each has its own TMA ring and producer.
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
constexpr int kNA = 7;                           // weight stages
constexpr int kNB = 6;                           // stages of the other operand
constexpr int kABytes = kTileRows * kChunk * 2;  // 16 KB: this CTA's 128 rows of G x 64 of K
constexpr int kBBytes = kN / 2 * kChunk * 2;     // 16 KB: this CTA's half of up to 256 dims x 64 of K
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
  // Grid: [slice pair][row-block pair][slice in the pair][rank].  Slices 2s and 2s + 1 of a
  // row block run side by side and start on the same weights (the widest prefixes reach
  // both), which they share through L2; the heavy first pair (every prefix reaches slice 0)
  // runs first, which keeps the tail of the launch short.
  int n_slices = 0;
#pragma unroll
  for (int kk = 0; kk < kMaxPrefix; ++kk)
    if (kk < p.n_prefix) n_slices = (p.prefix_end[kk] + kN - 1) / kN;
  const int64_t pairs = (p.m_rows + 2 * kTileRows - 1) / (2 * kTileRows);
  const int64_t cta = vblock >> 1;                     // [group][pair][slice in group]
  const int64_t per_group = pairs * 2;
  const int grp = static_cast<int>(cta / per_group);
  const int64_t rem = cta % per_group;
  const int64_t pair_i = rem / 2;
  const int slice = grp * 2 + static_cast<int>(rem % 2);
  const int64_t m0 = (pair_i * 2 + rank) * kTileRows;  // first row of G in this launch
  const int d0 = slice * kN;
  const int n = p.n_prefix;
  const bool idle = slice >= n_slices;  // an odd slice count leaves the last group half empty
  int k_first = idle ? n : 0;  // prefixes k_first .. n-1 reach this slice
#pragma unroll
  for (int k = 0; k < kMaxPrefix; ++k)
    if (!idle && k < n && p.prefix_end[k] <= d0) k_first = k + 1;
  const int nkc = static_cast<int>((p.kdim + kChunk - 1) / kChunk);  // K chunks per prefix

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNA; ++s) {
      mbar_init(&a_full[s], 1);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < kNB; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 8);  // the four epilogue warps of each CTA of the pair (leader's copy)
    }
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
    // warp 0: the weights (A operand); warp 6: the other side's transposed rows (B operand).
    // Both CTAs load their own parts into their own shared memory; completion is counted on
    // the leader's barrier, which the leader arms for the bytes of both.
    const bool wa = warp == 0;
    const int ns = wa ? kNA : kNB;
    uint64_t* fullb = wa ? a_full : b_full;
    uint64_t* emptyb = wa ? a_empty : b_empty;
    uint32_t it = 0;
    bool ok = true;
    for (int k = n - 1; k >= k_first && ok; --k) {
      const int nk = min(prefix_end_of(p, k), d0 + kN) - d0;
      const int half = nk / 2;  // B rows held by each CTA
      const int64_t wrow = static_cast<int64_t>(k) * p.w_rows_per_prefix;
      for (int c = 0; c < nkc; ++c, ++it) {
        const uint32_t st = it % ns, ph = (it / ns) & 1;
        if (!wait_bounded(&emptyb[st], ph ^ 1, abort_flag)) {
          fail(p, abort_flag);
          ok = false;
          break;
        }
        const uint32_t bar = mapa_shared(smem_u32(&fullb[st]), 0);
        if (rank == 0) mbar_arrive_expect_tx(&fullb[st], 2 * (wa ? kABytes : half * kChunk * 2));
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
          // one 128-row box when the half is full (one TMA instruction: the producer's issue
          // rate limits this loop), else 32-row boxes
          if (half == kN / 2)
            tma_load_2d_pair(sb + st * kBBytes, &tm_yt128, bar, static_cast<int>(p.b_col0 + c * kChunk),
                             d0 + static_cast<int>(rank) * half);
          else
            for (int r0 = 0; r0 < half; r0 += kBox)
              tma_load_2d_pair(sb + st * kBBytes + r0 * kChunk * 2, &tm_yt, bar,
                               static_cast<int>(p.b_col0 + c * kChunk), d0 + static_cast<int>(rank) * half + r0);
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
    uint32_t it = 0, pi = 0;
    bool ok = true;
    for (int k = n - 1; k >= k_first && ok; --k, ++pi) {
      const int nk = min(prefix_end_of(p, k), d0 + kN) - d0;
      const uint32_t a = pi & 1;
      // the epilogue must have read this accumulator's previous prefix
      if (pi >= 2 && !wait_bounded(&acc_empty[a], ((pi - 2) >> 1) & 1, abort_flag)) {
        fail(p, abort_flag);
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem + a * kN;
      const uint32_t idesc = AMN ? idesc_bf16_f32_amn(2 * kTileRows, static_cast<uint32_t>(nk))
                                 : idesc_bf16_f32(2 * kTileRows, static_cast<uint32_t>(nk));
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
          umma_bf16_pair(d, adesc, sdesc_kmajor_sw128(bs + kk * 32), idesc, (c != 0 || kk != 0) ? 1u : 0u);
        }
        umma_commit_pair(&a_empty[sta]);  // releases the stage in both CTAs
        umma_commit_pair(&b_empty[stb]);
      }
      if (ok) umma_commit_pair(&acc_full[a]);
    }
  } else if (warp >= 2 && warp < 6) {
    // ------------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int64_t gl = m0 + r;              // row within this launch
    const int64_t g = p.row0 + gl;          // row of G / X / crow
    const bool row_ok = gl < p.m_rows;
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    float* grow = p.G + g * p.d + d0;
    const uint16_t* xrow = p.X + g * p.d + d0;
    // prefixes that do not reach this slice contribute nothing to its slot
    if (row_ok && !p.accumulate && !idle)
      for (int k = 0; k < k_first; ++k) p.crow[(static_cast<int64_t>(slice) * n + k) * p.crow_rows + g] = 0.f;
    uint32_t pi = 0;
    bool ok = true;
    for (int k = n - 1; k >= k_first; --k, ++pi) {
      if (!ok) continue;
      const int nk = min(prefix_end_of(p, k), d0 + kN) - d0;
      const uint32_t a = pi & 1;
      if (!wait_bounded(&acc_full[a], (pi >> 1) & 1, abort_flag)) {
        fail(p, abort_flag);
        ok = false;
        continue;
      }
      tc_fence_after();
      const bool first = pi == 0 && !p.accumulate;  // the widest prefix writes G, the others add
      float rk = 0.f;
      for (int c = 0; c < nk; c += 32) {
        float v[32];
        tmem_ld32(tmem + lane_addr + a * kN + c, v);
        if (row_ok) {
#pragma unroll
          for (int j = 0; j < 32; j += 8) {
            const uint4 xv = *reinterpret_cast<const uint4*>(xrow + c + j);
            rk = fmaf(bf16_lo(xv.x), v[j + 0], rk);
            rk = fmaf(bf16_hi(xv.x), v[j + 1], rk);
            rk = fmaf(bf16_lo(xv.y), v[j + 2], rk);
            rk = fmaf(bf16_hi(xv.y), v[j + 3], rk);
            rk = fmaf(bf16_lo(xv.z), v[j + 4], rk);
            rk = fmaf(bf16_hi(xv.z), v[j + 5], rk);
            rk = fmaf(bf16_lo(xv.w), v[j + 6], rk);
            rk = fmaf(bf16_hi(xv.w), v[j + 7], rk);
          }
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            float4 o = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            if (!first) {
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
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&acc_empty[a]), 0));
      if (row_ok) {
        float* pc = p.crow + (static_cast<int64_t>(slice) * n + k) * p.crow_rows + g;
        *pc = p.accumulate ? *pc + rk : rk;
      }
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

// CTAs of one contraction: [slice pair][row-block pair][slice in the pair][rank]
unsigned grid_of(const GemmParams& p) {
  const int pn = p.prefix_end[p.n_prefix - 1];
  const int64_t blocks = (p.m_rows + kTileRows - 1) / kTileRows;
  const int64_t n_slices = (pn + kN - 1) / kN;
  const int64_t groups = (n_slices + 1) / 2;
  return static_cast<unsigned>(groups * ((blocks + 1) / 2) * 2 * 2);
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(split + gemm::grid_of(pn));
  cfg.blockDim = dim3(gemm::kThreads);
  cfg.dynamicSmemBytes = gemm::smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm::gemm_kernel_both, tk_w, tk_yt, tk_yt128, pk, tn_w, tn_yt, tn_yt128, pn,
                            split);
}

cudaError_t launch_gemm(const CUtensorMap& tm_w, const CUtensorMap& tm_yt, const CUtensorMap& tm_yt128,
                        const GemmParams& p, bool weights_mn, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(gemm::grid_of(p));
  cfg.blockDim = dim3(gemm::kThreads);
  cfg.dynamicSmemBytes = gemm::smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (weights_mn) return cudaLaunchKernelEx(&cfg, gemm::gemm_kernel<true>, tm_w, tm_yt, tm_yt128, p);
  return cudaLaunchKernelEx(&cfg, gemm::gemm_kernel<false>, tm_w, tm_yt, tm_yt128, p);
}

}  // namespace ufc
