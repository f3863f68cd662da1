// gemm_kernel.cu -- the gradient contraction of the Matryoshka loss as a dense tcgen05 GEMM
// over the bf16 weights m^k written by the weight kernel:
//
//     G[i, d] (+)= sum_k [d < p_k] sum_j m^k[i, j] * Y[j, d]
//
// (prefix-expanded: prefix k contributes to the first p_k dimensions only).  A CTA owns
// 128 rows of G and one 256-dimension slice [d0, d0 + 256); for every prefix reaching the
// slice it streams 64-column chunks of m^k (A operand, K-major) and of Y^T restricted to
// the slice (B operand, K-major, N = min(p_k, d0 + 256) - d0 rows) through a 4-stage TMA
// ring into one TMEM accumulator of 256 columns.  Prefixes are walked from the widest
// down, so the CTAs of the slices of one row block, which run side by side, read the same
// rows of m^4 first and share them through L2.
//
// Warps (128 threads): lane 0 of warp 0 issues the TMA loads, lane 0 of warp 1 the MMAs;
// afterwards all four warps move the accumulator (thread = row) to global memory.
#include "launch.h"
#include "ptx.cuh"

namespace ufc {
namespace gemm {

constexpr int kThreads = 128;
constexpr int kN = 256;                         // gradient slice width = TMEM columns
constexpr int kNS = 4;                          // operand stages
constexpr int kABytes = kTileRows * kChunk * 2;  // 16 KB: 128 rows of m^k x 64 columns
constexpr int kBBytes = kN * kChunk * 2;         // 32 KB: up to 256 dims of Y^T x 64 columns
constexpr int kBox = kBwdYtBox;                  // dims per Y^T TMA box
constexpr uint64_t kWaitLimitNs = 4000000000ull;

constexpr int off_a = 0;
constexpr int off_b = off_a + kNS * kABytes;
constexpr int off_bar = off_b + kNS * kBBytes;
constexpr int n_bars = 2 * kNS + 1;
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

template <bool ACC>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_yt,
                const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sa = smem + off_a;
  uint8_t* sb = smem + off_b;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + off_bar);
  uint64_t* empty = full + kNS;
  uint64_t* done = empty + kNS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + off_misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + off_misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // slices are the fast grid dimension: the CTAs of one row block run side by side
  const int64_t i0 = static_cast<int64_t>(blockIdx.y) * kTileRows;
  const int d0 = blockIdx.x * kN;
  const int n = p.n_prefix;
  int k_first = 0;  // prefixes k_first .. n-1 reach this slice
#pragma unroll
  for (int k = 0; k < kMaxPrefix; ++k)
    if (k < n && p.prefix_end[k] <= d0) k_first = k + 1;
  const int nj = static_cast<int>((p.kdim + kChunk - 1) / kChunk);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_yt);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
  // zero the accumulator: every MMA accumulates onto it (prefixes differ in width)
#pragma unroll
  for (int c = 0; c < kN; c += 32) tmem_st32_zero(tmem + lane_addr + c);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  bool ok = true;
  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------- TMA producer
    uint32_t it = 0;
    for (int k = n - 1; k >= k_first && ok; --k) {
      int pk = 0;
#pragma unroll
      for (int kk = 0; kk < kMaxPrefix; ++kk)
        if (kk == k) pk = p.prefix_end[kk];
      const int nk = min(pk, d0 + kN) - d0;
      const int arow = static_cast<int>(k * p.w_rows_per_prefix + i0);
      for (int jc = 0; jc < nj; ++jc, ++it) {
        const uint32_t st = it % kNS, ph = (it / kNS) & 1;
        if (!wait_bounded(&empty[st], ph ^ 1, abort_flag)) {
          fail(p, abort_flag);
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[st], kABytes + nk * kChunk * 2);
        tma_load_2d(sa + st * kABytes, &tm_w, &full[st], jc * kChunk, arow);
        for (int r0 = 0; r0 < nk; r0 += kBox)
          tma_load_2d(sb + st * kBBytes + r0 * kChunk * 2, &tm_yt, &full[st], jc * kChunk, d0 + r0);
      }
    }
    for (uint32_t q = 0; q < kNS && q < it; ++q) {  // let the last copies land
      const uint32_t u = it - 1 - q;
      mbar_wait(&full[u % kNS], (u / kNS) & 1, kWaitLimitNs);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------- MMA issuer
    uint32_t it = 0;
    for (int k = n - 1; k >= k_first && ok; --k) {
      int pk = 0;
#pragma unroll
      for (int kk = 0; kk < kMaxPrefix; ++kk)
        if (kk == k) pk = p.prefix_end[kk];
      const int nk = min(pk, d0 + kN) - d0;
      const uint32_t idesc = idesc_bf16_f32(kTileRows, static_cast<uint32_t>(nk));
      for (int jc = 0; jc < nj; ++jc, ++it) {
        const uint32_t st = it % kNS, ph = (it / kNS) & 1;
        if (!wait_bounded(&full[st], ph, abort_flag)) {
          fail(p, abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a = smem_u32(sa + st * kABytes), b = smem_u32(sb + st * kBBytes);
#pragma unroll
        for (int kk = 0; kk < kChunk / 16; ++kk)
          umma_bf16(tmem, sdesc_kmajor_sw128(a + kk * 32), sdesc_kmajor_sw128(b + kk * 32), idesc, 1u);
        umma_commit(&empty[st]);
      }
    }
    umma_commit(done);
  }
  __syncwarp();
  // ------------------------------------------------------------- epilogue (all 128 threads)
  if (!wait_bounded(done, 0, abort_flag)) {
    fail(p, abort_flag);
  } else if (!*abort_flag) {
    tc_fence_after();
    const int r = warp * 32 + lane;
    const int64_t gi = i0 + r;
    float* g = p.G + gi * p.d + d0;
#pragma unroll 1
    for (int c = 0; c < kN; c += 32) {
      float v[32];
      tmem_ld32(tmem + lane_addr + c, v);
      if (gi < p.m_rows && d0 + c < p.d) {
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          float4 o = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
          if constexpr (ACC) {
            const float4 prev = *reinterpret_cast<const float4*>(g + c + j);
            o.x += prev.x;
            o.y += prev.y;
            o.z += prev.z;
            o.w += prev.w;
          }
          *reinterpret_cast<float4*>(g + c + j) = o;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kN);
  }
}

template <bool ACC>
static cudaError_t setup_one() {
  return cudaFuncSetAttribute(gemm_kernel<ACC>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
}

}  // namespace gemm

cudaError_t gemm_kernel_setup() {
  cudaError_t e;
  if ((e = gemm::setup_one<false>()) != cudaSuccess) return e;
  return gemm::setup_one<true>();
}

cudaError_t launch_gemm(const CUtensorMap& tm_w, const CUtensorMap& tm_yt, const GemmParams& p, bool accumulate,
                        cudaStream_t stream) {
  int pn = p.prefix_end[p.n_prefix - 1];
  dim3 grid(static_cast<unsigned>((pn + gemm::kN - 1) / gemm::kN),
            static_cast<unsigned>((p.m_rows + kTileRows - 1) / kTileRows));
  if (accumulate)
    gemm::gemm_kernel<true><<<grid, gemm::kThreads, gemm::smem_bytes, stream>>>(tm_w, tm_yt, p);
  else
    gemm::gemm_kernel<false><<<grid, gemm::kThreads, gemm::smem_bytes, stream>>>(tm_w, tm_yt, p);
  return cudaGetLastError();
}

}  // namespace ufc
