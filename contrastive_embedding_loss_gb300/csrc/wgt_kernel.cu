// wgt_kernel.cu -- the backward weights of the Matryoshka contrastive loss, written to HBM.
//
// For every cell (i, j) off the diagonal and every prefix k the gradient of the loss
// with respect to the cosine, times the two inverse norms, is
//     m^k_ij = rho_i sigma_j dL/dcos^k_ij
// (CLIP/ROWS: e^{s_ij - tau} rho_i sigma_j (alpha_i + beta_j) with the softmax
// normalisers folded into alpha, beta; SigLIP: sigma(x_ij) rho_i sigma_j w_k t / N).
// On the max-shifted path (large or device-held tau) the row and column probabilities
// take their own shifts, m = w_k (sigma_j 2^(x + a_i) + 2^(x + log2 rho_i + b_j)), with
// a_i = log2(rho_i alpha_i / w_k) - u_i and b_j = log2(sigma_j beta_j / w_k) - v_j from the
// statistics (two exponentials per cell instead of one).
// This kernel recomputes the scores tile by tile exactly like the forward pass (128 x 256
// tcgen05 tiles, the K walk band by band into a cumulative TMEM accumulator, two
// accumulators so the MMA of one tile overlaps the epilogue of the other) and writes m^k
// as bf16 into a [prefix][row][column] array, 32 x 64 blocks per warp through TMA stores.
// For SigLIP it also sums the loss over the negatives.  Both gradient contractions,
// G_A = sum_k m^k B[:, :p_k] and G_B = sum_k (m^k)^T A[:, :p_k], are then dense GEMMs over
// these weights (gemm_kernel.cu): the backward computes the scores once.
//
// Warps (576 threads): 0 TMA, 1 MMA, 2..17 epilogue (warp w reads TMEM lanes 32 (w % 4)..
// and one 64-column quarter of the tile).
//
// Pairs.  Two CTAs (a cluster of 2 along the row blocks) compute their two 128-row blocks'
// score tiles together as one M = 256, N = 256 `tcgen05.mma.cta_group::2`: each CTA stages
// its own 128 rows of X and half (128 rows) of the Y tile, so a CTA's operand traffic per
// tile is two thirds of what a lone 128 x 256 tile needs (16 + 16 KB a K step instead of
// 16 + 32 KB) and three stages fit where two did.  The leader (rank 0) issues the MMAs and
// its barriers count both CTAs' copies; each CTA's epilogue reads its own TMEM.
#include <cuda_bf16.h>

#include <climits>

#include "launch.h"
#include "ptx.cuh"

namespace ufc {
namespace wgt {

constexpr int kCols = 256;
constexpr int kThreads = 576;
constexpr int kEpiWarp0 = 2;
constexpr int kEpiWarps = 16;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kNS = 3;                              // operand stages
constexpr int kXBytes = kTileRows * kChunk * 2;     // 16 KB: this CTA's 128 rows of X
constexpr int kYBytes = (kCols / 2) * kChunk * 2;   // 16 KB: this CTA's half of the Y tile
constexpr int kStageRows = 32;                      // one warp's rows of a weight block
constexpr int kStageBytes = kStageRows * kChunk * 2;  // 4 KB: [32 rows x 64 columns] bf16, 128-byte swizzle
constexpr int kColfBytes = kMaxPrefix * 2 * kCols * 4;  // [prefix][sigma, sigma*beta][256 columns]
constexpr uint64_t kWaitLimitNs = 4000000000ull;

constexpr int off_x = 0;
constexpr int off_y = off_x + kNS * kXBytes;
constexpr int off_stage = off_y + kNS * kYBytes;           // [16 warps][4 KB]
constexpr int off_colf = off_stage + kEpiWarps * kStageBytes;  // four buffers: two tile pairs
constexpr int off_bar = off_colf + 4 * kColfBytes;
constexpr int n_bars = 2 * kNS + 2 + 2 + 1;
constexpr int off_pend = off_bar + n_bars * 8;
constexpr int off_misc = off_pend + 4 * kMaxPrefix;
constexpr int smem_bytes = off_misc + 16 + 1024;
static_assert(smem_bytes <= 232448, "weight kernel shared memory");

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return mbar_wait_abortable(bar, parity, abort_flag, kWaitLimitNs);
}

__device__ __forceinline__ void fail(const WgtParams& p, volatile int* abort_flag) {
  *abort_flag = 1;
  if (p.status) atomicExch(p.status, kStatusTimeout);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Wait until at most `pending` of this thread's bulk store groups are incomplete (the immediate
// of cp.async.bulk.wait_group is a constant; more than 3 waits for all).
__device__ __forceinline__ void bulk_wait_upto(uint32_t pending) {
  switch (pending) {
    case 1: asm volatile("cp.async.bulk.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.bulk.wait_group 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.bulk.wait_group 3;" ::: "memory"); break;
    default: asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); break;
  }
}

// Sums over the warp's 32 rows (one per lane) of 8 columns' values v[0..7]: a reduce-scatter
// over lane bits 4, 3, 2 (each stage keeps half of the values, the upper half where the lane
// bit is set, and adds the partner's copy of it), then a butterfly over bits 1, 0.  Every lane
// ends with the total of column ((lane >> 2) & 7).  A fixed order for every lane.
__device__ __forceinline__ float colsum8(float (&v)[8], int lane) {
#pragma unroll
  for (int st = 0; st < 3; ++st) {
    const int m = 16 >> st, h = 4 >> st;
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float lo = v[i], hi = v[i + h];
      const float got = __shfl_xor_sync(0xffffffffu, upper ? lo : hi, m);
      v[i] = (upper ? hi : lo) + got;
    }
  }
  float t = v[0];
  t += __shfl_xor_sync(0xffffffffu, t, 2);
  t += __shfl_xor_sync(0xffffffffu, t, 1);
  return t;
}

// 8 cells: their weights as four packed bf16 pairs; (SigLIP, R3 != 0) adds the loss and
// the sigmoid of the negatives to acc (.x, .y).  c1, c2: shared addresses of the columns'
// factors.  CHECK evaluates the masks (padding rows and columns, the positive's cell).
template <int KIND, bool CHECK>
__device__ __forceinline__ uint4 cells8(const float* dot, uint32_t c1, uint32_t c2, float R1, float R2, float R3,
                                        float L, float b2, int col0, int ncols, int dcol, bool row_ok, float2& acc) {
  const float4 s1a = ld_shared_v4f(c1), s1b = ld_shared_v4f(c1 + 16);
  const float s1v[8] = {s1a.x, s1a.y, s1a.z, s1a.w, s1b.x, s1b.y, s1b.z, s1b.w};
  float s2v[8];
  if constexpr (KIND != KIND_SIGLIP) {
    const float4 s2a = ld_shared_v4f(c2), s2b = ld_shared_v4f(c2 + 16);
    s2v[0] = s2a.x; s2v[1] = s2a.y; s2v[2] = s2a.z; s2v[3] = s2a.w;
    s2v[4] = s2b.x; s2v[5] = s2b.y; s2v[6] = s2b.z; s2v[7] = s2b.w;
  }
  uint32_t packed[4];
  if constexpr (KIND == KIND_SIGLIP) {
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      float mv[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int jj = j + u;
        const float s1 = s1v[jj];
        bool keep = true;
        if constexpr (CHECK) {
          const int col = col0 + jj;
          keep = row_ok && col < ncols && col != dcol;
        }
        const float x2 = fmaf(R1 * s1, dot[jj], b2);
        const float e = ex2_approx(-fabsf(x2));
        const float d = 1.f + e;
        const float r = rcp_approx(d);
        const float sig = x2 >= 0.f ? r : e * r;
        float m = sig * (R2 * s1);
        if (R3 != 0.f) {  // this launch also sums the SigLIP loss
          const float l = fmaxf(x2, 0.f) + lg2_approx(d);
          acc.x += keep ? l : 0.f;
          acc.y += keep ? sig : 0.f;
        }
        if constexpr (CHECK) m = keep ? m : 0.f;
        mv[u] = m;
      }
      packed[j / 2] = pack_bf16x2(mv[0], mv[1]);
    }
  } else {
    // two cells per packed instruction: x = R1 sigma dot - L, e = 2^x, m = e (R2 sigma + R3 sigma beta)
    const float2 r1 = make_float2(R1, R1), r2 = make_float2(R2, R2), r3 = make_float2(R3, R3);
    const float2 nl = make_float2(-L, -L);
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      const float2 s1 = make_float2(s1v[j], s1v[j + 1]);
      const float2 s2 = make_float2(s2v[j], s2v[j + 1]);
      const float2 x = fma2(mul2(r1, s1), make_float2(dot[j], dot[j + 1]), nl);
      const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
      float2 m = mul2(e, fma2(r2, s1, mul2(r3, s2)));
      if constexpr (CHECK) {
        const int col = col0 + j;
        if (!(row_ok && col < ncols && col != dcol)) m.x = 0.f;
        if (!(row_ok && col + 1 < ncols && col + 1 != dcol)) m.y = 0.f;
      }
      packed[j / 2] = pack_bf16x2(m.x, m.y);
    }
  }
  return make_uint4(packed[0], packed[1], packed[2], packed[3]);
}

// The max-shifted variant of cells8 (CLIP/ROWS): R1 = L rho_i, A = a_i, Bl = log2 rho_i,
// wk = w_k; c2 holds b_j (CLIP).  Masks as in cells8.
template <int KIND, bool CHECK>
__device__ __forceinline__ uint4 cells8_shifted(const float* dot, uint32_t c1, uint32_t c2, float R1, float A, float Bl,
                                                float wk, int col0, int ncols, int dcol, bool row_ok) {
  const float4 s1a = ld_shared_v4f(c1), s1b = ld_shared_v4f(c1 + 16);
  const float s1v[8] = {s1a.x, s1a.y, s1a.z, s1a.w, s1b.x, s1b.y, s1b.z, s1b.w};
  float s2v[8];
  if constexpr (KIND == KIND_CLIP) {
    const float4 s2a = ld_shared_v4f(c2), s2b = ld_shared_v4f(c2 + 16);
    s2v[0] = s2a.x; s2v[1] = s2a.y; s2v[2] = s2a.z; s2v[3] = s2a.w;
    s2v[4] = s2b.x; s2v[5] = s2b.y; s2v[6] = s2b.z; s2v[7] = s2b.w;
  }
  uint32_t packed[4];
  const float2 r1 = make_float2(R1, R1), ra = make_float2(A, A), rb = make_float2(Bl, Bl), w2 = make_float2(wk, wk);
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    const float2 s1 = make_float2(s1v[j], s1v[j + 1]);
    const float2 x = mul2(mul2(r1, s1), make_float2(dot[j], dot[j + 1]));
    const float2 t1 = add2(x, ra);
    float2 m = mul2(s1, make_float2(ex2_approx(t1.x), ex2_approx(t1.y)));
    if constexpr (KIND == KIND_CLIP) {
      const float2 t2 = add2(add2(x, make_float2(s2v[j], s2v[j + 1])), rb);
      m = add2(m, make_float2(ex2_approx(t2.x), ex2_approx(t2.y)));
    }
    m = mul2(m, w2);
    if constexpr (CHECK) {
      const int col = col0 + j;
      if (!(row_ok && col < ncols && col != dcol)) m.x = 0.f;
      if (!(row_ok && col + 1 < ncols && col + 1 != dcol)) m.y = 0.f;
    }
    packed[j / 2] = pack_bf16x2(m.x, m.y);
  }
  return make_uint4(packed[0], packed[1], packed[2], packed[3]);
}

// Tiles in pairs (t even in accumulator 0, t + 1 in accumulator 1), band by band,
// alternating within a pair.  Step s -> (tile, band); producer, MMA and epilogue all walk it.
struct Schedule {
  int T, n;
  __device__ int steps() const { return T * n; }
  __device__ void at(int s, int& t, int& b) const {
    const int pair = s / (2 * n);
    const int rem = s - pair * 2 * n;
    const int tp = 2 * pair;
    const int width = (tp + 1 < T) ? 2 : 1;  // the last pair may hold one tile
    b = rem / width;
    t = tp + rem % width;
  }
};

// MERGE: the two widest prefixes' weights merged (WgtParams::merge); a separate instantiation,
// so that the kernels without it carry none of its code.
template <int KIND, bool SHIFTED, bool MERGE>
__global__ void __launch_bounds__(kThreads, 1)
    wgt_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_y,
               const __grid_constant__ CUtensorMap tm_w, const WgtParams p) {
  griddep_enter();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sx = smem + off_x;
  uint8_t* sy = smem + off_y;
  uint64_t* s_full = reinterpret_cast<uint64_t*>(smem + off_bar);
  uint64_t* s_empty = s_full + kNS;
  uint64_t* acc_full = s_empty + kNS;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  int* pend = reinterpret_cast<int*>(smem + off_pend);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + off_misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + off_misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // 0: the leader, which issues the pair's MMAs
  const int64_t il0 = static_cast<int64_t>(blockIdx.x) * kTileRows;  // first row within this launch
  const int64_t i0 = p.row0 + il0;                                    // first row of X
  const int split = blockIdx.y;
  const int n = p.n_prefix;
  const int t_begin = split * p.tiles_per_split;
  const int T = min(p.n_col_tiles, t_begin + p.tiles_per_split) - t_begin;
  const Schedule sched{T, n};

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 2 * kEpiWarps);  // the epilogue warps of both CTAs (leader's copy)
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
#pragma unroll
    for (int k = 0; k < kMaxPrefix; ++k) pend[k] = p.prefix_end[k];
    fence_mbar_init();
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_y);
    tma_prefetch_desc(&tm_w);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);  // the same columns in both SMs of the pair
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (T > 0 && warp == 0 && lane == 0) {
    // ------------------------------------------------------------- operand producer
    // Both CTAs copy their parts into their own shared memory; completion is counted on the
    // leader's barrier, which the leader arms for the bytes of both.
    uint32_t it = 0;
    bool ok = true;
    for (int s = 0; s < sched.steps() && ok; ++s) {
      int t, b;
      sched.at(s, t, b);
      const int j0 = static_cast<int>(p.col0) + (t_begin + t) * kCols;
      const int c0 = b == 0 ? 0 : pend[b - 1] / kChunk, c1 = pend[b] / kChunk;
      for (int c = c0; c < c1; ++c, ++it) {
        const uint32_t st = it % kNS, ph = (it / kNS) & 1;
        if (!wait_bounded(&s_empty[st], ph ^ 1, abort_flag)) {
          fail(p, abort_flag);
          ok = false;
          break;
        }
        const uint32_t bar = mapa_shared(smem_u32(&s_full[st]), 0);
        if (rank == 0) mbar_arrive_expect_tx(&s_full[st], 2 * (kXBytes + kYBytes));
        tma_load_2d_pair(sx + st * kXBytes, &tm_x, bar, c * kChunk, static_cast<int>(i0));
        tma_load_2d_pair(sy + st * kYBytes, &tm_y, bar, c * kChunk, j0 + static_cast<int>(rank) * (kCols / 2));
      }
    }
    if (rank == 0) {
      for (uint32_t k = 0; k < kNS && k < it; ++k) {  // let the last copies land
        const uint32_t q = it - 1 - k;
        mbar_wait(&s_full[q % kNS], (q / kNS) & 1, kWaitLimitNs);
      }
    } else {
      // the follower's copies are counted on the leader's barriers: wait until the MMAs that
      // read them (hence the copies) are done, i.e. the last stages are released
      for (uint32_t k = 0; k < kNS && k < it; ++k) {
        const uint32_t q = it - 1 - k;
        mbar_wait(&s_empty[q % kNS], (q / kNS) & 1, kWaitLimitNs);
      }
    }
  } else if (T > 0 && warp == 1 && lane == 0 && rank == 0) {
    // ------------------------------------------------------------- MMA issuer (leader)
    const uint32_t idesc = idesc_bf16_f32(2 * kTileRows, kCols);
    uint32_t it = 0;
    uint32_t uses0 = 0, uses1 = 0;  // uses of each accumulator (scalars: a runtime index would put them in local memory)
    bool ok = true;
    for (int s = 0; s < sched.steps() && ok; ++s) {
      int t, b;
      sched.at(s, t, b);
      const int a = t & 1;
      const uint32_t ua = a ? uses1 : uses0;
      if (ua > 0 && !wait_bounded(&acc_empty[a], (ua - 1) & 1, abort_flag)) {
        fail(p, abort_flag);
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem + a * kCols;
      const int c0 = b == 0 ? 0 : pend[b - 1] / kChunk, c1 = pend[b] / kChunk;
      for (int c = c0; c < c1; ++c, ++it) {
        const uint32_t st = it % kNS, ph = (it / kNS) & 1;
        if (!wait_bounded(&s_full[st], ph, abort_flag)) {
          fail(p, abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ax = smem_u32(sx + st * kXBytes), ay = smem_u32(sy + st * kYBytes);
#pragma unroll
        for (int kk = 0; kk < kChunk / 16; ++kk)  // bands accumulate: only a tile's first step starts fresh
          umma_bf16_pair(d, sdesc_kmajor_sw128(ax + kk * 32), sdesc_kmajor_sw128(ay + kk * 32), idesc,
                         (c != 0 || kk != 0) ? 1u : 0u);
        umma_commit_pair(&s_empty[st]);  // releases the stage in both CTAs
      }
      if (ok) umma_commit_pair(&acc_full[a]);
      if (a) ++uses1; else ++uses0;
    }
    umma_commit_pair(drain);
    mbar_wait(drain, 0, kWaitLimitNs);
  } else if (T > 0 && warp == 1 && lane == 0) {
    mbar_wait(drain, 0, kWaitLimitNs);  // the follower: the pair's last MMAs are done
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------- epilogue
    const int q = warp & 3;                       // TMEM lane quadrant (rows 32q..32q+31)
    const int ew = warp - kEpiWarp0;
    const int cq = ew >> 2;                       // column quarter (64 columns)
    const int r = q * 32 + lane;
    const int64_t gi = i0 + r;
    const bool row_ok = il0 + r < p.rows;
    const int etid = threadIdx.x - kEpiWarp0 * 32;
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t colf_s = smem_u32(smem + off_colf);
    uint8_t* stage = smem + off_stage + ew * kStageBytes;
    const uint32_t stage_row = smem_u32(stage) + (lane >> 3) * 1024 + (lane & 7) * 128;  // row `lane` of the block
    const uint32_t swz = lane & 7;
    // column factors of tile t live in buffer t & 3; a tile pair's factors are fetched by
    // cp.async while the previous pair is processed
    auto prefetch_colf = [&](int t) {
      const int64_t j0 = p.col0 + static_cast<int64_t>(t_begin + t) * kCols;
      const uint32_t dst = colf_s + (t & 3) * kColfBytes;
      for (int e = etid; e < n * 2 * kCols; e += kEpiThreads) {
        const int k = e / (2 * kCols), f = (e / kCols) & 1, c = e % kCols;
        const int64_t gj = j0 + c;
        const float* src = f == 0 ? p.rinv_y : p.beta_y;
        const bool v = src != nullptr && gj < p.ny;
        cp_async4_u32(dst + e * 4, v ? src + static_cast<int64_t>(k) * p.ny + gj : p.rinv_y, v ? 4u : 0u);
      }
    };
    for (int t = 0; t < 2 && t < T; ++t) prefetch_colf(t);
    cp_async_commit();
    // raw row factors of the next band (rho_i, and rho_i alpha_i for CLIP/ROWS), loaded one
    // band ahead
    float n_rho = 0.f, n_alpha = 0.f;
    auto load_row = [&](int k) {
      n_rho = row_ok ? p.rinv_x[static_cast<int64_t>(k) * p.nx + gi] : 0.f;
      if constexpr (KIND != KIND_SIGLIP)
        n_alpha = (row_ok && p.alpha_x) ? p.alpha_x[static_cast<int64_t>(k) * p.nx + gi] : 0.f;
    };
    if (T > 0) load_row(0);
    const float L = p.sc.t() * 1.4426950408889634f;
    const float b2 = p.sc.b() * 1.4426950408889634f;
    const float t_sc = p.sc.t();
    const int64_t slot_off = static_cast<int64_t>(split * 4 + cq) * n * p.nx + gi;
    const float siglip_loss = (KIND == KIND_SIGLIP && p.rowacc) ? 1.f : 0.f;
    const int64_t wrow = static_cast<int64_t>(il0) + q * 32;  // this warp's first row in the weight array
    const uint64_t l2_evict_first = l2_policy_evict_first();
    uint32_t uses = 0;  // uses of each accumulator so far (both advance together)
    bool ok = true;
    // merge: this row's sum over the tiles of W^{n-1} d^{n-1}; the CTA's 128-row block index
    float r5acc = 0.f;
    const int64_t rblk = i0 / kTileRows;
    // (lane 0) bulk store groups committed so far, and the count just after each tile's prefix
    // n-2 store (merge: how many later groups may still be pending when that block is added to)
    uint32_t ncommit = 0, c4_0 = 0, c4_1 = 0;
    // the schedule of Schedule::at as nested loops: tile pairs, bands, the pair's tiles
    for (int tp = 0; tp < T; tp += 2) {
      const int width = tp + 1 < T ? 2 : 1;
      // a tile pair begins (every warp reaches this point at the same step)
      named_bar_sync(1, kEpiThreads);          // all are done with the previous pair
      for (int u = 2; u < 4 && tp + u < T; ++u) prefetch_colf(tp + u);
      cp_async_commit();
      cp_async_wait<1>();                      // this pair's factors (fetched a pair ago) are in
      named_bar_sync(1, kEpiThreads);
      for (int b = 0; b < n; ++b, ++uses) {
        const int k = b;
        // this band's row factors, then the next band's (or the next pair's first) in flight
        const float rho = n_rho;
        float R2, R3;
        if constexpr (KIND == KIND_SIGLIP) {
          float ms = 0.f;
#pragma unroll
          for (int kk = 0; kk < kMaxPrefix; ++kk)
            if (kk == k) ms = p.m_scale[kk];
          R2 = rho * ms * t_sc;  // rho_i w_k t / N
          R3 = siglip_loss;
        } else if constexpr (SHIFTED) {
          R2 = n_alpha;          // a_i
          R3 = lg2_approx(rho);  // log2 rho_i
        } else {
          R2 = n_alpha;          // rho_i alpha_i
          R3 = rho;
        }
        float wk = 0.f;
        if constexpr (SHIFTED) {
#pragma unroll
          for (int kk = 0; kk < kMaxPrefix; ++kk)
            if (kk == k) wk = p.m_scale[kk];
        }
        const float R1 = L * rho;
        load_row(b + 1 < n ? b + 1 : 0);
        for (int u = 0; u < width; ++u) {
          const int t = tp + u;
          const int a = u;
          if (!ok) continue;
          if (!wait_bounded(&acc_full[a], uses & 1, abort_flag)) {
            fail(p, abort_flag);
            ok = false;
            continue;
          }
          tc_fence_after();
          // this warp's 64 columns as two 32-column halves, the second read once the first is
          // processed (32 fewer live registers: the SigLIP and max-shifted epilogues no longer
          // spill); the accumulator is released after the second read
          float v0[32], v1[32];
          const uint32_t ta = tmem + lane_addr + a * kCols + cq * 64;
          tmem_ld32(ta, v0);
          const int64_t j0 = p.col0 + static_cast<int64_t>(t_begin + t) * kCols;  // first column of Y
          const int64_t left = p.col0 + p.cols - j0;  // columns of this launch left in the tile
          const int ncols = left < kCols ? static_cast<int>(left) : kCols;
          const int64_t dtile = i0 - j0;  // uniform over the CTA: does this tile hold any positive?
          const bool check = ncols < kCols || (dtile > -kTileRows && dtile < kCols) || (il0 + kTileRows > p.rows);
          // tile column of this row's positive (none when a label matrix names the positives:
          // every cell is then written as a negative and the positives are patched afterwards)
          const int diag_col = p.no_diag ? INT_MIN : static_cast<int>(dtile) + r;
          const uint32_t cf = colf_s + (t & 3) * kColfBytes + cq * 64 * 4;
          const uint32_t c1 = cf + (k * 2 + 0) * kCols * 4;
          const uint32_t c2 = cf + (k * 2 + 1) * kCols * 4;
          // the previous TMA store of this warp must have read its staging block
          if (lane == 0) bulk_wait_read0();
          __syncwarp();
          float2 al = make_float2(0.f, 0.f);
          // four 8-column chunks of one half (vh: its 32 values; chb: its first chunk); the mask
          // test is hoisted out of the unrolled loops
          // merge, at prefix n-1: the stored weights W times the raw dots, into the row sum and
          // (over the warp's 32 rows) into this 32-row block's column sums
          const bool mtop = MERGE && k == n - 1;
          // this lane's column-sum slot of the tile's first 8-column chunk (lanes 4c hold column c)
          const int64_t gj_lane = j0 + cq * 64 + ((lane >> 2) & 7);
          float* const r5_lane = MERGE ? p.r5_col + (rblk * 4 + q) * p.ny + gj_lane : nullptr;
          const bool r5_writes = (lane & 3) == 0 && il0 < p.rows;
          auto r5_cells = [&](const uint4 pk, const float* vd, int ch) {
            const uint32_t w[4] = {pk.x, pk.y, pk.z, pk.w};
            float pr[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              pr[2 * e] = bf16_lo(w[e]) * vd[2 * e];
              pr[2 * e + 1] = bf16_hi(w[e]) * vd[2 * e + 1];
            }
            r5acc += ((pr[0] + pr[1]) + (pr[2] + pr[3])) + ((pr[4] + pr[5]) + (pr[6] + pr[7]));
            const float col = colsum8(pr, lane);
            if (r5_writes && gj_lane + ch * 8 < p.ny) r5_lane[ch * 8] = col;
          };
          // four 8-column chunks of one half (vh: its 32 values; chb: its first chunk); the mask
          // test is hoisted out of the unrolled loops
          auto chunks = [&](const float* vh, int chb) {
            const uint32_t dst = stage_row, f1 = c1 + chb * 32, f2 = c2 + chb * 32;
            const int col0 = cq * 64 + chb * 8;
            auto put = [&](int cc, const uint4 pk) {
              st_shared_v4(dst + (((chb + cc) ^ swz) << 4), pk);
              if constexpr (MERGE)
                if (mtop) r5_cells(pk, vh + cc * 8, chb + cc);
            };
            if constexpr (SHIFTED) {
              if (check) {
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                  put(cc, cells8_shifted<KIND, true>(vh + cc * 8, f1 + cc * 32, f2 + cc * 32, R1, R2, R3, wk,
                                                     col0 + cc * 8, ncols, diag_col, row_ok));
              } else {
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                  put(cc, cells8_shifted<KIND, false>(vh + cc * 8, f1 + cc * 32, f2 + cc * 32, R1, R2, R3, wk, 0, 0,
                                                      0, true));
              }
            } else if (check) {
#pragma unroll
              for (int cc = 0; cc < 4; ++cc)
                put(cc, cells8<KIND, true>(vh + cc * 8, f1 + cc * 32, f2 + cc * 32, R1, R2, R3, L, b2, col0 + cc * 8,
                                           ncols, diag_col, row_ok, al));
            } else {
#pragma unroll
              for (int cc = 0; cc < 4; ++cc)
                put(cc, cells8<KIND, false>(vh + cc * 8, f1 + cc * 32, f2 + cc * 32, R1, R2, R3, L, b2, 0, 0, 0, true,
                                            al));
            }
          };
          chunks(v0, 0);
          tmem_ld32(ta + 32, v1);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&acc_empty[a]), 0));  // the leader's copy
          chunks(v1, 4);
          fence_proxy_async_smem();
          __syncwarp();
          // a quarter wholly past the last column stores nothing, nor does the second CTA of
          // a pair that lies wholly past the launch's rows (its rows are not in the chunk)
          const bool stores = il0 < p.rows && j0 + cq * 64 < p.col0 + p.cols;  // (uniform over the warp)
          if (lane == 0 && stores) {
            // the weights are written once here and read back by the GEMMs much later: keep
            // them from evicting the score operands, which every CTA re-reads (merge: prefix
            // n-2's block is added to at prefix n-1, a few microseconds later, so it stays in L2
            // as a normal line)
            const int wc = static_cast<int>(j0 - p.col0 + cq * 64);
            const int wr = static_cast<int>(static_cast<int64_t>(k) * p.w_rows_per_prefix + wrow);
            if (MERGE && k == n - 2)
              tma_store_2d(&tm_w, stage, wc, wr);
            else
              tma_store_2d_hint(&tm_w, stage, wc, wr, l2_evict_first);
            bulk_commit();
            ++ncommit;
            if (MERGE && k == n - 2) (u ? c4_1 : c4_0) = ncommit;
            if (MERGE && mtop) {
              // prefix n-2's block of this tile (stored a snapshot or two ago) becomes
              // bf16(W^{n-1} + W^{n-2}): once that store has completed (the groups committed
              // after it may still run), the staging block, which holds W^{n-1}, is
              // reduce-added onto it in L2
              bulk_wait_upto(ncommit - (u ? c4_1 : c4_0));
              tma_reduce_add_2d_hint(&tm_w, stage, wc, wr - static_cast<int>(p.w_rows_per_prefix), l2_evict_first);
              bulk_commit();
              ++ncommit;
            }
          }
          if (KIND == KIND_SIGLIP && p.rowacc && row_ok) {
            float* pl = p.rowacc + slot_off + static_cast<int64_t>(k) * p.nx;
            if (t == 0 && !p.add_rows) *pl = al.x;
            else atomicAdd(pl, al.x);
            if (p.rowsig) {
              float* ps = p.rowsig + slot_off + static_cast<int64_t>(k) * p.nx;
              if (t == 0 && !p.add_rows) *ps = al.y;
              else atomicAdd(ps, al.y);
            }
          }
        }
      }
    }
    cp_async_wait<0>();
    if constexpr (MERGE)
      if (row_ok && T > 0) p.r5_row[static_cast<int64_t>(split * 4 + cq) * p.nx + gi] = r5acc;
    if (lane == 0) bulk_wait0();  // the weights are in global memory before the CTA exits
  }

  tc_fence_before();
  cluster_sync_all();  // no MMA, copy or remote arrive of the pair is still in flight
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

template <int KIND, bool SHIFTED>
static cudaError_t setup_one() {
  cudaError_t e = cudaFuncSetAttribute(wgt_kernel<KIND, SHIFTED, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem_bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(wgt_kernel<KIND, SHIFTED, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              smem_bytes);
}

}  // namespace wgt

cudaError_t wgt_kernel_setup() {
  cudaError_t e;
  if ((e = wgt::setup_one<KIND_CLIP, false>()) != cudaSuccess) return e;
  if ((e = wgt::setup_one<KIND_CLIP, true>()) != cudaSuccess) return e;
  if ((e = wgt::setup_one<KIND_SIGLIP, false>()) != cudaSuccess) return e;
  if ((e = wgt::setup_one<KIND_ROWS, false>()) != cudaSuccess) return e;
  return wgt::setup_one<KIND_ROWS, true>();
}

cudaError_t launch_wgt(int kind, const CUtensorMap& tm_x, const CUtensorMap& tm_y, const CUtensorMap& tm_w,
                       const WgtParams& p, dim3 grid, cudaStream_t stream) {
  using wgt::wgt_kernel;
  if (kind == KIND_SIGLIP && p.shifted) return cudaErrorInvalidValue;
  const dim3 g((grid.x + 1) / 2 * 2, grid.y, 1), blk(wgt::kThreads);  // CTA pairs along the row blocks
  const size_t sm = wgt::smem_bytes;
#define UF_WGT(K, SH)                                                                                      \
  (p.merge ? launch_pdl(wgt_kernel<K, SH, true>, g, blk, sm, stream, 2, tm_x, tm_y, tm_w, p)              \
           : launch_pdl(wgt_kernel<K, SH, false>, g, blk, sm, stream, 2, tm_x, tm_y, tm_w, p))
  if (kind == KIND_CLIP) return p.shifted ? UF_WGT(KIND_CLIP, true) : UF_WGT(KIND_CLIP, false);
  if (kind == KIND_SIGLIP) return UF_WGT(KIND_SIGLIP, false);
  return p.shifted ? UF_WGT(KIND_ROWS, true) : UF_WGT(KIND_ROWS, false);
#undef UF_WGT
}

}  // namespace ufc
