// fwd_kernel.cu -- forward statistics of the Matryoshka contrastive loss in one pass:
// per row i of X and prefix k the sum over the negatives of exp(s_ij - tau) (CLIP, ROWS)
// or of softplus(x_ij) (SigLIP, log2 units), and for CLIP also the same sums per column
// j of Y (so the column softmax needs no second pass over the grid).
//
// Tiles.  A CTA owns 128 rows of X and walks 256-row tiles of Y.  The score tile is one
// 128 x 256 tcgen05 MMA per K step (N = 256 keeps the tensor pipe at full rate; 128-wide
// tiles ran at about half rate on this part).  The K walk goes band by band (a band is
// the dimensions between consecutive prefix ends) and accumulates into one TMEM
// accumulator, so after band k the accumulator holds the prefix-k dot products: the
// epilogue reads that snapshot, releases the accumulator for the next band, and
// evaluates prefix k.  Two accumulators (512 TMEM columns) let the MMA run the next tile's
// band while the epilogue reads this one's.
//
// Epilogue.  16 warps: warp w reads TMEM lanes 32 (w % 4) .. +31 (its rows) and one
// quarter (64 columns) of the tile, half of it at a time.  Row-only sums (ROWS, SigLIP) use
// the 32x32b layout: a lane holds one row, read as two 32-column groups.  With column sums
// (CLIP) the 16x256b layout puts a column's 32 cells 4 to a lane on 8 lanes (two 16-row
// halves), so the column sums are in-thread adds and a 3-stage scatter over 8 lanes; the
// four row-quadrant warps of a column quarter combine through shared memory, and one of them
// writes the 128-row partial of every column to global memory (one slot per row block; a
// reduction kernel adds the slots in a fixed order).
//
// Shifts.  The default sums 2^(x - L) with x = tau log2(e) cos and the fixed shift L =
// tau log2(e): |cos| <= 1 keeps every term in [2^-2L, 1], normal fp32 while tau <= 40.
// Beyond that (or when tau is only known on the device) the same kernel runs twice: a
// max pass (kFwdMax) finds every row's and column's largest x, then a shifted pass
// (kFwdShifted) sums 2^(x - u_i) for the row and 2^(x - v_j) for the column, u and v
// those maxima, so the largest term of every sum is 1 whatever the scale.
#include <cuda_bf16.h>

#include <climits>

#include "launch.h"
#include "ptx.cuh"

namespace ufc {

namespace fwd {

constexpr int kCols = 256;                         // score tile N
constexpr int kThreads = 576;                      // warp 0 TMA, warp 1 MMA, warps 2..17 epilogue
constexpr int kEpiWarp0 = 2;
constexpr int kEpiWarps = 16;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kNS = 3;                             // operand stages
constexpr int kXBytes = kTileRows * kChunk * 2;    // 16 KB
constexpr int kYBytes = kCols * kChunk * 2;        // 32 KB
constexpr uint64_t kWaitLimitNs = 4000000000ull;

constexpr int off_x = 0;
constexpr int off_y = off_x + kNS * kXBytes;
constexpr int off_colf = off_y + kNS * kYBytes;                    // [4][kMaxPrefix][256] sigma_j
constexpr int off_colsh = off_colf + 4 * kMaxPrefix * kCols * 4;   // [4][kMaxPrefix][256] v_j (shifted, CLIP)
constexpr int off_rowf = off_colsh + 4 * kMaxPrefix * kCols * 4;   // [kMaxPrefix][128] L rho_i
constexpr int off_rowsh = off_rowf + kMaxPrefix * kTileRows * 4;   // [kMaxPrefix][128] u_i (shifted)
constexpr int off_cpart = off_rowsh + kMaxPrefix * kTileRows * 4;  // [2][4 quarters][4 quadrants][64]
constexpr int off_bar = off_cpart + 2 * 4 * 4 * 64 * 4;
constexpr int n_bars = 2 * kNS + 2 + 2 + 1;
constexpr int off_misc = off_bar + n_bars * 8;
constexpr int smem_bytes = off_misc + 16 + 1024;  // + slack for 1024-byte alignment
static_assert(smem_bytes <= 232448, "forward shared memory");

struct Params {
  int64_t nx, ny;
  int n_prefix;
  int prefix_end[kMaxPrefix];
  int n_col_tiles;      // ceil(ny / 256)
  int tiles_per_split;
  Scalars sc;           // tau or t, and b: L = scale log2(e) (also the fixed shift), b2 = bias log2(e)
  const float* rinv_x;  // [n][nx]
  const float* rinv_y;  // [n][ny]
  const float* shift_x; // kFwdShifted: [n][nx]
  const float* shift_y; // kFwdShifted, CLIP: [n][ny]
  int no_diag;          // the diagonal cells are not masked (SigLIP with a label matrix)
  float* rowacc;        // [split * 4 + quarter][n][nx]
  float* colacc;        // [row block][n][ny] (CLIP) or NULL
  int* status;
};

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return mbar_wait_abortable(bar, parity, abort_flag, kWaitLimitNs);
}

__device__ __forceinline__ void fail(const Params& p, volatile int* abort_flag) {
  *abort_flag = 1;
  if (p.status) atomicExch(p.status, kStatusTimeout);
}

// The row-only epilogues (ROWS, SigLIP) on the 32x32b TMEM layout: a lane holds one row and
// the warp's 64 columns of it arrive as two 32-column groups.  Each function takes group g
// (v: its 32 values; columns g*32 .. g*32+31 of the warp's quarter) and adds to rs, two
// interleaved row accumulators.  CHECK evaluates the masks (padding columns and rows, the
// positive's diagonal cell).

// Sums of 2^(R1 sigma_j dot - L) (CLIP/ROWS) or softplus(x) in log2 units (SigLIP).
template <int KIND, bool CHECK>
__device__ __forceinline__ void fwd_cells(const float (&v)[32], int g, const float* cf, float R1, float L, float b2,
                                          int col_base, int ncols, int dcol, bool row_ok, float2& rs) {
  const float2 r1 = make_float2(R1, R1), nl = make_float2(-L, -L);
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const int c = g * 32 + j;
    float2 val;
    if constexpr (KIND == KIND_SIGLIP) {
      float w[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float x2 = fmaf(R1 * cf[c + u], v[j + u], b2);
        w[u] = fmaxf(x2, 0.f) + lg2_approx(1.f + ex2_approx(-fabsf(x2)));
      }
      val = make_float2(w[0], w[1]);
    } else {
      // two cells per packed instruction
      const float2 x = fma2(mul2(r1, make_float2(cf[c], cf[c + 1])), make_float2(v[j], v[j + 1]), nl);
      val = make_float2(ex2_approx(x.x), ex2_approx(x.y));
    }
    if constexpr (CHECK) {
      const int col = col_base + c;
      if (!(row_ok && col < ncols && col != dcol)) val.x = 0.f;
      if (!(row_ok && col + 1 < ncols && col + 1 != dcol)) val.y = 0.f;
    }
    rs = add2(rs, val);
  }
}

// kFwdMax: the running maxima of x = R1 sigma_j dot.  Only padding is masked (to -inf).
template <bool CHECK>
__device__ __forceinline__ void fwd_cells_max(const float (&v)[32], int g, const float* cf, float R1, int col_base,
                                              int ncols, bool row_ok, float2& rm) {
  const float2 r1 = make_float2(R1, R1);
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const int c = g * 32 + j;
    // the same two roundings as fwd_cells_shifted, so that x - u_i <= 0 holds exactly there
    float2 val = mul2(mul2(r1, make_float2(cf[c], cf[c + 1])), make_float2(v[j], v[j + 1]));
    if constexpr (CHECK) {
      const int col = col_base + c;
      if (!(row_ok && col < ncols)) val.x = -INFINITY;
      if (!(row_ok && col + 1 < ncols)) val.y = -INFINITY;
    }
    rm = make_float2(fmaxf(rm.x, val.x), fmaxf(rm.y, val.y));
  }
}

// kFwdShifted: sums of 2^(x - U), U the row's shift.  Masks as in fwd_cells.
template <bool CHECK>
__device__ __forceinline__ void fwd_cells_shifted(const float (&v)[32], int g, const float* cf, float R1, float U,
                                                  int col_base, int ncols, int dcol, bool row_ok, float2& rs) {
  const float2 r1 = make_float2(R1, R1), nu = make_float2(-U, -U);
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const int c = g * 32 + j;
    const float2 x = mul2(mul2(r1, make_float2(cf[c], cf[c + 1])), make_float2(v[j], v[j + 1]));
    const float2 xr = add2(x, nu);
    float2 er = make_float2(ex2_approx(xr.x), ex2_approx(xr.y));
    if constexpr (CHECK) {
      const int col = col_base + c;
      if (!(row_ok && col < ncols && col != dcol)) er.x = 0.f;
      if (!(row_ok && col + 1 < ncols && col + 1 != dcol)) er.y = 0.f;
    }
    rs = add2(rs, er);
  }
}

// Reduce-scatter of NV values over the 2^STAGES lanes that differ in lane bits M0, M0/2, ...:
// each stage keeps half of the values (the upper half where the lane bit is set) and adds
// (MAX: takes the maximum of) the partner's other half, so lane bits (M0, M0/2, ...) select,
// from the most significant, which NV / 2^STAGES values a lane ends with in v[0..].
template <bool MAX, int NV, int M0, int STAGES>
__device__ __forceinline__ void reduce_scatter_bits(float (&v)[NV], int lane) {
#pragma unroll
  for (int st = 0; st < STAGES; ++st) {
    const int m = M0 >> st, h = NV >> (st + 1);
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float lo = v[i], hi = v[i + h];
      const float send = upper ? lo : hi;
      const float keep = upper ? hi : lo;
      const float got = __shfl_xor_sync(0xffffffffu, send, m);
      v[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
}

// The column-summing (CLIP) epilogue on the 16x256b TMEM layout: v[0..31] and v[32..63] are
// the warp's rows 0-15 and 16-31 (of its 32-row quadrant q), 64 columns; lane l = 4 g + c
// holds rows {g, g + 8} of each half and columns 8 r + 2 c + {0, 1}, r = 0..7 (register
// 4 r + 2 s + b of a half: row g + 8 s, column 8 r + 2 c + b).  A column's 32 cells then sit
// 4 to a lane on 8 lanes, so the column sums are in-thread adds and a 3-stage scatter over 8
// lanes (instead of 31 exchanges per 32 columns on the 32x32b layout), and a row's 16 cells
// per lane meet over 4 lanes.  MODE as in the kernel; rf, ru: this prefix's row factors
// L rho and (kFwdShifted) row shifts for the tile's 128 rows; cf, vs: the quarter's column
// factors sigma and (kFwdShifted) column shifts.  Returns the row value of the lane's own row
// (32 q + 16 (c >> 1) + g + 8 (c & 1)); the warp's 32-row column partials go to cp[0..63].
template <int MODE, bool CHECK>
__device__ __forceinline__ void fwd_cells16_half(const float (&v)[32], int h, const float* cf, const float* vs,
                                                 const float* rf, const float* ru, float L, int q, int lane,
                                                 int col_base, int ncols, int dtile, int rows_left, float2 (&rs)[4],
                                                 float2 (&cs)[8]) {
  const int g = lane >> 2, c4 = lane & 3;
  float R1[2], U[2];
#pragma unroll
  for (int sub = 0; sub < 2; ++sub) {
    const int row = q * 32 + 16 * h + g + 8 * sub;
    R1[sub] = rf[row];
    U[sub] = MODE == kFwdShifted ? ru[row] : 0.f;
  }
  const float2 nl = make_float2(-L, -L);
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int c = 8 * r + 2 * c4;  // column within the quarter
    const float2 sg = *reinterpret_cast<const float2*>(cf + c);
    float2 nv = make_float2(0.f, 0.f);
    if constexpr (MODE == kFwdShifted) {
      const float2 vv = *reinterpret_cast<const float2*>(vs + c);
      nv = make_float2(-vv.x, -vv.y);
    }
#pragma unroll
    for (int sub = 0; sub < 2; ++sub) {
      const int idx = 2 * h + sub;
      const float2 d = make_float2(v[r * 4 + 2 * sub], v[r * 4 + 2 * sub + 1]);
      const float2 r1s = mul2(make_float2(R1[sub], R1[sub]), sg);
      bool ok0 = true, ok1 = true;
      if constexpr (CHECK) {
        const int row = q * 32 + 16 * h + g + 8 * sub;
        const int col = col_base + c, dcol = dtile + row;
        const bool rok = row < rows_left;
        ok0 = rok && col < ncols;
        ok1 = rok && col + 1 < ncols;
        if constexpr (MODE != kFwdMax) {  // the max includes the positive; the sums leave it out
          ok0 = ok0 && col != dcol;
          ok1 = ok1 && col + 1 != dcol;
        }
      }
      if constexpr (MODE == kFwdMax) {
        float2 x = mul2(r1s, d);  // the same two roundings as the shifted pass
        if (!ok0) x.x = -INFINITY;
        if (!ok1) x.y = -INFINITY;
        rs[idx] = make_float2(fmaxf(rs[idx].x, x.x), fmaxf(rs[idx].y, x.y));
        cs[r] = make_float2(fmaxf(cs[r].x, x.x), fmaxf(cs[r].y, x.y));
      } else if constexpr (MODE == kFwdShifted) {
        const float2 x = mul2(r1s, d);
        const float2 xr = add2(x, make_float2(-U[sub], -U[sub]));
        const float2 xc = add2(x, nv);
        float2 er = make_float2(ex2_approx(xr.x), ex2_approx(xr.y));
        float2 ec = make_float2(ex2_approx(xc.x), ex2_approx(xc.y));
        if (!ok0) er.x = ec.x = 0.f;
        if (!ok1) er.y = ec.y = 0.f;
        rs[idx] = add2(rs[idx], er);
        cs[r] = add2(cs[r], ec);
      } else {
        const float2 x = fma2(r1s, d, nl);
        float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        if (!ok0) e.x = 0.f;
        if (!ok1) e.y = 0.f;
        rs[idx] = add2(rs[idx], e);
        cs[r] = add2(cs[r], e);
      }
    }
  }
}

// After both halves: the row values meet over the 4 lanes of a row group (lane bits 1, 0) and
// the column values over the 8 lanes that share c4 (lane bits 4, 3, 2), leaving the lane the
// columns 8 g + 2 c4 + {0, 1}, written to cp.  Returns the lane's own row value.
template <int MODE>
__device__ __forceinline__ float fwd_cells16_reduce(const float2 (&rs)[4], const float2 (&cs)[8], int lane,
                                                    float* cp) {
  const int g = lane >> 2, c4 = lane & 3;
  float rv[4], cv[16];
#pragma unroll
  for (int idx = 0; idx < 4; ++idx) rv[idx] = MODE == kFwdMax ? fmaxf(rs[idx].x, rs[idx].y) : rs[idx].x + rs[idx].y;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    cv[2 * r] = cs[r].x;
    cv[2 * r + 1] = cs[r].y;
  }
  reduce_scatter_bits<MODE == kFwdMax, 4, 2, 2>(rv, lane);
  reduce_scatter_bits<MODE == kFwdMax, 16, 16, 3>(cv, lane);
  *reinterpret_cast<float2*>(cp + 8 * g + 2 * c4) = make_float2(cv[0], cv[1]);
  return rv[0];
}

// The order in which tiles and bands are fed to the MMA: tiles in pairs (t even in
// accumulator 0, t + 1 in accumulator 1), band by band, alternating within a pair.
// Step index s -> (tile, band); the producer, the MMA issuer and the epilogue all walk it.
struct Schedule {
  int T, n;
  __device__ int steps() const { return T * n; }
};
// Walks the schedule one step at a time without divisions (every epilogue thread keeps one).
struct SchedIter {
  int T, n;
  int tp = 0, b = 0, u = 0;  // first tile of the pair, band, tile within the pair
  int width = 0;             // tiles in this pair (the last pair may hold one)
  __device__ SchedIter(int T_, int n_) : T(T_), n(n_), width(T_ > 1 ? 2 : 1) {}
  __device__ int t() const { return tp + u; }
  __device__ void next() {
    if (++u < width) return;
    u = 0;
    if (++b < n) return;
    b = 0;
    tp += 2;
    width = (tp + 1 < T) ? 2 : 1;
  }
};

template <int KIND, bool COLS, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_y, const Params p) {
  griddep_enter();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sx = smem + off_x;
  uint8_t* sy = smem + off_y;
  float* colf = reinterpret_cast<float*>(smem + off_colf);
  float* rowf = reinterpret_cast<float*>(smem + off_rowf);
  float* rowsh = reinterpret_cast<float*>(smem + off_rowsh);
  float* colsh = reinterpret_cast<float*>(smem + off_colsh);
  float* cpart = reinterpret_cast<float*>(smem + off_cpart);
  uint64_t* s_full = reinterpret_cast<uint64_t*>(smem + off_bar);
  uint64_t* s_empty = s_full + kNS;
  uint64_t* acc_full = s_empty + kNS;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + off_misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + off_misc + 4);
  // L = scale log2(e) and b2 = bias log2(e), read once from the host value or the device
  // scalar; the epilogue reloads them per snapshot (volatile) instead of pinning registers
  volatile float* s_scal = reinterpret_cast<volatile float*>(smem + off_misc + 8);
  const uint32_t scal_s = smem_u32(smem + off_misc + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kTileRows;
  const int split = blockIdx.y;
  const int n = p.n_prefix;
  const int t_begin = split * p.tiles_per_split;
  const int T = min(p.n_col_tiles, t_begin + p.tiles_per_split) - t_begin;
  const Schedule sched{T, n};
  // prefix k's end (selects over the parameter: a runtime index into a local copy would put
  // the copy in local memory); p_{-1} = 0
  auto pend = [&](int k) {
    int e = 0;
#pragma unroll
    for (int kk = 0; kk < kMaxPrefix; ++kk)
      if (kk == k) e = p.prefix_end[kk];
    return e;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    s_scal[0] = p.sc.t() * 1.4426950408889634f;
    s_scal[1] = p.sc.b() * 1.4426950408889634f;
    fence_mbar_init();
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_y);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (T > 0 && warp == 0 && lane == 0) {
    // ------------------------------------------------------------- operand producer
    uint32_t it = 0;
    bool ok = true;
    SchedIter si(T, n);
    for (int s = 0; s < sched.steps() && ok; ++s, si.next()) {
      const int t = si.t(), b = si.b;
      const int j0 = (t_begin + t) * kCols;
      const int c0 = pend(b - 1) / kChunk, c1 = pend(b) / kChunk;
      for (int c = c0; c < c1; ++c, ++it) {
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
    for (uint32_t k = 0; k < kNS && k < it; ++k) {  // let the last copies land
      const uint32_t q = it - 1 - k;
      mbar_wait(&s_full[q % kNS], (q / kNS) & 1, kWaitLimitNs);
    }
  } else if (T > 0 && warp == 1 && lane == 0) {
    // ------------------------------------------------------------- MMA issuer
    const uint32_t idesc = idesc_bf16_f32(kTileRows, kCols);
    uint32_t it = 0;
    uint32_t uses0 = 0, uses1 = 0;  // uses of each accumulator (scalars, as in the epilogue)
    bool ok = true;
    SchedIter si(T, n);
    for (int s = 0; s < sched.steps() && ok; ++s, si.next()) {
      const int t = si.t(), b = si.b;
      const int a = t & 1;
      const uint32_t ua = a ? uses1 : uses0;
      if (ua > 0 && !wait_bounded(&acc_empty[a], (ua - 1) & 1, abort_flag)) {
        fail(p, abort_flag);
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem + a * kCols;
      const int c0 = pend(b - 1) / kChunk, c1 = pend(b) / kChunk;
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
          umma_bf16(d, sdesc_kmajor_sw128(ax + kk * 32), sdesc_kmajor_sw128(ay + kk * 32), idesc,
                    (c != 0 || kk != 0) ? 1u : 0u);
        umma_commit(&s_empty[st]);
      }
      if (ok) umma_commit(&acc_full[a]);
      if (a) ++uses1; else ++uses0;
    }
    umma_commit(drain);
    mbar_wait(drain, 0, kWaitLimitNs);
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------- epilogue
    const int q = warp & 3;                       // TMEM lane quadrant (rows 32q..32q+31)
    const int cq = (warp - kEpiWarp0) >> 2;       // column quarter (64 columns)
    const int r = q * 32 + lane;
    const int64_t gi = i0 + r;
    const bool row_ok = gi < p.nx;
    // the row whose sums this lane keeps: its own (32x32b layout), or with the column sums on
    // the 16x256b layout the one fwd_cells16 leaves it
    const int r_own = COLS ? q * 32 + 16 * ((lane & 3) >> 1) + (lane >> 2) + 8 * (lane & 1) : r;
    const int64_t gi_own = i0 + r_own;
    const bool own_ok = gi_own < p.nx;
    const int etid = threadIdx.x - kEpiWarp0 * 32;
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    constexpr int CF = kMaxPrefix * kCols;  // floats per column-factor buffer
    if (cq == 0) {
      const float L = s_scal[0];
#pragma unroll
      for (int k = 0; k < kMaxPrefix; ++k)
        if (k < n) {
          rowf[k * kTileRows + r] = row_ok ? L * p.rinv_x[k * p.nx + gi] : 0.f;
          if constexpr (MODE == kFwdShifted) rowsh[k * kTileRows + r] = row_ok ? p.shift_x[k * p.nx + gi] : 0.f;
        }
    }
    // column factors of tile t live in colf[t & 3]; a tile pair's factors are fetched by
    // cp.async while the previous pair is processed
    auto prefetch_colf = [&](int t) {
      const int64_t j0 = static_cast<int64_t>(t_begin + t) * kCols;
      float* cf = colf + (t & 3) * CF;
      for (int e = etid; e < n * kCols; e += kEpiThreads) {
        const int k = e / kCols, c = e % kCols;
        const int64_t gj = j0 + c;
        const bool v = gj < p.ny;
        cp_async4(cf + k * kCols + c, p.rinv_y + (v ? k * p.ny + gj : 0), v ? 4u : 0u);
        if constexpr (MODE == kFwdShifted && COLS)
          cp_async4(colsh + (t & 3) * CF + k * kCols + c, p.shift_y + (v ? k * p.ny + gj : 0), v ? 4u : 0u);
      }
    };
    for (int t = 0; t < 2 && t < T; ++t) prefetch_colf(t);
    cp_async_commit();
    float acc_row[kMaxPrefix];
#pragma unroll
    for (int k = 0; k < kMaxPrefix; ++k) acc_row[k] = MODE == kFwdMax ? -INFINITY : 0.f;
    uint32_t uses0 = 0, uses1 = 0;  // uses of each accumulator (scalars: a runtime index would put them in local memory)
    uint32_t snap = 0;  // snapshots processed (selects the column-partial buffer)
    bool ok = true;
    SchedIter si(T, n);
    for (int s = 0; s < sched.steps(); ++s, si.next()) {
      const int t = si.t(), b = si.b;
      if ((t & 1) == 0 && b == 0) {
        // a tile pair begins (every warp reaches this point at the same step)
        named_bar_sync(1, kEpiThreads);          // all are done with the previous pair
        for (int u = 2; u < 4 && t + u < T; ++u) prefetch_colf(t + u);
        cp_async_commit();
        cp_async_wait<1>();                      // this pair's factors (fetched a pair ago) are in
        named_bar_sync(1, kEpiThreads);
      }
      const int a = t & 1;
      const int k = b;
      const int64_t j0 = static_cast<int64_t>(t_begin + t) * kCols;
      if (ok && !wait_bounded(&acc_full[a], (a ? uses1 : uses0) & 1, abort_flag)) {
        fail(p, abort_flag);
        ok = false;
      }
      if (ok) {
        tc_fence_after();
        // one half of the warp's 64 x 32 cells at a time (fewer live registers): COLS, 16 rows
        // on the 16x256b layout; otherwise 32 columns on the 32x32b layout
        float v[32];
        if constexpr (COLS)
          tmem_ld16x256_x8(tmem + lane_addr + a * kCols + cq * 64, v);
        else
          tmem_ld32(tmem + lane_addr + a * kCols + cq * 64, v);
        float2 rs16[4], cs16[8];  // COLS: the row and column accumulators of fwd_cells16_half
        if constexpr (COLS) {
          constexpr float kInit = MODE == kFwdMax ? -INFINITY : 0.f;
#pragma unroll
          for (int idx = 0; idx < 4; ++idx) rs16[idx] = make_float2(kInit, kInit);
#pragma unroll
          for (int rr = 0; rr < 8; ++rr) cs16[rr] = make_float2(kInit, kInit);
        }

        const float* cf = colf + (t & 3) * CF + k * kCols + cq * 64;
        const float R1 = rowf[k * kTileRows + r];
        const int64_t left = p.ny - j0;
        const int ncols = left < kCols ? static_cast<int>(left) : kCols;
        // tile column of this row's positive, if any (none when a label matrix names them)
        const int dcol = p.no_diag ? INT_MIN : static_cast<int>(i0 - j0) + r;
        // masks are only evaluated in the few tiles that need them (padding columns, the
        // positives' diagonal, padding rows); every other tile takes the unmasked path
        const int64_t dtile = i0 - j0;  // uniform over the CTA: does this tile hold any positive?
        const bool check = ncols < kCols || (dtile > -kTileRows && dtile < kCols) || (i0 + kTileRows > p.nx);
        float rs;
        if constexpr (COLS) {
          float* cp = cpart + (((snap & 1) * 4 + cq) * 4 + q) * 64;
          const float* vs = colsh + (t & 3) * CF + k * kCols + cq * 64;
          float L;
          asm volatile("ld.shared.f32 %0, [%1];" : "=f"(L) : "r"(scal_s));
          const int dt = p.no_diag ? INT_MIN / 2 : static_cast<int>(dtile);
          const int rows_left = p.nx - i0 < kTileRows ? static_cast<int>(p.nx - i0) : kTileRows;
          const float* rf = rowf + k * kTileRows;
          const float* ru = rowsh + k * kTileRows;
          for (int h = 0; h < 2; ++h) {
            if (h == 1) {  // the second 16-row half; then the accumulator is free for the MMA
              tmem_ld16x256_x8(tmem + lane_addr + (16u << 16) + a * kCols + cq * 64, v);
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&acc_empty[a]);
            }
            if (check)
              fwd_cells16_half<MODE, true>(v, h, cf, vs, rf, ru, L, q, lane, cq * 64, ncols, dt, rows_left, rs16,
                                           cs16);
            else
              fwd_cells16_half<MODE, false>(v, h, cf, vs, rf, ru, L, q, lane, cq * 64, ncols, dt, rows_left, rs16,
                                            cs16);
          }
          rs = fwd_cells16_reduce<MODE>(rs16, cs16, lane, cp);
        } else {
          float L = 0.f, b2 = 0.f, U = 0.f;
          if constexpr (MODE == kFwdShifted) {
            U = rowsh[k * kTileRows + r];
          } else if constexpr (MODE == kFwdSum) {
            // (a 32-bit shared address keeps the epilogue within its 96 registers)
            asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(L), "=f"(b2) : "r"(scal_s));
          }
          constexpr float kInit = MODE == kFwdMax ? -INFINITY : 0.f;
          float2 acc = make_float2(kInit, kInit);
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            if (g == 1) {  // the second 32 columns; then the accumulator is free for the MMA
              tmem_ld32(tmem + lane_addr + a * kCols + cq * 64 + 32, v);
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&acc_empty[a]);
            }
            if constexpr (MODE == kFwdMax) {
              if (check) fwd_cells_max<true>(v, g, cf, R1, cq * 64, ncols, row_ok, acc);
              else fwd_cells_max<false>(v, g, cf, R1, cq * 64, ncols, row_ok, acc);
            } else if constexpr (MODE == kFwdShifted) {
              if (check) fwd_cells_shifted<true>(v, g, cf, R1, U, cq * 64, ncols, dcol, row_ok, acc);
              else fwd_cells_shifted<false>(v, g, cf, R1, U, cq * 64, ncols, dcol, row_ok, acc);
            } else {
              if (check) fwd_cells<KIND, true>(v, g, cf, R1, L, b2, cq * 64, ncols, dcol, row_ok, acc);
              else fwd_cells<KIND, false>(v, g, cf, R1, L, b2, cq * 64, ncols, dcol, row_ok, acc);
            }
          }
          rs = MODE == kFwdMax ? fmaxf(acc.x, acc.y) : acc.x + acc.y;
        }
#pragma unroll
        for (int kk = 0; kk < kMaxPrefix; ++kk)
          if (kk == k) acc_row[kk] = MODE == kFwdMax ? fmaxf(acc_row[kk], rs) : acc_row[kk] + rs;
      }
      if (a) ++uses1; else ++uses0;
      if constexpr (COLS) {
        // combine the four row quadrants of this column quarter; one warp writes the partial
        named_bar_sync(2 + cq, 128);
        if (ok && q == 0) {
          const float* cp = cpart + (((snap & 1) * 4 + cq) * 4) * 64;
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            const int c = g * 32 + lane;
            const float sum = MODE == kFwdMax ? fmaxf(fmaxf(cp[c], cp[64 + c]), fmaxf(cp[128 + c], cp[192 + c]))
                                              : cp[c] + cp[64 + c] + cp[128 + c] + cp[192 + c];
            const int64_t gj = j0 + cq * 64 + c;
            if (gj < p.ny) p.colacc[(static_cast<int64_t>(blockIdx.x) * n + k) * p.ny + gj] = sum;
          }
        }
      }
      ++snap;
    }
    cp_async_wait<0>();
    if (own_ok && ok) {
      const int slot = split * 4 + cq;
#pragma unroll  // (a constant index keeps acc_row in registers)
      for (int k = 0; k < kMaxPrefix; ++k)
        if (k < n) p.rowacc[(static_cast<int64_t>(slot) * n + k) * p.nx + gi_own] = acc_row[k];
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int KIND, bool COLS, int MODE>
static cudaError_t setup_one() {
  return cudaFuncSetAttribute(fwd_kernel<KIND, COLS, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              smem_bytes);
}

}  // namespace fwd

cudaError_t fwd_kernel_setup() {
  cudaError_t e;
  if ((e = fwd::setup_one<KIND_CLIP, true, kFwdSum>()) != cudaSuccess) return e;
  if ((e = fwd::setup_one<KIND_CLIP, true, kFwdMax>()) != cudaSuccess) return e;
  if ((e = fwd::setup_one<KIND_CLIP, true, kFwdShifted>()) != cudaSuccess) return e;
  if ((e = fwd::setup_one<KIND_ROWS, false, kFwdSum>()) != cudaSuccess) return e;
  if ((e = fwd::setup_one<KIND_ROWS, false, kFwdMax>()) != cudaSuccess) return e;
  if ((e = fwd::setup_one<KIND_ROWS, false, kFwdShifted>()) != cudaSuccess) return e;
  return fwd::setup_one<KIND_SIGLIP, false, kFwdSum>();
}

cudaError_t launch_fwd(int kind, const CUtensorMap& tm_x, const CUtensorMap& tm_y, const FwdParams& q, dim3 grid,
                       cudaStream_t stream) {
  fwd::Params p;
  p.nx = q.nx;
  p.ny = q.ny;
  p.n_prefix = q.n_prefix;
  for (int k = 0; k < kMaxPrefix; ++k) p.prefix_end[k] = q.prefix_end[k];
  p.n_col_tiles = q.n_col_tiles;
  p.tiles_per_split = q.tiles_per_split;
  p.sc = q.sc;
  p.rinv_x = q.rinv_x;
  p.rinv_y = q.rinv_y;
  p.shift_x = q.shift_x;
  p.shift_y = q.shift_y;
  p.no_diag = q.no_diag;
  p.rowacc = q.rowacc;
  p.colacc = q.colacc;
  p.status = q.status;
  using fwd::fwd_kernel;
  constexpr int T = fwd::kThreads, S = fwd::smem_bytes;
  if (kind == KIND_SIGLIP && q.mode != kFwdSum) return cudaErrorInvalidValue;
  if (q.mode == kFwdShifted && (q.shift_x == nullptr || (kind == KIND_CLIP && q.shift_y == nullptr)))
    return cudaErrorInvalidValue;
  const dim3 blk(T);
  if (kind == KIND_CLIP) {
    if (q.mode == kFwdMax) return launch_pdl(fwd_kernel<KIND_CLIP, true, kFwdMax>, grid, blk, S, stream, 1, tm_x, tm_y, p);
    if (q.mode == kFwdShifted)
      return launch_pdl(fwd_kernel<KIND_CLIP, true, kFwdShifted>, grid, blk, S, stream, 1, tm_x, tm_y, p);
    return launch_pdl(fwd_kernel<KIND_CLIP, true, kFwdSum>, grid, blk, S, stream, 1, tm_x, tm_y, p);
  }
  if (kind == KIND_ROWS) {
    if (q.mode == kFwdMax) return launch_pdl(fwd_kernel<KIND_ROWS, false, kFwdMax>, grid, blk, S, stream, 1, tm_x, tm_y, p);
    if (q.mode == kFwdShifted)
      return launch_pdl(fwd_kernel<KIND_ROWS, false, kFwdShifted>, grid, blk, S, stream, 1, tm_x, tm_y, p);
    return launch_pdl(fwd_kernel<KIND_ROWS, false, kFwdSum>, grid, blk, S, stream, 1, tm_x, tm_y, p);
  }
  return launch_pdl(fwd_kernel<KIND_SIGLIP, false, kFwdSum>, grid, blk, S, stream, 1, tm_x, tm_y, p);
}

}  // namespace ufc
