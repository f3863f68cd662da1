// uf_contrastive.cu -- the C ABI: argument checks, the workspace plan, TMA tensor maps
// and the launch sequence on the caller's stream.  No allocation, no synchronisation.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/uf_contrastive.h"
#include "launch.h"

using namespace ufc;

namespace {

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// CTA slots of one wave for the forward and weight passes: both run one CTA per SM, and a
// GB300 has 152 SMs.  A constant, not the device's SM count: the split sets the size of the
// per-split partial-sum arrays, and the workspace size must be a function of the problem
// alone (it is queried before any device is chosen).
constexpr int64_t kWaveCtas = 152;

struct Split {
  int splits = 1;
  int tiles_per_split = 1;
};

// The column split of a pass over row_blocks x tiles score tiles (one CTA per row block and
// split).  s splits cost about waves(s) x (tiles per CTA + 1) tile times: a CTA's set-up and
// its last tile's epilogue, which nothing overlaps, come to about one tile.  Takes the fewest
// splits within 2 % of the cheapest (fewer partial sums to merge).
Split plan_split(int64_t row_blocks, int64_t tiles) {
  const int64_t s_max = tiles < 4 * kWaveCtas ? tiles : 4 * kWaveCtas;
  auto cost = [&](int64_t s) { return cdiv(row_blocks * s, kWaveCtas) * (cdiv(tiles, s) + 1); };
  int64_t best = cost(1);
  for (int64_t s = 2; s <= s_max; ++s) best = cost(s) < best ? cost(s) : best;
  int64_t s = 1;
  while (s < s_max && cost(s) * 100 > best * 102) ++s;
  Split r;
  r.tiles_per_split = static_cast<int>(cdiv(tiles, s));
  r.splits = static_cast<int>(cdiv(tiles, r.tiles_per_split));
  return r;
}

// Default size of the backward weight array (bf16 m^k of every prefix for a chunk of
// rows): a GB300 has 288 GB of HBM, so the N = 65536 workloads keep every row in one chunk.
constexpr size_t kDefaultWeightBytes = size_t(48) << 30;

// Sizes and offsets of every scratch array of one call.
struct Plan {
  int64_t na = 0, nb = 0, nmin = 0;
  int d = 0, n = 0;
  int kind = 0;
  bool grads = false;
  int64_t rb_a = 0;                  // 128-row blocks of A
  int64_t ftiles = 0;                // forward: 256-column tiles of B
  Split fwd_a, wgt;                  // column splits of the forward and of the weight pass
  int slices = 0;                    // 256-dimension slices of the gradient GEMMs
  int64_t lda = 0, ldb = 0;          // padded leading dimensions of A^T and B^T
  int64_t ldw = 0;                   // row stride of the weight array (elements)
  int64_t chunk = 0;                 // rows of A per weight chunk (multiple of 128)
  int64_t cchunk = 0;                // rows of B (weight columns) per weight chunk
  bool gsplit = false;               // gradient contractions split below the widest prefix
  int64_t g2_ld = 0;                 // columns of their G2 arrays
  bool merge = false;                // the two widest prefixes' weights merged (one chunk only)
  size_t fixed = 0;                  // bytes of everything but the weight array
  // offsets
  size_t o_rinv_a, o_rinv_b, o_pos, o_zr, o_zc, o_fa, o_fb, o_acc_a, o_acc_b, o_crow_a, o_crow_b, o_terms_a,
      o_terms_b, o_spart, o_done, o_g2a, o_g2b, o_at, o_bt, o_csum, o_sig, o_sh_a, o_sh_b, o_lab, o_lcount, o_w, total;
  size_t o_r5row = 0, o_r5col = 0, o_r5a = 0, o_r5b = 0;  // merged widest prefixes
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ws_limit: the workspace the caller provides (0: plan the default weight array).  The
// weight array takes what is left after the fixed part: every weight at once if it fits, else
// chunks of (rows of A) x (rows of B), about square (multiples of 128 x 256), so that both
// gradient contractions of a chunk stay wide.
bool make_plan(int64_t Na, int64_t Nb, int D, const int* prefixes, int n, int kind, bool grads, size_t ws_limit,
               Plan& P) {
  if (Na < 1 || Nb < 1 || D < 64 || D > 4096 || D % 64 != 0 || n < 1 || n > kMaxPrefix || !prefixes) return false;
  if (kind != KIND_CLIP && kind != KIND_SIGLIP && kind != KIND_ROWS) return false;
  if (kind == KIND_CLIP && Na != Nb) return false;
  // ROWS and SigLIP: the columns past Na are extra negatives (explicit hard negatives)
  if ((kind == KIND_ROWS || kind == KIND_SIGLIP) && Nb < Na) return false;
  if (Na > (int64_t(1) << 31) || Nb > (int64_t(1) << 31)) return false;
  for (int k = 0; k < n; ++k) {
    if (prefixes[k] <= 0 || prefixes[k] % 64 != 0 || prefixes[k] > D) return false;
    if (k && prefixes[k] <= prefixes[k - 1]) return false;
  }
  P.na = Na;
  P.nb = Nb;
  P.nmin = Na < Nb ? Na : Nb;
  P.d = D;
  P.n = n;
  P.kind = kind;
  P.grads = grads;
  P.rb_a = cdiv(Na, kTileRows);
  P.ftiles = cdiv(Nb, kFwdCols);
  P.fwd_a = plan_split(P.rb_a, P.ftiles);
  P.wgt = plan_split(P.rb_a, cdiv(Nb, kWgtCols));  // rows of A against 256-row tiles of B
  P.slices = static_cast<int>(cdiv(prefixes[n - 1], 256));
  P.lda = cdiv(Na, 64) * 64;
  P.ldb = cdiv(Nb, 64) * 64;
  P.ldw = P.ldb;

  const size_t f = sizeof(float);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  P.o_rinv_a = take(f * n * Na);
  P.o_rinv_b = take(f * n * Nb);
  P.o_pos = take(f * n * P.nmin);
  P.o_zr = take(f * n * Na);
  P.o_zc = take(f * n * Nb);
  P.o_fa = take(f * n * Na);
  P.o_fb = take(f * n * Nb);
  // row-statistic partials: forward (CLIP/ROWS), or the SigLIP loss sums of the weight pass
  int slots_a = 4 * P.fwd_a.splits;  // one slot per split and column quarter
  if (kind == KIND_SIGLIP && grads) slots_a = 4 * P.wgt.splits;
  P.o_acc_a = take(f * n * Na * slots_a);
  P.o_acc_b = take(kind == KIND_CLIP ? f * n * Nb * P.rb_a : 0);  // CLIP: 128-row column partials
  P.o_crow_a = take(grads ? f * n * Na * P.slices : 0);  // projection scalars, one slot per slice
  P.o_crow_b = take(grads ? f * n * Nb * P.slices : 0);
  P.o_terms_a = take(f * n * Na);
  P.o_terms_b = take(f * n * Nb);
  P.o_spart = take(sizeof(double) * kMaxPrefix * kStatsBlocks);  // statistics pass: per-block loss sums
  P.o_done = take(sizeof(unsigned));
  P.o_at = take(grads ? sizeof(uint16_t) * D * P.lda : 0);
  P.o_bt = take(grads ? sizeof(uint16_t) * D * P.ldb : 0);
  P.o_csum = take(grads ? f * Na : 0);  // per-row sums of the row scalars (logit-scale gradient)
  P.o_sig = take(grads && kind == KIND_SIGLIP ? f * n * Na * 4 * P.wgt.splits : 0);  // sigmoid sums (bias)
  // the max-shifted path's row and column shifts (taken for every call: the scale that
  // picks the path may live on the device)
  P.o_sh_a = take(kind != KIND_SIGLIP ? f * n * Na : 0);
  P.o_sh_b = take(kind == KIND_CLIP ? f * n * Nb : 0);
  // SigLIP with a label matrix: the positives' share of the row terms, positives per row
  P.o_lab = take(kind == KIND_SIGLIP ? f * n * Na : 0);
  P.o_lcount = take(kind == KIND_SIGLIP ? f * Na : 0);
  // A gradient contraction of at most one wave of CTA pairs (both sides together) is bound by
  // its heaviest unit, the slice group that every prefix reaches; there the prefixes below the
  // widest run as units of their own, which write their part of G to G2 (CLIP N = 4096: GEMMs
  // 0.234 -> 0.187 ms).  Larger grids balance over their waves without it.
  P.g2_ld = n >= 2 ? prefixes[n - 2] : 0;
  {
    const int64_t groups = cdiv(cdiv(prefixes[n - 1], 256), 2);
    const int64_t pairs = groups * (cdiv(Na, 2 * kTileRows) + cdiv(Nb, 2 * kTileRows));
    P.gsplit = grads && n >= 2 && pairs <= kWaveCtas / 2;
  }
  P.o_g2a = take(P.gsplit ? f * Na * P.g2_ld : 0);
  P.o_g2b = take(P.gsplit ? f * Nb * P.g2_ld : 0);
  P.fixed = o;
  P.o_w = o;
  P.chunk = 0;
  P.cchunk = 0;
  if (grads) {
    const int64_t rows_max = cdiv(Na, kTileRows) * kTileRows;
    const int64_t cols_max = cdiv(Nb, kWgtCols) * kWgtCols;
    const size_t per = sizeof(uint16_t) * static_cast<size_t>(n);  // bytes per (row, column) cell
    const size_t budget = ws_limit ? (ws_limit > o ? ws_limit - o : 0) : kDefaultWeightBytes;
    const size_t one_chunk = per * static_cast<size_t>(rows_max) * static_cast<size_t>(P.ldb);
    // The two widest prefixes' weights merged below p_{n-2} (a multiple of 512, so whole slice
    // groups): the gradient GEMMs then contract prefix n-1 only above it, 7 MMA passes of 9 for
    // the five-prefix ladder, for one more store of a weight block and the sums of prefix n-1's
    // row scalars in the weight pass.  Taken when every weight fits in one chunk with those sums
    // beside it and the contractions are long (not split); CLIP and ROWS only (SigLIP's weight
    // pass, heavier in its epilogue, loses more than its GEMMs gain: N = 16384 2.91 -> 3.10 ms).
    const size_t r5_bytes = align256(f * 4 * P.wgt.splits * Na) + align256(f * 4 * P.rb_a * Nb) + align256(f * Na) +
                            align256(f * Nb);  // (as taken below)
    const bool merge_ok = kind != KIND_SIGLIP && n >= 2 && prefixes[n - 2] % 512 == 0 && !P.gsplit;
    if (one_chunk <= budget) {
      P.chunk = rows_max;  // one chunk
      P.cchunk = Nb;
      P.ldw = P.ldb;
      P.merge = merge_ok && align256(one_chunk) + r5_bytes <= budget;
    } else {
      const double cells = static_cast<double>(budget / per);
      int64_t R = static_cast<int64_t>(std::sqrt(cells)) / kTileRows * kTileRows;
      if (R > rows_max) R = rows_max;
      if (R < kTileRows) R = kTileRows;
      int64_t C = static_cast<int64_t>(cells / static_cast<double>(R)) / kWgtCols * kWgtCols;
      if (C > cols_max) C = cols_max;
      if (C < kWgtCols) C = kWgtCols;  // the minimum chunk; a smaller workspace is rejected by the caller
      if (C == cols_max) {  // every column in one chunk (rows as the 1-D layout): the rest buys rows
        int64_t R2 = static_cast<int64_t>(cells / static_cast<double>(P.ldb)) / kTileRows * kTileRows;
        if (R2 > rows_max) R2 = rows_max;
        if (R2 < kTileRows) R2 = kTileRows;
        P.chunk = R2;
        P.cchunk = Nb;
        P.ldw = P.ldb;
      } else {
        P.chunk = R;
        P.cchunk = C;
        P.ldw = C;
      }
    }
    o = align256(o + per * static_cast<size_t>(P.chunk) * static_cast<size_t>(P.ldw));
    if (P.merge) {
      P.o_r5row = take(f * 4 * P.wgt.splits * Na);  // per (split, column quarter) row sums
      P.o_r5col = take(f * 4 * P.rb_a * Nb);        // per (128-row block, 32-row quadrant) column sums
      P.o_r5a = take(f * Na);
      P.o_r5b = take(f * Nb);
    }
  }
  P.total = o;
  return true;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// 2-D bf16 tensor map over a row-major [rows x cols] matrix with row stride ld
// elements, 128-byte swizzle, box = [box_rows x 64 columns].
bool encode_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

std::mutex g_init_mu;
uint64_t g_init_mask = 0;  // devices already set up (device ordinal < 64)
int g_sm_count[64];        // their SM counts

// ---- optional per-kernel timing (uf_contrastive_profile)
struct ProfRecord {
  int group;
  int launches;
  cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
std::atomic<bool> g_prof_on{false};
std::vector<ProfRecord> g_prof_pending;
std::vector<cudaEvent_t> g_prof_pool;
double g_prof_ms[UF_KERNEL_GROUPS];
int64_t g_prof_pairs[UF_KERNEL_GROUPS], g_prof_launches[UF_KERNEL_GROUPS];

cudaEvent_t prof_event() {
  if (!g_prof_pool.empty()) {
    cudaEvent_t e = g_prof_pool.back();
    g_prof_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Records a start event on construction and a stop event on destruction (profiling only).
struct ProfScope {
  bool on;
  ProfRecord rec{};
  cudaStream_t stream;
  ProfScope(int group, int launches, cudaStream_t s) : on(g_prof_on.load()), stream(s) {
    if (!on) return;
    std::lock_guard<std::mutex> lock(g_prof_mu);
    rec.group = group;
    rec.launches = launches;
    rec.start = prof_event();
    rec.stop = prof_event();
    cudaEventRecord(rec.start, stream);
  }
  ~ProfScope() {
    if (!on) return;
    cudaEventRecord(rec.stop, stream);
    std::lock_guard<std::mutex> lock(g_prof_mu);
    g_prof_pending.push_back(rec);
  }
};

}  // namespace

namespace ufc {
// SM count of the current device (read at uf_contrastive_init; queried here if the device was
// never initialised, e.g. by a launcher called from a test harness).
int current_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64 && g_sm_count[dev] > 0) return g_sm_count[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 1;
  return n;
}
}  // namespace ufc

extern "C" {

const char* uf_status_name(int status) {
  switch (status) {
    case UF_OK: return "ok";
    case UF_INVALID_ARGUMENT: return "invalid-argument";
    case UF_UNSUPPORTED: return "unsupported";
    case UF_WORKSPACE_TOO_SMALL: return "workspace-too-small";
    case UF_CUDA_ERROR: return "cuda-error";
    case UF_DEVICE_TIMEOUT: return "device-timeout";
    default: return "unknown";
  }
}

int uf_contrastive_version(void) { return 100; }

uf_status_t uf_contrastive_init(int device) {
  std::lock_guard<std::mutex> lock(g_init_mu);
  if (device < 0 || device >= 64) return UF_INVALID_ARGUMENT;
  if (g_init_mask & (uint64_t(1) << device)) return UF_OK;
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return UF_CUDA_ERROR;
  if (cudaSetDevice(device) != cudaSuccess) return UF_CUDA_ERROR;
  cudaDeviceProp prop;
  uf_status_t st = UF_OK;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess || prop.major != 10 || prop.minor != 3) {
    st = UF_CUDA_ERROR;
  } else if (wgt_kernel_setup() != cudaSuccess || gemm_kernel_setup() != cudaSuccess ||
             fwd_kernel_setup() != cudaSuccess ||
             aux_kernels_setup() != cudaSuccess || !get_encode()) {
    st = UF_CUDA_ERROR;
  }
  if (st == UF_OK && cudaDeviceGetAttribute(&g_sm_count[device], cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    st = UF_CUDA_ERROR;
  cudaSetDevice(prev);
  if (st == UF_OK) g_init_mask |= uint64_t(1) << device;
  return st;
}

size_t uf_contrastive_workspace_size(int64_t Na, int64_t Nb, int D, const int* prefixes, int n_prefix, int kind,
                                     int want_grads) {
  Plan P;
  if (!make_plan(Na, Nb, D, prefixes, n_prefix, kind, want_grads != 0, 0, P)) return 0;
  return P.total;
}

size_t uf_contrastive_workspace_min(int64_t Na, int64_t Nb, int D, const int* prefixes, int n_prefix, int kind,
                                    int want_grads) {
  Plan P;
  if (!make_plan(Na, Nb, D, prefixes, n_prefix, kind, want_grads != 0, 1, P)) return 0;  // the smallest weight chunk
  return P.total;
}

uf_status_t uf_contrastive_fwd_bwd(const void* A, const void* B, int64_t Na, int64_t Nb, int D, const int* prefixes,
                                   int n_prefix, int kind, float logit_scale, float bias,
                                   const float* prefix_weights, float* loss_per_prefix, float* row_terms,
                                   float* col_terms, float* dA, float* dB, void* workspace, size_t workspace_bytes,
                                   int* device_status, void* stream_handle) {
  return uf_contrastive_fwd_bwd_ex(A, B, Na, Nb, D, prefixes, n_prefix, kind, logit_scale, bias, nullptr, nullptr,
                                   nullptr, nullptr, prefix_weights, loss_per_prefix, row_terms, col_terms, dA, dB, nullptr, nullptr,
                                   workspace, workspace_bytes, device_status, stream_handle);
}

}  // extern "C"

namespace {

// Every buffer a call writes (the outputs, *device_status and the workspace) must overlap no
// other such buffer and no input: a kernel writing an output over an input that a later kernel
// reads, or over another output, would return garbage.  The inputs may overlap one another
// (A == B is a valid request).  pos_ids is checked by its first element (its length is only
// known on the device).
bool disjoint_buffers(const void* A, const void* B, int64_t Na, int64_t Nb, int D, int n, const float* scale_dev,
                      const float* bias_dev, const int64_t* pos_offsets, const int* pos_ids, const float* loss,
                      const float* row_terms, const float* col_terms, const float* dA, const float* dB,
                      const float* d_scale, const float* d_bias, const void* workspace, size_t workspace_bytes,
                      const int* status) {
  struct Range {
    uintptr_t lo, hi;  // [lo, hi); empty for a NULL pointer
  };
  auto range = [](const void* p, uint64_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return Range{a, p ? a + static_cast<uintptr_t>(bytes) : a};
  };
  const uint64_t f = sizeof(float), d = static_cast<uint64_t>(D), un = static_cast<uint64_t>(n);
  const uint64_t na = static_cast<uint64_t>(Na), nb = static_cast<uint64_t>(Nb);
  const Range written[] = {
      range(loss, f * un),          range(row_terms, f * un * na), range(col_terms, f * un * nb),
      range(dA, f * na * d),        range(dB, f * nb * d),         range(d_scale, f),
      range(d_bias, f),             range(status, sizeof(int)),    range(workspace, workspace_bytes),
  };
  const Range read[] = {
      range(A, 2 * na * d),  range(B, 2 * nb * d),
      range(scale_dev, f),   range(bias_dev, f),
      range(pos_offsets, sizeof(int64_t) * (na + 1)), range(pos_ids, sizeof(int)),
  };
  auto overlap = [](const Range& x, const Range& y) { return x.lo < x.hi && y.lo < y.hi && x.lo < y.hi && y.lo < x.hi; };
  const int nw = static_cast<int>(sizeof(written) / sizeof(written[0]));
  for (int i = 0; i < nw; ++i) {
    for (int j = i + 1; j < nw; ++j)
      if (overlap(written[i], written[j])) return false;
    for (const Range& r : read)
      if (overlap(written[i], r)) return false;
  }
  return true;
}

// The two-set loss of A against B, or (oneset) the one-set loss of the set A = B against
// itself: self-cells masked, labels required, dA = dX receives both roles of every cell
// (twice the A-side gradient, the weights being symmetric), no B-side GEMM.
uf_status_t run_loss(const void* A, const void* B, int64_t Na, int64_t Nb, int D, const int* prefixes,
                     int n_prefix, int kind, float logit_scale, float bias, const float* logit_scale_dev,
                     const float* bias_dev, const int64_t* pos_offsets, const int* pos_ids,
                     const float* prefix_weights, float* loss_per_prefix, float* row_terms, float* col_terms,
                     float* dA, float* dB, float* d_logit_scale, float* d_bias, void* workspace,
                     size_t workspace_bytes, int* device_status, void* stream_handle, bool oneset) {
  // ---- argument checks (nothing is enqueued on failure)
  if (!A || !B || !loss_per_prefix || !workspace) return UF_INVALID_ARGUMENT;
  if ((dA == nullptr) != (dB == nullptr)) return UF_INVALID_ARGUMENT;
  const bool grads = dA != nullptr;
  if ((d_logit_scale || d_bias) && !grads) return UF_INVALID_ARGUMENT;  // they come out of the backward
  if ((d_logit_scale && !aligned(d_logit_scale, 4)) || (d_bias && !aligned(d_bias, 4))) return UF_INVALID_ARGUMENT;
  if ((logit_scale_dev && !aligned(logit_scale_dev, 4)) || (bias_dev && !aligned(bias_dev, 4)))
    return UF_INVALID_ARGUMENT;
  const bool labels = pos_offsets != nullptr;
  if ((pos_offsets == nullptr) != (pos_ids == nullptr)) return UF_INVALID_ARGUMENT;
  if (labels && (!aligned(pos_offsets, 8) || !aligned(pos_ids, 4))) return UF_INVALID_ARGUMENT;
  if (labels && kind != KIND_SIGLIP) return UF_UNSUPPORTED;  // the pages define labelled positives for SigLIP
  Plan P;
  if (!make_plan(Na, Nb, D, prefixes, n_prefix, kind, grads, workspace_bytes, P)) return UF_INVALID_ARGUMENT;
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(workspace, 256) || !aligned(loss_per_prefix, 4))
    return UF_INVALID_ARGUMENT;
  if (grads && (!aligned(dA, 16) || !aligned(dB, 16))) return UF_INVALID_ARGUMENT;
  if ((row_terms && !aligned(row_terms, 4)) || (col_terms && !aligned(col_terms, 4))) return UF_INVALID_ARGUMENT;
  if (!disjoint_buffers(A, B, Na, Nb, D, n_prefix, logit_scale_dev, bias_dev, pos_offsets, pos_ids, loss_per_prefix,
                        row_terms, col_terms, dA, oneset ? nullptr : dB, d_logit_scale, d_bias, workspace,
                        workspace_bytes, device_status))
    return UF_INVALID_ARGUMENT;
  // host scalars are checked here; ones on the device by the first kernel (*device_status)
  if ((!logit_scale_dev && !std::isfinite(logit_scale)) || (!bias_dev && !std::isfinite(bias)))
    return UF_INVALID_ARGUMENT;
  float w[kMaxPrefix];
  for (int k = 0; k < kMaxPrefix; ++k) w[k] = 0.f;
  for (int k = 0; k < n_prefix; ++k) {
    w[k] = prefix_weights ? prefix_weights[k] : 1.f;
    if (!std::isfinite(w[k])) return UF_INVALID_ARGUMENT;
  }
  if (kind == KIND_SIGLIP) {
    if (!logit_scale_dev && !bias_dev && std::fabs(logit_scale) + std::fabs(bias) > kMaxSiglipRange)
      return UF_UNSUPPORTED;
    if (d_logit_scale && !logit_scale_dev && logit_scale == 0.f) return UF_UNSUPPORTED;  // taken as (sum W cos) / t
  } else if (!logit_scale_dev) {
    if (!(logit_scale > 0.f)) return UF_INVALID_ARGUMENT;
    if (logit_scale > kMaxLogitScale) return UF_UNSUPPORTED;
  }
  // CLIP/ROWS statistics with the fixed shift tau while tau <= 40 is known on the host;
  // the max-shifted path otherwise
  const bool shifted = kind != KIND_SIGLIP && (logit_scale_dev != nullptr || logit_scale > kFixedShiftMaxScale);
  const Scalars sc{logit_scale, bias, logit_scale_dev, bias_dev};
  if (workspace_bytes < P.total) return UF_WORKSPACE_TOO_SMALL;

  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return UF_CUDA_ERROR;
  if (uf_contrastive_init(dev) != UF_OK) return UF_CUDA_ERROR;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto F = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
  const uint16_t* A16 = static_cast<const uint16_t*>(A);
  const uint16_t* B16 = static_cast<const uint16_t*>(B);
  const int n = n_prefix;
  const bool siglip = kind == KIND_SIGLIP;
  float* shift_a = shifted ? F(P.o_sh_a) : nullptr;
  float* shift_b = shifted && kind == KIND_CLIP ? F(P.o_sh_b) : nullptr;

  // ---- tensor maps
  // [128 x 64] boxes for the owner rows, [256 x 64] for the walked rows, [64 dims x 64] for
  // the transposed operand of the gradient GEMM
  CUtensorMap tmA, tmB, tmAt, tmBt, tmAf, tmBf;
  if (!encode_map(&tmA, A, Na, D, D, kTileRows) || !encode_map(&tmB, B, Nb, D, D, kTileRows) ||
      !encode_map(&tmAf, A, Na, D, D, kWgtCols) || !encode_map(&tmBf, B, Nb, D, D, kFwdCols))
    return UF_CUDA_ERROR;
  uint16_t* At = reinterpret_cast<uint16_t*>(ws + P.o_at);
  uint16_t* Bt = reinterpret_cast<uint16_t*>(ws + P.o_bt);
  if (grads) {
    if (!encode_map(&tmAt, At, D, Na, P.lda, kGemmBBox) || !encode_map(&tmBt, Bt, D, Nb, P.ldb, kGemmBBox))
      return UF_CUDA_ERROR;
  } else {
    tmAt = tmA;
    tmBt = tmB;
  }

  cudaError_t e;
#define UF_CHECK(x)                 \
  do {                              \
    e = (x);                        \
    if (e != cudaSuccess) return UF_CUDA_ERROR; \
  } while (0)

  // ---- 1. inverse norms, positives' cosines, transposed copies
  PrepParams pp{};
  pp.kind = kind;
  pp.sc = sc;
  pp.status = device_status;
  pp.A = A16;
  pp.B = B16;
  pp.na = Na;
  pp.nb = Nb;
  pp.nmin = P.nmin;
  pp.d = D;
  pp.n_prefix = n;
  for (int k = 0; k < n; ++k) pp.prefix_end[k] = prefixes[k];
  pp.rinv_a = F(P.o_rinv_a);
  pp.rinv_b = F(P.o_rinv_b);
  pp.pos_cos = F(P.o_pos);
  pp.stats_done = reinterpret_cast<unsigned*>(ws + P.o_done);
  {
    ProfScope ps(UF_KERNEL_PREP, 1, stream);
    UF_CHECK(launch_prep(pp, stream));
  }
  if (grads) {
    TransposeParams tp{};
    tp.d = D;
    if (!oneset) {  // (one set: A^T is B^T)
      tp.X[tp.count] = A16;
      tp.Xt[tp.count] = At;
      tp.rows[tp.count] = Na;
      tp.ld[tp.count] = P.lda;
      ++tp.count;
    }
    tp.X[tp.count] = B16;
    tp.Xt[tp.count] = Bt;
    tp.rows[tp.count] = Nb;
    tp.ld[tp.count] = P.ldb;
    ++tp.count;
    ProfScope ps(UF_KERNEL_TRANSPOSE, 1, stream);
    UF_CHECK(launch_transpose(tp, stream));
  }

  // SigLIP with a label matrix: the positives' loss terms and counts (the dense passes score
  // every cell as a negative)
  LabelParams lp{};
  if (labels) {
    lp.offsets = pos_offsets;
    lp.ids = pos_ids;
    lp.A = A16;
    lp.B = B16;
    lp.na = Na;
    lp.nb = Nb;
    lp.d = D;
    lp.n_prefix = n;
    for (int k = 0; k < n; ++k) {
      lp.prefix_end[k] = prefixes[k];
      lp.weight[k] = w[k];
    }
    lp.sc = sc;
    lp.rinv_a = F(P.o_rinv_a);
    lp.rinv_b = F(P.o_rinv_b);
    lp.pos_term = F(P.o_lab);
    lp.lcount = F(P.o_lcount);
    lp.oneset = oneset ? 1 : 0;
    lp.status = device_status;
    ProfScope ps(UF_KERNEL_PREP, 1, stream);
    UF_CHECK(launch_labels(lp, stream));
  }

  float* terms_a = row_terms ? row_terms : F(P.o_terms_a);
  float* terms_b = col_terms ? col_terms : F(P.o_terms_b);
  StatsParams sp{};
  sp.kind = kind;
  sp.na = Na;
  sp.nb = Nb;
  sp.n_prefix = n;
  for (int k = 0; k < n; ++k) {
    sp.prefix_end[k] = prefixes[k];
    sp.weight[k] = w[k];
  }
  sp.sc = sc;
  sp.shift_a = shift_a;
  sp.shift_b = shift_b;
  sp.diag_pos = labels ? 0 : 1;
  sp.pos_term = labels ? F(P.o_lab) : nullptr;
  sp.rinv_a = F(P.o_rinv_a);
  sp.rinv_b = F(P.o_rinv_b);
  sp.pos_cos = F(P.o_pos);
  sp.zr = F(P.o_zr);
  sp.zc = F(P.o_zc);
  sp.fa = F(P.o_fa);
  sp.fb = F(P.o_fb);
  sp.terms_a = terms_a;
  sp.terms_b = terms_b;
  sp.loss = loss_per_prefix;
  sp.part = reinterpret_cast<double*>(ws + P.o_spart);
  sp.done = reinterpret_cast<unsigned*>(ws + P.o_done);

  // ---- 2. forward statistics (all kinds without gradients; CLIP/ROWS with them): one pass
  // over the grid gives every row sum and, for CLIP, every column sum (the max-shifted path
  // runs a max pass first for the shifts)
  if (!siglip || !grads) {
    FwdParams fp{};
    fp.nx = Na;
    fp.ny = Nb;
    fp.n_prefix = n;
    for (int k = 0; k < n; ++k) fp.prefix_end[k] = prefixes[k];
    fp.n_col_tiles = static_cast<int>(P.ftiles);
    fp.tiles_per_split = P.fwd_a.tiles_per_split;
    fp.sc = sc;
    fp.no_diag = labels && !oneset ? 1 : 0;  // one set: the diagonal cells are the self-cells, masked
    fp.rinv_x = F(P.o_rinv_a);
    fp.rinv_y = F(P.o_rinv_b);
    fp.rowacc = F(P.o_acc_a);
    fp.colacc = kind == KIND_CLIP ? F(P.o_acc_b) : nullptr;
    fp.status = device_status;
    const dim3 fgrid(static_cast<unsigned>(cdiv(Na, kTileRows)), P.fwd_a.splits, 1);
    if (shifted) {
      fp.mode = kFwdMax;
      {
        ProfScope ps(UF_KERNEL_FWD_TILE, 1, stream);
        UF_CHECK(launch_fwd(kind, tmA, tmBf, fp, fgrid, stream));
      }
      MaxReduceParams mp{};
      mp.n_prefix = n;
      mp.na = Na;
      mp.nb = Nb;
      mp.rowmax = fp.rowacc;
      mp.slots_a = 4 * P.fwd_a.splits;
      mp.colmax = fp.colacc;
      mp.blocks = static_cast<int>(P.rb_a);
      mp.u = shift_a;
      mp.v = shift_b;
      {
        ProfScope ps(UF_KERNEL_STATS, 1, stream);
        UF_CHECK(launch_max_reduce(mp, stream));
      }
      fp.mode = kFwdShifted;
      fp.shift_x = shift_a;
      fp.shift_y = shift_b;
    }
    {
      ProfScope ps(UF_KERNEL_FWD_TILE, 1, stream);
      UF_CHECK(launch_fwd(kind, tmA, tmBf, fp, fgrid, stream));
    }
    sp.rowacc_a = fp.rowacc;
    sp.slots_a = 4 * P.fwd_a.splits;
    if (kind == KIND_CLIP) {
      sp.rowacc_b = fp.colacc;
      sp.slots_b = static_cast<int>(P.rb_a);
    }
    ProfScope ps(UF_KERNEL_STATS, 1, stream);
    UF_CHECK(launch_stats(sp, stream));
  }
  if (!grads) {
    if (col_terms && kind != KIND_CLIP) UF_CHECK(cudaMemsetAsync(col_terms, 0, sizeof(float) * n * Nb, stream));
    return UF_OK;
  }

  // ---- 3. backward: per chunk of A's rows, the weight pass writes m^k (bf16, [k][i][j]);
  // one GEMM contracts the chunk's weights with B into dA's rows, another contracts their
  // transpose with the chunk of A into all of dB (added over chunks).  Both write G = dX
  // before its projection in place into dA / dB, and the projection scalars.
  // the two widest prefixes' weights merged (planned when they fit; not with a label matrix,
  // whose patch writes each prefix's exact weights, nor for the one-set loss)
  const bool wmerge = P.merge && !labels && !oneset;
  {
    uint16_t* W = reinterpret_cast<uint16_t*>(ws + P.o_w);
    const int64_t wrows = static_cast<int64_t>(n) * P.chunk;
    // the weight array as [n * chunk rows][Nb columns]: store, K-major and MN-major load boxes
    CUtensorMap tmWs, tmWk, tmWm, tmAt128, tmBt128;
    if (!encode_map(&tmAt128, At, D, Na, P.lda, 128) || !encode_map(&tmBt128, Bt, D, Nb, P.ldb, 128))
      return UF_CUDA_ERROR;
    if (!encode_map(&tmWs, W, wrows, P.cchunk, P.ldw, kWgtStoreRows) ||
        !encode_map(&tmWk, W, wrows, P.cchunk, P.ldw, kTileRows) || !encode_map(&tmWm, W, wrows, P.cchunk, P.ldw, 64))
      return UF_CUDA_ERROR;
    WgtParams wp{};
    wp.nx = Na;
    wp.ny = Nb;
    wp.n_prefix = n;
    for (int k = 0; k < n; ++k) wp.prefix_end[k] = prefixes[k];
    wp.sc = sc;
    wp.shifted = shifted ? 1 : 0;
    wp.no_diag = labels && !oneset ? 1 : 0;
    wp.rinv_x = F(P.o_rinv_a);
    wp.rinv_y = F(P.o_rinv_b);
    wp.alpha_x = siglip ? nullptr : F(P.o_fa);
    wp.beta_y = (kind == KIND_CLIP) ? F(P.o_fb) : nullptr;
    for (int k = 0; k < n; ++k)  // SigLIP: w_k / N (the kernel multiplies by t); shifted: w_k
      wp.m_scale[k] = shifted ? w[k] : static_cast<float>(w[k] / static_cast<double>(Na));
    wp.w_rows_per_prefix = P.chunk;
    wp.rowacc = siglip ? F(P.o_acc_a) : nullptr;  // the SigLIP loss sums
    wp.rowsig = (siglip && d_bias) ? F(P.o_sig) : nullptr;  // and, for the bias gradient, the sigmoid sums
    if (wmerge) {
      wp.merge = 1;
      wp.r5_row = F(P.o_r5row);
      wp.r5_col = F(P.o_r5col);
    }
    wp.status = device_status;
    GemmParams ga{}, gb{};
    for (GemmParams* g : {&ga, &gb}) {
      g->w_rows_per_prefix = P.chunk;
      g->d = D;
      g->n_prefix = n;
      for (int k = 0; k < n; ++k) g->prefix_end[k] = prefixes[k];
      g->status = device_status;
    }
    ga.G = dA;
    ga.X = A16;
    ga.crow = F(P.o_crow_a);
    ga.crow_rows = Na;
    gb.G = dB;
    gb.X = B16;
    gb.crow = F(P.o_crow_b);
    gb.crow_rows = Nb;
    ga.merge = gb.merge = wmerge ? 1 : 0;
    if (P.gsplit) {
      ga.split_rest = gb.split_rest = 1;
      ga.G2 = F(P.o_g2a);
      gb.G2 = F(P.o_g2b);
      ga.g2_ld = gb.g2_ld = P.g2_ld;
    }
    // The column split of one chunk's weight pass: the whole problem's for SigLIP (its row slots
    // of loss sums are sized by it); for CLIP and ROWS, which keep no per-split state, one sized
    // for the chunk's own row blocks, so a small chunk still fills the GPU.
    const Split wsplit = siglip ? P.wgt : plan_split(cdiv(P.chunk, kTileRows), cdiv(P.cchunk, kWgtCols));
    // Chunks: rows [r0, r0 + rows) of A against rows [c0, c0 + cols) of B.  dA's rows add over
    // the column chunks and dB's over the row chunks, each in a fixed order.  SigLIP's row loss
    // sums then add over the column chunks too (from zero; each slot has one owner thread, which
    // adds in program order).
    const bool col_chunks = P.cchunk < Nb;
    if (siglip && col_chunks) {
      UF_CHECK(cudaMemsetAsync(F(P.o_acc_a), 0, sizeof(float) * n * Na * 4 * P.wgt.splits, stream));
      if (wp.rowsig) UF_CHECK(cudaMemsetAsync(wp.rowsig, 0, sizeof(float) * n * Na * 4 * P.wgt.splits, stream));
    }
    for (int64_t r0 = 0; r0 < Na; r0 += P.chunk) {
      const int64_t rows = Na - r0 < P.chunk ? Na - r0 : P.chunk;
      for (int64_t c0 = 0; c0 < Nb; c0 += P.cchunk) {
        const int64_t cols = Nb - c0 < P.cchunk ? Nb - c0 : P.cchunk;
        wp.row0 = r0;
        wp.rows = rows;
        wp.col0 = c0;
        wp.cols = cols;
        wp.add_rows = col_chunks ? 1 : 0;
        wp.n_col_tiles = static_cast<int>(cdiv(cols, kWgtCols));
        const Split cs = siglip ? P.wgt : wsplit;
        wp.tiles_per_split = cs.tiles_per_split;
        const int splits = static_cast<int>(cdiv(wp.n_col_tiles, cs.tiles_per_split));
        {
          ProfScope ps(UF_KERNEL_BWD_TILE, 1, stream);
          UF_CHECK(launch_wgt(kind, tmA, tmB, tmWs, wp, dim3(static_cast<unsigned>(cdiv(rows, kTileRows)), splits),
                              stream));
        }
        if (labels) {  // the labelled positives' exact weights over the negative-cell ones
          LabelParams pq = lp;
          pq.W = W;
          pq.row0 = r0;
          pq.rows = rows;
          pq.col0 = c0;
          pq.cols = cols;
          pq.w_rows_per_prefix = P.chunk;
          pq.ldw = P.ldw;
          ProfScope ps(UF_KERNEL_BWD_TILE, 1, stream);
          UF_CHECK(launch_labels(pq, stream));
        }
        ga.m_rows = rows;
        ga.row0 = r0;
        ga.kdim = cols;
        ga.b_col0 = c0;
        ga.accumulate = c0 > 0;
        // A dA contraction of few waves (few rows: ROWS's queries, small batches) leaves SMs idle
        // in its last wave, which one grid with the dB contraction fills (ROWS 8192 x 262144:
        // GEMMs 14.0 -> 12.2 ms).  A long one runs alone: the two read the weights in different
        // orders, and mixed they share L2 worse (CLIP N = 65536: 23.7 -> 24.6 ms in one grid).
        const bool one_grid = !oneset && gemm_grid_pairs(ga) / (0.5 * g_sm_count[dev]) < kGemmOneGridWaves;
        ProfScope ps(UF_KERNEL_GEMM, oneset || one_grid ? 1 : 2, stream);
        if (oneset) {  // (the B side of the one-set loss is the A side's mirror)
          UF_CHECK(launch_gemm(tmWk, tmBt, tmBt128, ga, false, stream));
        } else {
          gb.m_rows = cols;
          gb.row0 = c0;
          gb.kdim = rows;
          gb.b_col0 = r0;
          gb.accumulate = r0 > 0;
          if (one_grid) {
            UF_CHECK(launch_gemm_both(tmWk, tmBt, tmBt128, ga, tmWm, tmAt, tmAt128, gb, stream));
          } else {
            UF_CHECK(launch_gemm(tmWk, tmBt, tmBt128, ga, false, stream));
            UF_CHECK(launch_gemm(tmWm, tmAt, tmAt128, gb, true, stream));
          }
        }
      }
    }
    if (siglip) {
      sp.rowacc_a = F(P.o_acc_a);
      sp.slots_a = 4 * P.wgt.splits;
      ProfScope ps(UF_KERNEL_STATS, 1, stream);
      UF_CHECK(launch_stats(sp, stream));
    }
    if (wmerge) {  // prefix n-1's row scalars from the weight pass's partial sums
      R5Params rp{};
      rp.na = Na;
      rp.nb = Nb;
      rp.row = F(P.o_r5row);
      rp.row_slots = 4 * P.wgt.splits;
      rp.col = F(P.o_r5col);
      rp.col_parts = static_cast<int>(4 * P.rb_a);
      rp.r5_a = F(P.o_r5a);
      rp.r5_b = F(P.o_r5b);
      ProfScope ps(UF_KERNEL_NORM_BWD, 1, stream);
      UF_CHECK(launch_r5(rp, stream));
    }
  }

  // ---- 4. projection term and diagonal correction
  {
    NormBwdParams qs[2] = {};
    const int n_sides = oneset ? 1 : 2;
    for (int side = 0; side < n_sides; ++side) {
      const bool xa = side == 0;
      NormBwdParams& q = qs[side];
      q.kind = kind;
      q.nx = xa ? Na : Nb;
      q.ny = xa ? Nb : Na;
      q.nmin = labels ? 0 : P.nmin;  // labelled positives went through the GEMMs with their exact weights
      q.n_total = Na;
      q.d = D;
      q.n_prefix = n;
      for (int k = 0; k < n; ++k) {
        q.prefix_end[k] = prefixes[k];
        q.weight[k] = w[k];
      }
      q.sc = sc;
      q.X = xa ? A16 : B16;
      q.Y = xa ? B16 : A16;
      q.rinv_x = F(xa ? P.o_rinv_a : P.o_rinv_b);
      q.rinv_y = F(xa ? P.o_rinv_b : P.o_rinv_a);
      q.pos_cos = F(P.o_pos);
      q.z_x = F(xa ? P.o_zr : P.o_zc);
      q.z_y = F(xa ? P.o_zc : P.o_zr);
      q.shift_x = xa ? shift_a : shift_b;
      q.shift_y = xa ? shift_b : shift_a;
      if (kind == KIND_ROWS) {
        q.x_is_query = xa ? 1 : 0;
        q.z_x = F(P.o_zr);
        q.z_y = F(P.o_zr);
        q.shift_x = shift_a;
        q.shift_y = shift_a;
      }
      q.crow = F(xa ? P.o_crow_a : P.o_crow_b);
      q.crow_slots = P.slices;
      q.csum = (xa && d_logit_scale) ? F(P.o_csum) : nullptr;
      q.G = xa ? dA : dB;
      if (wmerge) q.r5 = F(xa ? P.o_r5a : P.o_r5b);
      if (P.gsplit) {
        q.G2 = F(xa ? P.o_g2a : P.o_g2b);
        q.g2_ld = P.g2_ld;
      }
      q.double_out = oneset ? 1 : 0;
      q.dX = xa ? dA : dB;
    }
    ProfScope ps(UF_KERNEL_NORM_BWD, 1, stream);
    UF_CHECK(launch_norm_bwd(qs, n_sides, stream));
  }
  // ---- 5. gradients in the logit scale and the bias
  if (d_logit_scale || d_bias) {
    ScaleGradParams g{};
    g.kind = kind;
    g.na = Na;
    g.nmin = P.nmin;
    g.n_prefix = n;
    g.sc = sc;
    for (int k = 0; k < n; ++k) g.weight[k] = w[k];
    g.csum = d_logit_scale ? F(P.o_csum) : nullptr;
    g.rowsig = (siglip && d_bias) ? F(P.o_sig) : nullptr;
    g.sig_slots = 4 * P.wgt.splits;
    g.lcount = labels ? F(P.o_lcount) : nullptr;
    g.pos_cos = F(P.o_pos);
    g.d_scale = d_logit_scale;
    g.d_bias = d_bias;
    ProfScope ps(UF_KERNEL_NORM_BWD, 1, stream);
    UF_CHECK(launch_scale_grad(g, stream));
  }
  if (col_terms && kind != KIND_CLIP) UF_CHECK(cudaMemsetAsync(col_terms, 0, sizeof(float) * n * Nb, stream));
#undef UF_CHECK
  return UF_OK;
}

}  // namespace

extern "C" {

uf_status_t uf_contrastive_fwd_bwd_ex(const void* A, const void* B, int64_t Na, int64_t Nb, int D,
                                      const int* prefixes, int n_prefix, int kind, float logit_scale, float bias,
                                      const float* logit_scale_dev, const float* bias_dev,
                                      const int64_t* pos_offsets, const int* pos_ids,
                                      const float* prefix_weights, float* loss_per_prefix, float* row_terms,
                                      float* col_terms, float* dA, float* dB, float* d_logit_scale, float* d_bias,
                                      void* workspace, size_t workspace_bytes, int* device_status,
                                      void* stream_handle) {
  return run_loss(A, B, Na, Nb, D, prefixes, n_prefix, kind, logit_scale, bias, logit_scale_dev, bias_dev,
                  pos_offsets, pos_ids, prefix_weights, loss_per_prefix, row_terms, col_terms, dA, dB, d_logit_scale,
                  d_bias, workspace, workspace_bytes, device_status, stream_handle, false);
}

uf_status_t uf_contrastive_oneset_fwd_bwd(const void* X, int64_t N, int D, const int* prefixes, int n_prefix,
                                          float logit_scale, float bias, const float* logit_scale_dev,
                                          const float* bias_dev, const int64_t* pos_offsets, const int* pos_ids,
                                          const float* prefix_weights, float* loss_per_prefix, float* row_terms,
                                          float* dX, float* d_logit_scale, float* d_bias, void* workspace,
                                          size_t workspace_bytes, int* device_status, void* stream_handle) {
  if (!pos_offsets || !pos_ids) return UF_INVALID_ARGUMENT;  // a one-set batch names its pairs
  return run_loss(X, X, N, N, D, prefixes, n_prefix, KIND_SIGLIP, logit_scale, bias, logit_scale_dev, bias_dev,
                  pos_offsets, pos_ids, prefix_weights, loss_per_prefix, row_terms, nullptr, dX, dX, d_logit_scale,
                  d_bias, workspace, workspace_bytes, device_status, stream_handle, true);
}

uf_status_t uf_contrastive_selftest_wait(int* device_status, int limit_ms, void* stream_handle) {
  if (!device_status || !aligned(device_status, 4) || limit_ms < 1 || limit_ms > 10000) return UF_INVALID_ARGUMENT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return UF_CUDA_ERROR;
  if (uf_contrastive_init(dev) != UF_OK) return UF_CUDA_ERROR;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
  if (launch_wait_selftest(device_status, static_cast<uint64_t>(limit_ms) * 1000000ull, stream) != cudaSuccess)
    return UF_CUDA_ERROR;
  return UF_OK;
}

uf_status_t uf_contrastive_profile(int enable) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (enable) {
    for (auto& r : g_prof_pending) {
      g_prof_pool.push_back(r.start);
      g_prof_pool.push_back(r.stop);
    }
    g_prof_pending.clear();
    for (int g = 0; g < UF_KERNEL_GROUPS; ++g) {
      g_prof_ms[g] = 0.0;
      g_prof_pairs[g] = g_prof_launches[g] = 0;
    }
  }
  g_prof_on.store(enable != 0);
  return UF_OK;
}

uf_status_t uf_contrastive_profile_read(int group, double* total_ms, int64_t* pairs, int64_t* launches) {
  if (group < 0 || group >= UF_KERNEL_GROUPS) return UF_INVALID_ARGUMENT;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  for (auto& r : g_prof_pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)
      return UF_CUDA_ERROR;
    g_prof_ms[r.group] += ms;
    g_prof_pairs[r.group] += 1;
    g_prof_launches[r.group] += r.launches;
    g_prof_pool.push_back(r.start);
    g_prof_pool.push_back(r.stop);
  }
  g_prof_pending.clear();
  if (total_ms) *total_ms = g_prof_ms[group];
  if (pairs) *pairs = g_prof_pairs[group];
  if (launches) *launches = g_prof_launches[group];
  return UF_OK;
}

const char* uf_contrastive_profile_name(int group) {
  static const char* names[UF_KERNEL_GROUPS] = {"prep",     "transpose", "fwd_tile", "stats",
                                                "bwd_tile", "norm_bwd",  "gemm"};
  return (group >= 0 && group < UF_KERNEL_GROUPS) ? names[group] : "unknown";
}

}  // extern "C"
