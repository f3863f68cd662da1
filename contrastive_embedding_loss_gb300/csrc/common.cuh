// common.cuh -- parameters shared by the host launcher and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace ufc {

constexpr int kMaxPrefix = 8;
constexpr int kTileRows = 128;   // rows of X per CTA = UMMA M
constexpr int kChunk = 64;       // K elements per shared-memory stage: one 128-byte swizzle row

enum Kind : int { KIND_CLIP = 0, KIND_SIGLIP = 1, KIND_ROWS = 2 };

constexpr int kStatusTimeout = 5;  // == UF_DEVICE_TIMEOUT
constexpr int kStatusBadScalar = 1;  // == UF_INVALID_ARGUMENT: a logit scale / bias read on the device is out of range

// Largest logit scale the fixed-shift statistics take: every logit lies in [-tau, tau], so
// with the shift tau the smallest term e^{-2 tau} stays a normal fp32 up to tau ~ 43.
// Larger scales (and scales that only the device knows) take the max-shifted path.
constexpr float kFixedShiftMaxScale = 40.f;
// Largest logit scale accepted at all: the scores carry the fp32 error of a 1024-term
// dot product (~1e-6 of the cosine), which the softmax multiplies by the scale.
constexpr float kMaxLogitScale = 256.f;
// SigLIP: |t| + |b| bound (x = t cos + b stays well inside fp32's exp2 range in log2 units).
constexpr float kMaxSiglipRange = 80.f;

// The loss's two learned scalars (logit scale tau or t; SigLIP bias b): host values, or
// device fp32 scalars that every kernel reads when it starts (a captured CUDA graph then
// follows a scale that training updates in place).
struct Scalars {
  float scale, bias;
  const float* scale_ptr;  // device or NULL (then `scale`)
  const float* bias_ptr;   // device or NULL (then `bias`)
#ifdef __CUDACC__
  __device__ __forceinline__ float t() const { return scale_ptr ? __ldg(scale_ptr) : scale; }
  __device__ __forceinline__ float b() const { return bias_ptr ? __ldg(bias_ptr) : bias; }
#endif
};

}  // namespace ufc
