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

}  // namespace ufc
