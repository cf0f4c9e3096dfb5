// Shared device/host helpers of libmlora (internal header).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mlora.h"

namespace mlk {

constexpr int TILE_M = MLORA_TILE_M;   // routing / GEMM row tile
constexpr int RP = MLORA_MAX_RANK;     // padded rank of the bf16 / fp32 factor copies

// Device status bits (OR-ed by kernels, read by mlora_check_status).
constexpr int ST_RANGE = 1;
constexpr int ST_TIMEOUT = 2;

typedef __nv_bfloat16 bf16;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ float sigmoidf_(float u) { return 1.0f / (1.0f + __expf(-u)); }

__device__ __forceinline__ void raise_status(int* st, int bit) {
    if (st) atomicOr(st, bit);
}

// Host-side launch bookkeeping.
struct LaunchCounter {
    int64_t n = 0;
};

}  // namespace mlk
