// quant.cu -- the K/V quantiser and the E4M3 encoder as stand-alone entry
// points (same device code as the append inside the step).
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/wave.h"
#include "fp8.cuh"

namespace wave {

// One warp per row of D = 32 * kPer values.
template <int kPer>
__global__ void k_quantize_rows(const float* __restrict__ v, int64_t rows, uint8_t* __restrict__ codes,
                                float* __restrict__ scales) {
  constexpr int D = 32 * kPer;
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
    float x[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) x[e] = v[r * D + lane * kPer + e];
    float s;
    uint32_t packed = quantize_lane<kPer>(x, s);
#pragma unroll
    for (int e = 0; e < kPer; ++e) codes[r * D + lane * kPer + e] = (uint8_t)(packed >> (8 * e));
    if (lane == 0) scales[r] = s;
  }
}

// Generic D (multiple of 4): one warp per row, lanes stride over the row.
__global__ void k_quantize_rows_any(const float* __restrict__ v, int64_t rows, int D,
                                   uint8_t* __restrict__ codes, float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
    float amax = 0.f;
    for (int i = lane; i < D; i += 32) amax = fmaxf(amax, fabsf(v[r * D + i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = __fdiv_rn(amax, 448.0f);
    for (int i = lane; i < D; i += 32)
      codes[r * D + i] = (s == 0.f) ? 0 : e4m3_encode(__fdiv_rn(v[r * D + i], s));
    if (lane == 0) scales[r] = s;
  }
}

__global__ void k_encode(const float* __restrict__ in, int64_t n, uint8_t* __restrict__ out) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = e4m3_encode(in[i]);
}

static int blocks_for(int64_t work, int per_block) {
  int64_t b = (work + per_block - 1) / per_block;
  if (b > 152 * 16) b = 152 * 16;
  return b < 1 ? 1 : (int)b;
}

}  // namespace wave

using namespace wave;

extern "C" int wave_kv_quantize(const float* v, int64_t rows, int D, uint8_t* codes, float* scales,
                                void* stream) {
  if (!v || !codes || !scales || rows < 0 || D < 4 || D > 1024 || D % 4) return WAVE_EINVAL;
  if (rows == 0) return WAVE_OK;
  cudaStream_t st = (cudaStream_t)stream;
  const int grid = blocks_for(rows, 8);
  if (D == 128)
    k_quantize_rows<4><<<grid, 256, 0, st>>>(v, rows, codes, scales);
  else if (D == 64)
    k_quantize_rows<2><<<grid, 256, 0, st>>>(v, rows, codes, scales);
  else
    k_quantize_rows_any<<<grid, 256, 0, st>>>(v, rows, D, codes, scales);
  return cudaGetLastError() == cudaSuccess ? WAVE_OK : WAVE_ECUDA;
}

extern "C" int wave_fp8_encode(const float* in, int64_t n, uint8_t* out, void* stream) {
  if (!in || !out || n < 0) return WAVE_EINVAL;
  if (n == 0) return WAVE_OK;
  k_encode<<<blocks_for(n, 256), 256, 0, (cudaStream_t)stream>>>(in, n, out);
  return cudaGetLastError() == cudaSuccess ? WAVE_OK : WAVE_ECUDA;
}
