// synth_gpu.cu -- device twin of synth.c: the same counter-based generator,
// bit for bit, so that multi-gigabyte inputs (a 7B-class weight blob, a
// 65 GB FP8 history) can be drawn where they live.  Holds none of the decode
// step's arithmetic; see synth.c for the generator's definition.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#define SYNTH_G 0x9E3779B97F4A7C15ULL

__host__ __device__ static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static uint64_t key_of(uint64_t seed, uint64_t stream) {
  return mix64(seed * 0xD1B54A32D192ED03ULL + (stream + 1) * SYNTH_G);
}

__device__ static inline float normal_at(uint64_t key, uint64_t i) {
  uint32_t sum = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint64_t w = mix64(key + (4 * i + (uint64_t)j + 1) * SYNTH_G);
    sum += (uint32_t)(w & 0xFFFFF) + (uint32_t)((w >> 20) & 0xFFFFF) +
           (uint32_t)((w >> 40) & 0xFFFFF);
  }
  return (float)((int32_t)sum - 6 * 1048576) * (1.0f / 1048576.0f);
}

__global__ void k_normal_bf16(uint64_t key, uint64_t start, int64_t count,
                              float scale, __nv_bfloat16* out) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < count; j += stride)
    out[j] = __float2bfloat16_rn(__fmul_rn(normal_at(key, start + (uint64_t)j), scale));
}

__global__ void k_normal_f32(uint64_t key, uint64_t start, int64_t count, float* out) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < count; j += stride)
    out[j] = normal_at(key, start + (uint64_t)j);
}

// out[((s-s0)*H + h)*out_T + t][i] for t < t_count, as synth_kv_slab_f32.
__global__ void k_kv_slab(uint64_t key, int s0, int ns, int H, int T_ref, int t_count,
                          int D, int64_t out_T, float* out) {
  int64_t total = (int64_t)ns * H * t_count * D;
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += stride) {
    int i = (int)(e % D);
    int64_t rt = e / D;
    int t = (int)(rt % t_count);
    int64_t r = rt / t_count;
    int64_t s = s0 + r / H, h = r % H;
    uint64_t idx = (uint64_t)(((s * H + h) * T_ref + t) * D + i);
    out[(r * out_T + t) * D + i] = normal_at(key, idx);
  }
}

static int grid_for(int64_t n) {
  int64_t g = (n + 255) / 256;
  if (g > 152 * 32) g = 152 * 32;
  if (g < 1) g = 1;
  return (int)g;
}

extern "C" {

int synth_gpu_normal_bf16(uint64_t seed, uint64_t stream, uint64_t start, int64_t count,
                          float scale, void* out, void* cuda_stream) {
  if (count <= 0) return 0;
  k_normal_bf16<<<grid_for(count), 256, 0, (cudaStream_t)cuda_stream>>>(
      key_of(seed, stream), start, count, scale, (__nv_bfloat16*)out);
  return (int)cudaGetLastError();
}

int synth_gpu_normal_f32(uint64_t seed, uint64_t stream, uint64_t start, int64_t count,
                         float* out, void* cuda_stream) {
  if (count <= 0) return 0;
  k_normal_f32<<<grid_for(count), 256, 0, (cudaStream_t)cuda_stream>>>(
      key_of(seed, stream), start, count, out);
  return (int)cudaGetLastError();
}

int synth_gpu_kv_slab_f32(uint64_t seed, uint64_t stream, int s0, int ns, int H, int T_ref,
                          int t_count, int D, int64_t out_T, float* out, void* cuda_stream) {
  int64_t total = (int64_t)ns * H * t_count * D;
  if (total <= 0) return 0;
  k_kv_slab<<<grid_for(total), 256, 0, (cudaStream_t)cuda_stream>>>(
      key_of(seed, stream), s0, ns, H, T_ref, t_count, D, out_T, out);
  return (int)cudaGetLastError();
}

}  // extern "C"
