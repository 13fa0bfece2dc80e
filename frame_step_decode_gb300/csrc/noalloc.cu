// noalloc.cu -- wave_step_static: the frame step without any allocation.
//
// Some callers cannot allocate device memory: code that runs inside another
// runtime's memory pool or a process with a fixed device-memory budget, a
// plug-in that must not create allocations the host application does not
// track, or a real-time serving loop where cudaMalloc's implicit
// synchronisation is not allowed once the clock runs.  For them this entry
// point runs the same persistent step kernel as wave_step, with its whole
// workspace (residual, activations, split-K and attention partials, work
// list, RoPE table, barrier and error words) placed in one fixed, file-scope
// device array instead of memory from cudaMalloc.
//
// The array is kNoAllocScratchBytes (32 MiB) and exists on every GPU that
// loads this library, for the life of the process.  Calls share it and it
// keeps the last call's contents; the words that must start at zero are
// cleared on every call.  Two calls whose work overlaps on the GPU (other
// streams, or without waiting) race on it.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "../../include/wave.h"
#include "internal.h"

using namespace wave;

namespace {

constexpr size_t kNoAllocScratchBytes = 32u << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  }
  return fn;
}

bool encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, void* base, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  EncodeTiledFn fn = encoder();
  return fn && fn(m, dt, (cuuint32_t)rank, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The RoPE table, (cos, sin) of t * base^(-2i/D) evaluated in double.
__global__ void k_rope_table(float2* tab, int T_max, int half, int D, double base) {
  const int n = T_max * half;
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < n; e += gridDim.x * blockDim.x) {
    const int t = e / half, i = e - t * half;
    const double a = (double)t * pow(base, -2.0 * i / (double)D);
    tab[e] = make_float2((float)cos(a), (float)sin(a));
  }
}

int max_tiles(long long tiles, long long kb, int grid, int seg_cap) {
  const long long U = tiles * kb;
  const int G = stream_k_ctas(grid, U, (int)tiles, seg_cap);
  int mt = 1;
  for (int c = 0; c < G; ++c) {
    const long long u0 = U * c / G, u1 = U * (c + 1) / G;
    if (u1 <= u0) continue;
    const int n = (int)((u1 - 1) / kb - u0 / kb + 1);
    if (n > mt) mt = n;
  }
  return mt;
}

int max_segs(long long tiles, long long kb, int grid, int seg_cap) {
  const long long U = tiles * kb;
  const int G = stream_k_ctas(grid, U, (int)tiles, seg_cap);
  int ms = 1;
  for (long long t = 0; t < tiles; ++t) {
    const long long a = t * kb, b = (t + 1) * kb - 1;
    const int ca = (int)(((a + 1) * G + U - 1) / U - 1), cb = (int)(((b + 1) * G + U - 1) / U - 1);
    if (cb - ca + 1 > ms) ms = cb - ca + 1;
  }
  return ms;
}

}  // namespace

extern "C" int wave_step_static(const wave_config* cfg, int S_max, int T_max, int S, const void* weights,
                                uint8_t* kv_fp8, float* kv_scales, const int32_t* positions,
                                const void* x, void* y, void* stream) {
  // ---- arguments (the same rules as wave_create + wave_step)
  if (!cfg || !weights || !kv_fp8 || !kv_scales || !positions || !x || !y) return WAVE_EINVAL;
  if (cfg->n_layers < 1 || cfg->n_layers > 1024 || (cfg->head_dim != 64 && cfg->head_dim != 128) ||
      cfg->n_heads < 1 || cfg->d_model < 64 || cfg->d_model % 64 || cfg->d_model > 8192 ||
      (cfg->n_heads * cfg->head_dim) % 64 || cfg->ffn < 8 || cfg->ffn % 8 || !(cfg->rms_eps >= 0.f) ||
      !(cfg->rope_base > 0.f))
    return WAVE_EINVAL;
  if (S_max < 1 || S_max > 128 || T_max < 4 || T_max % 4 || S < 1 || S > S_max) return WAVE_EINVAL;
  const long long rows = (long long)cfg->n_layers * 2 * S_max * cfg->n_heads * T_max;
  if (rows >= (1LL << 31) || T_max > 65535 * kChunk) return WAVE_EINVAL;
  if (((uintptr_t)weights & 15) || ((uintptr_t)kv_fp8 & 15) || ((uintptr_t)kv_scales & 15) ||
      ((uintptr_t)positions & 3) || ((uintptr_t)x & 15) || ((uintptr_t)y & 15))
    return WAVE_EINVAL;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return WAVE_ECUDA;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return WAVE_ECUDA;
  if (major != 10 || minor != 3) return WAVE_EDEVICE;

  // ---- one-time set-up on this device: the scratch array's device address
  // (the host-side name of a __device__ array is not a device pointer).
  char* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_addr[dev]) {
      if (configure_step_kernel() != cudaSuccess) return WAVE_ECUDA;
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return WAVE_ECUDA;
      g_scratch_addr[dev] = ptr;
    }
    base = (char*)g_scratch_addr[dev];
  }
  int per_sm = 0;
  if (occupancy_per_sm(&per_sm) != cudaSuccess || per_sm < 1) return WAVE_ELAUNCH;

  // ---- workspace carve-up inside the scratch array
  const int d = cfg->d_model, H = cfg->n_heads, D = cfg->head_dim, F = cfg->ffn, HD = H * D;
  const long long n_off[6] = {d, 3LL * HD * d, (long long)d * HD, d, 2LL * F * d, (long long)d * F};
  long long off[6], layer_elems = 0;
  for (int i = 0; i < 6; ++i) {
    off[i] = layer_elems;
    layer_elems += n_off[i];
  }
  int tiles[kGemmKinds] = {0}, kblocks[kGemmKinds] = {0};
  tiles[kQKV] = (3 * HD + kTileM - 1) / kTileM;
  kblocks[kQKV] = (d + kKUnit - 1) / kKUnit;
  tiles[kO] = (d + kTileM - 1) / kTileM;
  kblocks[kO] = (HD + kKUnit - 1) / kKUnit;
  tiles[kGU] = (F + 63) / 64;
  kblocks[kGU] = (d + kKUnit - 1) / kKUnit;
  tiles[kDown] = (d + kTileM - 1) / kTileM;
  kblocks[kDown] = (F + kKUnit - 1) / kKUnit;
  int mt = 1;
  for (int k = 0; k < 4; ++k) {
    if (tiles[k] > 1024 || max_segs(tiles[k], kblocks[k], sms, gemm_seg_cap(k)) > 64) return WAVE_EINVAL;
    const int m = max_tiles(tiles[k], kblocks[k], sms, gemm_seg_cap(k));
    if (m > mt) mt = m;
  }
  const long long SP = (S_max + 15) / 16 * 16;
  const long long max_pieces =
      (long long)S_max * H * (((T_max + kChunk - 1) / kChunk + kPieceChunks - 1) / kPieceChunks);
  const size_t sizes[14] = {(size_t)(SP * d * 4),        (size_t)(SP * d * 2),
                            (size_t)(SP * 3 * HD * 4),   (size_t)(SP * HD * 2),
                            (size_t)(SP * F * 2),        (size_t)sms * mt * SP * kTileM * 4,
                            kCounterWords * 4,           (size_t)(max_pieces * (D + 4) * 4),
                            (size_t)(S_max * H * 8),     (size_t)(max_pieces * 32),
                            16,                          (size_t)T_max * (D / 2) * 8,
                            16,                          16};
  size_t offs[14], total = 0;
  for (int i = 0; i < 14; ++i) {
    offs[i] = total;
    total += (sizes[i] + 255) & ~(size_t)255;
  }
  if (total > kNoAllocScratchBytes) return WAVE_EINVAL;  // shape too large for the fixed scratch

  StepParams p;
  memset(&p, 0, sizeof(p));
  p.n_frames = 1;
  p.merge = needs_merge(T_max) ? 1 : 0;
  p.resid = (float*)(base + offs[0]);
  p.xn = (uint16_t*)(base + offs[1]);
  p.qkv = (float*)(base + offs[2]);
  p.attn = (uint16_t*)(base + offs[3]);
  p.u = (uint16_t*)(base + offs[4]);
  p.gemm_part = (float*)(base + offs[5]);
  p.tile_cnt = (int*)(base + offs[6]);
  p.att_ctr = p.tile_cnt + 2048;
  p.att_part = (float*)(base + offs[7]);
  p.sh_info = (int2*)(base + offs[8]);
  p.pieces = (int4*)(base + offs[9]);
  p.n_pieces = (int*)(base + offs[10]);
  float2* rope = (float2*)(base + offs[11]);
  p.rope = rope;
  p.bar = (unsigned*)(base + offs[12]);
  p.err = (int*)(base + offs[13]);

  // ---- tensor maps over the caller's weights / history and the scratch activations
  const int S_pad = (S + 15) / 16 * 16;
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  const cuuint64_t ud = d, uHD = HD, uF = F, uL = cfg->n_layers, ls = (cuuint64_t)layer_elems * 2;
  char* wb = (char*)weights;
  bool ok = true;
  {
    cuuint64_t dims[3] = {ud, 3 * uHD, uL}, str[2] = {ud * 2, ls};
    cuuint32_t box[3] = {kKBlk, kTileM, 1};
    ok = ok && encode(&p.tm_w[kQKV], BF, 3, wb + off[1] * 2, dims, str, box, SW);
  }
  {
    cuuint64_t dims[3] = {uHD, ud, uL}, str[2] = {uHD * 2, ls};
    cuuint32_t box[3] = {kKBlk, kTileM, 1};
    ok = ok && encode(&p.tm_w[kO], BF, 3, wb + off[2] * 2, dims, str, box, SW);
  }
  {
    cuuint64_t dims[4] = {ud, uF, 2, uL}, str[3] = {ud * 2, uF * ud * 2, ls};
    cuuint32_t box[4] = {kKBlk, 64, 1, 1};
    ok = ok && encode(&p.tm_w[kGU], BF, 4, wb + off[4] * 2, dims, str, box, SW);
  }
  {
    cuuint64_t dims[3] = {uF, ud, uL}, str[2] = {uF * 2, ls};
    cuuint32_t box[3] = {kKBlk, kTileM, 1};
    ok = ok && encode(&p.tm_w[kDown], BF, 3, wb + off[5] * 2, dims, str, box, SW);
  }
  {
    cuuint32_t box[2] = {kKBlk, (cuuint32_t)S_pad};
    cuuint64_t d1[2] = {ud, (cuuint64_t)SP}, s1[1] = {ud * 2};
    ok = ok && encode(&p.tm_x[kQKV], BF, 2, p.xn, d1, s1, box, SW);
    p.tm_x[kGU] = p.tm_x[kQKV];
    cuuint64_t d2[2] = {uHD, (cuuint64_t)SP}, s2[1] = {uHD * 2};
    ok = ok && encode(&p.tm_x[kO], BF, 2, p.attn, d2, s2, box, SW);
    cuuint64_t d3[2] = {uF, (cuuint64_t)SP}, s3[1] = {uF * 2};
    ok = ok && encode(&p.tm_x[kDown], BF, 2, p.u, d3, s3, box, SW);
  }
  {
    const cuuint64_t uD = D, n1 = (cuuint64_t)S_max * H * T_max;
    cuuint64_t dims[4] = {uD, n1, 2, uL}, str[3] = {uD, n1 * uD, 2 * n1 * uD};
    cuuint32_t box[4] = {(cuuint32_t)D, (cuuint32_t)kChunk, 2, 1};
    ok = ok && encode(&p.tm_kv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, kv_fp8, dims, str, box,
                      D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
    cuuint64_t sdims[3] = {n1, 2, uL}, sstr[2] = {n1 * 4, 2 * n1 * 4};
    cuuint32_t sbox[3] = {(cuuint32_t)kChunk, 2, 1};
    ok = ok && encode(&p.tm_sc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, kv_scales, sdims, sstr, sbox,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  if (!ok) return WAVE_ECUDA;

  p.L = cfg->n_layers;
  p.d = d;
  p.H = H;
  p.D = D;
  p.F = F;
  p.HD = HD;
  p.S = S;
  p.S_pad = S_pad;
  p.S_max = S_max;
  p.T_max = T_max;
  p.eps = cfg->rms_eps;
  for (int k = 0; k < 4; ++k) {
    p.tiles[k] = tiles[k];
    p.kblocks[k] = kblocks[k];
  }
  const int stride = gemm_stage_bytes(S_pad);
  const int nst = smem_layout().gemm_ring_bytes / stride;
  p.nstage = nst > kMaxStages ? kMaxStages : nst;
  p.max_tiles_per_cta = mt;
  p.layer_elems = layer_elems;
  p.off_g_attn = off[0];
  p.off_g_mlp = off[3];
  p.off_wo = off[2];
  p.off_wdown = off[5];
  p.weights = (const uint16_t*)weights;
  p.kv = kv_fp8;
  p.kv_scales = kv_scales;
  p.pos = positions;
  p.x = (const uint16_t*)x;
  p.y = (uint16_t*)y;
  p.timeout_ns = 2000000000LL;
  p.skip_cta = -1;
  p.skip_bar = -1;

  // ---- clear what must start at zero, rebuild the RoPE table, launch, wait
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(p.bar, 0, 16, st) != cudaSuccess || cudaMemsetAsync(p.err, 0, 16, st) != cudaSuccess)
    return WAVE_ECUDA;
  k_rope_table<<<64, 256, 0, st>>>(rope, T_max, D / 2, D, (double)cfg->rope_base);
  if (cudaGetLastError() != cudaSuccess) return WAVE_ECUDA;
  const cudaError_t e = launch_step(p, sms, st);
  if (e == cudaErrorCooperativeLaunchTooLarge) return WAVE_ELAUNCH;
  if (e != cudaSuccess) return WAVE_ECUDA;
  int err = 0;
  if (cudaMemcpyAsync(&err, p.err, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return WAVE_ECUDA;
  if (err & kErrTimeout) return WAVE_ETIMEOUT;
  if (err) return WAVE_EPOS;
  return WAVE_OK;
}
