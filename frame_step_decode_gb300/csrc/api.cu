// api.cu -- host side of the C ABI in include/wave.h: argument checks,
// workspace ownership, TMA tensor-map encoding and the single cooperative
// launch per frame.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <vector>

#include "../../include/wave.h"
#include "internal.h"

using namespace wave;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct wave_ctx {
  wave_config cfg;
  int S_max, S_pad_max, T_max, device, grid;
  long long layer_elems, off[6];
  int tiles[kGemmKinds], kblocks[kGemmKinds], max_tiles_per_cta;
  // workspace
  void* ws = nullptr;
  size_t ws_bytes = 0;
  float* resid;
  uint16_t *xn, *attn, *u;
  float* qkv;
  float* gemm_part;
  int* tile_cnt;
  float* att_part;
  int2* sh_info;
  int4* pieces;
  int* n_pieces;
  float2* rope;
  unsigned* bar;
  int* err;
  // cached tensor maps
  CUtensorMap tm_w[kGemmKinds], tm_x[kGemmKinds], tm_kv, tm_sc;
  const void* maps_wp = nullptr;  // W_p the kProj weight map was encoded for
  int32_t* zero_pos = nullptr;    // S_max zeros: chained frames start at position 0
  const void* maps_weights = nullptr;
  const void* maps_kv = nullptr;
  const void* maps_sc = nullptr;
  int maps_S = -1;
  cudaStream_t last_stream = nullptr;
  long long timeout_ns = 2000000000LL;
  int skip_cta = -1, skip_bar = -1;
  float* kv_dump = nullptr;
  long long* phase_ts = nullptr;
  long long* arrive_ts = nullptr;
  // hybrid model (wave_hybrid_create); cfg then describes its attention layers
  int hybrid = 0;
  wave_hybrid_config hcfg;
  long long hyb_M = 0, hyb_G = 0, hyb_off_w_in = 0, hyb_off_w_out = 0, hyb_off_a_log = 0;
  long long hyb_off_wqkv = 0, hyb_off_wo = 0;  // inside an attention block
  float* zx = nullptr;
  uint16_t* ssm_out = nullptr;
};

static EncodeTiledFn encode_fn() {
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

static bool shape_ok(const wave_config* c) {
  if (!c) return false;
  if (c->n_layers < 1 || c->n_layers > 1024) return false;
  if (c->head_dim != 64 && c->head_dim != 128) return false;
  if (c->n_heads < 1 || c->d_model < 64 || c->d_model % 64 || c->d_model > 8192) return false;
  if ((c->n_heads * c->head_dim) % 64) return false;
  if (c->ffn < 8 || c->ffn % 8) return false;
  if (!(c->rms_eps >= 0.f) || !(c->rope_base > 0.f)) return false;
  return true;
}

static void layout_offsets(const wave_config* c, long long* off, long long* layer_elems) {
  const long long d = c->d_model, HD = (long long)c->n_heads * c->head_dim, F = c->ffn;
  const long long n[6] = {d, 3 * HD * d, d * HD, d, 2 * F * d, d * F};
  long long o = 0;
  for (int i = 0; i < 6; ++i) {
    off[i] = o;
    o += n[i];
  }
  *layer_elems = o;
}

extern "C" size_t wave_weights_bytes(const wave_config* cfg) {
  if (!shape_ok(cfg)) return 0;
  long long off[6], le;
  layout_offsets(cfg, off, &le);
  return (size_t)(le * cfg->n_layers * 2);
}

extern "C" size_t wave_weight_offset(const wave_config* cfg, int layer, int which) {
  if (!shape_ok(cfg) || layer < 0 || layer >= cfg->n_layers || which < 0 || which > 5)
    return (size_t)-1;
  long long off[6], le;
  layout_offsets(cfg, off, &le);
  return (size_t)((le * layer + off[which]) * 2);
}

extern "C" const char* wave_strerror(int code) {
  switch (code) {
    case WAVE_OK: return "ok";
    case WAVE_EINVAL: return "invalid argument";
    case WAVE_ECUDA: return "CUDA call failed";
    case WAVE_ELAUNCH: return "persistent grid could not be launched co-resident";
    case WAVE_ETIMEOUT: return "a device-side wait timed out";
    case WAVE_EPOS: return "a session position was at or beyond T_max";
    case WAVE_EDEVICE: return "device is not sm_103";
    case WAVE_ENOMEM: return "device allocation failed";
    default: return "unknown error";
  }
}

// Stream-K split of tiles x kblocks over the grid: the most tiles one CTA touches.
static int max_tiles_touched(long long tiles, long long kb, int grid, int seg_cap) {
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

// Most segments (CTAs) any one tile is split into.
static int max_segments(long long tiles, long long kb, int grid, int seg_cap) {
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

static int device_check(int* dev, int* sms) {
  if (cudaGetDevice(dev) != cudaSuccess) return WAVE_ECUDA;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, *dev) != cudaSuccess) return WAVE_ECUDA;
  if (prop.major != 10 || prop.minor != 3) return WAVE_EDEVICE;
  if (!encode_fn()) return WAVE_ECUDA;
  if (configure_step_kernel() != cudaSuccess) return WAVE_ECUDA;
  *sms = prop.multiProcessorCount;
  return WAVE_OK;
}

static int build_ctx(wave_ctx* h, int S_max, int T_max, int in_rows, int d_inner);

extern "C" int wave_create(const wave_config* cfg, int S_max, int T_max, wave_t** out) {
  if (!out || !shape_ok(cfg) || S_max < 1 || S_max > 128 || T_max < 4 || T_max % 4) return WAVE_EINVAL;
  const long long rows = (long long)cfg->n_layers * 2 * S_max * cfg->n_heads * T_max;
  if (rows >= (1LL << 31) || T_max > 65535 * kChunk) return WAVE_EINVAL;
  int dev = 0, sms = 0;
  int rc = device_check(&dev, &sms);
  if (rc) return rc;
  wave_ctx* h = new wave_ctx();
  h->cfg = *cfg;
  h->device = dev;
  h->grid = sms;
  layout_offsets(cfg, h->off, &h->layer_elems);
  rc = build_ctx(h, S_max, T_max, 0, 0);
  if (rc) {
    delete h;
    return rc;
  }
  *out = h;
  return WAVE_OK;
}

// Tiles, workspace and RoPE table of a handle whose cfg (and, for the hybrid
// model, hcfg) is set.  On failure nothing stays allocated.
static int build_ctx(wave_ctx* h, int S_max, int T_max, int in_rows, int d_inner) {
  const wave_config* cfg = &h->cfg;
  h->S_max = S_max;
  h->S_pad_max = (S_max + 15) / 16 * 16;
  h->T_max = T_max;
  const int d = cfg->d_model, HD = cfg->n_heads * cfg->head_dim, F = cfg->ffn, H = cfg->n_heads,
            D = cfg->head_dim;
  h->tiles[kQKV] = (3 * HD + kTileM - 1) / kTileM;
  h->kblocks[kQKV] = (d + kKUnit - 1) / kKUnit;
  h->tiles[kO] = (d + kTileM - 1) / kTileM;
  h->kblocks[kO] = (HD + kKUnit - 1) / kKUnit;
  h->tiles[kGU] = (F + 63) / 64;
  h->kblocks[kGU] = (d + kKUnit - 1) / kKUnit;
  h->tiles[kDown] = F ? (d + kTileM - 1) / kTileM : 0;
  h->kblocks[kDown] = (F + kKUnit - 1) / kKUnit;
  h->tiles[kProj] = h->hybrid ? 0 : (d + kTileM - 1) / kTileM;
  h->kblocks[kProj] = (d + kKUnit - 1) / kKUnit;
  h->tiles[kIn] = (in_rows + kTileM - 1) / kTileM;
  h->kblocks[kIn] = (d + kKUnit - 1) / kKUnit;
  h->tiles[kOut] = d_inner ? (d + kTileM - 1) / kTileM : 0;
  h->kblocks[kOut] = (d_inner + kKUnit - 1) / kKUnit;
  int mt = 1;
  for (int k = 0; k < kGemmKinds; ++k) {
    if (h->tiles[k] > 1024) return WAVE_EINVAL;
    int m = max_tiles_touched(h->tiles[k], h->kblocks[k], h->grid, gemm_seg_cap(k));
    if (m > mt) mt = m;
    if (max_segments(h->tiles[k], h->kblocks[k], h->grid, gemm_seg_cap(k)) > 64) return WAVE_EINVAL;
  }
  h->max_tiles_per_cta = mt;

  // workspace carve-up (256-byte aligned pieces)
  const long long SP = h->S_pad_max;
  const long long max_pieces =
      (long long)S_max * H * (((T_max + kChunk - 1) / kChunk + kPieceChunks - 1) / kPieceChunks);
  struct Part { void** dst; size_t bytes; };
  std::vector<Part> parts = {
      {(void**)&h->resid, (size_t)(SP * d * 4)},
      {(void**)&h->xn, (size_t)(SP * d * 2)},
      {(void**)&h->qkv, (size_t)(SP * 3 * HD * 4)},
      {(void**)&h->attn, (size_t)(SP * HD * 2)},
      {(void**)&h->u, (size_t)(SP * F * 2)},
      {(void**)&h->gemm_part, (size_t)h->grid * mt * SP * kTileM * 4},
      {(void**)&h->tile_cnt, kCounterWords * 4},
      {(void**)&h->att_part, (size_t)(max_pieces * (D + 4) * 4)},
      {(void**)&h->sh_info, (size_t)(S_max * H * 8)},
      {(void**)&h->pieces, (size_t)(max_pieces * 32)},
      {(void**)&h->n_pieces, 16},
      {(void**)&h->rope, (size_t)T_max * (D / 2) * 8},
      {(void**)&h->bar, 16},
      {(void**)&h->err, 16},
      {(void**)&h->zero_pos, (size_t)S_max * 4},
      {(void**)&h->zx, (size_t)(SP * in_rows * 4)},
      {(void**)&h->ssm_out, (size_t)(SP * d_inner * 2)},
  };
  size_t total = 0;
  for (auto& pt : parts) total += (pt.bytes + 255) & ~(size_t)255;
  if (cudaMalloc(&h->ws, total) != cudaSuccess) return WAVE_ENOMEM;
  h->ws_bytes = total;
  if (cudaMemset(h->ws, 0, total) != cudaSuccess) {
    cudaFree(h->ws);
    h->ws = nullptr;
    return WAVE_ECUDA;
  }
  size_t o = 0;
  for (auto& pt : parts) {
    *pt.dst = (char*)h->ws + o;
    o += (pt.bytes + 255) & ~(size_t)255;
  }
  // RoPE table: angle t * base^(-2i/D), evaluated in double, stored as fp32.
  std::vector<float2> tab((size_t)T_max * (D / 2));
  for (int t = 0; t < T_max; ++t)
    for (int i = 0; i < D / 2; ++i) {
      const double th = pow((double)cfg->rope_base, -2.0 * i / (double)D);
      const double a = (double)t * th;
      tab[(size_t)t * (D / 2) + i] = make_float2((float)cos(a), (float)sin(a));
    }
  if (cudaMemcpy(h->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice) !=
      cudaSuccess) {
    cudaFree(h->ws);
    h->ws = nullptr;
    return WAVE_ECUDA;
  }
  // co-residency: one CTA per SM must fit
  int per_sm = 0;
  if (occupancy_per_sm(&per_sm) != cudaSuccess || per_sm < 1) {
    cudaFree(h->ws);
    h->ws = nullptr;
    return WAVE_ELAUNCH;
  }
  return WAVE_OK;
}

// ---------------------------------------------------------- hybrid model
static bool hybrid_ok(const wave_hybrid_config* c) {
  if (!c) return false;
  if (c->n_layers < 1 || c->n_layers > 1024 || c->attn_every < 1 || c->n_layers % c->attn_every) return false;
  if (c->d_model < 64 || c->d_model % 64 || c->d_model > 8192) return false;
  if (c->head_dim != 64 && c->head_dim != 128) return false;
  if (c->n_heads < 1 || (c->n_heads * c->head_dim) % 64) return false;
  if (c->ssm_head_dim != kSsmP || c->ssm_state != kSsmN) return false;
  if (c->ssm_heads < 4 || c->ssm_heads % 4 || c->ssm_heads > kSsmMaxHeads) return false;
  if (!(c->rms_eps >= 0.f) || !(c->rope_base > 0.f)) return false;
  return true;
}

static void hybrid_layout(const wave_hybrid_config* c, long long* M, long long* A, long long* w_in,
                          long long* w_out, long long* a_log, long long* wqkv, long long* wo) {
  const long long d = c->d_model, di = (long long)c->ssm_heads * c->ssm_head_dim;
  const long long HD = (long long)c->n_heads * c->head_dim;
  const long long rows = 2 * di + 2 * c->ssm_state + c->ssm_heads;
  *w_in = d;
  *w_out = d + rows * d;
  *a_log = *w_out + d * di;
  *M = *a_log + (3LL * c->ssm_heads + 7) / 8 * 8;
  *wqkv = d;
  *wo = d + 3 * HD * d;
  *A = *wo + d * HD;
}

extern "C" size_t wave_hybrid_weights_bytes(const wave_hybrid_config* cfg) {
  if (!hybrid_ok(cfg)) return 0;
  long long M, A, a, b, c, q, o;
  hybrid_layout(cfg, &M, &A, &a, &b, &c, &q, &o);
  const int e = cfg->attn_every;
  return (size_t)((cfg->n_layers / e) * ((e - 1) * M + A) * 2);
}

extern "C" size_t wave_hybrid_layer_offset(const wave_hybrid_config* cfg, int layer) {
  if (!hybrid_ok(cfg) || layer < 0 || layer > cfg->n_layers) return (size_t)-1;
  long long M, A, a, b, c, q, o;
  hybrid_layout(cfg, &M, &A, &a, &b, &c, &q, &o);
  return (size_t)(hyb_layer_offset(M, (cfg->attn_every - 1) * M + A, cfg->attn_every, layer) * 2);
}

extern "C" int wave_hybrid_create(const wave_hybrid_config* hc, int S_max, int T_max, wave_t** out) {
  if (!out || !hybrid_ok(hc) || S_max < 1 || S_max > 128 || T_max < 4 || T_max % 4) return WAVE_EINVAL;
  const int La = hc->n_layers / hc->attn_every;
  const long long rows = (long long)La * 2 * S_max * hc->n_heads * T_max;
  if (rows >= (1LL << 31) || T_max > 65535 * kChunk) return WAVE_EINVAL;
  int dev = 0, sms = 0;
  int rc = device_check(&dev, &sms);
  if (rc) return rc;
  wave_ctx* h = new wave_ctx();
  h->hybrid = 1;
  h->hcfg = *hc;
  // cfg describes the attention layers (their history and maps)
  h->cfg.n_layers = La;
  h->cfg.d_model = hc->d_model;
  h->cfg.n_heads = hc->n_heads;
  h->cfg.head_dim = hc->head_dim;
  h->cfg.ffn = 0;
  h->cfg.rms_eps = hc->rms_eps;
  h->cfg.rope_base = hc->rope_base;
  h->device = dev;
  h->grid = sms;
  long long A;
  hybrid_layout(hc, &h->hyb_M, &A, &h->hyb_off_w_in, &h->hyb_off_w_out, &h->hyb_off_a_log, &h->hyb_off_wqkv,
                &h->hyb_off_wo);
  h->hyb_G = (hc->attn_every - 1) * h->hyb_M + A;
  for (int i = 0; i < 6; ++i) h->off[i] = 0;
  h->layer_elems = h->hyb_G;
  const int di = hc->ssm_heads * hc->ssm_head_dim;
  rc = build_ctx(h, S_max, T_max, 2 * di + 2 * hc->ssm_state + hc->ssm_heads, di);
  if (rc) {
    delete h;
    return rc;
  }
  *out = h;
  return WAVE_OK;
}

extern "C" void wave_destroy(wave_t* h) {
  if (!h) return;
  cudaDeviceSynchronize();
  cudaFree(h->ws);
  delete h;
}

static bool enc(CUtensorMap* m, CUtensorMapDataType dt, int rank, void* base, const cuuint64_t* dims,
                const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return encode_fn()(m, dt, (cuuint32_t)rank, base, dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int encode_hybrid_weight_maps(wave_ctx* h, const void* weights) {
  const wave_hybrid_config& c = h->hcfg;
  const cuuint64_t d = c.d_model, HD = (cuuint64_t)c.n_heads * c.head_dim;
  const cuuint64_t di = (cuuint64_t)c.ssm_heads * c.ssm_head_dim;
  const cuuint64_t rows = 2 * di + 2 * c.ssm_state + c.ssm_heads;
  const cuuint64_t e = c.attn_every, groups = c.n_layers / c.attn_every;
  const cuuint64_t M2 = (cuuint64_t)h->hyb_M * 2, G2 = (cuuint64_t)h->hyb_G * 2;
  char* base = (char*)weights;
  char* attn0 = base + (e - 1) * M2;  // the first attention block
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  {  // attention Wqkv [La][3HD][d], one attention block per group
    cuuint64_t dims[3] = {d, 3 * HD, groups}, str[2] = {d * 2, G2};
    cuuint32_t box[3] = {kKBlk, kTileM, 1};
    if (!enc(&h->tm_w[kQKV], BF, 3, attn0 + h->hyb_off_wqkv * 2, dims, str, box, SW)) return WAVE_ECUDA;
  }
  {  // attention Wo [La][d][HD]
    cuuint64_t dims[3] = {HD, d, groups}, str[2] = {HD * 2, G2};
    cuuint32_t box[3] = {kKBlk, kTileM, 1};
    if (!enc(&h->tm_w[kO], BF, 3, attn0 + h->hyb_off_wo * 2, dims, str, box, SW)) return WAVE_ECUDA;
  }
  if (e > 1) {
    {  // W_in [group][place][rows][d]
      cuuint64_t dims[4] = {d, rows, e - 1, groups}, str[3] = {d * 2, M2, G2};
      cuuint32_t box[4] = {kKBlk, kTileM, 1, 1};
      if (!enc(&h->tm_w[kIn], BF, 4, base + h->hyb_off_w_in * 2, dims, str, box, SW)) return WAVE_ECUDA;
    }
    {  // W_out [group][place][d][d_inner]
      cuuint64_t dims[4] = {di, d, e - 1, groups}, str[3] = {di * 2, M2, G2};
      cuuint32_t box[4] = {kKBlk, kTileM, 1, 1};
      if (!enc(&h->tm_w[kOut], BF, 4, base + h->hyb_off_w_out * 2, dims, str, box, SW)) return WAVE_ECUDA;
    }
  }
  return WAVE_OK;
}

static int encode_weight_maps(wave_ctx* h, const void* weights) {
  if (h->hybrid) return encode_hybrid_weight_maps(h, weights);
  const wave_config& c = h->cfg;
  const cuuint64_t d = c.d_model, HD = (cuuint64_t)c.n_heads * c.head_dim, F = c.ffn, L = c.n_layers;
  const cuuint64_t ls = (cuuint64_t)h->layer_elems * 2;  // layer stride in bytes
  char* base = (char*)weights;
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  {  // Wqkv [L][3HD][d]
    cuuint64_t dims[3] = {d, 3 * HD, L}, str[2] = {d * 2, ls};
    cuuint32_t box[3] = {kKBlk, kTileM, 1};
    if (!enc(&h->tm_w[kQKV], BF, 3, base + h->off[1] * 2, dims, str, box, SW)) return WAVE_ECUDA;
  }
  {  // Wo [L][d][HD]
    cuuint64_t dims[3] = {HD, d, L}, str[2] = {HD * 2, ls};
    cuuint32_t box[3] = {kKBlk, kTileM, 1};
    if (!enc(&h->tm_w[kO], BF, 3, base + h->off[2] * 2, dims, str, box, SW)) return WAVE_ECUDA;
  }
  {  // Wgu [L][2][F][d]
    cuuint64_t dims[4] = {d, F, 2, L}, str[3] = {d * 2, F * d * 2, ls};
    cuuint32_t box[4] = {kKBlk, 64, 1, 1};
    if (!enc(&h->tm_w[kGU], BF, 4, base + h->off[4] * 2, dims, str, box, SW)) return WAVE_ECUDA;
  }
  {  // Wdown [L][d][F]
    cuuint64_t dims[3] = {F, d, L}, str[2] = {F * 2, ls};
    cuuint32_t box[3] = {kKBlk, kTileM, 1};
    if (!enc(&h->tm_w[kDown], BF, 3, base + h->off[5] * 2, dims, str, box, SW)) return WAVE_ECUDA;
  }
  return WAVE_OK;
}

static int encode_act_maps(wave_ctx* h, int S_pad) {
  const wave_config& c = h->cfg;
  const cuuint64_t d = c.d_model, HD = (cuuint64_t)c.n_heads * c.head_dim, F = c.ffn;
  const cuuint64_t R = h->S_pad_max;
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  cuuint32_t box[2] = {kKBlk, (cuuint32_t)S_pad};
  {
    cuuint64_t dims[2] = {d, R}, str[1] = {d * 2};
    if (!enc(&h->tm_x[kQKV], BF, 2, h->xn, dims, str, box, SW)) return WAVE_ECUDA;
    h->tm_x[kGU] = h->tm_x[kQKV];
  }
  {
    cuuint64_t dims[2] = {HD, R}, str[1] = {HD * 2};
    if (!enc(&h->tm_x[kO], BF, 2, h->attn, dims, str, box, SW)) return WAVE_ECUDA;
  }
  if (F) {
    cuuint64_t dims[2] = {F, R}, str[1] = {F * 2};
    if (!enc(&h->tm_x[kDown], BF, 2, h->u, dims, str, box, SW)) return WAVE_ECUDA;
  }
  if (h->hybrid) {
    h->tm_x[kIn] = h->tm_x[kQKV];
    const cuuint64_t di = (cuuint64_t)h->hcfg.ssm_heads * h->hcfg.ssm_head_dim;
    cuuint64_t dims[2] = {di, R}, str[1] = {di * 2};
    if (!enc(&h->tm_x[kOut], BF, 2, h->ssm_out, dims, str, box, SW)) return WAVE_ECUDA;
  }
  return WAVE_OK;
}

static int encode_kv_map(wave_ctx* h, uint8_t* kv, float* scales) {
  const wave_config& c = h->cfg;
  const cuuint64_t D = c.head_dim, L = c.n_layers;
  const cuuint64_t n1 = (cuuint64_t)h->S_max * c.n_heads * h->T_max;  // slots of one (layer, K|V)
  {
    cuuint64_t dims[4] = {D, n1, 2, L}, str[3] = {D, n1 * D, 2 * n1 * D};
    cuuint32_t box[4] = {(cuuint32_t)D, (cuuint32_t)kChunk, 2, 1};
    const auto SW = (D == 128) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (!enc(&h->tm_kv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, kv, dims, str, box, SW)) return WAVE_ECUDA;
  }
  {
    cuuint64_t dims[3] = {n1, 2, L}, str[2] = {n1 * 4, 2 * n1 * 4};
    cuuint32_t box[3] = {(cuuint32_t)kChunk, 2, 1};
    if (!enc(&h->tm_sc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, scales, dims, str, box,
             CU_TENSOR_MAP_SWIZZLE_NONE))
      return WAVE_ECUDA;
  }
  return WAVE_OK;
}

// One launch of `frames` frames (positions + f in frame f); positions are
// advanced by `frames` on the device at the end when `advance` is set.
static int launch_frames(wave_t* h, int S, int frames, const void* weights, uint8_t* kv_fp8,
                         float* kv_scales, const int32_t* positions, int32_t* advance, const void* x,
                         void* y, void* stream, uint16_t* x_chain = nullptr, float* ssm_state = nullptr) {
  if (!h || !weights || !kv_fp8 || !kv_scales || !positions || !x || !y) return WAVE_EINVAL;
  if (S < 1 || S > h->S_max || frames < 1 || frames > kMaxFrames) return WAVE_EINVAL;
  if (((uintptr_t)weights & 15) || ((uintptr_t)kv_fp8 & 15) || ((uintptr_t)kv_scales & 15) ||
      ((uintptr_t)positions & 3) || ((uintptr_t)x & 15) || ((uintptr_t)y & 15))
    return WAVE_EINVAL;
  cudaStream_t st = (cudaStream_t)stream;
  const int S_pad = (S + 15) / 16 * 16;
  if (weights != h->maps_weights) {
    int rc = encode_weight_maps(h, weights);
    if (rc) return rc;
    h->maps_weights = weights;
  }
  if (kv_fp8 != h->maps_kv || kv_scales != h->maps_sc) {
    int rc = encode_kv_map(h, kv_fp8, kv_scales);
    if (rc) return rc;
    h->maps_kv = kv_fp8;
    h->maps_sc = kv_scales;
  }
  if (S_pad != h->maps_S) {
    int rc = encode_act_maps(h, S_pad);
    if (rc) return rc;
    h->maps_S = S_pad;
  }
  StepParams p;
  memset(&p, 0, sizeof(p));
  for (int k = 0; k < kGemmKinds; ++k) {
    p.tm_w[k] = h->tm_w[k];
    p.tm_x[k] = h->tm_x[k];
    p.tiles[k] = h->tiles[k];
    p.kblocks[k] = h->kblocks[k];
  }
  p.tm_kv = h->tm_kv;
  p.tm_sc = h->tm_sc;
  const wave_config& c = h->cfg;
  p.L = c.n_layers;
  p.d = c.d_model;
  p.H = c.n_heads;
  p.D = c.head_dim;
  p.F = c.ffn;
  p.HD = c.n_heads * c.head_dim;
  p.S = S;
  p.S_pad = S_pad;
  p.S_max = h->S_max;
  p.T_max = h->T_max;
  p.eps = c.rms_eps;
  const int stride = gemm_stage_bytes(S_pad);
  int nst = smem_layout().gemm_ring_bytes / stride;
  p.nstage = nst > kMaxStages ? kMaxStages : nst;
  p.max_tiles_per_cta = h->max_tiles_per_cta;
  p.layer_elems = h->layer_elems;
  p.off_g_attn = h->off[0];
  p.off_g_mlp = h->off[3];
  p.off_wo = h->off[2];
  p.off_wdown = h->off[5];
  p.weights = (const uint16_t*)weights;
  p.kv = kv_fp8;
  p.kv_scales = kv_scales;
  p.pos = positions;
  p.x = (const uint16_t*)x;
  p.y = (uint16_t*)y;
  p.n_frames = frames;
  p.pos_advance = advance;
  p.depth = x_chain ? 1 : 0;
  p.merge = needs_merge(h->T_max) ? 1 : 0;
  if (h->hybrid) {
    const wave_hybrid_config& hc = h->hcfg;
    p.hybrid = 1;
    p.L = hc.n_layers;  // the layer loop; cfg.n_layers counts the attention layers
    p.attn_every = hc.attn_every;
    p.ssm_heads = hc.ssm_heads;
    p.d_inner = hc.ssm_heads * hc.ssm_head_dim;
    p.in_rows = 2 * p.d_inner + 2 * hc.ssm_state + hc.ssm_heads;
    p.hyb_M = h->hyb_M;
    p.hyb_G = h->hyb_G;
    p.hyb_off_w_in = h->hyb_off_w_in;
    p.hyb_off_a_log = h->hyb_off_a_log;
    p.zx = h->zx;
    p.ssm_out = h->ssm_out;
    p.ssm_state = ssm_state;
    // the output projection's L2 prefetch walks attention blocks: one per group
    p.layer_elems = h->hyb_G;
    p.off_wo = (hc.attn_every - 1) * h->hyb_M + h->hyb_off_wo;
    p.off_g_attn = 0;
  }
  p.x_chain = x_chain;
  p.resid = h->resid;
  p.xn = h->xn;
  p.qkv = h->qkv;
  p.attn = h->attn;
  p.u = h->u;
  p.gemm_part = h->gemm_part;
  p.tile_cnt = h->tile_cnt;
  p.att_ctr = h->tile_cnt + 2048;
  p.att_part = h->att_part;
  p.sh_info = h->sh_info;
  p.pieces = h->pieces;
  p.n_pieces = h->n_pieces;
  p.rope = h->rope;
  p.bar = h->bar;
  p.err = h->err;
  p.timeout_ns = h->timeout_ns;
  p.skip_cta = h->skip_cta;
  p.skip_bar = h->skip_bar;
  if (frames == 1) {  // the profiling and testing hooks are sized for one frame
    p.kv_dump = h->kv_dump;
    p.phase_ts = h->phase_ts;
    p.arrive_ts = h->arrive_ts;
  }
  if (cudaMemsetAsync(h->bar, 0, 4, st) != cudaSuccess) return WAVE_ECUDA;
  cudaError_t e = launch_step(p, h->grid, st);
  h->last_stream = st;
  if (e == cudaErrorCooperativeLaunchTooLarge) return WAVE_ELAUNCH;
  if (e != cudaSuccess) return WAVE_ECUDA;
  return WAVE_OK;
}

extern "C" int wave_step(wave_t* h, int S, const void* weights, uint8_t* kv_fp8, float* kv_scales,
                         const int32_t* positions, const void* x, void* y, void* stream) {
  if (h && h->hybrid) return WAVE_EINVAL;
  return launch_frames(h, S, 1, weights, kv_fp8, kv_scales, positions, nullptr, x, y, stream);
}

extern "C" int wave_depth(wave_t* h, int S, int steps, const void* weights, const void* w_proj,
                          uint8_t* kv_fp8, float* kv_scales, const void* x0, void* xs, void* y,
                          void* stream) {
  if (!h || h->hybrid || !w_proj || !x0 || !xs || !y) return WAVE_EINVAL;
  if (S < 1 || S > h->S_max || steps < 1 || steps > kMaxFrames || steps > h->T_max) return WAVE_EINVAL;
  if (((uintptr_t)w_proj & 15) || ((uintptr_t)x0 & 15) || ((uintptr_t)xs & 15) || ((uintptr_t)y & 15))
    return WAVE_EINVAL;
  const wave_config& c = h->cfg;
  const cuuint64_t d = c.d_model;
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  if (w_proj != h->maps_wp) {  // W_p [d][d] as a one-layer stack
    cuuint64_t dims[3] = {d, d, 1}, str[2] = {d * 2, d * d * 2};
    cuuint32_t box[3] = {kKBlk, kTileM, 1};
    if (!enc(&h->tm_w[kProj], BF, 3, (void*)w_proj, dims, str, box, SW)) return WAVE_ECUDA;
    h->maps_wp = w_proj;
  }
  {  // the outputs y [steps * S][d], read back S_pad rows at a time
    const int S_pad = (S + 15) / 16 * 16;
    cuuint64_t dims[2] = {d, (cuuint64_t)steps * S}, str[1] = {d * 2};
    cuuint32_t box[2] = {kKBlk, (cuuint32_t)S_pad};
    if (!enc(&h->tm_x[kProj], BF, 2, y, dims, str, box, SW)) return WAVE_ECUDA;
  }
  cudaStream_t st = (cudaStream_t)stream;
  if (xs != x0 && cudaMemcpyAsync(xs, x0, (size_t)S * d * 2, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return WAVE_ECUDA;
  return launch_frames(h, S, steps, weights, kv_fp8, kv_scales, h->zero_pos, nullptr, xs, y, stream,
                       (uint16_t*)xs);
}

extern "C" int wave_hybrid_step(wave_t* h, int S, const void* weights, uint8_t* kv_fp8, float* kv_scales,
                                float* ssm_state, const int32_t* positions, const void* x, void* y,
                                void* stream) {
  if (!h || !h->hybrid || !ssm_state || ((uintptr_t)ssm_state & 15)) return WAVE_EINVAL;
  return launch_frames(h, S, 1, weights, kv_fp8, kv_scales, positions, nullptr, x, y, stream, nullptr,
                       ssm_state);
}

extern "C" int wave_beat(wave_t* h, int S, int frames, const void* weights, uint8_t* kv_fp8,
                         float* kv_scales, int32_t* positions, int advance, const void* x, void* y,
                         void* stream) {
  if (h && h->hybrid) return WAVE_EINVAL;
  return launch_frames(h, S, frames, weights, kv_fp8, kv_scales, positions, advance ? positions : nullptr,
                       x, y, stream);
}

extern "C" int wave_status(wave_t* h) {
  if (!h) return WAVE_EINVAL;
  if (cudaStreamSynchronize(h->last_stream) != cudaSuccess) return WAVE_ECUDA;
  int e = 0;
  if (cudaMemcpy(&e, h->err, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return WAVE_ECUDA;
  if (e == 0) return WAVE_OK;
  if (cudaMemset(h->err, 0, 4) != cudaSuccess) return WAVE_ECUDA;
  if (e & kErrTimeout) return WAVE_ETIMEOUT;
  return WAVE_EPOS;
}

extern "C" int wave_set_timeout_ns(wave_t* h, long long ns) {
  if (!h || ns <= 0) return WAVE_EINVAL;
  h->timeout_ns = ns;
  return WAVE_OK;
}

extern "C" int wave_debug_skip_barrier(wave_t* h, int cta, int barrier) {
  if (!h) return WAVE_EINVAL;
  h->skip_cta = cta;
  h->skip_bar = barrier;
  return WAVE_OK;
}

extern "C" int wave_debug_dump_kv(wave_t* h, float* dst) {
  if (!h) return WAVE_EINVAL;
  h->kv_dump = dst;
  return WAVE_OK;
}

extern "C" int wave_debug_phase_times(wave_t* h, long long* dst) {
  if (!h) return WAVE_EINVAL;
  h->phase_ts = dst;
  return WAVE_OK;
}

extern "C" int wave_debug_arrival_times(wave_t* h, long long* dst) {
  if (!h) return WAVE_EINVAL;
  h->arrive_ts = dst;
  return WAVE_OK;
}

extern "C" int wave_grid_size(wave_t* h) { return h ? h->grid : WAVE_EINVAL; }

extern "C" int wave_barriers_per_step(wave_t* h) {
  if (!h) return WAVE_EINVAL;
  return h->hybrid ? hybrid_barriers_per_step(h->hcfg.n_layers, h->hcfg.attn_every, h->T_max)
                   : barriers_per_step(h->cfg.n_layers, h->T_max);
}
