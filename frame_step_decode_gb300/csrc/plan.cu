// plan.cu -- host-side set-up shared by every entry point of the step
// library (see plan.h).
#include <math.h>
#include <string.h>

#include "plan.h"

namespace wave {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

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

static bool enc(CUtensorMap* m, CUtensorMapDataType dt, int rank, void* base, const cuuint64_t* dims,
                const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  EncodeTiledFn fn = encode_fn();
  return fn && fn(m, dt, (cuuint32_t)rank, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool decoder_shape_ok(const wave_config* c) {
  if (!c) return false;
  if (c->n_layers < 1 || c->n_layers > 1024) return false;
  if (c->head_dim != 64 && c->head_dim != 128) return false;
  if (c->n_heads < 1 || c->d_model < 64 || c->d_model % 64 || c->d_model > 8192) return false;
  if ((c->n_heads * c->head_dim) % 64) return false;
  if (c->ffn < 8 || c->ffn % 8) return false;
  if (!(c->rms_eps >= 0.f) || !(c->rope_base > 0.f)) return false;
  return true;
}

bool hybrid_shape_ok(const wave_hybrid_config* c) {
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

void decoder_layout(const wave_config* c, long long* off, long long* layer_elems) {
  const long long d = c->d_model, HD = (long long)c->n_heads * c->head_dim, F = c->ffn;
  const long long n[6] = {d, 3 * HD * d, d * HD, d, 2 * F * d, d * F};
  long long o = 0;
  for (int i = 0; i < 6; ++i) {
    off[i] = o;
    o += n[i];
  }
  *layer_elems = o;
}

void hybrid_layout(const wave_hybrid_config* c, long long* M, long long* A, long long* w_in, long long* w_out,
                   long long* a_log, long long* wqkv, long long* wo) {
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

int device_check(int* dev, int* sms) {
  if (cudaGetDevice(dev) != cudaSuccess) return WAVE_ECUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev) != cudaSuccess ||
      cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess)
    return WAVE_ECUDA;
  if (major != 10 || minor != 3) return WAVE_EDEVICE;
  if (!encode_fn()) return WAVE_ECUDA;
  if (configure_step_kernel() != cudaSuccess) return WAVE_ECUDA;
  int per_sm = 0;
  if (occupancy_per_sm(&per_sm) != cudaSuccess || per_sm < 1) return WAVE_ELAUNCH;
  return WAVE_OK;
}

bool capacity_ok(int S_max, int T_max, long long history_rows) {
  if (S_max < 1 || S_max > 128 || T_max < 4 || T_max % 4) return false;
  if (history_rows >= (1LL << 31) || T_max > 65535 * kChunk) return false;
  return true;
}

// Stream-K split of tiles x kb units over the grid: the most tiles one CTA
// touches, and the most segments (CTAs) one tile is split into.
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

static int plan_gemms(Plan* pl) {
  const wave_config* cfg = &pl->cfg;
  const int d = cfg->d_model, HD = cfg->n_heads * cfg->head_dim, F = cfg->ffn;
  pl->tiles[kQKV] = (3 * HD + kTileM - 1) / kTileM;
  pl->kblocks[kQKV] = (d + kKUnit - 1) / kKUnit;
  pl->tiles[kO] = (d + kTileM - 1) / kTileM;
  pl->kblocks[kO] = (HD + kKUnit - 1) / kKUnit;
  pl->tiles[kGU] = (F + 63) / 64;
  pl->kblocks[kGU] = (d + kKUnit - 1) / kKUnit;
  pl->tiles[kDown] = F ? (d + kTileM - 1) / kTileM : 0;
  pl->kblocks[kDown] = (F + kKUnit - 1) / kKUnit;
  pl->tiles[kProj] = pl->hybrid ? 0 : (d + kTileM - 1) / kTileM;
  pl->kblocks[kProj] = (d + kKUnit - 1) / kKUnit;
  pl->tiles[kIn] = (pl->in_rows + kTileM - 1) / kTileM;
  pl->kblocks[kIn] = (d + kKUnit - 1) / kKUnit;
  pl->tiles[kOut] = pl->d_inner ? (d + kTileM - 1) / kTileM : 0;
  pl->kblocks[kOut] = (pl->d_inner + kKUnit - 1) / kKUnit;
  int mt = 1;
  for (int k = 0; k < kGemmKinds; ++k) {
    if (pl->tiles[k] > 1024) return WAVE_EINVAL;
    const int m = max_tiles_touched(pl->tiles[k], pl->kblocks[k], pl->grid, gemm_seg_cap(k));
    if (m > mt) mt = m;
    if (max_segments(pl->tiles[k], pl->kblocks[k], pl->grid, gemm_seg_cap(k)) > 64) return WAVE_EINVAL;
  }
  pl->max_tiles_per_cta = mt;
  return WAVE_OK;
}

// The packed layout: per decoder layer [g_attn][Wqkv][Wo][g_mlp][Wgu][Wdown],
// per hybrid group (attn_every - 1) selective-state blocks [g][W_in][W_out]
// [A_log, dt_bias, D padded to 8] then one attention block [g][Wqkv][Wo];
// every matrix as packed_matrix_elems of its projection's tiles and units.
static void plan_packed(Plan* pl) {
  const long long d = pl->cfg.d_model;
  auto mat = [&](int kind) { return packed_matrix_elems(pl->tiles[kind], pl->kblocks[kind]); };
  if (!pl->hybrid) {
    const long long n[6] = {d, mat(kQKV), mat(kO), d, mat(kGU), mat(kDown)};
    long long o = 0;
    for (int i = 0; i < 6; ++i) {
      pl->pk_off[i] = o;
      o += n[i];
    }
    pl->pk_layer = o;
    pl->pk_total = o * pl->cfg.n_layers;
  } else {
    const wave_hybrid_config& hc = pl->hcfg;
    pl->pk_w_in = d;
    pl->pk_w_out = d + mat(kIn);
    pl->pk_a_log = pl->pk_w_out + (pl->d_inner ? mat(kOut) : 0);
    pl->pk_M = pl->pk_a_log + (3LL * hc.ssm_heads + 7) / 8 * 8;
    pl->pk_wqkv = d;
    pl->pk_wo = d + mat(kQKV);
    pl->pk_A = pl->pk_wo + mat(kO);
    pl->pk_layer = (hc.attn_every - 1) * pl->pk_M + pl->pk_A;
    pl->pk_total = pl->pk_layer * (hc.n_layers / hc.attn_every);
  }
}

int plan_decoder(Plan* pl, const wave_config* cfg, int S_max, int T_max, int grid) {
  if (!decoder_shape_ok(cfg)) return WAVE_EINVAL;
  const long long rows = (long long)cfg->n_layers * 2 * S_max * cfg->n_heads * T_max;
  if (!capacity_ok(S_max, T_max, rows)) return WAVE_EINVAL;
  *pl = Plan();
  pl->cfg = *cfg;
  pl->S_max = S_max;
  pl->S_pad_max = (S_max + 15) / 16 * 16;
  pl->T_max = T_max;
  pl->grid = grid;
  decoder_layout(cfg, pl->off, &pl->layer_elems);
  const int rc = plan_gemms(pl);
  plan_packed(pl);
  return rc;
}

int plan_hybrid(Plan* pl, const wave_hybrid_config* hc, int S_max, int T_max, int grid) {
  if (!hybrid_shape_ok(hc)) return WAVE_EINVAL;
  const int La = hc->n_layers / hc->attn_every;
  const long long rows = (long long)La * 2 * S_max * hc->n_heads * T_max;
  if (!capacity_ok(S_max, T_max, rows)) return WAVE_EINVAL;
  *pl = Plan();
  pl->hybrid = 1;
  pl->hcfg = *hc;
  // cfg describes the attention layers (their history and maps)
  pl->cfg.n_layers = La;
  pl->cfg.d_model = hc->d_model;
  pl->cfg.n_heads = hc->n_heads;
  pl->cfg.head_dim = hc->head_dim;
  pl->cfg.ffn = 0;
  pl->cfg.rms_eps = hc->rms_eps;
  pl->cfg.rope_base = hc->rope_base;
  pl->S_max = S_max;
  pl->S_pad_max = (S_max + 15) / 16 * 16;
  pl->T_max = T_max;
  pl->grid = grid;
  long long A;
  hybrid_layout(hc, &pl->hyb_M, &A, &pl->hyb_off_w_in, &pl->hyb_off_w_out, &pl->hyb_off_a_log, &pl->hyb_off_wqkv,
                &pl->hyb_off_wo);
  pl->hyb_G = (hc->attn_every - 1) * pl->hyb_M + A;
  pl->layer_elems = pl->hyb_G;
  pl->d_inner = hc->ssm_heads * hc->ssm_head_dim;
  pl->in_rows = 2 * pl->d_inner + 2 * hc->ssm_state + hc->ssm_heads;
  const int rc = plan_gemms(pl);
  plan_packed(pl);
  return rc;
}

size_t carve_workspace(const Plan& pl, char* base, Workspace* ws) {
  const wave_config& c = pl.cfg;
  const long long SP = pl.S_pad_max, d = c.d_model, HD = (long long)c.n_heads * c.head_dim, F = c.ffn;
  const long long H = c.n_heads, D = c.head_dim;
  const long long max_pieces =
      (long long)pl.S_max * H * (((pl.T_max + kChunk - 1) / kChunk + kPieceChunks - 1) / kPieceChunks);
  struct Part {
    void** dst;
    size_t bytes;
  };
  Workspace w;
  const Part parts[] = {
      {(void**)&w.resid, (size_t)(SP * d * 4)},
      {(void**)&w.xn, (size_t)(SP * d * 2)},
      {(void**)&w.qkv, (size_t)(SP * 3 * HD * 4)},
      {(void**)&w.attn, (size_t)(SP * HD * 2)},
      {(void**)&w.u, (size_t)(SP * F * 2)},
      {(void**)&w.gemm_part, 2 * (size_t)pl.grid * pl.max_tiles_per_cta * SP * kTileM * 4},
      {(void**)&w.tile_cnt, kCounterWords * 4},
      {(void**)&w.att_part, (size_t)(max_pieces * (D + 4) * 4)},
      {(void**)&w.sh_info, (size_t)(pl.S_max * H * 8)},
      {(void**)&w.pieces, (size_t)(max_pieces * 32)},
      {(void**)&w.n_pieces, 16},
      {(void**)&w.sh_cnt, (size_t)pl.S_max * H * 4},
      {(void**)&w.rope, (size_t)pl.T_max * (D / 2) * 8},
      {(void**)&w.bar, 16},
      {(void**)&w.err, 16},
      {(void**)&w.zero_pos, (size_t)pl.S_max * 4},
      {(void**)&w.zx, (size_t)(SP * pl.in_rows * 4)},
      {(void**)&w.ssm_out, (size_t)(SP * pl.d_inner * 2)},
  };
  size_t o = 0;
  for (const Part& pt : parts) {
    if (base) *pt.dst = base + o;
    o += (pt.bytes + 255) & ~(size_t)255;
  }
  if (base && ws) *ws = w;
  return o;
}

void rope_table(const Plan& pl, std::vector<float2>* tab) {
  const int D = pl.cfg.head_dim, T = pl.T_max;
  tab->resize((size_t)T * (D / 2));
  for (int t = 0; t < T; ++t)
    for (int i = 0; i < D / 2; ++i) {
      const double th = pow((double)pl.cfg.rope_base, -2.0 * i / (double)D);
      const double a = (double)t * th;
      (*tab)[(size_t)t * (D / 2) + i] = make_float2((float)cos(a), (float)sin(a));
    }
}

// A packed projection matrix as a tensor of 128-byte rows (64 bf16): a
// 128-row box is one contiguous 16 KB block, unit (t, kb) the two blocks at
// rows ((t * kunits + kb) * 2 + bx) * 128.  Outer dims: layers (decoder) or
// place-in-group and group (hybrid).
static bool enc_packed(CUtensorMap* m, const char* base, int tiles, int kunits, int rank, const cuuint64_t* outer,
                       const cuuint64_t* outer_stride_bytes) {
  cuuint64_t dims[4] = {64, (cuuint64_t)tiles * kunits * 2 * 128, 1, 1}, str[3] = {128, 0, 0};
  cuuint32_t box[4] = {64, 128, 1, 1};
  for (int i = 0; i < rank - 2; ++i) {
    dims[2 + i] = outer[i];
    str[1 + i] = outer_stride_bytes[i];
  }
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, (void*)base, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

static int encode_hybrid_weight_maps(const Plan& pl, const void* weights, Maps* m) {
  const wave_hybrid_config& c = pl.hcfg;
  const cuuint64_t e = c.attn_every, groups = c.n_layers / c.attn_every;
  const cuuint64_t M2 = (cuuint64_t)pl.pk_M * 2, G2 = (cuuint64_t)pl.pk_layer * 2;
  const char* base = (const char*)weights;
  const char* attn0 = base + (e - 1) * M2;  // the first attention block
  {  // attention Wqkv and Wo, one attention block per group
    const cuuint64_t outer[1] = {groups}, ostr[1] = {G2};
    if (!enc_packed(&m->tm_w[kQKV], attn0 + pl.pk_wqkv * 2, pl.tiles[kQKV], pl.kblocks[kQKV], 3, outer, ostr))
      return WAVE_ECUDA;
    if (!enc_packed(&m->tm_w[kO], attn0 + pl.pk_wo * 2, pl.tiles[kO], pl.kblocks[kO], 3, outer, ostr))
      return WAVE_ECUDA;
  }
  if (e > 1) {  // W_in and W_out [group][place]
    const cuuint64_t outer[2] = {e - 1, groups}, ostr[2] = {M2, G2};
    if (!enc_packed(&m->tm_w[kIn], base + pl.pk_w_in * 2, pl.tiles[kIn], pl.kblocks[kIn], 4, outer, ostr))
      return WAVE_ECUDA;
    if (!enc_packed(&m->tm_w[kOut], base + pl.pk_w_out * 2, pl.tiles[kOut], pl.kblocks[kOut], 4, outer, ostr))
      return WAVE_ECUDA;
  }
  return WAVE_OK;
}

int encode_weight_maps(const Plan& pl, const void* weights, Maps* m) {
  if (pl.hybrid) return encode_hybrid_weight_maps(pl, weights, m);
  const char* base = (const char*)weights;
  const cuuint64_t outer[1] = {(cuuint64_t)pl.cfg.n_layers}, ostr[1] = {(cuuint64_t)pl.pk_layer * 2};
  const int kinds[4] = {kQKV, kO, kGU, kDown}, which[4] = {1, 2, 4, 5};
  for (int i = 0; i < 4; ++i)
    if (!enc_packed(&m->tm_w[kinds[i]], base + pl.pk_off[which[i]] * 2, pl.tiles[kinds[i]], pl.kblocks[kinds[i]],
                    3, outer, ostr))
      return WAVE_ECUDA;
  return WAVE_OK;
}

int encode_act_maps(const Plan& pl, const Workspace& ws, int S_pad, Maps* m) {
  const wave_config& c = pl.cfg;
  const cuuint64_t d = c.d_model, HD = (cuuint64_t)c.n_heads * c.head_dim, F = c.ffn;
  const cuuint64_t R = pl.S_pad_max;
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  cuuint32_t box[2] = {kKBlk, (cuuint32_t)S_pad};
  {
    cuuint64_t dims[2] = {d, R}, str[1] = {d * 2};
    if (!enc(&m->tm_x[kQKV], BF, 2, ws.xn, dims, str, box, SW)) return WAVE_ECUDA;
    m->tm_x[kGU] = m->tm_x[kQKV];
  }
  {
    cuuint64_t dims[2] = {HD, R}, str[1] = {HD * 2};
    if (!enc(&m->tm_x[kO], BF, 2, ws.attn, dims, str, box, SW)) return WAVE_ECUDA;
  }
  if (F) {
    cuuint64_t dims[2] = {F, R}, str[1] = {F * 2};
    if (!enc(&m->tm_x[kDown], BF, 2, ws.u, dims, str, box, SW)) return WAVE_ECUDA;
  }
  if (pl.hybrid) {
    m->tm_x[kIn] = m->tm_x[kQKV];
    const cuuint64_t di = (cuuint64_t)pl.d_inner;
    cuuint64_t dims[2] = {di, R}, str[1] = {di * 2};
    if (!enc(&m->tm_x[kOut], BF, 2, ws.ssm_out, dims, str, box, SW)) return WAVE_ECUDA;
  }
  return WAVE_OK;
}

int encode_kv_maps(const Plan& pl, uint8_t* kv, float* scales, Maps* m) {
  const wave_config& c = pl.cfg;
  const cuuint64_t D = c.head_dim, L = c.n_layers;
  const cuuint64_t n1 = (cuuint64_t)pl.S_max * c.n_heads * pl.T_max;  // slots of one (layer, K|V)
  {
    cuuint64_t dims[4] = {D, n1, 2, L}, str[3] = {D, n1 * D, 2 * n1 * D};
    cuuint32_t box[4] = {(cuuint32_t)D, (cuuint32_t)kChunk, 2, 1};
    const auto SW = (D == 128) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (!enc(&m->tm_kv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, kv, dims, str, box, SW)) return WAVE_ECUDA;
  }
  {
    cuuint64_t dims[3] = {n1, 2, L}, str[2] = {n1 * 4, 2 * n1 * 4};
    cuuint32_t box[3] = {(cuuint32_t)(kChunk * kScaleGroup), 2, 1};  // a group of chunks, K and V planes
    if (!enc(&m->tm_sc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, scales, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE))
      return WAVE_ECUDA;
  }
  return WAVE_OK;
}

int encode_proj_maps(const Plan& pl, const void* w_proj, void* y, int S, int steps, Maps* m) {
  const cuuint64_t d = pl.cfg.d_model;
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  {
    cuuint64_t dims[3] = {d, d, 1}, str[2] = {d * 2, d * d * 2};
    cuuint32_t box[3] = {kKBlk, kTileM, 1};
    if (!enc(&m->tm_w[kProj], BF, 3, (void*)w_proj, dims, str, box, SW)) return WAVE_ECUDA;
  }
  {
    const int S_pad = (S + 15) / 16 * 16;
    cuuint64_t dims[2] = {d, (cuuint64_t)steps * S}, str[1] = {d * 2};
    cuuint32_t box[2] = {kKBlk, (cuuint32_t)S_pad};
    if (!enc(&m->tm_x[kProj], BF, 2, y, dims, str, box, SW)) return WAVE_ECUDA;
  }
  return WAVE_OK;
}

static void act_sections(const Plan& pl, int* n1, int* n2) {
  const int HD = pl.cfg.n_heads * pl.cfg.head_dim;
  *n1 = 3 * HD > pl.in_rows ? 3 * HD : pl.in_rows;
  *n2 = HD > pl.d_inner ? HD : pl.d_inner;
}

long long act_record_floats(const Plan& pl) {
  int n1, n2;
  act_sections(pl, &n1, &n2);
  return 5LL * pl.cfg.d_model + n1 + n2 + pl.cfg.ffn;
}

bool launch_args_ok(const Plan& pl, int S, int frames, const void* weights, const void* kv, const void* kv_scales,
                    const void* positions, const void* x, const void* y) {
  if (!weights || !kv || !kv_scales || !positions || !x || !y) return false;
  if (S < 1 || S > pl.S_max || frames < 1 || frames > kMaxFrames) return false;
  if (((uintptr_t)weights & 15) || ((uintptr_t)kv & 15) || ((uintptr_t)kv_scales & 15) ||
      ((uintptr_t)positions & 3) || ((uintptr_t)x & 15) || ((uintptr_t)y & 15))
    return false;
  return true;
}

void fill_params(StepParams* p, const Plan& pl, const Workspace& ws, const Maps& m, int S, const void* weights,
                 uint8_t* kv, float* kv_scales, const int32_t* positions, const void* x, void* y, int frames) {
  memset(p, 0, sizeof(*p));
  for (int k = 0; k < kGemmKinds; ++k) {
    p->tm_w[k] = m.tm_w[k];
    p->tm_x[k] = m.tm_x[k];
    p->tiles[k] = pl.tiles[k];
    p->kblocks[k] = pl.kblocks[k];
  }
  p->tm_kv = m.tm_kv;
  p->tm_sc = m.tm_sc;
  const wave_config& c = pl.cfg;
  const int S_pad = (S + 15) / 16 * 16;
  p->L = c.n_layers;
  p->d = c.d_model;
  p->H = c.n_heads;
  p->D = c.head_dim;
  p->F = c.ffn;
  p->HD = c.n_heads * c.head_dim;
  p->S = S;
  p->S_pad = S_pad;
  p->S_max = pl.S_max;
  p->T_max = pl.T_max;
  p->eps = c.rms_eps;
  const int nst = smem_layout().gemm_ring_bytes / gemm_stage_bytes(S_pad);
  p->nstage = nst > kMaxStages ? kMaxStages : nst;
  p->max_tiles_per_cta = pl.max_tiles_per_cta;
  p->layer_elems = pl.pk_layer;
  p->off_g_attn = pl.pk_off[0];
  p->off_g_mlp = pl.pk_off[3];
  p->weights = (const uint16_t*)weights;
  p->kv = kv;
  p->kv_scales = kv_scales;
  p->pos = positions;
  p->x = (const uint16_t*)x;
  p->y = (uint16_t*)y;
  p->n_frames = frames;
  if (pl.hybrid) {
    const wave_hybrid_config& hc = pl.hcfg;
    p->hybrid = 1;
    p->L = hc.n_layers;  // the layer loop; cfg.n_layers counts the attention layers
    p->attn_every = hc.attn_every;
    p->ssm_heads = hc.ssm_heads;
    p->d_inner = pl.d_inner;
    p->in_rows = pl.in_rows;
    p->hyb_M = pl.pk_M;
    p->hyb_G = pl.pk_layer;
    p->hyb_off_a_log = pl.pk_a_log;
    p->zx = ws.zx;
    p->ssm_out = ws.ssm_out;
    p->layer_elems = pl.pk_layer;
    p->off_g_attn = 0;
  }
  p->resid = ws.resid;
  p->xn = ws.xn;
  p->qkv = ws.qkv;
  p->attn = ws.attn;
  p->u = ws.u;
  p->gemm_part = ws.gemm_part;
  p->part_bank = (long long)pl.grid * pl.max_tiles_per_cta * pl.S_pad_max * kTileM;
  p->tile_cnt = ws.tile_cnt;
  p->done_cnt = ws.tile_cnt + kDoneCntOff;
  p->qkv_done = ws.tile_cnt + kQkvDoneOff;
  p->head_cnt = ws.tile_cnt + kHeadCntOff;
  p->sh_cnt = ws.sh_cnt;
  p->att_ctr = ws.tile_cnt + kAttCtrOff;
  p->att_part = ws.att_part;
  p->sh_info = ws.sh_info;
  p->pieces = ws.pieces;
  p->n_pieces = ws.n_pieces;
  p->rope = ws.rope;
  p->bar = ws.bar;
  p->err = ws.err;
  p->timeout_ns = 2000000000LL;
  p->skip_cta = -1;
  p->skip_bar = -1;
  p->skip_sig = -1;
  p->skip_sig_kind = -1;
  act_sections(pl, &p->act_n1, &p->act_n2);
  p->act_rec = act_record_floats(pl);
}

}  // namespace wave
