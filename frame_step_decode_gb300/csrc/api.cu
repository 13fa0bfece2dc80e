// api.cu -- host side of the C ABI in include/wave.h: argument checks,
// workspace ownership and the single cooperative launch per frame.  The
// plan, carve-up, tensor maps and parameter block come from plan.cu, shared
// with the no-allocation entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <vector>

#include "../../include/wave.h"
#include "internal.h"
#include "plan.h"

using namespace wave;

struct wave_ctx {
  Plan pl;
  int device = 0;
  void* ws_block = nullptr;
  Workspace ws;
  int* err_host = nullptr;      // pinned host word the kernel mirrors the error bits into
  int* err_host_dev = nullptr;  // its device-side address
  // cached tensor maps and what they were encoded for
  Maps maps;
  const void* maps_weights = nullptr;
  const void* maps_kv = nullptr;
  const void* maps_sc = nullptr;
  int maps_S = -1;
  cudaStream_t last_stream = nullptr;
  long long timeout_ns = 2000000000LL;
  int skip_cta = -1, skip_bar = -1, skip_sig = -1, skip_sig_kind = -1;
  float* kv_dump = nullptr;
  float* act_dump = nullptr;
  int act_dump_n = 0;
  long long* phase_ts = nullptr;
  long long* arrive_ts = nullptr;
};

extern "C" size_t wave_weights_bytes(const wave_config* cfg) {
  if (!decoder_shape_ok(cfg)) return 0;
  long long off[6], le;
  decoder_layout(cfg, off, &le);
  return (size_t)(le * cfg->n_layers * 2);
}

extern "C" size_t wave_weight_offset(const wave_config* cfg, int layer, int which) {
  if (!decoder_shape_ok(cfg) || layer < 0 || layer >= cfg->n_layers || which < 0 || which > 5)
    return (size_t)-1;
  long long off[6], le;
  decoder_layout(cfg, off, &le);
  return (size_t)((le * layer + off[which]) * 2);
}

extern "C" size_t wave_packed_weights_bytes(const wave_config* cfg) {
  Plan pl;
  if (plan_decoder(&pl, cfg, 1, 4, 1) != WAVE_OK) return 0;
  return (size_t)pl.pk_total * 2;
}

extern "C" int wave_pack_weights(const wave_config* cfg, const void* src, void* dst, void* stream) {
  Plan pl;
  if (!src || !dst || src == dst || ((uintptr_t)src & 15) || ((uintptr_t)dst & 15) ||
      plan_decoder(&pl, cfg, 1, 4, 1) != WAVE_OK)
    return WAVE_EINVAL;
  return pack_weights(pl, src, dst, (cudaStream_t)stream);
}

extern "C" size_t wave_hybrid_packed_weights_bytes(const wave_hybrid_config* cfg) {
  Plan pl;
  if (plan_hybrid(&pl, cfg, 1, 4, 1) != WAVE_OK) return 0;
  return (size_t)pl.pk_total * 2;
}

extern "C" int wave_hybrid_pack_weights(const wave_hybrid_config* cfg, const void* src, void* dst, void* stream) {
  Plan pl;
  if (!src || !dst || src == dst || ((uintptr_t)src & 15) || ((uintptr_t)dst & 15) ||
      plan_hybrid(&pl, cfg, 1, 4, 1) != WAVE_OK)
    return WAVE_EINVAL;
  return pack_weights(pl, src, dst, (cudaStream_t)stream);
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

static void free_ctx(wave_ctx* h) {
  if (h->ws_block) cudaFree(h->ws_block);
  if (h->err_host) cudaFreeHost(h->err_host);
  delete h;
}

// Workspace, error mirror and RoPE table of a handle whose plan is set.
static int build_ctx(wave_ctx* h) {
  const size_t total = carve_workspace(h->pl, nullptr, nullptr);
  if (cudaMalloc(&h->ws_block, total) != cudaSuccess) {
    h->ws_block = nullptr;
    return WAVE_ENOMEM;
  }
  if (cudaMemset(h->ws_block, 0, total) != cudaSuccess) return WAVE_ECUDA;
  carve_workspace(h->pl, (char*)h->ws_block, &h->ws);
  if (cudaHostAlloc((void**)&h->err_host, 16, cudaHostAllocMapped) != cudaSuccess) {
    h->err_host = nullptr;
    return WAVE_ENOMEM;
  }
  *(volatile int*)h->err_host = 0;
  if (cudaHostGetDevicePointer((void**)&h->err_host_dev, h->err_host, 0) != cudaSuccess) return WAVE_ECUDA;
  std::vector<float2> tab;
  rope_table(h->pl, &tab);
  if (cudaMemcpy(h->ws.rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess)
    return WAVE_ECUDA;
  return WAVE_OK;
}

extern "C" int wave_create(const wave_config* cfg, int S_max, int T_max, wave_t** out) {
  if (!out || !decoder_shape_ok(cfg)) return WAVE_EINVAL;
  int dev = 0, sms = 0;
  Plan pl;
  // shape and capacity first (no device needed), then the device
  if (plan_decoder(&pl, cfg, S_max, T_max, 1) != WAVE_OK) return WAVE_EINVAL;
  int rc = device_check(&dev, &sms);
  if (rc) return rc;
  wave_ctx* h = new wave_ctx();
  h->device = dev;
  rc = plan_decoder(&h->pl, cfg, S_max, T_max, sms);
  if (!rc) rc = build_ctx(h);
  if (rc) {
    free_ctx(h);
    return rc;
  }
  *out = h;
  return WAVE_OK;
}

extern "C" size_t wave_hybrid_weights_bytes(const wave_hybrid_config* cfg) {
  if (!hybrid_shape_ok(cfg)) return 0;
  long long M, A, a, b, c, q, o;
  hybrid_layout(cfg, &M, &A, &a, &b, &c, &q, &o);
  const int e = cfg->attn_every;
  return (size_t)((cfg->n_layers / e) * ((e - 1) * M + A) * 2);
}

extern "C" size_t wave_hybrid_layer_offset(const wave_hybrid_config* cfg, int layer) {
  if (!hybrid_shape_ok(cfg) || layer < 0 || layer > cfg->n_layers) return (size_t)-1;
  long long M, A, a, b, c, q, o;
  hybrid_layout(cfg, &M, &A, &a, &b, &c, &q, &o);
  return (size_t)(hyb_layer_offset(M, (cfg->attn_every - 1) * M + A, cfg->attn_every, layer) * 2);
}

extern "C" int wave_hybrid_create(const wave_hybrid_config* hc, int S_max, int T_max, wave_t** out) {
  if (!out || !hybrid_shape_ok(hc)) return WAVE_EINVAL;
  int dev = 0, sms = 0;
  Plan pl;
  if (plan_hybrid(&pl, hc, S_max, T_max, 1) != WAVE_OK) return WAVE_EINVAL;
  int rc = device_check(&dev, &sms);
  if (rc) return rc;
  wave_ctx* h = new wave_ctx();
  h->device = dev;
  rc = plan_hybrid(&h->pl, hc, S_max, T_max, sms);
  if (!rc) rc = build_ctx(h);
  if (rc) {
    free_ctx(h);
    return rc;
  }
  *out = h;
  return WAVE_OK;
}

extern "C" void wave_destroy(wave_t* h) {
  if (!h) return;
  cudaDeviceSynchronize();
  free_ctx(h);
}

// One launch of `frames` frames (positions + f in frame f); positions are
// advanced by `frames` on the device at the end when `advance` is set.
static int launch_frames(wave_t* h, int S, int frames, const void* weights, uint8_t* kv_fp8,
                         float* kv_scales, const int32_t* positions, int32_t* advance, const void* x,
                         void* y, void* stream, uint16_t* x_chain = nullptr, float* ssm_state = nullptr) {
  if (!h || !launch_args_ok(h->pl, S, frames, weights, kv_fp8, kv_scales, positions, x, y)) return WAVE_EINVAL;
  cudaStream_t st = (cudaStream_t)stream;
  const int S_pad = (S + 15) / 16 * 16;
  if (weights != h->maps_weights) {
    int rc = encode_weight_maps(h->pl, weights, &h->maps);
    if (rc) return rc;
    h->maps_weights = weights;
  }
  if (kv_fp8 != h->maps_kv || kv_scales != h->maps_sc) {
    int rc = encode_kv_maps(h->pl, kv_fp8, kv_scales, &h->maps);
    if (rc) return rc;
    h->maps_kv = kv_fp8;
    h->maps_sc = kv_scales;
  }
  if (S_pad != h->maps_S) {
    int rc = encode_act_maps(h->pl, h->ws, S_pad, &h->maps);
    if (rc) return rc;
    h->maps_S = S_pad;
  }
  StepParams p;
  fill_params(&p, h->pl, h->ws, h->maps, S, weights, kv_fp8, kv_scales, positions, x, y, frames);
  p.pos_advance = advance;
  p.depth = x_chain ? 1 : 0;
  p.x_chain = x_chain;
  p.ssm_state = ssm_state;
  p.err_out = h->err_host_dev;
  p.timeout_ns = h->timeout_ns;
  p.skip_cta = h->skip_cta;
  p.skip_bar = h->skip_bar;
  p.skip_sig = h->skip_sig;
  p.skip_sig_kind = h->skip_sig_kind;
  p.act_dump = h->act_dump;
  p.act_dump_n = h->act_dump ? (S < h->act_dump_n ? S : h->act_dump_n) : 0;
  if (frames == 1) {  // the profiling and testing hooks below are sized for one frame
    p.kv_dump = h->kv_dump;
    p.phase_ts = h->phase_ts;
    p.arrive_ts = h->arrive_ts;
  }
  if (cudaMemsetAsync(h->ws.bar, 0, 8, st) != cudaSuccess) return WAVE_ECUDA;
  cudaError_t e = launch_step(p, h->pl.grid, st);
  h->last_stream = st;
  if (e == cudaErrorCooperativeLaunchTooLarge) return WAVE_ELAUNCH;
  if (e != cudaSuccess) return WAVE_ECUDA;
  return WAVE_OK;
}

extern "C" int wave_step(wave_t* h, int S, const void* weights, uint8_t* kv_fp8, float* kv_scales,
                         const int32_t* positions, const void* x, void* y, void* stream) {
  if (h && h->pl.hybrid) return WAVE_EINVAL;
  return launch_frames(h, S, 1, weights, kv_fp8, kv_scales, positions, nullptr, x, y, stream);
}

extern "C" int wave_depth(wave_t* h, int S, int steps, const void* weights, const void* w_proj,
                          uint8_t* kv_fp8, float* kv_scales, const void* x0, void* xs, void* y,
                          void* stream) {
  if (!h || h->pl.hybrid || !w_proj || !x0 || !xs || !y) return WAVE_EINVAL;
  if (S < 1 || S > h->pl.S_max || steps < 1 || steps > kMaxFrames || steps > h->pl.T_max) return WAVE_EINVAL;
  if (((uintptr_t)w_proj & 15) || ((uintptr_t)x0 & 15) || ((uintptr_t)xs & 15) || ((uintptr_t)y & 15))
    return WAVE_EINVAL;
  if (encode_proj_maps(h->pl, w_proj, y, S, steps, &h->maps) != WAVE_OK) return WAVE_ECUDA;
  cudaStream_t st = (cudaStream_t)stream;
  if (xs != x0 &&
      cudaMemcpyAsync(xs, x0, (size_t)S * h->pl.cfg.d_model * 2, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return WAVE_ECUDA;
  return launch_frames(h, S, steps, weights, kv_fp8, kv_scales, h->ws.zero_pos, nullptr, xs, y, stream,
                       (uint16_t*)xs);
}

extern "C" int wave_hybrid_step(wave_t* h, int S, const void* weights, uint8_t* kv_fp8, float* kv_scales,
                                float* ssm_state, const int32_t* positions, const void* x, void* y,
                                void* stream) {
  if (!h || !h->pl.hybrid || !ssm_state || ((uintptr_t)ssm_state & 15)) return WAVE_EINVAL;
  return launch_frames(h, S, 1, weights, kv_fp8, kv_scales, positions, nullptr, x, y, stream, nullptr,
                       ssm_state);
}

extern "C" int wave_beat(wave_t* h, int S, int frames, const void* weights, uint8_t* kv_fp8,
                         float* kv_scales, int32_t* positions, int advance, const void* x, void* y,
                         void* stream) {
  if (h && h->pl.hybrid) return WAVE_EINVAL;
  return launch_frames(h, S, frames, weights, kv_fp8, kv_scales, positions, advance ? positions : nullptr,
                       x, y, stream);
}

extern "C" int wave_status(wave_t* h) {
  if (!h) return WAVE_EINVAL;
  // The kernel's last CTA copies the device error word into this pinned host
  // word when a launch ends; the caller has synchronised, so it is current.
  const int e = *(volatile int*)h->err_host;
  if (e == 0) return WAVE_OK;
  *(volatile int*)h->err_host = 0;
  // clear the device word behind the launches already on the handle's stream
  if (cudaMemsetAsync(h->ws.err, 0, 4, h->last_stream) != cudaSuccess) return WAVE_ECUDA;
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

extern "C" int wave_debug_skip_signal(wave_t* h, int which, int index) {
  if (!h || (index >= 0 && (which < 0 || which > 8))) return WAVE_EINVAL;
  h->skip_sig = index;
  h->skip_sig_kind = which;
  return WAVE_OK;
}

extern "C" int wave_debug_dump_kv(wave_t* h, float* dst) {
  if (!h) return WAVE_EINVAL;
  h->kv_dump = dst;
  return WAVE_OK;
}

extern "C" long long wave_debug_act_record_floats(wave_t* h) {
  if (!h) return WAVE_EINVAL;
  return act_record_floats(h->pl);
}

extern "C" int wave_debug_dump_acts(wave_t* h, float* dst, int n_sessions) {
  if (!h || (dst && (n_sessions < 1 || n_sessions > h->pl.S_max)) || ((uintptr_t)dst & 15)) return WAVE_EINVAL;
  h->act_dump = dst;
  h->act_dump_n = dst ? n_sessions : 0;
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

extern "C" int wave_grid_size(wave_t* h) { return h ? h->pl.grid : WAVE_EINVAL; }

extern "C" int wave_phases_per_step(wave_t* h) {
  if (!h) return WAVE_EINVAL;
  return h->pl.hybrid ? phases_per_step(h->pl.hcfg.n_layers, true, h->pl.hcfg.attn_every)
                      : phases_per_step(h->pl.cfg.n_layers, false, 1);
}

extern "C" int wave_barriers_per_step(wave_t* h) {
  if (!h) return WAVE_EINVAL;
  return h->pl.hybrid ? hybrid_barriers_per_step(h->pl.hcfg.n_layers, h->pl.hcfg.attn_every, h->pl.T_max)
                      : barriers_per_step(h->pl.cfg.n_layers, h->pl.T_max);
}
