// noalloc.cu -- wave_step_static: the frame step without any allocation.
//
// Some callers cannot allocate device memory: code that runs inside another
// runtime's memory pool or a process with a fixed device-memory budget, a
// plug-in that must not create allocations the host application does not
// track, or a real-time serving loop where cudaMalloc's implicit
// synchronisation is not allowed once the clock runs.  For them this entry
// point runs the same persistent step kernel as wave_step, on the same plan
// (plan.cu builds both), with its whole workspace (residual, activations,
// split-K and attention partials, work list, RoPE table, barrier and error
// words) placed in one fixed, file-scope device array instead of memory from
// cudaMalloc.
//
// The array is kNoAllocScratchBytes (32 MiB) and exists on every GPU that
// loads this library, for the life of the process.  Calls share it and it
// keeps the last call's contents; the words that must start at zero are
// cleared on every call, and the RoPE table is copied in whenever the shape
// differs from the previous call's on that device.  Two calls whose work
// overlaps on the GPU (other streams, or without waiting) race on it.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "../../include/wave.h"
#include "internal.h"
#include "plan.h"

using namespace wave;

namespace {

constexpr size_t kNoAllocScratchBytes = 32u << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Per device: the scratch array's device address (looked up once, with that
// device current) and the shape whose RoPE table the scratch holds.
struct DeviceState {
  void* addr = nullptr;
  bool have_table = false;
  wave_config cfg;
  int S_max = 0, T_max = 0;
};
std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

bool same_shape(const DeviceState& d, const wave_config* c, int S_max, int T_max) {
  return d.have_table && d.S_max == S_max && d.T_max == T_max && d.cfg.n_layers == c->n_layers &&
         d.cfg.d_model == c->d_model && d.cfg.n_heads == c->n_heads && d.cfg.head_dim == c->head_dim &&
         d.cfg.ffn == c->ffn && d.cfg.rms_eps == c->rms_eps && d.cfg.rope_base == c->rope_base;
}

}  // namespace

extern "C" int wave_step_static(const wave_config* cfg, int S_max, int T_max, int S, const void* weights,
                                uint8_t* kv_fp8, float* kv_scales, const int32_t* positions,
                                const void* x, void* y, void* stream) {
  // ---- arguments (the rules of wave_create + wave_step), before any device call
  Plan pl;
  if (!cfg || plan_decoder(&pl, cfg, S_max, T_max, 1) != WAVE_OK) return WAVE_EINVAL;
  if (!launch_args_ok(pl, S, 1, weights, kv_fp8, kv_scales, positions, x, y)) return WAVE_EINVAL;
  int dev = 0, sms = 0;
  const int rc = device_check(&dev, &sms);
  if (rc) return rc;
  if (dev < 0 || dev >= kMaxDevices) return WAVE_ECUDA;
  if (plan_decoder(&pl, cfg, S_max, T_max, sms) != WAVE_OK) return WAVE_EINVAL;
  // the workspace must fit the fixed array: larger shapes are refused
  if (carve_workspace(pl, nullptr, nullptr) > kNoAllocScratchBytes) return WAVE_EINVAL;

  cudaStream_t st = (cudaStream_t)stream;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& ds = g_dev[dev];
  // ---- one-time set-up on this device: the host-side name of a __device__
  // array is not a device address; look the address up with the device current
  if (!ds.addr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return WAVE_ECUDA;
    ds.addr = ptr;
  }
  Workspace ws;
  carve_workspace(pl, (char*)ds.addr, &ws);
  // ---- the RoPE table, built on the host exactly as wave_create builds it,
  // copied in when this device's scratch does not hold this shape's table
  if (!same_shape(ds, cfg, S_max, T_max)) {
    std::vector<float2> tab;
    rope_table(pl, &tab);
    ds.have_table = false;
    if (cudaMemcpyAsync(ws.rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)  // the host table is freed on return
      return WAVE_ECUDA;
    ds.have_table = true;
    ds.cfg = *cfg;
    ds.S_max = S_max;
    ds.T_max = T_max;
  }

  // ---- tensor maps over the caller's weights / history and the scratch activations
  Maps maps;
  const int S_pad = (S + 15) / 16 * 16;
  if (encode_weight_maps(pl, weights, &maps) || encode_kv_maps(pl, kv_fp8, kv_scales, &maps) ||
      encode_act_maps(pl, ws, S_pad, &maps))
    return WAVE_ECUDA;
  StepParams p;
  fill_params(&p, pl, ws, maps, S, weights, kv_fp8, kv_scales, positions, x, y, 1);

  // ---- clear what must start at zero (barrier and exit counters, the error
  // word; the kernel zeroes its tile and attention counters itself), launch, wait
  if (cudaMemsetAsync(ws.bar, 0, 16, st) != cudaSuccess || cudaMemsetAsync(ws.err, 0, 16, st) != cudaSuccess)
    return WAVE_ECUDA;
  const cudaError_t e = launch_step(p, pl.grid, st);
  if (e == cudaErrorCooperativeLaunchTooLarge) return WAVE_ELAUNCH;
  if (e != cudaSuccess) return WAVE_ECUDA;
  int err = 0;
  if (cudaMemcpyAsync(&err, ws.err, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return WAVE_ECUDA;
  if (err & kErrTimeout) return WAVE_ETIMEOUT;
  if (err) return WAVE_EPOS;
  return WAVE_OK;
}
