// plan.h -- host-side set-up shared by the handle API (api.cu) and the
// no-allocation entry point (noalloc.cu): shape checks, the weight-blob
// layout, the stream-K plan of the projections, the workspace carve-up, the
// RoPE table, tensor-map encoding and the kernel's parameter block.  Both
// entry points build their launches through these functions only, so that
// they run the same kernel on the same plan.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <vector>

#include "../../include/wave.h"
#include "internal.h"

namespace wave {

// Everything derived from a shape, a capacity and the grid, before any pointer.
struct Plan {
  wave_config cfg;           // decoder shape; for the hybrid model, its attention blocks
  int hybrid = 0;
  wave_hybrid_config hcfg;   // the hybrid shape (hybrid only)
  int S_max = 0, S_pad_max = 0, T_max = 0, grid = 0;
  long long off[6] = {0, 0, 0, 0, 0, 0};  // decoder blob: g_attn, Wqkv, Wo, g_mlp, Wgu, Wdown
  long long layer_elems = 0;              // decoder: one layer; hybrid: one group of layers
  long long hyb_M = 0, hyb_G = 0;         // hybrid: elements of a selective-state block / a group
  long long hyb_off_w_in = 0, hyb_off_w_out = 0, hyb_off_a_log = 0;  // inside a selective-state block
  long long hyb_off_wqkv = 0, hyb_off_wo = 0;                        // inside an attention block
  int in_rows = 0, d_inner = 0;
  int tiles[kGemmKinds] = {0}, kblocks[kGemmKinds] = {0};
  int max_tiles_per_cta = 1;
  // The packed blob the step reads (see wave_pack_weights): the same tensors
  // in the same order, every projection matrix as tile blocks.
  long long pk_off[6] = {0, 0, 0, 0, 0, 0};  // decoder: offsets inside a packed layer
  long long pk_layer = 0;                     // decoder: one packed layer; hybrid: one packed group
  long long pk_M = 0, pk_A = 0;               // hybrid: packed selective-state / attention block
  long long pk_w_in = 0, pk_w_out = 0, pk_a_log = 0, pk_wqkv = 0, pk_wo = 0;  // inside those blocks
  long long pk_total = 0;                     // elements of the packed blob
};

// Elements of one packed projection matrix: `tiles` row tiles x `kunits`
// 128-column units, each unit two 128-row x 64-column blocks of 8192 elements.
inline long long packed_matrix_elems(int tiles, int kunits) { return (long long)tiles * kunits * 2 * 8192; }

// The library-owned device buffers of a step, carved out of one block.
struct Workspace {
  float* resid = nullptr;
  uint16_t* xn = nullptr;
  float* qkv = nullptr;
  uint16_t* attn = nullptr;
  uint16_t* u = nullptr;
  float* gemm_part = nullptr;
  int* tile_cnt = nullptr;
  float* att_part = nullptr;
  int2* sh_info = nullptr;
  int4* pieces = nullptr;
  int* n_pieces = nullptr;
  int* sh_cnt = nullptr;
  float2* rope = nullptr;
  unsigned* bar = nullptr;   // [0] grid barrier counter, [1] exit counter (zeroed before each launch)
  int* err = nullptr;
  int32_t* zero_pos = nullptr;
  float* zx = nullptr;
  uint16_t* ssm_out = nullptr;
};

// Tensor maps of one launch.
struct Maps {
  CUtensorMap tm_w[kGemmKinds], tm_x[kGemmKinds], tm_kv, tm_sc;
};

bool decoder_shape_ok(const wave_config* c);
bool hybrid_shape_ok(const wave_hybrid_config* c);
void decoder_layout(const wave_config* c, long long off[6], long long* layer_elems);
// Hybrid blob: element counts of a selective-state block (M) and of an
// attention block (A), and the offsets inside them.
void hybrid_layout(const wave_hybrid_config* c, long long* M, long long* A, long long* w_in,
                   long long* w_out, long long* a_log, long long* wqkv, long long* wo);
// The current device, its SM count, and whether it is sm_103 with the driver
// entry points and kernel attributes the step needs.
int device_check(int* dev, int* sms);
// Capacity checks shared by every entry point (S_max, T_max, history rows).
bool capacity_ok(int S_max, int T_max, long long history_rows);
// Stream-K plan of a decoder / hybrid shape on `grid` CTAs.  WAVE_OK, or
// WAVE_EINVAL when a projection has too many tiles or segments.
int plan_decoder(Plan* pl, const wave_config* cfg, int S_max, int T_max, int grid);
int plan_hybrid(Plan* pl, const wave_hybrid_config* hc, int S_max, int T_max, int grid);
// Bytes of the workspace of a plan; with base != nullptr, the pointers into
// [base, base + bytes) (256-byte aligned pieces).
size_t carve_workspace(const Plan& pl, char* base, Workspace* ws);
// RoPE table (cos, sin) of t * base^(-2i/D) for t < T_max, i < D/2,
// evaluated in double on the host and stored as fp32 pairs.
void rope_table(const Plan& pl, std::vector<float2>* tab);
// Tensor maps over the caller's weights, the history and the workspace's
// activation buffers (S_pad rows per activation box).
int encode_weight_maps(const Plan& pl, const void* weights, Maps* m);
int encode_act_maps(const Plan& pl, const Workspace& ws, int S_pad, Maps* m);
int encode_kv_maps(const Plan& pl, uint8_t* kv, float* scales, Maps* m);
// The kernel parameter block of one launch; the testing and profiling hooks
// are left off (null / -1) and the error mirror unset.
void fill_params(StepParams* p, const Plan& pl, const Workspace& ws, const Maps& m, int S,
                 const void* weights, uint8_t* kv, float* kv_scales, const int32_t* positions,
                 const void* x, void* y, int frames);
// The inner depth loop's maps: W_p [d][d] as a one-layer weight stack, and
// the outputs y [steps * S][d] read back S_pad rows at a time.
int encode_proj_maps(const Plan& pl, const void* w_proj, void* y, int S, int steps, Maps* m);
// Floats per record of the activation dump (the testing hook of wave.h):
// 5 d + max(3 H D, in_rows) + max(H D, d_inner) + F.
long long act_record_floats(const Plan& pl);
// Reorder the blob laid out as wave_weight_offset / wave_hybrid_layer_offset
// describe into the packed blob of the plan (device to device, on stream).
int pack_weights(const Plan& pl, const void* src, void* dst, cudaStream_t stream);
// Argument checks of a launch on the host (null pointers, S, frames, alignment).
bool launch_args_ok(const Plan& pl, int S, int frames, const void* weights, const void* kv,
                    const void* kv_scales, const void* positions, const void* x, const void* y);

}  // namespace wave
