/*
 * wave.h -- C ABI of the frame-locked batched decode step for one GB300
 * (sm_103a).  One call advances every live session by one 80 ms frame through
 * all decoder layers in a single persistent GPU launch; each bf16 weight is
 * read from HBM once per step and shared by all S sessions.
 *
 * The operation follows the pages' description of the frame step:
 *   - "PersonaPlex 7B, 80 sessions, one H100" (narilabs blog): "What Real-time
 *     Means for a Full-duplex Agent" (one 80 ms frame per forward pass),
 *     "Compressing the Temporal KV cache" (bf16 weights and activations, FP8
 *     temporal K/V cache), "A server built around the conversation clock"
 *     (every session on one clock, fixed-shape batches, slots filled by new
 *     sessions without changing execution);
 *   - dotwave.ai case study, "02 / The solution" and "04 / Under the hood"
 *     (weights shared across sessions, state resident between beats, no CPU
 *     round trip between operations, profiles per session capacity and
 *     context length).
 * The decoder layer itself (RMSNorm, QKV, RoPE, FP8 K/V append, attention,
 * output projection, SwiGLU MLP) is not spelled out on the pages; the
 * readings taken are listed with wave_step below.
 *
 * Conventions.  Every pointer passed to wave_step / wave_kv_quantize /
 * wave_fp8_encode is a DEVICE pointer owned by the caller.  Nothing returned
 * by this library needs freeing except a handle (wave_destroy).  Functions
 * return WAVE_OK (0) or a negative WAVE_E* code; no function aborts the
 * process or traps the GPU.  A handle is used by one stream at a time.
 */
#ifndef WAVE_H_
#define WAVE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define WAVE_OK 0
#define WAVE_EINVAL (-1)   /* bad argument: null pointer, size out of range, misalignment */
#define WAVE_ECUDA (-2)    /* a CUDA runtime/driver call failed */
#define WAVE_ELAUNCH (-3)  /* the persistent grid could not be made co-resident */
#define WAVE_ETIMEOUT (-4) /* a device-side wait (grid barrier, async copy) gave up */
#define WAVE_EPOS (-5)     /* a session's position was at or beyond T_max */
#define WAVE_EDEVICE (-6)  /* the current device is not an sm_103 GPU */
#define WAVE_ENOMEM (-7)   /* device allocation failed */

/* Decoder shape.  Constraints checked by wave_create: head_dim is 64 or 128;
 * d_model (at most 8192), n_heads*head_dim and ffn are multiples of 64, 64
 * and 8. */
typedef struct {
  int n_layers, d_model, n_heads, head_dim, ffn;
  float rms_eps, rope_base;
} wave_config;

typedef struct wave_ctx wave_t; /* opaque; owns only its device workspace */

/*
 * Create a step context for at most S_max sessions (1..128) and a history of
 * T_max slots per session (a multiple of 4): the dotwave.ai case study ("04 /
 * Under the hood") builds one engine profile per model, session capacity and
 * context length, and a handle is that profile here.  Allocates the device
 * workspace on the current device (activations, partial sums, the RoPE
 * cos/sin table, barrier words; about 0.5 MB + S_max * (2.1 * d_model + ...)
 * bytes, e.g. ~60 MB for the 7B-class shape at S_max = 128) and one pinned,
 * device-mapped host word for the error status.  Returns WAVE_EINVAL for a
 * bad shape, WAVE_EDEVICE off sm_103, WAVE_ENOMEM/WAVE_ECUDA on failure;
 * *out is set only on success.
 */
int wave_create(const wave_config* cfg, int S_max, int T_max, wave_t** out);

/* Free the workspace (the end of the per-session state's residence that
 * the dotwave.ai case study, "02 / The solution", keeps between beats; the
 * caller's history buffers are untouched).  Waits for the device to finish
 * the handle's work first.  NULL is a no-op. */
void wave_destroy(wave_t* h);

/* Bytes of the bf16 weight blob for cfg (see wave_weight_offset): the bf16
 * weights of the narilabs blog, "Compressing the Temporal KV cache", laid
 * out as below.  0 for an invalid shape. */
size_t wave_weights_bytes(const wave_config* cfg);

/*
 * Byte offset inside the weight blob of one tensor of one layer (the pages
 * fix no layout; this is the library's, in nn.Linear [out][in] order so
 * that every row streams contiguously).  which:
 *   0 g_attn  [d]            RMSNorm gain before attention
 *   1 Wqkv    [3*H*D][d]     rows: q (H*D), then k (H*D), then v (H*D)
 *   2 Wo      [d][H*D]
 *   3 g_mlp   [d]            RMSNorm gain before the MLP
 *   4 Wgu     [2*F][d]       rows: gate (F), then up (F)
 *   5 Wdown   [d][F]
 * All bf16, each matrix [out][in] with the in-dimension contiguous; layers are
 * stored one after another in this order.  Returns (size_t)-1 on bad input.
 */
size_t wave_weight_offset(const wave_config* cfg, int layer, int which);

/*
 * The packed weight blob the step reads.  The blob of wave_weight_offset
 * (row-major [out][in] matrices) is the interchange layout; the step reads
 * the same tensors in the same order with every projection matrix stored as
 * blocks of 128 rows x 64 inputs (16 KB, row-major inside a block), ordered
 * by 128-row tile, then by 64-input block, rows and inputs beyond the matrix
 * zero (the gate/up matrix's tile t holds gate rows 64t..64t+63, then up rows
 * 64t..64t+63).  Every 16 KB the projections stream is then one contiguous
 * block, which HBM serves at its streaming rate; the row-major tiles' 128-byte
 * rows, kilobytes apart, cost DRAM page switches.  The pages fix no layout
 * (the weights are bf16: the narilabs blog, "Compressing the Temporal KV
 * cache").  The RMSNorm gains are copied as they are.
 *
 * wave_packed_weights_bytes: bytes of the packed blob (0 for a bad shape);
 * the same as wave_weights_bytes when d_model, n_heads * head_dim and ffn
 * are multiples of 128.  wave_pack_weights: reorder src (the blob of
 * wave_weight_offset) into dst (wave_packed_weights_bytes, distinct from
 * src); both device pointers, 16-byte aligned; asynchronous on `stream`.
 * WAVE_EINVAL for bad arguments.
 */
size_t wave_packed_weights_bytes(const wave_config* cfg);
int wave_pack_weights(const wave_config* cfg, const void* src, void* dst, void* stream);

/*
 * One frame for sessions 0..S-1 (1 <= S <= S_max).  Asynchronous: enqueues
 * two operations on `stream` (an 8-byte memset of the barrier and exit
 * counters and one cooperative kernel launch) and returns; nothing is
 * synchronised.
 *
 *   weights    the packed bf16 blob (wave_pack_weights), 16-byte aligned, read only.
 *   kv_fp8     uint8 [L][2][S_max][H][T_max][D] E4M3 codes (index 0 = K, 1 = V),
 *              16-byte aligned.  Slots 0..pos[s]-1 are read; slot pos[s] of every
 *              (layer, K|V, s, head) is written; no other byte is touched.
 *   kv_scales  float [L][2][S_max][H][T_max], 16-byte aligned: one scale per
 *              (layer, K|V, session, head, token) with value = code * scale.
 *   positions  int32 [S]: pos[s] is the RoPE position of this frame and the
 *              cache slot it writes; attention spans slots 0..pos[s] inclusive.
 *              A negative pos[s] marks an empty slot of the fixed-shape batch
 *              (no session there this frame): its cache is not touched and
 *              y[s] = x[s] bit for bit.  Input only: the caller advances
 *              positions between frames.
 *   x          bf16 [S][d] input activations; y bf16 [S][d] output (may alias x);
 *              both 16-byte aligned.
 *
 * Readings of what the pages leave open: bf16 rounding only at the projection
 * inputs (normed x, attention output, SwiGLU output) and at y, fp32 elsewhere;
 * RMSNorm r / sqrt(mean(r^2) + eps) * g; rotate-half RoPE, pairs (i, i+D/2),
 * angle pos * base^(-2i/D); the current token's K/V are quantised first and
 * read back quantised; scale = amax/448 in fp32, code = E4M3-RNE-satfinite of
 * v/scale (fp32 division), all-zero codes and scale 0 for a zero row; softmax
 * scale 1/sqrt(D); SwiGLU silu(gate) * up; no biases, no final norm.
 *
 * A session whose pos is at or beyond T_max gets no cache write and a zero
 * attention output; the step records WAVE_EPOS for wave_status.
 * Returns WAVE_EINVAL for bad arguments (checked on the host before any
 * launch), WAVE_ELAUNCH/WAVE_ECUDA if the launch fails.
 */
int wave_step(wave_t* h, int S, const void* weights, uint8_t* kv_fp8, float* kv_scales,
              const int32_t* positions, const void* x, void* y, void* stream);

/*
 * Several frames in one launch: the beat of the dotwave.ai case study ("01 /
 * The challenge", "Measurement notes": two 80 ms model steps per beat, a
 * 160 ms deadline; "02 / The solution": state stays ready between beats).
 * Frame f (0 <= f < frames) reads x[f] and writes y[f] (x, y bf16
 * [frames][S][d], 16-byte aligned) and runs every session at position
 * pos[s] + f; a negative pos[s] stays an empty slot in every frame.  The
 * results equal `frames` wave_step calls with the positions advanced by one
 * between them.  With advance != 0 the kernel adds `frames` to every
 * non-negative pos[s] after the last frame (positions roll on the device;
 * nothing crosses to the host between beats); with advance == 0 positions is
 * only read.  1 <= frames <= 64; the other arguments, the error behaviour
 * and the asynchrony are those of wave_step.  The wave_debug_* hooks apply to
 * single-frame launches only.
 */
int wave_beat(wave_t* h, int S, int frames, const void* weights, uint8_t* kv_fp8, float* kv_scales,
              int32_t* positions, int advance, const void* x, void* y, void* stream);

/*
 * The inner depth loop: `steps` dependent steps of the model in one launch
 * (the narilabs blog, "Predictable GPU execution": the Depformer's
 * autoregressive loop of 8 steps per frame, captured with the frame).  Step
 * k runs every session at depth position k over a depth cache of T_max >=
 * steps slots (kv_fp8 / kv_scales as in wave_step; slots 0..k-1 hold this
 * call's earlier steps, so nothing carries over from an earlier call), and
 * takes as input
 *     x_0 = x0,   x_k = bf16(W_p y_{k-1})  (fp32 accumulation),
 * W_p a bf16 [d][d] matrix (row n = output n, 16-byte aligned).  x0 is bf16
 * [S][d]; xs is caller scratch bf16 [steps][S][d] that receives x_0..x_{k}
 * (xs may equal x0); y is bf16 [steps][S][d], the outputs of every step.
 * 1 <= steps <= min(64, T_max).  Errors and asynchrony as wave_step (it
 * enqueues one device-to-device copy of x0 before the launch).  The wave_debug_*
 * hooks apply to single-frame launches only.
 */
int wave_depth(wave_t* h, int S, int steps, const void* weights, const void* w_proj, uint8_t* kv_fp8,
               float* kv_scales, const void* x0, void* xs, void* y, void* stream);

/*
 * The hybrid recurrent step (e.g. 48 layers of width 4096, an attention
 * block every sixth layer, 64 state heads of 64 x 128: the NemotronH-style
 * thinker of the vllm-omni recipe page, "Summary", whose recurrent state is
 * FP32 per the dotwave.ai profile.json): n_layers pre-norm residual blocks
 * without MLPs; layer l is an attention block (RMSNorm, QKV, RoPE, FP8 K/V
 * append, attention over the history, O; as wave_step's attention half) when
 * l % attn_every == attn_every - 1, else a Mamba2-style selective-state
 * block: zxbcdt = W_in xn split [z d_i | x d_i | B N | C N | dt Hs] (one
 * group, no conv1d); per head dt = softplus(dt + dt_bias), a = exp(-exp(A_log)
 * dt); per head dim p and state n: h = a h + dt x_p B_n (fp32 state, in
 * place), y_p = sum_n C_n h + D x_p; r += W_out bf16(y silu(z)).
 * Constraints: n_layers % attn_every == 0, ssm_head_dim 64, ssm_state 128,
 * ssm_heads a multiple of 4 and at most 1024, the attention shapes of wave_config.
 */
typedef struct {
  int n_layers, d_model, attn_every;  /* layers; width; an attention block every attn_every layers */
  int n_heads, head_dim;              /* attention blocks (head_dim 64 or 128) */
  int ssm_heads, ssm_head_dim, ssm_state;
  float rms_eps, rope_base;
} wave_hybrid_config;

/* Bytes of the hybrid bf16 weight blob and of the start of layer `layer`
 * (layer == n_layers gives the total).  Per layer, [out][in] matrices:
 * selective-state block: g[d], W_in[2 d_i + 2 N + Hs][d] (z, x, B, C, dt
 * rows), W_out[d][d_i], A_log[Hs], dt_bias[Hs], D[Hs] (this last block padded
 * to 8 elements); attention block: g[d], Wqkv[3 H D][d], Wo[d][H D].  Groups
 * of attn_every layers: (attn_every - 1) selective-state blocks, then one
 * attention block.  0 / (size_t)-1 for an invalid config or layer. */
size_t wave_hybrid_weights_bytes(const wave_hybrid_config* cfg);
size_t wave_hybrid_layer_offset(const wave_hybrid_config* cfg, int layer);

/* The hybrid step's packed blob: the blob of wave_hybrid_layer_offset with
 * every projection matrix (W_in, W_out, Wqkv, Wo) packed as for
 * wave_pack_weights; gains and the A_log / dt_bias / D block copied as they
 * are.  Sizes and arguments as wave_packed_weights_bytes / wave_pack_weights. */
size_t wave_hybrid_packed_weights_bytes(const wave_hybrid_config* cfg);
int wave_hybrid_pack_weights(const wave_hybrid_config* cfg, const void* src, void* dst, void* stream);

/* A handle for the hybrid step (the attention blocks' history as in
 * wave_create, with n_layers / attn_every layers).  Release with
 * wave_destroy.  wave_step / wave_beat / wave_depth refuse a hybrid handle. */
int wave_hybrid_create(const wave_hybrid_config* cfg, int S_max, int T_max, wave_t** out);

/* One frame of the hybrid model for sessions 0..S-1.  weights: the hybrid
 * packed blob (wave_hybrid_pack_weights).  kv_fp8 / kv_scales:
 * the attention blocks' history ([La][2][S_max][H][T_max][D], La = n_layers /
 * attn_every; as wave_step).  ssm_state: fp32 [Lm][S_max][Hs][64][128]
 * (Lm = n_layers - La), 16-byte aligned, read and written in place; an empty
 * slot's (negative position) state is not touched.  Other arguments, errors
 * and asynchrony as wave_step. */
int wave_hybrid_step(wave_t* h, int S, const void* weights, uint8_t* kv_fp8, float* kv_scales,
                     float* ssm_state, const int32_t* positions, const void* x, void* y, void* stream);

/*
 * The error status of the handle's launches, read without synchronising
 * anything: every launch's last CTA copies the device error word into a
 * pinned host word as the kernel ends, and wave_status reads that word.  So
 * call it after the caller has synchronised with the launches it asks
 * about (stream or event synchronisation); before that it reports only the
 * launches already finished.  The bits are sticky across launches until
 * read: a non-OK result clears them (host word now, device word by an
 * asynchronous memset enqueued on the handle's last stream).  Returns
 * WAVE_OK, WAVE_ETIMEOUT (a device wait gave up; that step's outputs are
 * undefined, the GPU context stays usable) or WAVE_EPOS; WAVE_ECUDA if the
 * clearing memset could not be enqueued.  This is the step's own failure
 * report: the pages describe none (their only recovery, the vllm-omni recipe
 * page's eager fallback in "Notes", is a second code path this library does
 * not have), so errors become status codes and no device wait is unbounded.
 */
int wave_status(wave_t* h);

/* Static description of a return code (see wave_status). */
const char* wave_strerror(int code);

/*
 * FP8 quantiser of the K/V append, on its own: for each of `rows` rows of D
 * fp32 values (row-major, device), scale = amax/448 and codes = E4M3(v/scale)
 * exactly as wave_step writes them.  Used to prefill a history.  Writes
 * codes [rows][D] and scales [rows].  Asynchronous on `stream`.
 * D must be a multiple of 4 in [4, 1024].
 */
int wave_kv_quantize(const float* v, int64_t rows, int D, uint8_t* codes, float* scales,
                     void* stream);

/* Element-wise E4M3 encoder of the step (round to nearest even, saturate to
 * +-448, sign kept): out[i] = E4M3(in[i]).  Asynchronous on `stream`. */
int wave_fp8_encode(const float* in, int64_t n, uint8_t* out, void* stream);

/*
 * wave_step for callers that cannot allocate device memory (inside another
 * runtime's memory pool or a fixed device-memory budget, a plug-in that must
 * not create untracked allocations, or a real-time loop where cudaMalloc's
 * implicit synchronisation is not allowed).  No source page describes such
 * a call: it is an interface addition of this library.
 *
 * Same arguments and layouts as wave_create(cfg, S_max, T_max) followed by
 * wave_step(S, ...), but no handle and no allocation: the workspace lives in
 * one fixed 32 MiB device array of the library, present on every GPU that
 * loads it until the process exits.  Shapes whose workspace does not fit
 * (roughly: S_max * (2.1 d + 3 H*D + 0.5 F) * 4 bytes of activations plus
 * split-K and attention partials plus a T_max * D * 4-byte RoPE table)
 * return WAVE_EINVAL.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress); make that first call before any stream
 * capture.  Unlike wave_step the call waits for its step to finish on
 * `stream` and returns the step's status (WAVE_OK, WAVE_EPOS, WAVE_ETIMEOUT)
 * directly.  All calls share the array: calls that overlap on the GPU (from
 * several streams or threads at once) race and must not be made.
 */
int wave_step_static(const wave_config* cfg, int S_max, int T_max, int S, const void* weights,
                     uint8_t* kv_fp8, float* kv_scales, const int32_t* positions, const void* x,
                     void* y, void* stream);

/* ---- testing hooks (fault tests without a GPU fault) ---------------------
 * Limit for every device-side wait of later steps, in nanoseconds (default
 * 2e9).  A wait that runs out sets WAVE_ETIMEOUT and the kernel returns. */
int wave_set_timeout_ns(wave_t* h, long long ns);
/* Make CTA `cta` skip its arrival at grid barrier number `barrier` (0-based)
 * in later steps, so that the others' waits run out; cta < 0 disables. */
int wave_debug_skip_barrier(wave_t* h, int cta, int barrier);
/* Make later steps never publish the readiness of one item, so that the
 * wait for it runs out at a phase hand-over without a grid barrier: which =
 * 0 the QKV tile `index` (attention waits), 1 the gate/up tile `index` (the
 * down projection waits), 2 the attention rows of head `index` (the output
 * projection waits), 3 the output-projection tile `index` (the second
 * RMSNorm waits), 4 the down-projection tile `index` (the next layer's first
 * RMSNorm waits), 5 the RMSNorm row `index` (the next projection waits);
 * in the hybrid step also 6 the selective-state in-projection tile `index`
 * (the state items wait), 7 the finished state items of CTA `index` (the
 * out-projection waits), 8 the selective-state out-projection tile `index`
 * (the next RMSNorm waits).  index < 0 disables. */
int wave_debug_skip_signal(wave_t* h, int which, int index);
/* Make later steps also write, for every session with a valid position, the
 * fp32 K (after RoPE) and V rows they quantise into dst, a device buffer of
 * [L][2][S_max][H][D] floats, so that tests can check the append bit for bit
 * against a reference quantiser.  dst = NULL disables. */
int wave_debug_dump_kv(wave_t* h, float* dst);
/* Activation dump: make later launches (any number of frames) record, for
 * sessions 0..n_sessions-1, every phase's input and output as fp32 values
 * into dst (device, 16-byte aligned): [frames][layers][n_sessions][R] floats,
 * R = wave_debug_act_record_floats(h), layers = the model's layer count.
 * Record of a layer, in this order (d model width, F the MLP width; N1 =
 * max(3 H D, the hybrid in-projection rows), N2 = max(H D, the hybrid
 * d_inner)):
 *   [0, d)          the layer's input residual (fp32)
 *   [d, 2d)         its RMS-normed input xn (bf16 values)
 *   [2d, 2d+N1)     the input projection's output: q, k, v before RoPE, or the
 *                   selective-state block's z, x, B, C, dt (fp32)
 *   [.., +N2)       the attention output (bf16) or the gated mixer output (bf16)
 *   [.., +d)        decoder: residual after O; hybrid: the block's output residual
 *   [.., +d)        decoder: the MLP's normed input (bf16)
 *   [.., +F)        decoder: the SwiGLU output u (bf16)
 *   [.., +d)        decoder: the layer's output residual (fp32)
 * The last layer's output residual is not recorded (y holds it, rounded).
 * The dump runs a second instantiation of the step kernel that differs from
 * the usual one only by these copies.  dst = NULL disables. */
int wave_debug_dump_acts(wave_t* h, float* dst, int n_sessions);
long long wave_debug_act_record_floats(wave_t* h);
/* Profiling hook: make later steps record %globaltimer (ns) into dst, a device
 * buffer of wave_barriers_per_step(h) + 2 int64: [0] at kernel entry, [1+b]
 * when grid barrier b released CTA 0, and the last entry at kernel exit.
 * dst = NULL disables. */
int wave_debug_phase_times(wave_t* h, long long* dst);
/* Profiling hook: later steps write, into the device buffer dst of
 * wave_phases_per_step(h) x wave_grid_size(h) int64, the globaltimer value
 * at which each CTA finished each phase ([phase][cta]; the prologue, then
 * each layer's phases in order: decoder [first RMSNorm from layer 1 on],
 * QKV, attention, O, second RMSNorm, gate/up, down; hybrid [RMSNorm from
 * layer 1 on], in-projection (or QKV), state update (or attention),
 * out-projection (or O)), so that the spread of a phase's finishing times
 * and the critical path can be read.  dst = NULL disables. */
int wave_debug_arrival_times(wave_t* h, long long* dst);
/* Grid size (CTAs, one per SM), grid barriers and phases per step, for
 * tests and tools. */
int wave_grid_size(wave_t* h);
int wave_barriers_per_step(wave_t* h);
int wave_phases_per_step(wave_t* h);

#ifdef __cplusplus
}
#endif
#endif /* WAVE_H_ */
