// internal.h -- shared definitions of the step library (host and device).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace wave {

constexpr int kThreads = 256;     // 8 warps: TMA producer, MMA issuer, 4 epilogue warps, 2 more
                                  // (all 8 run attention and the norms)
constexpr int kWarps = kThreads / 32;
constexpr int kTileM = 128;       // weight rows per GEMM tile = tcgen05 M
constexpr int kKBlk = 64;         // K elements per TMA box (128 B of bf16, the swizzle span)
constexpr int kKStage = 2;        // boxes per ring stage: a stream-K unit is kKUnit K elements
constexpr int kKUnit = kKBlk * kKStage;
constexpr int kChunk = 32;        // attention tokens per async-copy chunk (2 x 16)
constexpr int kAttStages = 3;     // stages per attention warp (two in flight while one is read)
// The K and V scales of kScaleGroup chunks come in one copy (a box of both
// planes), into one of two buffers per warp: a quarter of the copies of one
// per chunk (measured 0.8 us per layer faster).
constexpr int kScaleGroup = 4;
constexpr int kScaleBufBytes = 2 * kScaleGroup * kChunk * 4;  // [K|V][kScaleGroup * kChunk] fp32
#ifndef WAVE_PIECE_CHUNKS
#define WAVE_PIECE_CHUNKS 16
#endif
constexpr int kPieceChunks = WAVE_PIECE_CHUNKS;  // chunks per attention work piece
// GEMM ring depth cap.  At S = 80 four stages fill the ring; smaller S fit
// five to seven, but a fifth and sixth stage measured 0.4-2.5% slower per
// step (S = 1 to 48), presumably because the weights issued ahead of a
// hand-over then compete with the previous phase's last copies.
constexpr int kMaxStages = 4;
constexpr int kTmemCols = 256;    // two fp32 accumulators of up to 128 columns

enum ErrBits : int { kErrTimeout = 1, kErrPos = 2 };

// Device error word bits -> public codes live in api.cu.

enum GemmKind : int { kQKV = 0, kO = 1, kGU = 2, kDown = 3, kProj = 4, kIn = 5, kOut = 6 };
constexpr int kGemmKinds = 7;
// Selective-state blocks of the hybrid model: head dim and state size the
// state phase is laid out for (8 warps x 8 rows, 32 lanes x 4 states).
constexpr int kSsmP = 64;
constexpr int kSsmN = 128;
// State items in flight per CTA (34 KB each, 102 KB for three).  Three
// measured 0.4-0.9% faster per step than four or five on the 48-layer hybrid
// shape (56 sessions x 64 state heads, ~24 items per CTA per block).
constexpr int kSsmStages = 3;
// A_log, dt_bias and D of every head are staged after the items in flight:
// 3 x 34 KB + 3 x 1024 x 4 B fit the 200 KB ring.
constexpr int kSsmMaxHeads = 1024;
static_assert(kSsmStages * (kSsmP * kSsmN + 512) * 4 + 3 * kSsmMaxHeads * 4 <= 200 * 1024,
              "state stages and per-head parameters exceed the ring");

struct StepParams {
  CUtensorMap tm_w[kGemmKinds];  // weights of the projections (see GemmKind)
  CUtensorMap tm_x[kGemmKinds];  // their activation inputs: xn, attn, xn, u, y, xn, ssm_out (box rows = S_pad)
  CUtensorMap tm_kv;     // the FP8 history as [D][S_max*H*T_max][K|V][L]: one box = a chunk's K and V
  CUtensorMap tm_sc;     // the scales as [S_max*H*T_max][K|V][L]: one box = a chunk's K and V scales
  // shape
  int L, d, H, D, F, HD, S, S_pad, S_max, T_max;
  float eps;
  int nstage;            // GEMM ring depth for this S
  int tiles[kGemmKinds], kblocks[kGemmKinds];
  int max_tiles_per_cta; // partial-sum slots per CTA
  long long layer_elems, off_g_attn, off_g_mlp;  // the packed blob: layer stride, RMSNorm gains
  // caller buffers
  const uint16_t* weights;
  uint8_t* kv;
  float* kv_scales;
  const int32_t* pos;
  const uint16_t* x;     // [n_frames][S][d]
  uint16_t* y;           // [n_frames][S][d]
  int n_frames;          // frames run back to back in this launch (positions + f in frame f)
  int32_t* pos_advance;  // if set: positions += n_frames at the end (empty slots stay empty)
  int depth;             // frames chained: x[f] = bf16(W_p y[f-1]) (the kProj GEMM) before frame f
  uint16_t* x_chain;     // where those inputs go (the buffer x points at)
  // hybrid model (selective-state blocks with an attention block every attn_every layers)
  int hybrid, attn_every, ssm_heads, d_inner, in_rows;
  long long hyb_M, hyb_G;      // packed elements of one Mamba block and of one group of attn_every layers
  long long hyb_off_a_log;     // inside a packed Mamba block: A_log, dt_bias, D
  float* zx;             // [S_pad][in_rows] fp32 in-projection output (z | x | B | C | dt)
  uint16_t* ssm_out;     // [S_pad][d_inner] bf16 gated mixer output
  float* ssm_state;      // caller's [Lm][S_max][Hs][P][N] fp32 state
  // workspace
  float* resid;          // [S_pad_max][d] fp32 residual stream
  uint16_t* xn;          // [S_pad_max][d] bf16 normed input of QKV / gate-up
  float* qkv;            // [S_max][3*H*D] fp32
  uint16_t* attn;        // [S_pad_max][H*D] bf16 attention output
  uint16_t* u;           // [S_pad_max][F] bf16 SwiGLU output
  float* gemm_part;      // [2 banks][G][max_tiles_per_cta][S_pad][128] split-K partials
  long long part_bank;   // floats per bank of gemm_part
  int* tile_cnt;         // [2 banks][2][1024] per tile: segments arrived, final reducers done
  int* done_cnt;         // [kind] tiles of that projection finished (and published) in this frame
  int* qkv_done;         // [1024] per QKV tile: history layer + 1 once its q, k, v rows are written
  int* head_cnt;         // [H] (session, head) attention rows written in this frame
  int* sh_cnt;           // [S_max*H] pieces of a (session, head) finished in this frame
  int* att_ctr;          // [L] attention work counters
  float* att_part;       // [max pieces][D + 4] (acc, m, l) per attention piece
  int2* sh_info;         // [S_max*H] (first partial slot, pieces) per (session, head)
  int4* pieces;          // [2 * max pieces] (sh, c_lo | c_hi << 16, pieces of sh, first slot), (pos, 0, 0, 0)
  int* n_pieces;         // [0] work-list entries, [1] sessions with a valid position
  const float2* rope;    // [T_max][D/2] (cos, sin)
  unsigned* bar;         // [0] grid barrier counter, [1] CTAs finished (both zeroed before each launch)
  int* err;              // error bits (sticky until wave_status)
  long long timeout_ns;
  int skip_cta, skip_bar;
  int skip_sig;          // testing hook: item (tile, head or norm row) never published, of ...
  int skip_sig_kind;     // ... this kind (wave_debug_skip_signal's `which`); skip_sig -1: off
  float* kv_dump;        // testing hook: [L][2][S_max][H][D] pre-quantisation K/V, or null
  float* act_dump;       // testing hook: [frames][L][act_dump_n][act_rec] phase inputs/outputs, or null
  int act_dump_n;        // sessions 0..act_dump_n-1 are recorded
  int act_n1, act_n2;    // record sections: input-projection output, mixer output (floats)
  long long act_rec;     // floats per record
  int* err_out;          // if set: the last CTA to finish copies *err here (a mapped host word)
  long long* phase_ts;   // profiling hook: globaltimer at start, after each barrier, at end
  long long* arrive_ts;  // profiling hook: [phase][cta] globaltimer when each CTA finished each phase
};

// CTAs taking part in a stream-K GEMM phase of `tiles` tiles and U units:
// every participating span is non-empty, and at least U / (seg_cap * tiles)
// units long, so that a tile has at most seg_cap + 1 segments.
// Counter words of the workspace (zeroed at each frame's start): two banks of
// two words per GEMM tile (1024 tiles at most; consecutive projections with
// no grid barrier between them use different banks), the gate/up tiles'
// done flags, then one attention work counter per layer (1024 layers at most).
constexpr int kTileCntWords = 2048;
constexpr int kDoneCntOff = 2 * kTileCntWords;   // per projection kind: tiles finished so far this frame
constexpr int kHeadsDone = 8;                    // done_cnt[8]: heads whose attention rows are all written
constexpr int kNormRows = 9;                     // done_cnt[9]: RMSNorm rows written this frame
constexpr int kSsmDone = 10;                     // done_cnt[10]: selective-state items finished this frame
constexpr int kQkvDoneOff = kDoneCntOff + 32;
constexpr int kHeadCntOff = kQkvDoneOff + 1024;  // per head: (session, head) rows written this frame
constexpr int kAttCtrOff = kHeadCntOff + 1024;
constexpr int kCounterWords = kAttCtrOff + 1024;
// The bank of a projection's counters and partial slots.
__host__ __device__ inline int gemm_bank(int kind) { return (kind == kO || kind == kDown || kind == kOut) ? 1 : 0; }
// Frames one launch may run back to back (wave_beat).
constexpr int kMaxFrames = 64;

__host__ __device__ inline int stream_k_ctas(int grid, long long U, int tiles, int seg_cap) {
  long long g = grid;
  if (U < g) g = U;
  if ((long long)seg_cap * tiles < g) g = (long long)seg_cap * tiles;
  return (int)g;
}
// Segments per tile at most: a tile split many ways (small models) pays one
// L2 round trip per pair of segments in its reduction, more than the extra
// streaming a few CTAs more per tile would save; the depth loop's W_p, at ~4.
__host__ __device__ inline int gemm_seg_cap(int kind) { return kind == kProj ? 4 : 8; }
// Element offset of layer l in a hybrid blob (groups of attn_every layers:
// attn_every - 1 Mamba blocks, then the attention block).
__host__ __device__ inline long long hyb_layer_offset(long long M, long long G, int e, int l) {
  return (long long)(l / e) * G + (long long)(l % e) * M;
}

// Host-side launch (step.cu).
cudaError_t launch_step(const StepParams& p, int grid, cudaStream_t stream);
cudaError_t configure_step_kernel();
cudaError_t occupancy_per_sm(int* blocks);
int barriers_per_step(int L, int T_max);  // of the decoder kernel without the dump hook
int phases_per_step(int L, bool hybrid, int attn_every);
int barriers_per_launch(int L, int T_max, int frames, bool advance, bool depth);
int hybrid_barriers_per_step(int L, int attn_every, int T_max);
// Dynamic shared memory layout shared by host checks and the kernel.
struct SmemLayout {
  int ring_off, ring_bytes;      // attention K and V tiles / state blocks / norm rows (union)
  int gemm_ring_bytes;           // the GEMM ring: ring, attention scales, prologue scratch and
                                 // query scratch together (none of those is live in a GEMM phase)
  int ascale_off;                // attention K/V scales: kWarps x 2 x kScaleBufBytes
  int xbuf_off;                  // prologue scratch (work-list positions), 4352 B
  int qscr_off;                  // per-warp query scratch (kWarps x 512 B)
  int red_off;                   // reduction scratch (256 words)
  int bar_off;                   // mbarriers
  int misc_off;                  // tmem address, flags
  int total;
};
__host__ __device__ inline SmemLayout smem_layout() {
  SmemLayout s;
  s.ring_off = 0;
  s.ring_bytes = 200 * 1024;
  s.ascale_off = s.ring_off + s.ring_bytes;
  s.xbuf_off = s.ascale_off + kWarps * 2 * kScaleBufBytes;  // 16 KB
  s.qscr_off = s.xbuf_off + 64 * 17 * 4;             // 3 KB: q as f16 hi + lo per warp
  s.red_off = s.qscr_off + kWarps * 512;             // 1 KB: one int per thread
  s.bar_off = s.red_off + 1024;                      // 64 mbarriers
  s.misc_off = s.bar_off + 64 * 8;
  s.total = s.misc_off + 64 + 1024;                  // + alignment slack
  s.gemm_ring_bytes = s.red_off - s.ring_off;
  return s;
}
// Bytes of one GEMM ring stage at S_pad sessions: kKStage weight boxes
// (128 rows x 128 B) and kKStage activation boxes (S_pad rows x 128 B, each
// padded to the 1024-byte swizzle atom).
__host__ __device__ inline int gemm_act_box_stride(int S_pad) { return (S_pad * 128 + 1023) & ~1023; }
__host__ __device__ inline int gemm_stage_bytes(int S_pad) {
  return kKStage * (16384 + gemm_act_box_stride(S_pad));
}
__host__ __device__ inline int attn_stage_bytes(int D) {  // K tile + V tile (scales live apart)
  return 2 * kChunk * D;
}

}  // namespace wave
