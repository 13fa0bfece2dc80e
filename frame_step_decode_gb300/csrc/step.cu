// step.cu -- the persistent frame-step kernel: one cooperative launch runs
// every layer for all S sessions, with no CPU round trip between operations
// (dotwave.ai case study, "02 / The solution" and "04 / Under the hood").
// One grid barrier per frame (after its prologue); every other hand-over
// between phases is a bounded wait on a count or flag in global memory, for
// exactly the data the next phase reads.
//
// Decoder layer l:
//   norm     RMSNorm rows of the fp32 residual -> bf16 xn           (CUDA cores)
//   QKV      xn . Wqkv^T -> fp32 q,k,v                              (tcgen05, stream-K)
//   attn     per (session, head) piece: RoPE(q); the piece holding the
//            current slot also RoPEs k, quantises k and v to E4M3 and
//            appends them at slot pos; then split-T flash-decode over the
//            FP8 history (mma.sync f16 with in-register dequantisation);
//            the warp finishing a split pair's last piece merges its
//            partials -> bf16 attention output                 (TMA + mma.sync)
//   O        resid += attn . Wo^T                                  (tcgen05, stream-K)
//   norm     RMSNorm -> xn
//   GU       u = bf16(silu(xn . Wg^T) * (xn . Wu^T))               (tcgen05, stream-K)
//   down     resid += u . Wdown^T (y = bf16(resid) after the last layer)
// Around the layers: a prologue (work list, residual from x, first norm);
// several frames per launch (beats) with positions + f; chained frames (the
// depth loop) with x_f = bf16(W_p y_{f-1}) between them.  The hybrid model
// (step_kernel<true, ...>) replaces the MLP half by nothing and, in all but every
// attn_every-th layer, attention by a selective-state block: in-projection,
// state update, out-projection + residual.
//
// Roles inside the 8-warp CTA during GEMM phases: warp 0 issues TMA loads of
// weight/activation tiles into a shared-memory ring, warp 1 issues tcgen05
// MMAs into a double-buffered TMEM accumulator, warps 2..5 drain TMEM into
// split-K partial slots; the split tile a CTA's span ends in is then summed
// by all its threads.  Attention, the norms and the state update use all 8
// warps.  Every wait is bounded (globaltimer) and reports WAVE_ETIMEOUT
// through the device error word instead of hanging.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "fp8.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace wave {

struct Ctx {
  uint8_t* smem;
  uint32_t sbase;       // shared-space address of smem
  uint32_t tmem;        // TMEM base address of the two accumulators
  unsigned bar_target;  // thread 0: next grid-barrier target
  int bar_index;
  uint32_t ring_it;     // GEMM ring stage counter (producer and MMA threads)
  uint32_t acc_it;      // accumulator counter (MMA and epilogue threads)
  uint32_t att_it;      // attention chunk counter (per warp)
  uint32_t norm_it;     // norm-row copy counter (all threads)
  int frame;            // frame of the launch being computed
  uint32_t ssm_it;      // state-block copy counter (all threads)
  SmemLayout lay;
};

// mbarrier slots (byte offsets from bar_off)
__device__ __forceinline__ uint32_t bar_full(const Ctx& c, int i) { return c.sbase + c.lay.bar_off + 8 * i; }
__device__ __forceinline__ uint32_t bar_empty(const Ctx& c, int i) { return c.sbase + c.lay.bar_off + 64 + 8 * i; }
__device__ __forceinline__ uint32_t bar_accf(const Ctx& c, int i) { return c.sbase + c.lay.bar_off + 128 + 8 * i; }
__device__ __forceinline__ uint32_t bar_acce(const Ctx& c, int i) { return c.sbase + c.lay.bar_off + 144 + 8 * i; }
__device__ __forceinline__ uint32_t bar_att(const Ctx& c, int w, int st) {
  return c.sbase + c.lay.bar_off + 160 + 8 * (w * kAttStages + st);
}
__device__ __forceinline__ uint32_t bar_drain(const Ctx& c) {
  return c.sbase + c.lay.bar_off + 160 + 8 * kWarps * kAttStages;
}
__device__ __forceinline__ uint32_t bar_norm(const Ctx& c) {
  return c.sbase + c.lay.bar_off + 168 + 8 * kWarps * kAttStages;
}
__device__ __forceinline__ uint32_t bar_ssm(const Ctx& c, int i) {
  return c.sbase + c.lay.bar_off + 176 + 8 * kWarps * kAttStages + 8 * i;
}
static_assert(176 + 8 * kWarps * kAttStages + 8 * kSsmStages <= 64 * 8, "mbarrier slots exceed their region");
static_assert(kAttStages <= kScaleGroup, "a scale buffer would be refilled before its last chunk is read");
static_assert(kSsmStages * (kSsmP * kSsmN + 512) * 4 <= 200 * 1024, "state stages exceed the ring");
__device__ __forceinline__ volatile int* misc_word(const Ctx& c, int i) {
  return (volatile int*)(c.smem + c.lay.misc_off + 4 * i);
}

// Profiling hook: this CTA has finished its next phase (call with the CTA's
// threads past the phase); the mark count is a shared-memory word.
__device__ __forceinline__ void mark_phase(const StepParams& p, const Ctx& c) {
  if (p.arrive_ts && threadIdx.x == 0) {
    const int m = (*misc_word(c, 8))++;
    p.arrive_ts[(size_t)m * gridDim.x + blockIdx.x] = globaltimer();
  }
}

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void set_err(const StepParams& p, int bits) { atomicOr(p.err, bits); }
__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Wait (bounded) until *f >= v, the flag written with st_release by another
// CTA; false if the wait gave up (timeout here or elsewhere).
__device__ __noinline__ bool wait_flag_ge(const StepParams& p, const int* f, int v) {
  if ((int)ld_acquire((const unsigned*)f) >= v) return true;
  const long long t0 = globaltimer();
  for (uint32_t it = 0;; ++it) {
    if ((int)ld_acquire((const unsigned*)f) >= v) return true;
    if ((it & 15) == 15) {
      if (*(volatile int*)p.err & kErrTimeout) return false;
      if (globaltimer() - t0 > p.timeout_ns) {
        set_err(p, kErrTimeout);
        return false;
      }
    }
  }
}
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// The same wait with a smaller footprint, for call sites under register
// pressure: bounded by a spin count that approximates the timeout.
__device__ __forceinline__ bool wait_flag_ge_light(const StepParams& p, const int* f, int v) {
  const uint32_t max_it = (uint32_t)min(p.timeout_ns / 128, 0x7fffffffLL) + 1u;
  for (uint32_t it = 0; it < max_it; ++it) {
    if ((int)ld_acquire((const unsigned*)f) >= v) return true;
    __nanosleep(128);
    if ((it & 63) == 63 && (*(volatile int*)p.err & kErrTimeout)) return false;
  }
  set_err(p, kErrTimeout);
  return false;
}

// What a testing hook may withhold (wave_debug_skip_signal's `which`).
enum SigKind : int {
  kSigQkv = 0, kSigGu = 1, kSigAttn = 2, kSigO = 3, kSigDown = 4, kSigNorm = 5,
  kSigIn = 6, kSigSsm = 7, kSigOut = 8  // the hybrid's selective-state blocks
};
__device__ __forceinline__ int sig_of(int kind) {
  return kind == kQKV ? kSigQkv : kind == kGU ? kSigGu : kind == kO ? kSigO : kind == kDown ? kSigDown
       : kind == kIn ? kSigIn : kind == kOut ? kSigOut : -1;
}

// Projections whose next phase starts without a grid barrier publish every
// finished tile: the QKV tiles one flag each (attention waits for its
// head's tiles), both a count of finished tiles (gate/up: the down
// projection waits for the count to cover every tile).
__device__ __forceinline__ bool publishes(int kind) { return kind != kProj; }
__device__ __forceinline__ void publish_tile(const StepParams& p, int kind, int t, int layer) {
  if (kind == kQKV) st_release(p.qkv_done + t, layer + 1);
  atomicAdd(p.done_cnt + kind, 1);  // after the release (or the fence before it)
}

// ------------------------------------------------------------- grid barrier
// All CTAs arrive on one counter (zeroed before the launch) and wait until it
// reaches (barrier index + 1) * grid.  Every thread's generic writes are made
// visible to the async proxy first (the next phase reads some of them by TMA)
// and released with the arrival; the waiting thread's acquire load orders the
// next phase after the other CTAs' writes.  The wait gives up after
// timeout_ns or when another CTA has recorded an error.
__device__ bool grid_sync(const StepParams& p, Ctx& c) {
  fence_proxy_async_global();
  fence_proxy_async_smem();  // this phase's generic shared accesses before the next one's copies
  __syncthreads();
  if (threadIdx.x == 0) {
    c.bar_target += gridDim.x;
    __threadfence();
    bool skip = ((int)blockIdx.x == p.skip_cta && c.bar_index == p.skip_bar);
    if (!skip) atomicAdd(p.bar, 1u);
    int ok = 1;
    long long t0 = globaltimer();
    for (uint32_t it = 0;; ++it) {
      unsigned v = ld_acquire(p.bar);
      if ((int)(v - c.bar_target) >= 0) break;
      if (*(volatile int*)p.err & kErrTimeout) { ok = 0; break; }
      if ((it & 15) == 15 && globaltimer() - t0 > p.timeout_ns) {
        set_err(p, kErrTimeout);
        ok = 0;
        break;
      }
    }
    *misc_word(c, 2) = ok;  // the acquire load above orders what follows
    if (p.phase_ts && blockIdx.x == 0) p.phase_ts[1 + c.bar_index] = globaltimer();
  }
  c.bar_index++;
  __syncthreads();
  return *misc_word(c, 2) != 0;
}

// ------------------------------------------------------------------- norm
// xn[s] = bf16(r * rstd * g), rstd = 1/sqrt(mean(r^2) + eps); one row per CTA
// (rows strided over CTAs).  One thread bulk-copies the residual row (at
// layer 0 the bf16 input row x) and g into the idle GEMM ring, so that the
// whole row arrives in one round trip with no register staging, then the
// block reduces the sum of squares and writes xn.  Returns false if the copy
// wait gave up.
// wait_cnt / wait_target: the residual rows are final once *wait_cnt (the
// producing projection's finished-tile count) reaches wait_target (null: a
// grid barrier came before).  With publish, every row written adds one to
// the norm-rows count the next projection waits for (the frame's first norm
// runs before a grid barrier and before the counts are zeroed, and does not).
__device__ bool norm_phase(const StepParams& p, Ctx& c, const uint16_t* g, bool from_x, bool publish,
                           const int* wait_cnt = nullptr, int wait_target = 0) {
  float* red = (float*)(c.smem + c.lay.red_off);
  if (wait_cnt && (int)blockIdx.x < p.S) {
    if (threadIdx.x == 0) {
      const bool ok0 = wait_flag_ge(p, wait_cnt, wait_target);
      fence_proxy_async_global();  // the row copies below come after those tiles' writes
      *misc_word(c, 6) = ok0 ? 1 : 0;
    }
    __syncthreads();
    if (!*misc_word(c, 6)) return false;
  }
  const int d = p.d, d4 = d / 4, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float* rrow = (float*)(c.smem + c.lay.ring_off);                       // d fp32
  const uint16_t* grow = (const uint16_t*)(c.smem + c.lay.ring_off + 4 * d);  // d bf16
  const uint16_t* xrow = (const uint16_t*)(c.smem + c.lay.ring_off + 6 * d);  // d bf16 (layer 0)
  const uint32_t nbar = bar_norm(c);
  for (int s = blockIdx.x; s < p.S; s += gridDim.x) {
    if (tid == 0) {
      fence_proxy_async_smem();  // earlier generic accesses to this area come first
      mbar_arrive_expect_tx(nbar, (from_x ? 4u : 6u) * (uint32_t)d);  // row + g
      if (from_x)
        bulk_load(c.sbase + c.lay.ring_off + 6 * d, p.x + ((size_t)c.frame * p.S + s) * d, 2u * d, nbar);
      else
        bulk_load(c.sbase + c.lay.ring_off, p.resid + (size_t)s * d, 4u * d, nbar);
      bulk_load(c.sbase + c.lay.ring_off + 4 * d, g, 2u * d, nbar);
    }
    // one thread waits (bounded) and the block takes its decision
    if (tid == 0) {
      const bool ok0 = mbar_wait(nbar, c.norm_it & 1u, p.timeout_ns, p.err);
      if (!ok0) set_err(p, kErrTimeout);
      *misc_word(c, 6) = ok0 ? 1 : 0;
    }
    c.norm_it++;
    __syncthreads();
    if (!*misc_word(c, 6)) return false;
    float ss = 0.f;
#pragma unroll 1
    for (int i4 = tid; i4 < d4; i4 += kThreads) {
      float4 v;
      if (from_x) {
        const uint2 xb = *(const uint2*)(xrow + 4 * i4);
        v = make_float4(bf16_to_f32((uint16_t)(xb.x & 0xFFFF)), bf16_to_f32((uint16_t)(xb.x >> 16)),
                        bf16_to_f32((uint16_t)(xb.y & 0xFFFF)), bf16_to_f32((uint16_t)(xb.y >> 16)));
        ((float4*)rrow)[i4] = v;
        ((float4*)(p.resid + (size_t)s * d))[i4] = v;
      } else {
        v = ((const float4*)rrow)[i4];
      }
      ss = fmaf(v.x, v.x, ss);
      ss = fmaf(v.y, v.y, ss);
      ss = fmaf(v.z, v.z, ss);
      ss = fmaf(v.w, v.w, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) tot += red[w];
    const float rstd = 1.0f / sqrtf(tot / (float)d + p.eps);
#pragma unroll 1
    for (int i4 = tid; i4 < d4; i4 += kThreads) {
      const float4 v = ((const float4*)rrow)[i4];
      const uint2 gb = *(const uint2*)(grow + 4 * i4);
      const float g0 = bf16_to_f32((uint16_t)(gb.x & 0xFFFF)), g1 = bf16_to_f32((uint16_t)(gb.x >> 16));
      const float g2 = bf16_to_f32((uint16_t)(gb.y & 0xFFFF)), g3 = bf16_to_f32((uint16_t)(gb.y >> 16));
      uint2 o;
      o.x = (uint32_t)f32_to_bf16((v.x * rstd) * g0) | ((uint32_t)f32_to_bf16((v.y * rstd) * g1) << 16);
      o.y = (uint32_t)f32_to_bf16((v.z * rstd) * g2) | ((uint32_t)f32_to_bf16((v.w * rstd) * g3) << 16);
      *(uint2*)(p.xn + (size_t)s * d + 4 * i4) = o;
    }
    fence_proxy_async_global();  // the next projection reads xn by TMA
    __syncthreads();
    if (publish && threadIdx.x == 0 && !(p.skip_sig == s && p.skip_sig_kind == kSigNorm)) {
      __threadfence();
      atomicAdd(p.done_cnt + kNormRows, 1);
    }
  }
  fence_proxy_async_smem();  // the next phase's copies overwrite this area
  return true;
}

// ------------------------------------------------------------ GEMM (tcgen05)
struct Span { long long u0, u1; };
__device__ __forceinline__ Span cta_span(long long U, int G, int c) {
  return Span{U * c / G, U * (c + 1) / G};
}
// Last CTA whose span starts at or before unit u (the owner of u).
__device__ __forceinline__ int owner_of(long long U, int G, long long u) {
  return (int)(((u + 1) * G + U - 1) / U - 1);
}


__device__ __forceinline__ float4 ld4cg(const float* q) { return __ldcg((const float4*)q); }
__device__ __forceinline__ void add4(float4& a, const float4& b) {
  a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
}
// Sum, in segment order, of the float4 at element offsets o[0..NI) of each
// of a tile's partial slots (the first at `first`, the others at part +
// seg[1..nseg)); the NI loads of a segment in flight together.  kOne: the
// tile has one segment (no partner slots).
template <bool kOne, int NI>
__device__ __forceinline__ void seg_sumn(const float* first, const float* part, const long long* seg, int nseg,
                                         const size_t* o, float4* a) {
#pragma unroll
  for (int k = 0; k < NI; ++k) a[k] = __ldcg((const float4*)(first + o[k]));
  if constexpr (!kOne) {
    for (int j = 1; j < nseg; ++j) {
      const float* bk = part + seg[j];
      float4 tv[NI];
#pragma unroll
      for (int k = 0; k < NI; ++k) tv[k] = __ldcg((const float4*)(bk + o[k]));
#pragma unroll
      for (int k = 0; k < NI; ++k) add4(a[k], tv[k]);
    }
  }
}
// The same for four offsets passed one by one.
template <bool kOne>
__device__ __forceinline__ void seg_sum4(const float* first, const float* part, const long long* seg,
                                         int nseg, size_t o0, size_t o1, size_t o2, size_t o3,
                                         float4& a0, float4& a1, float4& a2, float4& a3) {
  a0 = ld4cg(first + o0); a1 = ld4cg(first + o1); a2 = ld4cg(first + o2); a3 = ld4cg(first + o3);
  if constexpr (!kOne) {
    for (int j = 1; j < nseg; ++j) {
      const float* bk = part + seg[j];
      const float4 t0 = ld4cg(bk + o0), t1 = ld4cg(bk + o1), t2 = ld4cg(bk + o2), t3 = ld4cg(bk + o3);
      add4(a0, t0); add4(a1, t1); add4(a2, t2); add4(a3, t3);
    }
  }
}
__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }
// u[n..n+3] = bf16(silu(gate) * up) for one session row (F % 4 == 0).
__device__ __forceinline__ void swiglu_store(uint16_t* urow, int n, int F, const float4& g, const float4& u) {
  if (n >= F) return;
  uint2 o;
  o.x = (uint32_t)f32_to_bf16(silu_mul(g.x, u.x)) | ((uint32_t)f32_to_bf16(silu_mul(g.y, u.y)) << 16);
  o.y = (uint32_t)f32_to_bf16(silu_mul(g.z, u.z)) | ((uint32_t)f32_to_bf16(silu_mul(g.w, u.w)) << 16);
  *(uint2*)(urow + n) = o;
}
// resid[s][n..n+3] = old + v (and y = bf16 of it after the last layer; an
// empty slot, negative position, passes x through unchanged).
__device__ __forceinline__ void resid_store(const StepParams& p, int s, int n, float4 old, const float4& v,
                                            bool last_layer, int frame) {
  add4(old, v);
  *(float4*)(p.resid + (size_t)s * p.d + n) = old;
  if (last_layer) {
    const size_t at = ((size_t)frame * p.S + s) * p.d + n;
    uint2 o;
    if (p.pos[s] < 0) {
      o = *(const uint2*)(p.x + at);
    } else {
      o.x = (uint32_t)f32_to_bf16(old.x) | ((uint32_t)f32_to_bf16(old.y) << 16);
      o.y = (uint32_t)f32_to_bf16(old.z) | ((uint32_t)f32_to_bf16(old.w) << 16);
    }
    *(uint2*)(p.y + at) = o;
  }
}

// Finish tile t of GEMM `kind` from its partial sums: the first segment's
// slot at `first`, the others at part + seg[1..nseg), summed in segment order.
// Flat float4 items over the valid columns; this thread takes items et,
// et + step, ...
template <bool kOne>
__device__ __forceinline__ void finish_tile(const StepParams& p, int kind, int t, const float* first,
                                         const float* part, const long long* seg, int nseg, int et, int step,
                                         bool last_layer, int frame) {
  if (kind == kGU) {
    // item (s, r4): gate rows 4r4..4r4+3 and the up rows 64 below them; five
    // items per pass, their ten loads per segment in flight together
    constexpr int GI = 5;
    const int F = p.F, items = p.S * 16;
#pragma unroll 1
    for (int i0 = et; i0 < items; i0 += GI * step) {
      int iv[GI];
      size_t ov[2 * GI];
#pragma unroll
      for (int k = 0; k < GI; ++k) {
        iv[k] = (i0 + k * step < items) ? i0 + k * step : i0;
        ov[k] = (size_t)(iv[k] >> 4) * kTileM + 4 * (iv[k] & 15);
        ov[GI + k] = ov[k] + 64;
      }
      float4 a[2 * GI];
      seg_sumn<kOne, 2 * GI>(first, part, seg, nseg, ov, a);
#pragma unroll
      for (int k = 0; k < GI; ++k)
        if (k == 0 || iv[k] != i0)
          swiglu_store(p.u + (size_t)(iv[k] >> 4) * F, t * 64 + 4 * (iv[k] & 15), F, a[k], a[GI + k]);
    }
  } else if (kind == kProj) {
    // item (s, r4): the next frame's input x[frame][s][n..n+3] in bf16; four items per pass
    const int d = p.d, items = p.S * 32;
#pragma unroll 1
    for (int i0 = et; i0 < items; i0 += 4 * step) {
      int iv[4];
      size_t ov[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        iv[k] = (i0 + k * step < items) ? i0 + k * step : i0;
        ov[k] = (size_t)(iv[k] >> 5) * kTileM + 4 * (iv[k] & 31);
      }
      float4 a[4];
      seg_sum4<kOne>(first, part, seg, nseg, ov[0], ov[1], ov[2], ov[3], a[0], a[1], a[2], a[3]);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int n = t * kTileM + 4 * (iv[k] & 31);
        if ((k == 0 || iv[k] != i0) && n < d) {
          uint2 o;
          o.x = (uint32_t)f32_to_bf16(a[k].x) | ((uint32_t)f32_to_bf16(a[k].y) << 16);
          o.y = (uint32_t)f32_to_bf16(a[k].z) | ((uint32_t)f32_to_bf16(a[k].w) << 16);
          *(uint2*)(p.x_chain + ((size_t)frame * p.S + (iv[k] >> 5)) * d + n) = o;
        }
      }
    }
  } else if (kind == kQKV || kind == kIn) {
    // item (s, r4): output rows 4r4..4r4+3 of the tile (fp32); five items per
    // pass (two passes for a tile finished by one CTA at S = 80)
    constexpr int QI = 5;
    const int N = (kind == kQKV) ? 3 * p.HD : p.in_rows, items = p.S * 32;
    float* dst = (kind == kQKV) ? p.qkv : p.zx;
#pragma unroll 1
    for (int i0 = et; i0 < items; i0 += QI * step) {
      int iv[QI];
      size_t ov[QI];
#pragma unroll
      for (int k = 0; k < QI; ++k) {
        iv[k] = (i0 + k * step < items) ? i0 + k * step : i0;
        ov[k] = (size_t)(iv[k] >> 5) * kTileM + 4 * (iv[k] & 31);
      }
      float4 a[QI];
      seg_sumn<kOne, QI>(first, part, seg, nseg, ov, a);
#pragma unroll
      for (int k = 0; k < QI; ++k) {
        const int n = t * kTileM + 4 * (iv[k] & 31);
        if ((k == 0 || iv[k] != i0) && n < N) *(float4*)(dst + (size_t)(iv[k] >> 5) * N + n) = a[k];
      }
    }
  } else {
    // item (s, r4): output rows 4r4..4r4+3 of the tile, residual added; four
    // items per pass, their old values' and partials' loads in flight together
    const int d = p.d, items = p.S * 32;
#pragma unroll 1
    for (int i0 = et; i0 < items; i0 += 4 * step) {
      int iv[4], nv[4];
      size_t ov[4];
      float4 old[4], a[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        iv[k] = (i0 + k * step < items) ? i0 + k * step : i0;
        nv[k] = t * kTileM + 4 * (iv[k] & 31);
        ov[k] = (size_t)(iv[k] >> 5) * kTileM + 4 * (iv[k] & 31);
        old[k] = (nv[k] < d) ? __ldcg((const float4*)(p.resid + (size_t)(iv[k] >> 5) * d + nv[k]))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      seg_sum4<kOne>(first, part, seg, nseg, ov[0], ov[1], ov[2], ov[3], a[0], a[1], a[2], a[3]);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if ((k == 0 || iv[k] != i0) && nv[k] < d) resid_store(p, iv[k] >> 5, nv[k], old[k], a[k], last_layer, frame);
    }
  }
}

// wait_cnt / wait_target: the activations this projection reads are final
// once *wait_cnt reaches wait_target (the norm-rows count, the gate/up tile
// count, the heads-done count; null: a grid barrier came before).  The
// producer issues the first ring of weights before it waits.
__device__ void gemm_phase(const StepParams& p, Ctx& c, int kind, int layer, bool last_layer,
                           const int* wait_cnt = nullptr, int wait_target = 0) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = p.kblocks[kind];
  const long long U = (long long)p.tiles[kind] * KB;
  // Split over min(grid, units, seg_cap * tiles) CTAs: every participating
  // span is non-empty, the owners of a tile's units are consecutive CTAs, and
  // a tile has at most seg_cap + 1 segments (the plan checks 64, the size of
  // the reduction's segment table).
  const int G = stream_k_ctas(gridDim.x, U, p.tiles[kind], gemm_seg_cap(kind)), cta = blockIdx.x;
  const Span sp = (cta < G) ? cta_span(U, G, cta) : Span{0, 0};
  const int S_pad = p.S_pad, nst = p.nstage;
  // a stage: kKStage weight boxes, then kKStage activation boxes
  const uint32_t b_bytes = (uint32_t)S_pad * 128u;
  const uint32_t b_stride = (uint32_t)gemm_act_box_stride(S_pad);
  const uint32_t stride = (uint32_t)gemm_stage_bytes(S_pad);
  const uint32_t ring = c.sbase + c.lay.ring_off;

  // The stream-K span as units (t, kb); weights have no input dependency,
  // the activations may still be being written by other CTAs (no grid
  // barrier between the phases).
  const bool wait_inputs = wait_cnt != nullptr;
  int* const cnt = p.tile_cnt + gemm_bank(kind) * kTileCntWords;
  float* const part = p.gemm_part + (size_t)gemm_bank(kind) * (size_t)p.part_bank;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const CUtensorMap* wm = &p.tm_w[kind];
      const CUtensorMap* xm = &p.tm_x[kind];
      // the projection between chained frames reads the previous frame's y rows
      const int xrow0 = (kind == kProj) ? (c.frame - 1) * p.S : 0;
      // weights: unit (t, kb) of a packed matrix is two contiguous 16 KB
      // blocks (128 rows x 64 K each, the ragged edges zero-filled by the
      // packing); the projection between chained frames reads W_p as a plain
      // [d][d] matrix instead
      auto load_w = [&](uint32_t a, uint32_t fb, int t, int kb) {
#pragma unroll
        for (int bx = 0; bx < kKStage; ++bx) {
          const uint32_t wa = a + (uint32_t)bx * 16384u;
          const int row = ((t * KB + kb) * kKStage + bx) * kTileM;
          if (kind == kProj) {
            tma_load_3d(wa, wm, (kb * kKStage + bx) * kKBlk, t * kTileM, 0, fb, pol);
          } else if (kind == kIn || kind == kOut) {  // hybrid Mamba blocks: (place in group, group)
            tma_load_4d(wa, wm, 0, row, layer % p.attn_every, layer / p.attn_every, fb, pol);
          } else {
            tma_load_3d(wa, wm, 0, row, layer, fb, pol);
          }
        }
      };
      auto load_x = [&](uint32_t a, uint32_t fb, int kb) {
#pragma unroll
        for (int bx = 0; bx < kKStage; ++bx)
          tma_load_2d(a + (uint32_t)kKStage * 16384u + (uint32_t)bx * b_stride, xm, (kb * kKStage + bx) * kKBlk,
                      xrow0, fb);
      };
      bool fail = false;
      // with inputs to wait for, the first ring's worth of weights is issued
      // before the first wait, so that it streams while other CTAs finish
      const long long n_pre = wait_inputs ? min((long long)nst, sp.u1 - sp.u0) : 0;
      const uint32_t it0 = c.ring_it;
      long long n_w = 0;  // units of the first ring whose weights are issued
      for (; n_w < n_pre; ++n_w) {
        const long long u = sp.u0 + n_w;
        const uint32_t it = it0 + (uint32_t)n_w, slot = it % nst;
        if (!mbar_wait(bar_empty(c, slot), ((it / nst) & 1u) ^ 1u, p.timeout_ns, p.err)) {
          set_err(p, kErrTimeout);
          fail = true;
          break;
        }
        mbar_arrive_expect_tx(bar_full(c, slot), (uint32_t)kKStage * (16384u + b_bytes));
        load_w(ring + slot * stride, bar_full(c, slot), (int)(u / KB), (int)(u % KB));
      }
      // every gate/up tile of this layer is done (one count; they finish
      // together), then the activation boxes of the first ring
      if (!fail && wait_inputs) {
        fail = !wait_flag_ge(p, wait_cnt, wait_target);
        fence_proxy_async_global();  // the TMA reads below come after those rows' writes
      }
      for (long long i = 0; !fail && i < n_pre; ++i) {
        const long long u = sp.u0 + i;
        const uint32_t slot = (it0 + (uint32_t)i) % nst;
        load_x(ring + slot * stride, bar_full(c, slot), (int)(u % KB));
      }
      c.ring_it = it0 + (uint32_t)n_w;
      for (long long u = sp.u0 + n_pre; !fail && u < sp.u1; ++u) {
        const int t = (int)(u / KB), kb = (int)(u % KB);
        const uint32_t slot = c.ring_it % nst, ph = (c.ring_it / nst) & 1u;
        if (!mbar_wait(bar_empty(c, slot), ph ^ 1u, p.timeout_ns, p.err)) {
          set_err(p, kErrTimeout);
          fail = true;
          break;
        }
        const uint32_t fb = bar_full(c, slot);
        mbar_arrive_expect_tx(fb, (uint32_t)kKStage * (16384u + b_bytes));
        const uint32_t a = ring + slot * stride;
        load_w(a, fb, t, kb);
        load_x(a, fb, kb);
        c.ring_it++;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kTileM, S_pad);
      bool fail = false;
      for (long long u = sp.u0; !fail && u < sp.u1;) {
        const int t = (int)(u / KB);
        const long long e = min(sp.u1, (long long)(t + 1) * KB);
        const uint32_t b = c.acc_it & 1u;
        if (!mbar_wait(bar_acce(c, b), ((c.acc_it >> 1) & 1u) ^ 1u, p.timeout_ns, p.err)) {
          set_err(p, kErrTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t dt = c.tmem + b * 128u;
        const int k0 = (int)(u - (long long)t * KB), k1 = (int)(e - (long long)t * KB);
        for (int kb = k0; kb < k1; ++kb) {
          const uint32_t slot = c.ring_it % nst, ph = (c.ring_it / nst) & 1u;
          if (!mbar_wait(bar_full(c, slot), ph, p.timeout_ns, p.err)) {
            set_err(p, kErrTimeout);
            fail = true;
            break;
          }
          tc_fence_after();
          const uint32_t a = ring + slot * stride, bs = a + (uint32_t)kKStage * 16384u;
#pragma unroll
          for (int kk = 0; kk < 4 * kKStage; ++kk) {
            const uint32_t bx = (uint32_t)kk >> 2, off = (uint32_t)(kk & 3) * 32u;
            tc_mma_bf16(dt, sdesc_sw128(a + bx * 16384u + off), sdesc_sw128(bs + bx * b_stride + off), idesc,
                        (kb > k0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(bar_empty(c, slot));
          c.ring_it++;
        }
        if (fail) break;
        tc_commit(bar_accf(c, b));
        c.acc_it++;
        u = e;
      }
    }
    __syncwarp();
  } else if (warp >= 6) {
    // idle during GEMMs
  } else {
    const int q = warp & 3, r = q * 32 + lane;
    const int MT = p.max_tiles_per_cta;
    const int first_tile = (int)(sp.u0 / KB);
    for (long long u = sp.u0; u < sp.u1;) {
      const int t = (int)(u / KB);
      const long long tb = (long long)t * KB, te = tb + KB;
      const long long e = min(sp.u1, te);
      const int nseg = owner_of(U, G, te - 1) - owner_of(U, G, tb) + 1;
      const uint32_t b = c.acc_it & 1u;
      // one thread waits, the four warps take the same decision
      volatile int* wflag = misc_word(c, 4 + (int)b);
      if (threadIdx.x == 64)
        *wflag = mbar_wait(bar_accf(c, b), (c.acc_it >> 1) & 1u, p.timeout_ns, p.err) ? 1 : 0;
      named_bar(1, 128);
      if (!*wflag) {
        if (threadIdx.x == 64) set_err(p, kErrTimeout);
        break;
      }
      tc_fence_after();
      const uint32_t tb_addr = c.tmem + ((uint32_t)(q * 32) << 16) + b * 128u;
      // Store this segment's sums as a partial slot ([column][128 rows] fp32).
      float* slot = part + ((size_t)cta * MT + (t - first_tile)) * (size_t)S_pad * kTileM;
      for (int col = 0; col < S_pad; col += 16) {
        float v[16];
        tmem_ld16(tb_addr + col, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) slot[(size_t)(col + i) * kTileM + r] = v[i];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_acce(c, b));
      if (nseg == 1) {
        // whole tile here: the four epilogue warps finish it from the slot
        named_bar(1, 128);
        finish_tile<true>(p, kind, t, slot, part, nullptr, 1, threadIdx.x - 64, 128, last_layer, c.frame);
        if (publishes(kind)) {  // publish the tile to the next phase
          fence_proxy_async_global();
          named_bar(1, 128);
          if (threadIdx.x == 64 && !(p.skip_sig == t && p.skip_sig_kind == sig_of(kind))) {
            __threadfence();
            publish_tile(p, kind, t, layer);
          }
        }
      } else {
        // split tile: count this segment in (one thread releases the four
        // warps' stores, which the named barrier orders before it)
        named_bar(1, 128);
        if (threadIdx.x == 64) {
          __threadfence();
          atomicAdd(cnt + t, 1);
        }
      }
      c.acc_it++;
      u = e;
    }
  }

  // Each CTA finishes the tile its span ends in, when that tile is split: once
  // every segment has arrived (bounded wait), the CTAs whose spans end inside
  // the tile (m of them) sum its partials in segment order, all threads taking
  // a share of the flat float4 items.
  __syncthreads();
  if (cta >= G) return;
  const int t = (int)((sp.u1 - 1) / KB);
  const long long tb = (long long)t * KB, te = tb + KB;
  const int c_first = owner_of(U, G, tb), c_last = owner_of(U, G, te - 1);
  const int nseg = c_last - c_first + 1;
  if (nseg == 1) return;
  const int m = (c_last - c_first) + (cta_span(U, G, c_last).u1 == te ? 1 : 0);
  const int idx = cta - c_first;
  const int MT = p.max_tiles_per_cta;
  long long* seg = (long long*)(c.smem + c.lay.red_off);  // partial-slot offsets (from part), segment order
  for (int j = threadIdx.x; j < nseg; j += kThreads) {
    const int cj = c_first + j;
    const int ftj = (int)(cta_span(U, G, cj).u0 / KB);
    seg[j] = ((long long)cj * MT + (t - ftj)) * (long long)S_pad * kTileM;
  }
  if (threadIdx.x == 0) {
    int ok = (*(volatile int*)p.err & kErrTimeout) ? 0 : 1;
    const long long t0 = globaltimer();
    for (uint32_t it = 0; ok; ++it) {
      if ((int)ld_acquire((const unsigned*)(cnt + t)) >= nseg) break;
      if ((it & 15) == 15) {
        if (*(volatile int*)p.err & kErrTimeout) { ok = 0; break; }
        if (globaltimer() - t0 > p.timeout_ns) {
          set_err(p, kErrTimeout);
          ok = 0;
          break;
        }
      }
    }
    *misc_word(c, 3) = ok;
  }
  __syncthreads();
  if (!*misc_word(c, 3)) return;
  finish_tile<false>(p, kind, t, part + seg[0], part, seg, nseg, idx * kThreads + threadIdx.x, m * kThreads,
              last_layer, c.frame);
  const bool pub = publishes(kind);
  if (pub) fence_proxy_async_global();  // the next phase may read these rows by TMA
  __syncthreads();
  // the last final contributor to finish re-arms the tile's counters (and
  // publishes the tile where the next phase waits for it: every
  // contributor's writes came before its count, so they come before that)
  if (threadIdx.x == 0) {
    if (pub) __threadfence();
    if (atomicAdd(cnt + 1024 + t, 1) == m - 1) {
      cnt[t] = 0;
      cnt[1024 + t] = 0;
      if (pub && !(p.skip_sig == t && p.skip_sig_kind == sig_of(kind))) publish_tile(p, kind, t, layer);
    }
  }
}

// --------------------------------------------------------------- merge
// Combine the split-T partials of one (session, head) cut into np pieces,
// in piece order: M = max m_i, L = sum l_i 2^(m_i - M), o = sum acc_i
// 2^(m_i - M) / L, written as bf16.  One warp, lane i owning dims
// [i*D/32, (i+1)*D/32); up to kMergeMax pieces' loads in flight at once.
// Run by the warp that finishes the (session, head)'s last piece.
constexpr int kMergeMax = 8;
template <int D>
__device__ __forceinline__ void merge_item(const StepParams& p, int first, int np, int s, int h, int lane) {
  constexpr int DPL = D / 32;
  float M = -INFINITY, Ls = 0.f, o[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) o[e] = 0.f;
  if (np > kMergeMax) {
    for (int i = 0; i < np; ++i) M = fmaxf(M, __ldcg(p.att_part + (size_t)(first + i) * (D + 4) + D));
  }
  for (int i0 = 0; i0 < np; i0 += kMergeMax) {
    float mv[kMergeMax], lv[kMergeMax], ov[kMergeMax][DPL];
#pragma unroll
    for (int i = 0; i < kMergeMax; ++i) {
      if (i0 + i < np) {
        const float* pp = p.att_part + (size_t)(first + i0 + i) * (D + 4);
        const float2 ml = __ldcg((const float2*)(pp + D));
        mv[i] = ml.x;
        lv[i] = ml.y;
#pragma unroll
        for (int e = 0; e < DPL; ++e) ov[i][e] = __ldcg(pp + lane * DPL + e);
      }
    }
    if (np <= kMergeMax) {
#pragma unroll
      for (int i = 0; i < kMergeMax; ++i)
        if (i < np) M = fmaxf(M, mv[i]);
    }
#pragma unroll
    for (int i = 0; i < kMergeMax; ++i) {
      if (i0 + i < np) {
        const float wgt = ex2(mv[i] - M);
        Ls += lv[i] * wgt;
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[e] += ov[i][e] * wgt;
      }
    }
  }
  const float inv = 1.0f / Ls;
  uint16_t* od = p.attn + (size_t)s * p.HD + h * D + lane * DPL;
#pragma unroll
  for (int e = 0; e < DPL; ++e) od[e] = f32_to_bf16(o[e] * inv);
}

// A (session, head)'s bf16 attention output is written (by this warp): count
// it for its head; the count that completes a head (every live session)
// adds one to the heads-done word the output projection waits for.
__device__ __forceinline__ void attn_row_done(const StepParams& p, int h, int la, int lane) {
  fence_proxy_async_global();  // the output projection reads these rows by TMA
  __syncwarp();
  if (lane == 0 && !(p.skip_sig == h && p.skip_sig_kind == kSigAttn)) {
    __threadfence();
    const int n_valid = __ldcg(p.n_pieces + 1);
    if (atomicAdd(p.head_cnt + h, 1) == (la + 1) * n_valid - 1) {
      __threadfence();
      atomicAdd(p.done_cnt + kHeadsDone, 1);
    }
  }
}

// ---------------------------------------------------------------- attention
// Byte offset inside a TMA tile written with the 128-byte (D = 128) or
// 64-byte (D = 64) swizzle: the 16-byte chunk index (address bits 4..6) is
// XORed with the 128-byte row index (bits 7..9), masked to the swizzle span.
template <int D>
__device__ __forceinline__ uint32_t swz(uint32_t off) {
  constexpr uint32_t m = (D == 128) ? 7u : 3u;
  return off ^ (((off >> 7) & m) << 4);
}

template <int D>
__device__ void attention_phase(const StepParams& p, Ctx& c, int layer) {
  constexpr int DPL = D / 32;    // dims per lane for row-wise work
  constexpr int KQB = D / 4;     // K bytes per lane per token (score mma)
  constexpr int KST = D / 16;    // k-steps of the score mma over the head dim
  constexpr int VB = D / 8;      // V bytes per lane per token (P.V mma)
  constexpr int MTV = D / 16;    // m-tiles of the P.V mma (16 head dims each)
  constexpr int kMT = kChunk / 16;  // 16-token tiles per chunk
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t4 = lane & 3;       // thread-in-group of the mma fragments
  const int g = lane >> 2;       // group of the mma fragments
  const int NW = gridDim.x * kWarps;
  const int gw = blockIdx.x * kWarps + warp;
  const int n_pieces = __ldcg(p.n_pieces);
  const int H = p.H, HD = p.HD;
  const int stage_bytes = attn_stage_bytes(D);
  uint8_t* wbuf = c.smem + c.lay.ring_off + warp * kAttStages * stage_bytes;
  const uint32_t wbuf_s = c.sbase + c.lay.ring_off + warp * kAttStages * stage_bytes;
  __half* qs_hi = (__half*)(c.smem + c.lay.qscr_off + warp * 512);
  __half* qs_lo = qs_hi + 128;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
  const uint64_t kv_policy = policy_evict_first();

  // Dynamic assignment over the longest-first list: warp gw starts with entry
  // gw, then takes the next unclaimed entry from the layer's counter.
  int* ctr = p.att_ctr + layer;
  for (int pi = gw; pi < n_pieces;) {
    const int4 pc = __ldcg(p.pieces + 2 * pi);
    const int P = __ldcg(p.pieces + 2 * pi + 1).x;
    const int sh = pc.x, c_lo = pc.y & 0xFFFF, c_hi = pc.y >> 16, np = pc.z, first = pc.w;
    const int s = sh / H, h = sh - s * H;
    const int nch = P / kChunk + 1;
    const bool tail = (c_hi == nch);
    const float* qrow = p.qkv + (size_t)s * 3 * HD + h * D;
    const float2* cs = p.rope + (size_t)P * (D / 2);
    const size_t rowK = ((((size_t)layer * 2 + 0) * p.S_max + s) * H + h) * (size_t)p.T_max;
    const size_t rowV = ((((size_t)layer * 2 + 1) * p.S_max + s) * H + h) * (size_t)p.T_max;
    // start the copies first: the q / k / v work below overlaps their latency
    const int n = c_hi - c_lo;
    auto issue = [&](int ci, int st) {
      const uint32_t base = wbuf_s + st * stage_bytes;
      const uint32_t fb = bar_att(c, warp, st);
      // one box holds the chunk's K tile then its V tile; the first chunk of
      // each group of kScaleGroup in the piece also brings the group's K and
      // V scales, into the warp's buffer (group & 1).  A buffer is refilled
      // two groups later, when the issue is kAttStages <= kScaleGroup chunks
      // ahead of a read that is already past the group it held.
      const int xrow = sh * p.T_max + ci * kChunk;
      const int gk = ci - c_lo;
      const bool grp = (gk % kScaleGroup) == 0;
      mbar_arrive_expect_tx(fb, 2u * kChunk * D + (grp ? (uint32_t)kScaleBufBytes : 0u));
      tma_load_4d(base, &p.tm_kv, 0, xrow, 0, layer, fb, kv_policy);
      if (grp) {
        const uint32_t sc_s = c.sbase + c.lay.ascale_off + (warp * 2 + (gk / kScaleGroup) % 2) * kScaleBufBytes;
        tma_load_3d(sc_s, &p.tm_sc, xrow, 0, layer, fb, kv_policy);
      }
    };
    if (lane == 0) {
      for (int k = 0; k < min(n, kAttStages); ++k) issue(c_lo + k, (c.att_it + k) % kAttStages);
    }
    __syncwarp();
    // q (and for the tail piece k and v) come from QKV tiles that other CTAs
    // may still be finishing (no grid barrier between the two phases): wait
    // for their readiness flags, lanes 0..2 one tile each in parallel, while
    // the chunk copies above are in flight
    bool aborted;
    {
      bool ready = true;
      if (lane < (tail ? 3 : 1)) ready = wait_flag_ge_light(p, p.qkv_done + (lane * HD + h * D) / kTileM, layer + 1);
      // the flags' acquire orders the q, k, v reads below for the whole warp
      aborted = __any_sync(0xffffffffu, !ready);
    }

    // RoPE of q (and k) in fp32: lane i holds dims [i*DPL, (i+1)*DPL); its
    // rotate-half partner dims are in lane i^16.
    float rq[DPL], rk[DPL], vv[DPL];
    {
      float x[DPL], y[DPL];
#pragma unroll
      for (int e = 0; e < DPL; ++e) x[e] = __ldcg(qrow + lane * DPL + e);
#pragma unroll
      for (int e = 0; e < DPL; ++e) y[e] = __shfl_xor_sync(0xffffffffu, x[e], 16);
#pragma unroll
      for (int e = 0; e < DPL; ++e) {
        const float2 t = cs[(lane & 15) * DPL + e];
        rq[e] = (lane < 16) ? (x[e] * t.x - y[e] * t.y) : (y[e] * t.y + x[e] * t.x);
      }
    }
    uint32_t kcodes = 0, vcodes = 0;
    float ks_new = 0.f, vs_new = 0.f;
    if (tail && !aborted) {
      float x[DPL], y[DPL];
#pragma unroll
      for (int e = 0; e < DPL; ++e) x[e] = __ldcg(qrow + HD + lane * DPL + e);
#pragma unroll
      for (int e = 0; e < DPL; ++e) y[e] = __shfl_xor_sync(0xffffffffu, x[e], 16);
#pragma unroll
      for (int e = 0; e < DPL; ++e) {
        const float2 t = cs[(lane & 15) * DPL + e];
        rk[e] = (lane < 16) ? (x[e] * t.x - y[e] * t.y) : (y[e] * t.y + x[e] * t.x);
        vv[e] = __ldcg(qrow + 2 * HD + lane * DPL + e);
      }
      if (p.kv_dump) {
        float* dk = p.kv_dump + ((((size_t)layer * 2 + 0) * p.S_max + s) * H + h) * D + lane * DPL;
        float* dv = p.kv_dump + ((((size_t)layer * 2 + 1) * p.S_max + s) * H + h) * D + lane * DPL;
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
          dk[e] = rk[e];
          dv[e] = vv[e];
        }
      }
      kcodes = quantize_lane<DPL>(rk, ks_new);
      vcodes = quantize_lane<DPL>(vv, vs_new);
      uint8_t* kdst = p.kv + (rowK + P) * D + lane * DPL;
      uint8_t* vdst = p.kv + (rowV + P) * D + lane * DPL;
      if constexpr (DPL == 4) {
        *(uint32_t*)kdst = kcodes;
        *(uint32_t*)vdst = vcodes;
      } else {
        *(uint16_t*)kdst = (uint16_t)kcodes;
        *(uint16_t*)vdst = (uint16_t)vcodes;
      }
      if (lane == 0) {
        p.kv_scales[rowK + P] = ks_new;
        p.kv_scales[rowV + P] = vs_new;
      }
    }
    // q as an f16 pair hi + lo (|q - hi - lo| <~ 2^-22 |q|), so that the
    // tensor-core dot products keep close to fp32 accuracy.
#pragma unroll
    for (int e = 0; e < DPL; ++e) {
      const __half hi = __float2half_rn(rq[e]);
      qs_hi[lane * DPL + e] = hi;
      qs_lo[lane * DPL + e] = __float2half_rn(rq[e] - __half2float(hi));
    }
    __syncwarp();
    // B fragments of the score mma: column 0 = q_hi (lanes 0..3), column 1 =
    // q_lo (lanes 4..7), zero elsewhere, so that one mma yields both partial
    // products; lane t4 holds dims [t4*D/4, (t4+1)*D/4), k-step j takes
    // dims +4j..+4j+3.
    uint32_t qb0[KST], qb1[KST];
    {
      const uint32_t* wq = (const uint32_t*)(((lane < 4) ? qs_hi : qs_lo) + t4 * (D / 4));
#pragma unroll
      for (int j = 0; j < KST; ++j) {
        qb0[j] = (lane < 8) ? wq[2 * j] : 0u;
        qb1[j] = (lane < 8) ? wq[2 * j + 1] : 0u;
      }
    }


    // acc[j]: c0 + c1 = o[dim of row g], c2 + c3 = o[dim of row g+8] of P.V
    // m-tile j (w_hi and w_lo parts; real in lanes with t4 == 0; units of R).
    float acc[MTV][4];
#pragma unroll
    for (int j = 0; j < MTV; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    float m_run = -INFINITY, l_run = 0.f, R = 0.f;

    for (int k = 0; !aborted && k < n; ++k) {
      const int ci = c_lo + k;
      const uint32_t it = c.att_it + k;
      const int st = it % kAttStages;
      if (!mbar_wait(bar_att(c, warp, st), (it / kAttStages) & 1u, p.timeout_ns, p.err)) {
        set_err(p, kErrTimeout);
        aborted = true;
        break;
      }
      uint8_t* kt = wbuf + st * stage_bytes;
      uint8_t* vt = kt + kChunk * D;
      float* ksm = (float*)(c.smem + c.lay.ascale_off + (warp * 2 + (k / kScaleGroup) % 2) * kScaleBufBytes) +
                   (k % kScaleGroup) * kChunk;
      float* vsm = ksm + kScaleGroup * kChunk;
      const bool last = tail && (ci == nch - 1);
      const int valid = last ? (P - ci * kChunk + 1) : kChunk;
      if (last) {  // the current slot: use the codes just written
        const int rr = P - ci * kChunk;
        const uint32_t off = swz<D>((uint32_t)(rr * D + lane * DPL));
        if constexpr (DPL == 4) {
          *(uint32_t*)(kt + off) = kcodes;
          *(uint32_t*)(vt + off) = vcodes;
        } else {
          *(uint16_t*)(kt + off) = (uint16_t)kcodes;
          *(uint16_t*)(vt + off) = (uint16_t)vcodes;
        }
        if (lane == 0) {
          ksm[rr] = ks_new;
          vsm[rr] = vs_new;
        }
        __syncwarp();
      }

      // ---- scores S[token] = K . q: 4 m-tiles of 16 tokens, interleaved so
      // that 8 accumulators (m-tile x {q_hi, q_lo}) form independent chains;
      // A = codes of tokens g and g+8 (the lane's KQB bytes), B = q (column 0).
      float cac[kMT][4];
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) cac[mt][0] = cac[mt][1] = cac[mt][2] = cac[mt][3] = 0.f;
#pragma unroll
      for (int ch = 0; ch < KQB / 16; ++ch) {
        uint32_t ka[kMT][4], kb[kMT][4];
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt) {
          const uint4 a = *(const uint4*)(kt + swz<D>((uint32_t)((mt * 16 + g) * D + t4 * KQB + ch * 16)));
          const uint4 b = *(const uint4*)(kt + swz<D>((uint32_t)((mt * 16 + g + 8) * D + t4 * KQB + ch * 16)));
          ka[mt][0] = a.x; ka[mt][1] = a.y; ka[mt][2] = a.z; ka[mt][3] = a.w;
          kb[mt][0] = b.x; kb[mt][1] = b.y; kb[mt][2] = b.z; kb[mt][3] = b.w;
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = ch * 4 + jj;
#pragma unroll
          for (int mt = 0; mt < kMT; ++mt) {
            uint32_t a0, a1, a2, a3;
            e4m3x4_to_f16x2x2(ka[mt][jj], a0, a2);
            e4m3x4_to_f16x2x2(kb[mt][jj], a1, a3);
            mma_f16_16816(cac[mt], a0, a1, a2, a3, qb0[j], qb1[j]);
          }
        }
      }
      float sc[kMT][2];  // [m-tile][token g, token g+8], real where t4 == 0
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        sc[mt][0] = cac[mt][0] + cac[mt][1];  // token g: q_hi part + q_lo part
        sc[mt][1] = cac[mt][2] + cac[mt][3];  // token g + 8
      }
      // ---- online softmax (base 2) over the lanes with t4 == 0
      float mx = -INFINITY, vmax = 0.f;
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int tok = mt * 16 + g + 8 * e;
          const bool ok = tok < valid;
          const float v = ok ? sc[mt][e] * ksm[tok] * scale_log2 : -INFINITY;
          sc[mt][e] = v;
          mx = fmaxf(mx, v);
          vmax = ok ? fmaxf(vmax, vsm[tok]) : vmax;
        }
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
      }
      const float m_new = fmaxf(m_run, mx);
      const float alpha = ex2(m_run - m_new);
      // acc holds values in units of R; move to units of the chunk's largest
      // V scale so that the weights p * vs / R stay in [0, 1].
      const float R_new = (vmax > 0.f) ? vmax : 1.f;
      const float rescale = (R > 0.f) ? alpha * (R / R_new) : 0.f;
      l_run *= alpha;
#pragma unroll
      for (int j = 0; j < MTV; ++j) {
        acc[j][0] *= rescale;
        acc[j][1] *= rescale;
        acc[j][2] *= rescale;
        acc[j][3] *= rescale;
      }
      R = R_new;
      m_run = m_new;
      const float inv_R = 1.0f / R_new;
      // weights w = p * vs / R as f16 hi + lo, packed {token g, token g+8}
      uint32_t whi[kMT], wlo[kMT];
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        float w2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int tok = mt * 16 + g + 8 * e;
          const float pr = ex2(sc[mt][e] - m_new);
          l_run += pr;
          w2[e] = (tok < valid) ? pr * (vsm[tok] * inv_R) : 0.f;
        }
        const __half2 hi = __floats2half2_rn(w2[0], w2[1]);
        const float2 hf = __half22float2(hi);
        const __half2 lo = __floats2half2_rn(w2[0] - hf.x, w2[1] - hf.y);
        whi[mt] = *(const uint32_t*)&hi;
        wlo[mt] = *(const uint32_t*)&lo;
      }
      // ---- O += V^T . w: per 16-token group, A = V codes (rows = head dims,
      // columns = tokens), B = w (column 0).  Lane t4 < 4 gathers the weights
      // of tokens 2t4, 2t4+1, 2t4+8, 2t4+9 from lanes 8*t4 and 8*t4+4.
      const int srcA = 8 * t4, srcB = 8 * t4 + 4;
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        const uint32_t hA = __shfl_sync(0xffffffffu, whi[mt], srcA);
        const uint32_t hB = __shfl_sync(0xffffffffu, whi[mt], srcB);
        const uint32_t lA = __shfl_sync(0xffffffffu, wlo[mt], srcA);
        const uint32_t lB = __shfl_sync(0xffffffffu, wlo[mt], srcB);
        // column 0 of B = w_hi (lanes 0..3), column 1 = w_lo (lanes 4..7)
        const uint32_t xA = (lane < 4) ? hA : lA, xB = (lane < 4) ? hB : lB;
        const uint32_t bw0 = (lane < 8) ? prmt(xA, xB, 0x5410u) : 0u;
        const uint32_t bw1 = (lane < 8) ? prmt(xA, xB, 0x7632u) : 0u;
        const int r0 = mt * 16 + 2 * t4;
        const int rows[4] = {r0, r0 + 1, r0 + 8, r0 + 9};
        uint32_t vw[4][VB / 4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const uint32_t off = swz<D>((uint32_t)(rows[a] * D + g * VB));
          if constexpr (VB == 16) {
            const uint4 w4 = *(const uint4*)(vt + off);
            vw[a][0] = w4.x;
            vw[a][1] = w4.y;
            vw[a][2 % (VB / 4)] = w4.z;
            vw[a][3 % (VB / 4)] = w4.w;
          } else {
            const uint2 w2 = *(const uint2*)(vt + off);
            vw[a][0] = w2.x;
            vw[a][1] = w2.y;
          }
          if (rows[a] >= valid) {
#pragma unroll
            for (int w = 0; w < VB / 4; ++w) vw[a][w] = 0u;
          }
        }
        // f01[b] = f16 pair {tok r0 byte b, tok r0+1 byte b}; f23 likewise
        uint32_t f01[VB], f23[VB];
#pragma unroll
        for (int w = 0; w < VB / 4; ++w) {
          e4m3x4_to_f16x2x2(prmt(vw[0][w], vw[1][w], 0x5140u), f01[4 * w + 0], f01[4 * w + 1]);
          e4m3x4_to_f16x2x2(prmt(vw[0][w], vw[1][w], 0x7362u), f01[4 * w + 2], f01[4 * w + 3]);
          e4m3x4_to_f16x2x2(prmt(vw[2][w], vw[3][w], 0x5140u), f23[4 * w + 0], f23[4 * w + 1]);
          e4m3x4_to_f16x2x2(prmt(vw[2][w], vw[3][w], 0x7362u), f23[4 * w + 2], f23[4 * w + 3]);
        }
        // m-tile j: row g <-> byte j, row g+8 <-> byte j + VB/2
#pragma unroll
        for (int j = 0; j < MTV; ++j) {
          const uint32_t a0 = f01[j], a1 = f01[j + VB / 2], a2 = f23[j], a3 = f23[j + VB / 2];
          mma_f16_16816(acc[j], a0, a1, a2, a3, bw0, bw1);
        }
      }
      if (last) fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && k + kAttStages < n) issue(ci + kAttStages, st);
      __syncwarp();
    }
    if (aborted) {
      // let this warp's copies in flight land before returning
      for (int k = 0; k < n; ++k) {
        const uint32_t it = c.att_it + k;
        mbar_wait(bar_att(c, warp, it % kAttStages), (it / kAttStages) & 1u, 100000000LL, p.err);
      }
      return;
    }
    c.att_it += n;

    // ---- finish the piece: l over the lanes with t4 == 0
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) l_run += __shfl_xor_sync(0xffffffffu, l_run, o);
    // lane (g, 0): m-tile j row g -> dim g*VB + j, row g+8 -> dim g*VB + VB/2 + j
    if (np == 1) {
      if (t4 == 0) {
        const float f = R / l_run;
        uint16_t* o = p.attn + (size_t)s * HD + h * D + g * VB;
#pragma unroll
        for (int j = 0; j < MTV; ++j) {
          o[j] = f32_to_bf16((acc[j][0] + acc[j][1]) * f);
          o[VB / 2 + j] = f32_to_bf16((acc[j][2] + acc[j][3]) * f);
        }
      }
      attn_row_done(p, h, layer, lane);
    } else {
      // split (session, head): store this piece's (acc, m, l) and count it;
      // the warp whose piece completes the count merges them
      float* part = p.att_part + (size_t)(first + c_lo / kPieceChunks) * (D + 4);
      if (t4 == 0) {
#pragma unroll
        for (int j = 0; j < MTV; ++j) {
          part[g * VB + j] = (acc[j][0] + acc[j][1]) * R;
          part[g * VB + VB / 2 + j] = (acc[j][2] + acc[j][3]) * R;
        }
        if (lane == 0) {
          part[D] = m_run;
          part[D + 1] = l_run;
        }
      }
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        __threadfence();  // this piece's partial before its count
        last = atomicAdd(p.sh_cnt + sh, 1) == (layer + 1) * np - 1;
        if (last) __threadfence();  // every piece's partial before the reads below
      }
      if (__shfl_sync(0xffffffffu, last, 0)) {
        merge_item<D>(p, first, np, s, h, lane);
        attn_row_done(p, h, layer, lane);
      }
    }
    // the next piece is claimed once this warp is free (a piece claimed
    // ahead would wait behind the current one while other warps run dry
    // at the end of the list; the claim's latency hides behind the other
    // warps' copies)
    int nxt = 0;
    if (lane == 0) nxt = NW + atomicAdd(ctr, 1);
    pi = __shfl_sync(0xffffffffu, nxt, 0);
  }
}

// ------------------------------------------------------- selective state
// The Mamba2-style mixer of hybrid layer l (its lm-th selective-state block)
// for every (session, head): dt = softplus(dt + dt_bias), a = exp(-exp(A_log)
// dt); per head dim p and state n: h = a h + dt x_p B_n (the fp32 state,
// written back in place); y_p = sum_n C_n h + D x_p; out = bf16(y_p silu(z_p)).
// (session, head) items are dealt round-robin to CTAs; a CTA's 8 warps work
// on one item together (warp w: rows 8w..8w+7, lane: states 4 lane..+3)
// while thread 0 keeps kSsmStages of its next items in flight by bulk copy:
// the 32 KB state block and the item's x, z, B, C and dt from the in-
// projection output, so that an item's arithmetic reads shared memory only.
// An empty slot (negative position) leaves its state alone and writes zeros.
// Returns false if a copy wait gave up.
constexpr int kSsmSide = 64 + 64 + kSsmN + kSsmN + 4;              // x, z, B, C, dt group (floats)
constexpr int kSsmStageF = kSsmP * kSsmN + ((kSsmSide + 31) / 32) * 32;  // floats per stage
// The items read the in-projection's rows once every tile of this block's
// in-projection is published (wait_target on its finished-tile count; 0: a
// grid barrier came before); every CTA counts its items done in the
// selective-state count when they are written, which the out-projection
// waits for.
__device__ __forceinline__ bool ssm_phase(const StepParams& p, Ctx& c, int lm, int l, int wait_target) {
  static_assert(kWarps * 8 == kSsmP && 32 * 4 == kSsmN, "state phase layout");
  constexpr uint32_t kBlk = kSsmP * kSsmN * 4;
  constexpr uint32_t kTx = kBlk + (64 + 64 + kSsmN + kSsmN + 4) * 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hs = p.ssm_heads, di = p.d_inner, R = p.in_rows, N = kSsmN;
  const int items = p.S * Hs;
  const int my = (items > (int)blockIdx.x) ? (items - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const uint16_t* prm = p.weights + hyb_layer_offset(p.hyb_M, p.hyb_G, p.attn_every, l) + p.hyb_off_a_log;
  float* state_l = p.ssm_state + (size_t)lm * p.S_max * Hs * kSsmP * kSsmN;
  const uint32_t ring_s = c.sbase + c.lay.ring_off;
  const float* ring = (const float*)(c.smem + c.lay.ring_off);
  // A_log, dt_bias, D of every head, once per phase, after the stages
  float* prm_s = (float*)(c.smem + c.lay.ring_off) + kSsmStages * kSsmStageF;
  auto issue = [&](int k) {  // thread 0
    const int i = (int)blockIdx.x + k * (int)gridDim.x, s = i / Hs, hh = i - s * Hs;
    const uint32_t st = (c.ssm_it + (uint32_t)k) % kSsmStages, b = bar_ssm(c, st);
    if (p.pos[s] < 0) {
      mbar_arrive(b);  // nothing to copy for an empty slot
    } else {
      const uint32_t dst = ring_s + st * kSsmStageF * 4;
      const float* zrow = p.zx + (size_t)s * R;
      mbar_arrive_expect_tx(b, kTx);
      bulk_load_hint(dst, state_l + (size_t)i * kSsmP * kSsmN, kBlk, b, policy_evict_first());
      bulk_load(dst + kBlk, zrow + di + hh * kSsmP, 64 * 4, b);                 // x
      bulk_load(dst + kBlk + 256, zrow + hh * kSsmP, 64 * 4, b);                // z
      bulk_load(dst + kBlk + 512, zrow + 2 * di, kSsmN * 4, b);                 // B
      bulk_load(dst + kBlk + 512 + kSsmN * 4, zrow + 2 * di + N, kSsmN * 4, b);  // C
      bulk_load(dst + kBlk + 512 + 2 * kSsmN * 4, zrow + 2 * di + 2 * N + (hh & ~3), 16, b);  // dt
    }
  };
  if (wait_target > 0 && my > 0) {
    if (threadIdx.x == 0) {
      const bool ok0 = wait_flag_ge(p, p.done_cnt + kIn, wait_target);
      fence_proxy_async_global();  // the copies below read those tiles' rows
      *misc_word(c, 7) = ok0 ? 1 : 0;
    }
    __syncthreads();
    if (!*misc_word(c, 7)) return false;
  }
  if (threadIdx.x == 0) {
    fence_proxy_async_smem();  // earlier generic accesses to the ring come first
    for (int k = 0; k < min(my, kSsmStages); ++k) issue(k);
  }
  for (int i = threadIdx.x; i < 3 * Hs; i += kThreads) prm_s[i] = bf16_to_f32(prm[i]);
  for (int k = 0; k < my; ++k) {
    const int i = (int)blockIdx.x + k * (int)gridDim.x, s = i / Hs, hh = i - s * Hs;
    const uint32_t st = (c.ssm_it + (uint32_t)k) % kSsmStages;
    volatile int* flag = misc_word(c, (k & 1) ? 10 : 7);  // alternating: no word is rewritten while read
    if (threadIdx.x == 0) {
      const bool ok0 = mbar_wait(bar_ssm(c, st), ((c.ssm_it + (uint32_t)k) / kSsmStages) & 1u, p.timeout_ns, p.err);
      if (!ok0) set_err(p, kErrTimeout);
      *flag = ok0 ? 1 : 0;
    }
    // one barrier per item: every thread is past item k - 1 (its reads of
    // that stage fenced), so the stage it used is refilled now
    __syncthreads();
    if (!*flag) return false;
    if (threadIdx.x == 0 && k >= 1 && k - 1 + kSsmStages < my) issue(k - 1 + kSsmStages);
    uint16_t* orow = p.ssm_out + (size_t)s * di + hh * kSsmP + warp * 8;
    if (p.pos[s] < 0) {
      if (lane < 8) orow[lane] = 0;
    } else {
      const float* blk = ring + st * kSsmStageF;
      const float* xs = blk + kSsmP * kSsmN;
      const float* zs = xs + 64;
      const float* Bs = zs + 64;
      const float* Cs = Bs + kSsmN;
      const float* dts = Cs + kSsmN;
      const float dtr = dts[hh & 3] + prm_s[Hs + hh];
      const float dt = dtr > 0.f ? dtr + log1pf(expf(-dtr)) : log1pf(expf(dtr));
      const float a = expf(-expf(prm_s[hh]) * dt);
      const float Dh = prm_s[2 * Hs + hh];
      const float4 B4 = ((const float4*)Bs)[lane];
      const float4 C4 = ((const float4*)Cs)[lane];
      float* gst = state_l + (size_t)i * kSsmP * kSsmN;
      float yv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int pr = warp * 8 + j;
        const float tx = dt * xs[pr];
        float4 h = *(const float4*)(blk + pr * N + 4 * lane);
        h.x = fmaf(a, h.x, tx * B4.x);
        h.y = fmaf(a, h.y, tx * B4.y);
        h.z = fmaf(a, h.z, tx * B4.z);
        h.w = fmaf(a, h.w, tx * B4.w);
        __stcs((float4*)(gst + pr * N + 4 * lane), h);  // streamed: read again only next frame
        yv[j] = C4.x * h.x + C4.y * h.y + C4.z * h.z + C4.w * h.w;
      }
      // y over the 32 lanes of each of the 8 rows by recursive halving: lane
      // bits 4, 3, 2 pick a half of the rows at each of the first three
      // levels (4 + 2 + 1 shuffles), bits 1, 0 sum the last value; lane l
      // then holds row 4 b4 + 2 b3 + b2 whole
      {
        const bool h4 = lane & 16, h3 = lane & 8, h2 = lane & 4;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float send = h4 ? yv[j] : yv[j + 4];
          const float keep = h4 ? yv[j + 4] : yv[j];
          yv[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float send = h3 ? yv[j] : yv[j + 2];
          const float keep = h3 ? yv[j + 2] : yv[j];
          yv[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
        {
          const float send = h2 ? yv[0] : yv[1];
          const float keep = h2 ? yv[1] : yv[0];
          yv[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
        yv[0] += __shfl_xor_sync(0xffffffffu, yv[0], 2);
        yv[0] += __shfl_xor_sync(0xffffffffu, yv[0], 1);
      }
      if ((lane & 3) == 0) {
        const int j = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
        const int pr = warp * 8 + j;
        const float xp = xs[pr], zp = zs[pr];
        const float yp = yv[0] + Dh * xp;
        orow[j] = f32_to_bf16(yp * zp / (1.0f + expf(-zp)));
      }
    }
    fence_proxy_async_smem();  // this stage's reads come before its refill
  }
  c.ssm_it += (uint32_t)my;
  __syncthreads();           // every thread is past the last item before the ring is reused
  if (wait_target > 0 && my > 0) {
    fence_proxy_async_global();  // the out-projection reads these rows by TMA
    __syncthreads();
    if (threadIdx.x == 0 && !(p.skip_sig == (int)blockIdx.x && p.skip_sig_kind == kSigSsm)) {
      __threadfence();
      atomicAdd(p.done_cnt + kSsmDone, my);
    }
  }
  return true;
}

// ---------------------------------------------------------------- prologue
// One CTA turns positions into the attention work list: each (session, head)
// history of pos+1 slots is cut into pieces of up to kPieceChunks chunks.
// The list is ordered by piece length, longest first (a counting sort over
// the kPieceChunks possible lengths); the attention phase's warps claim its
// entries in that order, which balances their loads.  A piece's slot
// for its partial result is first + c_lo / kPieceChunks, first being the
// first slot of its (session, head).
static_assert(kThreads <= 256, "the reduction scratch holds one word per thread");
static_assert(kPieceChunks % kWarps == 0, "each warp scans kPieceChunks / kWarps length classes");
static_assert(kThreads % 32 == 0 && kThreads / 32 <= 8, "lanes scan kThreads/32 entries");
__device__ void build_pieces(const StepParams& p, Ctx& c) {
  int* red = (int*)(c.smem + c.lay.red_off);     // per-thread slot counts -> first slots
  int* tab = (int*)(c.smem + c.lay.ring_off);    // [length class][thread] counts -> offsets
  int* cbase = tab + kPieceChunks * kThreads;    // [length class] totals -> list offsets
  int* spos = (int*)(c.smem + c.lay.xbuf_off);   // positions, -1 where invalid
  const int N = p.S * p.H, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int s = tid; s < p.S; s += kThreads) {
    const int P0 = p.pos[s];
    const int P = (P0 < 0) ? P0 : P0 + c.frame;  // frame f of a launch is at position + f
    // a negative position is an empty slot; one at or beyond T_max an error
    spos[s] = (P >= 0 && P < p.T_max) ? P : -1;
    if (P >= p.T_max) set_err(p, kErrPos);
  }
  __syncthreads();
  const int b0 = (int)((long long)N * tid / kThreads), b1 = (int)((long long)N * (tid + 1) / kThreads);
  int cc[kPieceChunks];
#pragma unroll
  for (int k = 0; k < kPieceChunks; ++k) cc[k] = 0;
  int slots = 0;
  for (int sh = b0; sh < b1; ++sh) {
    const int P = spos[sh / p.H];
    if (P < 0) continue;
    const int nch = P / kChunk + 1, nf = nch / kPieceChunks, ts = nch % kPieceChunks;
    cc[kPieceChunks - 1] += nf;
#pragma unroll
    for (int k = 0; k < kPieceChunks - 1; ++k) cc[k] += (ts == k + 1) ? 1 : 0;
    slots += nf + (ts ? 1 : 0);
  }
#pragma unroll
  for (int k = 0; k < kPieceChunks; ++k) tab[k * kThreads + tid] = cc[k];
  red[tid] = slots;
  __syncthreads();
  for (int k = kPieceChunks - 1 - warp; k >= 0; k -= kWarps) {  // exclusive scan over threads
    constexpr int per = kThreads / 32;
    int* row = tab + k * kThreads;
    int v[per], sum = 0;
#pragma unroll
    for (int i = 0; i < per; ++i) {
      v[i] = row[lane * per + i];
      sum += v[i];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    int run = incl - sum;
#pragma unroll
    for (int i = 0; i < per; ++i) {
      row[lane * per + i] = run;
      run += v[i];
    }
    if (lane == 31) cbase[k] = incl;
  }
  __syncthreads();
  if (tid == 0) {
    int off = 0;
    for (int k = kPieceChunks - 1; k >= 0; --k) {  // longest pieces first
      const int t = cbase[k];
      cbase[k] = off;
      off += t;
    }
    *p.n_pieces = off;
    int nv = 0;
    for (int s = 0; s < p.S; ++s) nv += (spos[s] >= 0) ? 1 : 0;
    p.n_pieces[1] = nv;  // sessions whose attention rows the output projection waits for
    int run = 0;
    for (int i = 0; i < kThreads; ++i) {
      const int v = red[i];
      red[i] = run;
      run += v;
    }
  }
  __syncthreads();
  int at[kPieceChunks];
#pragma unroll
  for (int k = 0; k < kPieceChunks; ++k) at[k] = cbase[k] + tab[k * kThreads + tid];
  int first = red[tid];
  for (int sh = b0; sh < b1; ++sh) {
    const int P = spos[sh / p.H];
    if (P < 0) {
      p.sh_info[sh] = make_int2(0, 0);
      continue;
    }
    const int nch = P / kChunk + 1;
    const int np = (nch + kPieceChunks - 1) / kPieceChunks;
    p.sh_info[sh] = make_int2(first, np);
    for (int q = 0; q < np; ++q) {
      const int lo = q * kPieceChunks, hi = min(nch, lo + kPieceChunks);
      int idx = 0;
#pragma unroll
      for (int k = 0; k < kPieceChunks; ++k)
        if (hi - lo == k + 1) idx = at[k]++;
      p.pieces[2 * idx] = make_int4(sh, lo | (hi << 16), np, first);
      p.pieces[2 * idx + 1] = make_int4(P, 0, 0, 0);
    }
    first += np;
  }
  // empty slots and sessions with an invalid position get a zero attention output
  for (int s = 0; s < p.S; ++s)
    if (spos[s] < 0)
      for (int i = tid; i < p.HD; i += kThreads) p.attn[(size_t)s * p.HD + i] = 0;
  fence_proxy_async_smem();  // the ring area is refilled by copies later
  __syncthreads();
}

// ------------------------------------------------------------ testing hook
// Activation dump: copies rows 0..act_dump_n-1 of a workspace buffer (fp32
// or bf16, row stride ld, n values per row) into section `off` of the
// record of (frame, layer, session).  Runs on all CTAs right after the grid
// barrier that ends the buffer's producing phase; the buffer is only read
// until the next barrier, so the copy sees its final values.
enum ActSection : int { kActIn = 0, kActXn1, kActProj, kActMix, kActMid, kActXn2, kActU, kActOut };
__device__ __forceinline__ long long act_off(const StepParams& p, int sec) {
  const long long d = p.d, n1 = p.act_n1, n2 = p.act_n2;
  switch (sec) {
    case kActIn: return 0;
    case kActXn1: return d;
    case kActProj: return 2 * d;
    case kActMix: return 2 * d + n1;
    case kActMid: return 2 * d + n1 + n2;
    case kActXn2: return 3 * d + n1 + n2;
    case kActU: return 4 * d + n1 + n2;
    default: return 4 * d + n1 + n2 + p.F;
  }
}
template <typename T>
__device__ __noinline__ void act_dump_rows(const StepParams& p, int frame, int layer, int sec, const T* src,
                                           int ld, int n) {
  const int ns = p.act_dump_n;
  const long long off = act_off(p, sec);
  const int total = ns * n;
  for (int i = blockIdx.x * kThreads + threadIdx.x; i < total; i += gridDim.x * kThreads) {
    const int s = i / n, e = i - s * n;
    float v;
    if constexpr (sizeof(T) == 2) v = bf16_to_f32(__ldcg((const unsigned short*)src + (size_t)s * ld + e));
    else v = __ldcg((const float*)src + (size_t)s * ld + e);
    p.act_dump[(((long long)frame * p.L + layer) * ns + s) * p.act_rec + off + e] = v;
  }
}

// ------------------------------------------------------------------ kernel
// kHybrid selects the hybrid model's layer loop at compile time, so that each
// model's kernel is register-allocated for its own phases only.  kDump adds
// the activation-dump testing hook; launches without it run the kernel that
// has no trace of it (same phases, same arithmetic).
template <bool kHybrid, bool kDump>
__global__ void __launch_bounds__(kThreads, 1) step_kernel(const __grid_constant__ StepParams p) {
  extern __shared__ uint8_t smem_raw[];
  Ctx c;
  {  // align the shared-space address to 1024 B (swizzle atoms, TMA boxes)
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    c.smem = smem_raw + pad;
    c.sbase = raw + pad;
  }
  c.lay = smem_layout();
  c.bar_target = 0;
  c.bar_index = 0;
  c.ring_it = c.acc_it = c.att_it = c.norm_it = 0;
  c.frame = 0;
  c.ssm_it = 0;
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(bar_full(c, i), 1);
      mbar_init(bar_empty(c, i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_accf(c, i), 1);
      mbar_init(bar_acce(c, i), 4);
    }
    for (int w = 0; w < kWarps; ++w)
      for (int st = 0; st < kAttStages; ++st) mbar_init(bar_att(c, w, st), 1);
    *misc_word(c, 8) = 0;  // phase marks of the profiling hook
    mbar_init(bar_drain(c), 1);
    mbar_init(bar_norm(c), 1);
    for (int i = 0; i < kSsmStages; ++i) mbar_init(bar_ssm(c, i), 1);
    fence_mbar_init();
    for (int i = 0; i < (p.depth ? kGemmKinds : 4); ++i) {
      prefetch_tmap(&p.tm_w[i]);
      prefetch_tmap(&p.tm_x[i]);
    }
    prefetch_tmap(&p.tm_kv);
    prefetch_tmap(&p.tm_sc);
  }
  if (warp == 1) {
    tmem_alloc(c.sbase + c.lay.misc_off, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  c.tmem = *(volatile uint32_t*)(c.smem + c.lay.misc_off);

  if (p.phase_ts && blockIdx.x == 0 && threadIdx.x == 0) p.phase_ts[0] = globaltimer();
  bool ok = true;
  for (int f = 0; ok && f < p.n_frames; ++f) {
    c.frame = f;
    // the previous frame's last reductions (resid, y) finish before this
    // frame's prologue reloads the residual
    if (f > 0 && !(ok = grid_sync(p, c))) break;
    // chained frames: this frame's input is the previous output projected
    if constexpr (!kHybrid) {
      if (f > 0 && p.depth) {
        gemm_phase(p, c, kProj, 0, false);
        if (!(ok = grid_sync(p, c))) break;
      }
    }
    // phase 0: work list, counter reset, residual and first norm
    for (int i = blockIdx.x * kThreads + threadIdx.x; i < kCounterWords; i += gridDim.x * kThreads)
      p.tile_cnt[i] = 0;
    for (int i = blockIdx.x * kThreads + threadIdx.x; i < p.S * p.H; i += gridDim.x * kThreads) p.sh_cnt[i] = 0;
    if (blockIdx.x == gridDim.x - 1) build_pieces(p, c);
    const bool n0 = norm_phase(p, c, p.weights + p.off_g_attn, true, false);
    if (!(ok = grid_sync(p, c) && n0)) break;
    mark_phase(p, c);

    // Within a frame no grid barrier separates the phases: each waits, by
    // counts and flags in global memory, for exactly the data it reads, its
    // weights or history already streaming.  Norm rows wait for the finished
    // tiles of the projection that wrote the residual; a projection waits
    // for the norm rows, the attention rows or the gate/up tiles it reads;
    // attention waits per piece for its head's QKV tiles.  Counts grow over
    // the frame, so a target is the phase's ordinal times its per-phase
    // count.  (The dump kernel adds a barrier before each dump.)
    for (int l = 0; ok && l < p.L; ++l) {
      // decoder layer: attention half + MLP half; hybrid model: an attention
      // block every attn_every layers, selective-state blocks otherwise, no MLP
      constexpr bool hyb = kHybrid;
      const int e = hyb ? p.attn_every : 1;
      const bool attn_layer = !hyb || (l % e == e - 1);
      const int li = (hyb && attn_layer) ? l / e : l;  // attention weights / history index
      const bool last = (l == p.L - 1);
      const uint16_t* wl = hyb ? p.weights + hyb_layer_offset(p.hyb_M, p.hyb_G, e, l)
                               : p.weights + (size_t)l * p.layer_elems;
      if (l > 0) {
        // the residual is final once the previous block's output projection
        // has finished every tile
        int wk, wt;
        if constexpr (kHybrid) {
          const int lp = l - 1;
          const bool pa = (lp % e == e - 1);
          wk = pa ? kO : kOut;
          wt = (pa ? lp / e + 1 : lp - lp / e + 1) * p.tiles[wk];
        } else {
          wk = kDown;
          wt = l * p.tiles[kDown];
        }
        if constexpr (kDump) {
          if (!(ok = grid_sync(p, c))) break;
        }
        const bool nok = norm_phase(p, c, wl + p.off_g_attn, false, true, kDump ? nullptr : p.done_cnt + wk, wt);
        ok = nok;
        if (!ok) break;
        if constexpr (kDump) {
          if (!(ok = grid_sync(p, c))) break;
        } else {
          __syncthreads();
        }
        mark_phase(p, c);
      }
      if (kDump) {  // the layer's input residual and its normed input
        act_dump_rows(p, c.frame, l, kActIn, p.resid, p.d, p.d);
        act_dump_rows(p, c.frame, l, kActXn1, p.xn, p.d, p.d);
      }
      // the block's input projection: QKV, or the selective-state in-projection,
      // once this layer's norm rows are written (counted from the frame's
      // second norm: two per decoder layer, one per hybrid layer; layer 0's
      // follows the prologue's grid barrier)
      const int n_rows = (hyb ? l : 2 * l) * p.S;
      gemm_phase(p, c, attn_layer ? kQKV : kIn, li, false, l > 0 ? p.done_cnt + kNormRows : nullptr, n_rows);
      // attention and the selective-state phase start without a grid barrier:
      // a piece waits for the QKV tiles it reads, the state items for every
      // tile of the in-projection (the dump kernel takes a barrier to read
      // the projection's output whole)
      if (kDump) {
        if (!(ok = grid_sync(p, c))) break;
      } else {
        __syncthreads();
      }
      mark_phase(p, c);
      if (kDump) {
        if (attn_layer) act_dump_rows(p, c.frame, l, kActProj, p.qkv, 3 * p.HD, 3 * p.HD);
        else act_dump_rows(p, c.frame, l, kActProj, p.zx, p.in_rows, p.in_rows);
      }
      if (attn_layer) {
        // split histories are merged by the warp that finishes their last
        // piece; the output projection waits for every head's rows, its
        // weights already streaming
        if (p.D == 128) attention_phase<128>(p, c, li); else attention_phase<64>(p, c, li);
        if constexpr (kDump) {
          if (!(ok = grid_sync(p, c))) break;
          act_dump_rows(p, c.frame, l, kActMix, p.attn, p.HD, p.HD);
        } else {
          __syncthreads();  // the CTA's warps leave the shared ring before the projection refills it
          if (*(volatile int*)p.err & kErrTimeout) { ok = false; break; }
        }
        mark_phase(p, c);
      } else if constexpr (kHybrid) {
        const int lm = l - l / e;
        const bool sok = ssm_phase(p, c, lm, l, kDump ? 0 : (lm + 1) * p.tiles[kIn]);
        if constexpr (kDump) {
          if (!(ok = grid_sync(p, c) && sok)) break;
        } else {
          __syncthreads();
          ok = sok;
          if (!ok) break;
        }
        mark_phase(p, c);
        if (kDump) act_dump_rows(p, c.frame, l, kActMix, p.ssm_out, p.d_inner, p.d_inner);
      }
      // and its output projection + residual: O (once every head's rows are
      // written; with no live session there is none to wait for), or the
      // selective-state out-projection
      if constexpr (kHybrid) {
        // the out-projection: O once every head's rows are written (with no
        // live session there is none to wait for), the selective-state one
        // once every item of the block is
        const int lm = l - l / e;
        if (attn_layer)
          gemm_phase(p, c, kO, li, last, __ldcg(p.n_pieces + 1) > 0 ? p.done_cnt + kHeadsDone : nullptr,
                     (li + 1) * p.H);
        else
          gemm_phase(p, c, kOut, li, last, kDump ? nullptr : p.done_cnt + kSsmDone, (lm + 1) * p.S * p.ssm_heads);
      } else {
        gemm_phase(p, c, kO, li, false, __ldcg(p.n_pieces + 1) > 0 ? p.done_cnt + kHeadsDone : nullptr,
                   (li + 1) * p.H);
        if constexpr (kDump) {
          if (!(ok = grid_sync(p, c))) break;
          act_dump_rows(p, c.frame, l, kActMid, p.resid, p.d, p.d);
        } else {
          __syncthreads();
        }
        mark_phase(p, c);
        const bool nok2 = norm_phase(p, c, wl + p.off_g_mlp, false, true, kDump ? nullptr : p.done_cnt + kO,
                                     (l + 1) * p.tiles[kO]);
        ok = nok2;
        if (!ok) break;
        if constexpr (kDump) {
          if (!(ok = grid_sync(p, c))) break;
          act_dump_rows(p, c.frame, l, kActXn2, p.xn, p.d, p.d);
        } else {
          __syncthreads();
        }
        mark_phase(p, c);
        gemm_phase(p, c, kGU, l, false, p.done_cnt + kNormRows, (2 * l + 1) * p.S);
        if constexpr (kDump) {  // the dump reads u whole
          if (!(ok = grid_sync(p, c))) break;
          act_dump_rows(p, c.frame, l, kActU, p.u, p.F, p.F);
        } else {
          __syncthreads();
        }
        mark_phase(p, c);
        gemm_phase(p, c, kDown, l, last, p.done_cnt + kGU, (l + 1) * p.tiles[kGU]);
      }
      if (kDump && !last) {  // the block's output residual (the last layer's is y, rounded)
        if (!(ok = grid_sync(p, c))) break;
        act_dump_rows(p, c.frame, l, kHybrid ? kActMid : kActOut, p.resid, p.d, p.d);
      }
      // the next phase (a norm, or the next frame's prologue) reuses the ring
      __syncthreads();
      mark_phase(p, c);
      if (*(volatile int*)p.err & kErrTimeout) { ok = false; break; }
    }
  }
  // rolling positions: every frame has read them; advance once all are done
  if (ok && p.pos_advance) {
    ok = grid_sync(p, c);
    if (ok && blockIdx.x == 0)
      for (int s = threadIdx.x; s < p.S; s += kThreads)
        if (p.pos_advance[s] >= 0) p.pos_advance[s] += p.n_frames;
  }

  if (!ok) {
    // Abort path: let outstanding tensor-core work finish before TMEM is freed.
    if (warp == 1 && (threadIdx.x & 31) == 0) {
      tc_commit(bar_drain(c));
      mbar_wait(bar_drain(c), 0, 100000000LL, p.err);
    }
    if (warp == 0 && (threadIdx.x & 31) == 0) {
      // wait (bounded) for the most recent ring loads
      const uint32_t nst = (uint32_t)p.nstage;
      for (uint32_t k = 0; k < nst && k < c.ring_it; ++k) {
        const uint32_t it = c.ring_it - 1 - k;
        long long t0 = globaltimer();
        while (!mbar_try_wait(bar_full(c, it % nst), (it / nst) & 1u) && globaltimer() - t0 < 100000000LL) {
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (p.phase_ts && blockIdx.x == 0 && threadIdx.x == 0) p.phase_ts[1 + c.bar_index] = globaltimer();
  if (warp == 1) tmem_dealloc(c.tmem, kTmemCols);
  // the last CTA to finish copies the error word to the caller-visible host
  // word, so that reading the status needs no copy or synchronisation
  if (p.err_out && threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.bar + 1, 1u) == gridDim.x - 1) {
      const int e = atomicOr(p.err, 0);
      *(volatile int*)p.err_out = e;
      __threadfence_system();
    }
  }
}

// The four instantiations: decoder / hybrid, without / with the dump hook.
static const void* const kKernels[4] = {(const void*)step_kernel<false, false>, (const void*)step_kernel<true, false>,
                                        (const void*)step_kernel<false, true>, (const void*)step_kernel<true, true>};

cudaError_t configure_step_kernel() {
  for (const void* fn : kKernels) {
    const cudaError_t e =
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_layout().total);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_step(const StepParams& p, int grid, cudaStream_t stream) {
  void* args[] = {(void*)&p};
  const void* fn = kKernels[(p.hybrid ? 1 : 0) + (p.act_dump ? 2 : 0)];
  return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kThreads), args, (size_t)smem_layout().total,
                                     stream);
}

int barriers_per_step(int L, int T_max) { return 1; }  // the prologue's
// Phase marks of one frame (the profiling hook): the prologue, then per
// layer its norms and phases, in the layer loop's order.
int phases_per_step(int L, bool hybrid, int attn_every) {
  if (!hybrid) return 1 + L * 6 + (L - 1);  // QKV, attention, O, norm2, gate/up, down; norm1 after layer 0
  int n = 1;
  for (int l = 0; l < L; ++l) n += (l > 0 ? 1 : 0) + 3;  // norm, in-projection, mixer or attention, out
  return n;
}
int hybrid_barriers_per_step(int L, int attn_every, int T_max) {
  return 1;  // the prologue's; every other hand-over is a count or a flag
}
int barriers_per_launch(int L, int T_max, int frames, bool advance, bool depth) {
  return frames * barriers_per_step(L, T_max) + (frames - 1) * (depth ? 2 : 1) + (advance ? 1 : 0);
}

cudaError_t occupancy_per_sm(int* blocks) {
  int lo = 1 << 30;
  for (const void* fn : kKernels) {
    int a = 0;
    const cudaError_t e =
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, fn, kThreads, (size_t)smem_layout().total);
    if (e != cudaSuccess) return e;
    if (a < lo) lo = a;
  }
  *blocks = lo;
  return cudaSuccess;
}

}  // namespace wave
