// pack.cu -- the packed weight blob the step reads.
//
// Every projection matrix W [N][K] (row n = output n, K contiguous) is
// stored as blocks of 128 rows x 64 columns (16 KB, row-major inside the
// block), ordered by 128-row tile, then by 64-column block; a stream-K unit
// (a tile's 128 columns) is then two adjacent blocks, 32 KB of contiguous
// memory, and every TMA box the projections load is one contiguous block.
// A row-major tile box (128 rows of 128 bytes, 8-22 KB apart) costs the
// projections about a fifth of their HBM rate in DRAM page switches.  The
// gate/up matrix keeps its pairing: the tile t block holds gate rows
// 64t..64t+63, then up rows 64t..64t+63.  Rows and columns beyond the matrix
// are zeros.  Vectors (RMSNorm gains, the selective-state parameters) are
// copied as they are.
#include <cuda_runtime.h>
#include <stdint.h>

#include "plan.h"

namespace wave {

// One packed matrix from a row-major one.  gu_F > 0: the gate/up pairing,
// the source holding F gate rows then F up rows.  Each thread moves 16 bytes
// (8 bf16; K is a multiple of 8, so a chunk is inside K or wholly beyond it).
__global__ void k_pack_matrix(const uint16_t* __restrict__ src, int N, int K, int gu_F, int tiles, int kunits,
                              uint16_t* __restrict__ dst) {
  const long long chunks = (long long)tiles * kunits * 2 * 128 * 8;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < chunks;
       i += (long long)gridDim.x * blockDim.x) {
    const int c8 = (int)(i & 7);
    const int r = (int)((i >> 3) & 127);
    const long long blk = i >> 10;
    const int t = (int)(blk / (2 * kunits)), j = (int)(blk - (long long)t * 2 * kunits);
    long long row;
    bool ok;
    if (gu_F > 0) {
      const int f = t * 64 + (r & 63);
      ok = f < gu_F;
      row = (r < 64) ? f : (long long)gu_F + f;
    } else {
      row = (long long)t * 128 + r;
      ok = row < N;
    }
    const int col = j * 64 + c8 * 8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (ok && col < K) v = *(const uint4*)(src + row * K + col);
    *(uint4*)(dst + blk * 8192 + r * 64 + c8 * 8) = v;
  }
}

static int pack_matrix(const uint16_t* src, int N, int K, int gu_F, int tiles, int kunits, uint16_t* dst,
                       cudaStream_t st) {
  const long long chunks = (long long)tiles * kunits * 2 * 128 * 8;
  const int blocks = (int)((chunks + 255) / 256 < 4096 ? (chunks + 255) / 256 : 4096);
  k_pack_matrix<<<blocks, 256, 0, st>>>(src, N, K, gu_F, tiles, kunits, dst);
  return cudaGetLastError() == cudaSuccess ? WAVE_OK : WAVE_ECUDA;
}

static int copy_vec(const uint16_t* src, long long n, uint16_t* dst, cudaStream_t st) {
  return cudaMemcpyAsync(dst, src, (size_t)n * 2, cudaMemcpyDeviceToDevice, st) == cudaSuccess ? WAVE_OK
                                                                                                : WAVE_ECUDA;
}

int pack_weights(const Plan& pl, const void* src_v, void* dst_v, cudaStream_t st) {
  const uint16_t* src = (const uint16_t*)src_v;
  uint16_t* dst = (uint16_t*)dst_v;
  const int d = pl.cfg.d_model, HD = pl.cfg.n_heads * pl.cfg.head_dim;
  int rc = WAVE_OK;
  if (!pl.hybrid) {
    const int F = pl.cfg.ffn;
    for (int l = 0; !rc && l < pl.cfg.n_layers; ++l) {
      const uint16_t* s = src + (long long)l * pl.layer_elems;
      uint16_t* o = dst + (long long)l * pl.pk_layer;
      rc = copy_vec(s + pl.off[0], d, o + pl.pk_off[0], st);
      if (!rc) rc = pack_matrix(s + pl.off[1], 3 * HD, d, 0, pl.tiles[kQKV], pl.kblocks[kQKV], o + pl.pk_off[1], st);
      if (!rc) rc = pack_matrix(s + pl.off[2], d, HD, 0, pl.tiles[kO], pl.kblocks[kO], o + pl.pk_off[2], st);
      if (!rc) rc = copy_vec(s + pl.off[3], d, o + pl.pk_off[3], st);
      if (!rc) rc = pack_matrix(s + pl.off[4], 2 * F, d, F, pl.tiles[kGU], pl.kblocks[kGU], o + pl.pk_off[4], st);
      if (!rc) rc = pack_matrix(s + pl.off[5], d, F, 0, pl.tiles[kDown], pl.kblocks[kDown], o + pl.pk_off[5], st);
    }
    return rc;
  }
  const wave_hybrid_config& hc = pl.hcfg;
  const int e = hc.attn_every;
  for (int l = 0; !rc && l < hc.n_layers; ++l) {
    const uint16_t* s = src + hyb_layer_offset(pl.hyb_M, pl.hyb_G, e, l);
    uint16_t* o = dst + hyb_layer_offset(pl.pk_M, pl.pk_layer, e, l);
    rc = copy_vec(s, d, o, st);  // the block's RMSNorm gain
    if (l % e == e - 1) {
      if (!rc)
        rc = pack_matrix(s + pl.hyb_off_wqkv, 3 * HD, d, 0, pl.tiles[kQKV], pl.kblocks[kQKV], o + pl.pk_wqkv, st);
      if (!rc) rc = pack_matrix(s + pl.hyb_off_wo, d, HD, 0, pl.tiles[kO], pl.kblocks[kO], o + pl.pk_wo, st);
    } else {
      if (!rc)
        rc = pack_matrix(s + pl.hyb_off_w_in, pl.in_rows, d, 0, pl.tiles[kIn], pl.kblocks[kIn], o + pl.pk_w_in, st);
      if (!rc)
        rc = pack_matrix(s + pl.hyb_off_w_out, d, pl.d_inner, 0, pl.tiles[kOut], pl.kblocks[kOut], o + pl.pk_w_out,
                         st);
      if (!rc) rc = copy_vec(s + pl.hyb_off_a_log, 3LL * hc.ssm_heads, o + pl.pk_a_log, st);
    }
  }
  return rc;
}

}  // namespace wave
