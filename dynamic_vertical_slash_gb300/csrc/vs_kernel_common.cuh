// Device helpers shared by the attention kernels: geometry from the arena
// header, per-unit masks, fast exp2, the bar-chunk gather.
#pragma once
#include "sm100_ptx.cuh"
#include "vs_common.cuh"

namespace vs {

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bit c (c < 4) set iff some lane of the warp has a set bit among bits
// [16 c, 16 c + 16) of its 64-bit mask: the 16-column chunks of a unit that
// hold any mask entry of the warp's 32 rows.  Warp-collective; the result is
// warp-uniform, so it may steer tcgen05.ld / tcgen05.st.
__device__ __forceinline__ uint32_t chunk_occupancy16(uint64_t mask) {
  uint32_t mine = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) mine |= ((mask >> (16 * c)) & 0xFFFFull) ? (1u << c) : 0u;
  return __reduce_or_sync(0xffffffffu, mine);
}

__device__ __forceinline__ Geo geo_from(const ArenaHeader* h, int Hkv, int d) {
  Geo G;
  G.B = h->B;
  G.Nq = h->Nq;
  G.Nk = h->Nk;
  G.Hq = h->Hq;
  G.Hkv = Hkv;
  G.d = d;
  G.g = h->Hq / Hkv;
  G.world = h->world;
  G.q_rank = h->q_rank;
  G.kv_rank = h->kv_rank;
  G.WG = h->WG;
  G.WL = h->WL;
  G.EMAX = h->EMAX;
  G.KVP = h->KVP;
  G.N_global = h->N_global;
  return G;
}

// Slash-tile masks of the 128 rows of query tile t against the 64 keys
// starting at local key c (query-major passes): bit k of row n's mask is set
// iff offset n_g - m_g(c + k) is selected, key c + k is not a selected column
// (vertical entries belong to the bars), and the key exists (c + k >= 0; c < 0
// only without striping).  The 64 keys are globally contiguous (unstriped, or
// c block-aligned).  Built by one warp: the lane's rows are rr * 32 + lane
// (rr = 0..3), returned in m[rr].  Within a 64-row block the rows' global
// positions are contiguous, so the offset windows of its 64 rows lie in three
// consecutive bitmap words; lanes 0-5 load the words of both blocks and lanes
// 6-7 the two column-bitmap words (one memory round trip per tile), and every
// row's window is cut out of the shuffled words.
__device__ __forceinline__ void slash_tile_masks(const Geo& G, const uint64_t* offbits, const uint64_t* colbits,
                                                 int t, int64_t c, int Nq, int lane, uint64_t (&m)[4]) {
  const int64_t m0 = (c >= 0) ? kpos_g(G, c) : c;
  int64_t L0[2];
#pragma unroll
  for (int blk = 0; blk < 2; ++blk) L0[blk] = qpos_g(G, int64_t(t) * kQTile + 64 * blk) - m0 - 63;
  uint64_t wv = 0;
  if (lane < 6) {
    const int64_t w = ((lane < 3 ? L0[0] : L0[1]) >> 6) + lane % 3;
    wv = (w >= 0 && w < G.WG) ? __ldg(offbits + w) : 0ull;
  } else if (lane < 8) {
    const int64_t w = (m0 >> 6) + (lane - 6);
    wv = (w >= 0 && w < G.WG) ? __ldg(colbits + w) : 0ull;
  }
  uint64_t W[6];
#pragma unroll
  for (int j = 0; j < 6; ++j) W[j] = __shfl_sync(0xffffffffu, wv, j);
  const uint64_t C0 = __shfl_sync(0xffffffffu, wv, 6), C1 = __shfl_sync(0xffffffffu, wv, 7);
  const int shc = int(m0 & 63);
  const uint64_t colw = shc ? ((C0 >> shc) | (C1 << (64 - shc))) : C0;
  const uint64_t keep = ~colw & ((c < 0) ? ((~0ull) << (-c)) : ~0ull);
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int blk = rr >> 1;
    const int o = int(L0[blk] & 63) + (rr & 1) * 32 + lane;  // bit offset in the block's first word, 0..126
    const uint64_t a = (o >> 6) ? W[3 * blk + 1] : W[3 * blk];
    const uint64_t b = (o >> 6) ? W[3 * blk + 2] : W[3 * blk + 1];
    const int sh = o & 63;
    const uint64_t x = sh ? ((a >> sh) | (b << (64 - sh))) : a;
    const int64_t nl = int64_t(t) * kQTile + rr * 32 + lane;
    m[rr] = nl < Nq ? (__brevll(x) & keep) : 0ull;
  }
}

// Key-major slash mask of one key (local index kl) against the 64 rows
// starting at local row r0: bit i set iff offset n_g(r0 + i) - m_g(kl) is
// selected and row r0 + i exists.  The caller clears the whole mask when the
// key is a selected column of the head.
__device__ __forceinline__ uint64_t slash_col_mask(const Geo& G, const uint64_t* offbits, int64_t kl, int64_t r0) {
  const int64_t base = qpos_g(G, r0) - kpos_g(G, kl);
  uint64_t m = bits64(offbits, base, G.WG);
  const int64_t rows = int64_t(G.Nq) - r0;
  if (rows < 64) m &= (rows <= 0) ? 0ull : ((1ull << rows) - 1);
  if (r0 < 0) m &= ~low_bits(-r0);  // rows before the query window
  return m;
}

// Block-cover counterpart of slash_col_mask: bit i set iff row r0 + i exists,
// is causal for the key (n_g >= m_g), and the 64 x 64 block of (row, key)
// lies on an active block diagonal (bdbits).  The unit's 64 rows are globally
// contiguous, so they span at most two row blocks.
__device__ __forceinline__ uint64_t block_col_mask(const Geo& G, const uint64_t* bdbits, int64_t kl, int64_t r0) {
  const int64_t n0 = qpos_g(G, r0), m = kpos_g(G, kl);
  const uint64_t a = bits64(bdbits, (n0 >> 6) - (m >> 6), G.WG);  // bit 0: rows' first block, bit 1: the next
  const uint64_t lo = low_bits(64 - (n0 & 63));
  uint64_t mask = ((a & 1ull) ? lo : 0ull) | ((a & 2ull) ? ~lo : 0ull);
  mask &= ~low_bits(m - n0);  // causal rows
  if (r0 < 0) mask &= ~low_bits(-r0);  // rows before the query window
  return mask & low_bits(int64_t(G.Nq) - r0);
}

// Issues the cp.async gather of `nrows` key rows (index list `keys`, -1 =
// zero row) of a [*, Hkv, d] bf16 tensor into a 128B-swizzled K-major tile:
// row r, 16-byte chunk j of half hf lands at dst + hf*rows*128 + r*128 +
// ((j ^ (r & 7)) * 16).  Called by all 32 lanes of a warp.
template <int D>
__device__ __forceinline__ void gather_rows(uint32_t dst, int rows_in_tile, const uint8_t* base, int64_t s_tok,
                                            const int32_t* keys, int nrows, int lane) {
  constexpr int NH = D / 64;
  for (int idx = lane; idx < nrows * 8 * NH; idx += 32) {
    const int r = idx / (8 * NH);
    const int rem = idx % (8 * NH);
    const int hf = rem / 8, j = rem % 8;
    const int key = __ldg(keys + r);
    const uint8_t* src = base + (key >= 0 ? int64_t(key) * s_tok * 2 : 0) + hf * 128 + j * 16;
    const uint32_t d = dst + hf * rows_in_tile * 128 + r * 128 + ((j ^ (r & 7)) << 4);
    cp_async_16(d, src, key >= 0 ? 16u : 0u);
  }
}

}  // namespace vs
