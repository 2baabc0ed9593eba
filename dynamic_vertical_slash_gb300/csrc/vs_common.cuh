// Definitions shared by the library's host code and kernels: the index arena
// layout, global-position maps of the striped mode, and small device helpers.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include "../../include/vs.h"

namespace vs {

constexpr int kBlk = 64;        // key block / stripe granularity (section 4.1 (ii), 4.2 (ii))
constexpr int kQTile = 128;     // query rows per tcgen05 tile (MMA M = 128)
constexpr int kKTile = 64;      // keys per slash tile / query-major bar chunk
constexpr int kBarK = 128;      // keys per key-major bar chunk (MMA M = 128)
constexpr int kRowTile = 64;    // query rows per key-major unit
constexpr int kBarSplitTiles = 256;  // row tiles per key-major bar work item
constexpr int32_t kArenaMagic = 0x56534958;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Index arena.  All offsets are bytes from the arena base; every section is
// 256-byte aligned.  Per (b, h) records are indexed by bh = b * Hq + h.
struct ArenaHeader {
  int32_t status;   // device status word (vs_status)
  int32_t magic;
  int32_t B, Hq, Nq, Nk, kv, ks;
  int32_t world, stripe, q_rank, kv_rank;
  int64_t N_global;
  int32_t WG;       // uint64 words per global bitmap (selected offsets / columns)
  int32_t WL;       // uint64 words per local-key bitmap
  int32_t EMAX;     // capacity of the e / f lists
  int32_t KVP;      // capacity of the vertical list (kv rounded up to 128)
  int32_t sheared;  // 1: unstriped sheared cover; 0: block-aligned striped cover
  int32_t block_cover;  // 1: slashes cover whole 64 x 64 blocks (bdbits); 0: the exact token mask
  int64_t off_offbits, off_colbits, off_elist, off_ecount, off_flist, off_fcount;
  int64_t off_vlist, off_vcount, off_vlocbits, off_vlocpre, off_counts;
  int64_t total_bytes;
  int64_t off_bdbits;
  int32_t pack;  // GQA packing: g (query-major tiles of 128 / g tokens x g heads), 0 = one head per tile
};
static_assert(sizeof(ArenaHeader) <= 256, "arena header exceeds 256 bytes");

// Device view of an arena.
struct ArenaView {
  const ArenaHeader* hdr;
  const uint64_t* offbits;   // [BH][WG]   bit o: offset o selected
  const uint64_t* colbits;   // [BH][WG]   bit c: column c selected (global)
  const int32_t* elist;      // [BH][EMAX] query-major slash list (ascending)
  const int32_t* ecount;     // [BH]
  const int32_t* flist;      // [BH][EMAX] key-major slash list (ascending)
  const int32_t* fcount;     // [BH]
  const int32_t* vlist;      // [BH][KVP]  local key index of selected columns in this shard (-1 pad)
  const int32_t* vcount;     // [BH]
  const uint64_t* vlocbits;  // [BH][WL]   bit k: local key k is a selected column
  const int32_t* vlocpre;    // [BH][WL]   selected columns in words before w
  const uint64_t* bdbits;    // [BH][WG]   block mode: bit D: a selected slash passes through block diagonal D
};

__host__ __device__ inline ArenaView arena_view(const void* base) {
  const uint8_t* p = static_cast<const uint8_t*>(base);
  const ArenaHeader* h = reinterpret_cast<const ArenaHeader*>(p);
  ArenaView v;
  v.hdr = h;
  v.offbits = reinterpret_cast<const uint64_t*>(p + h->off_offbits);
  v.colbits = reinterpret_cast<const uint64_t*>(p + h->off_colbits);
  v.elist = reinterpret_cast<const int32_t*>(p + h->off_elist);
  v.ecount = reinterpret_cast<const int32_t*>(p + h->off_ecount);
  v.flist = reinterpret_cast<const int32_t*>(p + h->off_flist);
  v.fcount = reinterpret_cast<const int32_t*>(p + h->off_fcount);
  v.vlist = reinterpret_cast<const int32_t*>(p + h->off_vlist);
  v.vcount = reinterpret_cast<const int32_t*>(p + h->off_vcount);
  v.vlocbits = reinterpret_cast<const uint64_t*>(p + h->off_vlocbits);
  v.vlocpre = reinterpret_cast<const int32_t*>(p + h->off_vlocpre);
  v.bdbits = reinterpret_cast<const uint64_t*>(p + h->off_bdbits);
  return v;
}

// The low n bits set (n clipped to [0, 64]).
__host__ __device__ __forceinline__ uint64_t low_bits(int64_t n) {
  return n >= 64 ? ~0ull : (n <= 0 ? 0ull : ((1ull << n) - 1));
}

// Plain (host-side) copy of the geometry the kernels need, passed by value.
struct Geo {
  int B, Nq, Nk, Hq, Hkv, d, g;
  int world, q_rank, kv_rank;
  int WG, WL, EMAX, KVP;
  int64_t N_global;
};

// Local 64-token block j of the query (key) tensor is global block
// world * j + q_rank (kv_rank): the striped shards of a ring (ranks below
// world) and contiguous windows of the sequence (world 1, rank = the window's
// first block, e.g. the two chunks of a ZigZag worker) are both of this form.
// Global position of a local query row / key:
__host__ __device__ __forceinline__ int64_t qpos_g(const Geo& G, int64_t l) {
  return (int64_t(G.world) * (l >> 6) + G.q_rank) * kBlk + (l & 63);
}
__host__ __device__ __forceinline__ int64_t kpos_g(const Geo& G, int64_t l) {
  return (int64_t(G.world) * (l >> 6) + G.kv_rank) * kBlk + (l & 63);
}

// The first local 64-row block whose rows can attend global key position
// m_g: the smallest rb >= 0 with qpos_g(64 rb + 63) >= m_g.
__host__ __device__ __forceinline__ int64_t first_causal_row_block(int world, int q_rank, int64_t m_g) {
  const int64_t num = (m_g >> 6) - q_rank;
  return num <= 0 ? 0 : (num + world - 1) / world;
}

// Local index of global key position x in a key window of Nk tokens, or -1
// when the window does not hold it.
__host__ __device__ __forceinline__ int64_t local_key_of(int world, int kv_rank, int64_t Nk, int64_t x) {
  const int64_t rb = (x >> 6) - kv_rank;
  if (rb < 0 || rb % world) return -1;
  const int64_t lb = rb / world;
  return lb < Nk / kBlk ? lb * kBlk + (x & 63) : -1;
}

// Bits [lo, lo + 64) of a bitmap of `nwords` words; positions outside the
// bitmap read as 0.  Bit j of the result is bitmap bit lo + j.
__device__ __forceinline__ uint64_t bits64(const uint64_t* bm, int64_t lo, int nwords) {
  const int64_t w = lo >> 6;  // floor division (arithmetic shift)
  const int sh = int(lo & 63);
  const uint64_t a = (w >= 0 && w < nwords) ? __ldg(bm + w) : 0ull;
  const uint64_t b = (w + 1 >= 0 && w + 1 < nwords) ? __ldg(bm + w + 1) : 0ull;
  return sh ? ((a >> sh) | (b << (64 - sh))) : a;
}

// Number of entries of an ascending list that are <= x (binary search).
__device__ __forceinline__ int count_le(const int32_t* list, int n, int64_t x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(list + mid) <= x) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// Query-major work of the tile of R tokens starting at local row r0 (R = 128,
// or 128 / g with GQA packing) of head bh: its slash units are
// elist[lo, lo + nslash) (the entries e <= r0 + R - 1 whose 64 keys
// c = r0 + R - 64 - e start before Nk), its bar chunks the first nbar chunks
// of the vertical list (those whose first column is not after, on global
// positions, the tile's last row).
struct TileWork {
  int lo, nslash, nbar;
};
__device__ __forceinline__ TileWork tile_work(const ArenaView& av, const Geo& G, int64_t bh, int64_t r0, int R) {
  TileWork w;
  const int32_t* elist = av.elist + bh * G.EMAX;
  const int ne = __ldg(av.ecount + bh);
  const int64_t last_row = r0 + R - 1;
  w.lo = count_le(elist, ne, r0 + R - 64 - G.Nk);
  w.nslash = count_le(elist, ne, last_row) - w.lo;
  const int32_t* vlist = av.vlist + bh * G.KVP;
  const int vc = __ldg(av.vcount + bh);
  const int64_t last_g = qpos_g(G, last_row);
  int lo = 0, hi = (vc + kKTile - 1) / kKTile;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (kpos_g(G, __ldg(vlist + mid * kKTile)) <= last_g) lo = mid + 1;
    else hi = mid;
  }
  w.nbar = lo;
  return w;
}

}  // namespace vs
