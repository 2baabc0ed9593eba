// Sparse attention forward on the Vertical-Slash mask (tcgen05 / TMEM / TMA).
//
// One CTA owns one query tile (128 rows of one query head, or with GQA
// packing 128 / g tokens of the g heads of a KV group) and walks its units
//   * slash tiles: 64 keys starting at local key c = r0 + R - 64 - e for every
//     entry e of the head's query-major list that reaches the tile, by TMA;
//   * bar chunks: 64 selected columns gathered with cp.async
// two at a time: a pair of units is one 128-key block, so S = Q K^T is one
// M=128, N=128 MMA chain and O += P V one K=128 chain (an odd last unit
// leaves the second half of its pair masked and out of the PV chain).
//
// Warp roles (384 threads): warp 0 loads the K blocks, warp 11 the V
// blocks, warp 10 publishes, per unit, the few words every row's mask is cut
// from, warp 1 issues the MMAs (the whole warp runs the loop, an elected lane
// issues), warps 2-9 run the softmax: every pair goes through all eight, the
// two warps of a TMEM lane quarter holding the same 32 rows, one the pair's
// first unit and one its second.  fp32 online softmax on the exact token mask
// in registers, P (bf16) over the first half of the unit's own score columns.
//
// TMEM columns: O [0, d), score buffers S_j [128 + 128 j, +128) for j < 3
// (unit u's scores in [64 u, +64), then its P as bf16 pairs in [64 u,
// +32)).  Q sits in shared memory (one TMA load per tile), so every S = Q K^T
// chain reads both operands from there.  S of pair i goes to buffer i % 3.
// The MMA order is S0 S1 S2, then per pair i: PV_i (once P_i is stored),
// S_{i+3} into buffer i % 3 (the pipe runs them in order, so PV_i has read
// P_i by then): the scores of the next two pairs are computed while pair i
// is in softmax.  P_i overwrites scores the softmax already holds, so it is
// stored without waiting for any PV.  The row's reference maximum is lazy
// (it moves only for the row's first entries or an entry 2^64 above it); the
// two threads of a row agree on it through a named barrier of their two
// warps, and before O is rescaled every PV issued so far has completed.
//
// Shared memory: the tile's Q, a ring of five slots that each hold K or V
// of one pair (128 rows), filled and released in the MMA's order K0 K1 K2
// V0 K3 V1 K4 ..., and a ring of per-pair mask records.
#include "vs_internal.h"
#include "vs_kernel_common.cuh"

namespace vs {
namespace {

constexpr int kFwdThreads = 384;
constexpr int kFwdRecWarp = 10;
constexpr int kFwdVWarp = 11;
constexpr int kFwdSoftmax = 256;  // softmax threads (warps 2-9): two per row, one per unit of a pair
constexpr int kPairKeys = 2 * kKTile;
constexpr int kFwdSlots = 5;
constexpr int kRecRing = 8;
constexpr int kSBufs = 3;  // score buffers: S of pair i + 3 is issued right after pair i's PV
constexpr uint32_t kColO = 0, kColS = 128, kTmemCols = 512;
constexpr float kRefSlack = 18446744073709551616.0f;  // 2^64: largest masked pair sum accepted against the reference

// What a unit's 128 row masks are cut from (written by the loader).
//   slash tile: bits [L0 + i, L0 + i + 64) of the head's offset bitmap give
//     row i of a 64-row block (reversed: bit k <-> offset base - k), with
//     L0 = n_g(block row 0) - m_g(first key) - 63; W holds the three bitmap
//     words from floor(L0 / 64) of both blocks, lo6 = L0 mod 64, and keep
//     clears the selected columns (owned by the bars) and keys before 0;
//   bar chunk: the 64 keys' global positions, ascending (padding last), so a
//     row's mask is the prefix of keys at or before it.
struct MaskRec {
  int kind;  // 0: no unit (odd last pair), 1: slash tile, 2: bar chunk
  int lo6[2];         // bit offsets of the row blocks' windows in W
  uint64_t W[6];      // per row block, three words of the offset bitmap around its window
  uint64_t keep[2];   // per row block: keys that may be set (not a selected column, existing, and
                      // in block-cover mode on an active block diagonal of that row block)
  int64_t kg[kKTile];
};

// The mask of the row whose token is the tile's token r (bit k: key k of the
// unit), from its unit's record.
template <bool BLOCK>
__device__ __forceinline__ uint64_t rec_row_mask(const MaskRec& rc, int kind, int r, int64_t ng) {
  if (kind == 1) {
    const int blk = r >> 6;
    const int o = rc.lo6[blk] + (r & 63);
    const uint64_t a = rc.W[3 * blk + (o >> 6)], b = rc.W[3 * blk + (o >> 6) + 1];
    const int sh = o & 63;
    const uint64_t x = sh ? ((a >> sh) | (b << (64 - sh))) : a;
    return __brevll(x) & rc.keep[BLOCK ? blk : 0];
  }
  if (kind == 2) {
    int pos = 0;
#pragma unroll
    for (int step = 32; step > 0; step >>= 1)
      if (rc.kg[pos + step - 1] <= ng) pos += step;
    const int cnt = (rc.kg[kKTile - 1] <= ng) ? kKTile : pos;
    return cnt == kKTile ? ~0ull : ((1ull << cnt) - 1);
  }
  return 0ull;
}

template <int D>
struct FwdSmem {
  static constexpr int NH = D / 64;
  uint8_t slot[kFwdSlots][NH][kPairKeys * 128];  // K or V of one pair, 128B-swizzled, per d-half
  uint8_t q[NH][kQTile * 128];                    // the tile's Q: A operand of every S = Q K^T
  MaskRec rec[kRecRing][2];                      // mask records of a pair's two units
  uint64_t q_full;  // the tile's Q (TMA)
  uint64_t slot_full[kFwdSlots], slot_empty[kFwdSlots];
  uint64_t rec_full[kRecRing], rec_empty[kRecRing];
  uint64_t s_full[kSBufs], p_full[kSBufs];  // per score buffer
  uint64_t pv_done[kSBufs];  // PV of pair i completes on pv_done[i % kSBufs]
  uint64_t o_final, teardown;
  float red_m[2][kQTile];  // per half (unit of a pair): masked maximum, for re-basing
  float red_l[2][kQTile];  // per half: row sum
  uint32_t tmem_base;
  int abort_flag;
};

struct FwdParams {
  const void* arena;
  const uint8_t* q;  // Q base (bytes)
  const uint8_t* k;
  const uint8_t* v;
  int64_t sq[3], sk[3], sv[3], so[3];
  int B, Nq, Hq, Hkv;
  float scale_log2;
  uint8_t* o;
  float* lse;
  float* o_acc;
  int* err;
};

// The order in which the MMA consumes K / V blocks (and the loader fills the
// slot ring): K0, K1, then per pair i: V_i, K_{i+2}.  One loop with one call
// of f, so that its body is emitted once per warp role (the roles' loops
// share the SM's instruction cache).
template <typename F>
__device__ __forceinline__ void for_each_block(int P, F&& f) {
  const int head = P < kSBufs ? P : kSBufs;  // K blocks before the first V
  const int mid = P > kSBufs ? P - kSBufs : 0;  // pairs followed by a K block
#pragma unroll 1
  for (int c = 0; c < 2 * P; ++c) {
    int kind, i;
    if (c < head) {
      kind = 0;
      i = c;
    } else if (c - head < 2 * mid) {
      const int e = c - head;
      kind = (e & 1) ? 0 : 1;
      i = (e >> 1) + ((e & 1) ? kSBufs : 0);
    } else {
      kind = 1;
      i = mid + (c - head - 2 * mid);
    }
    f(kind, i);
  }
}

// Re-basing helpers, out of line (rare: a row's first entries, or an entry
// 2^64 above the reference), so the common path keeps its registers.
// Masked maximum (log2 units) of one unit's 64 scores of the row, -inf if the
// mask is empty.  Warp-collective.
__device__ __noinline__ float fwd_unit_max(uint32_t taddr, uint64_t mask, float scale_log2) {
  uint32_t sr[64];
  tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
  tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
  tmem_ld_wait();
  float mx[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) mx[k] = -INFINITY;
#pragma unroll
  for (int k = 0; k < 64; ++k)
    if ((mask >> k) & 1ull) mx[k & 7] = fmaxf(mx[k & 7], __uint_as_float(sr[k]) * scale_log2);
  return fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
}
// O[row, c] *= alpha for the `ncols` accumulator columns at taddr.  Warp-collective.
__device__ __noinline__ void fwd_scale_o(uint32_t taddr, int ncols, float alpha) {
#pragma unroll 1
  for (int cc = 0; cc < ncols; cc += 16) {
    uint32_t ov[16];
    tmem_ld16(taddr + cc, ov);
    tmem_ld_wait();
#pragma unroll
    for (int k = 0; k < 16; ++k) ov[k] = __float_as_uint(__uint_as_float(ov[k]) * alpha);
    tmem_st16(taddr + cc, ov);
  }
  tmem_st_wait();
}

// The kernel body, compiled once per mask reading (BLOCK: block-cover
// slashes) so that neither reading carries the other's code.
template <int D, bool BLOCK>
__device__ __forceinline__ void fwd_body(const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmQ,
                                         const CUtensorMap& tmQp, const FwdParams& p) {
  constexpr int NH = D / 64;
  extern __shared__ uint8_t smem_raw[];
  FwdSmem<D>& s = *reinterpret_cast<FwdSmem<D>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  const ArenaView av = arena_view(p.arena);
  const Geo G = geo_from(av.hdr, p.Hkv, D);
  // A tile is R = 128 rows of one query head, or with GQA packing (gp = g)
  // R = 128 / g tokens of the g heads of a KV group: tile row r is token
  // r / gp of head h + r % gp.  Heavy (late) tiles first.
  const int gp = av.hdr->pack;
  const int R = gp ? kQTile / gp : kQTile;
  int t, b, h, hk;
  if (gp) {
    const int BHK = p.B * p.Hkv, TS = (p.Nq + R - 1) / R;
    if (int(blockIdx.x) >= TS * BHK) return;  // the grid is sized for unpacked tiles
    t = TS - 1 - int(blockIdx.x) / BHK;
    b = int(blockIdx.x) % BHK / p.Hkv;
    hk = int(blockIdx.x) % p.Hkv;
    h = hk * gp;
  } else {
    const int T = (p.Nq + kQTile - 1) / kQTile, BH = p.B * p.Hq;
    t = T - 1 - int(blockIdx.x) / BH;
    b = int(blockIdx.x) % BH / p.Hq;
    h = int(blockIdx.x) % p.Hq;
    hk = h / G.g;
  }
  const int bh = b * p.Hq + h;  // the lists of this head serve the whole tile
  const int64_t r0 = int64_t(t) * R;

  // Work list of this tile.
  // a workspace already holding an error makes the call skip its work
  const bool arena_ok = (av.hdr->status == 0) && (av.hdr->magic == kArenaMagic) &&
                        (*reinterpret_cast<volatile int*>(p.err) == 0);
  const TileWork tw = arena_ok ? tile_work(av, G, bh, r0, R) : TileWork{0, 0, 0};
  const int32_t* elist = av.elist + int64_t(bh) * G.EMAX + tw.lo;  // this tile's slash units
  const int32_t* vlist = av.vlist + int64_t(bh) * G.KVP;
  const int nslash = tw.nslash, nbar = tw.nbar;
  const int U = nslash + nbar;
  const int P = (U + 1) / 2;  // pairs
  // a pair holds a gathered (bar) half
  auto gathered = [&](int i) { return 2 * i + 1 >= nslash && 2 * i + 1 < U || 2 * i >= nslash; };

  if (threadIdx.x == 0) {
    if (!arena_ok && av.hdr->status) raise_error(p.err, av.hdr->status);
    else if (!arena_ok && av.hdr->magic != kArenaMagic) raise_error(p.err, VS_ERR_ARG);
    s.abort_flag = 0;
    mbar_init(&s.q_full, 1);
    for (int i = 0; i < kFwdSlots; ++i) {
      mbar_init(&s.slot_full[i], 1);
      mbar_init(&s.slot_empty[i], 1);
    }
    for (int i = 0; i < kRecRing; ++i) {
      mbar_init(&s.rec_full[i], 1);
      mbar_init(&s.rec_empty[i], kFwdSoftmax);
    }
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], kFwdSoftmax);
    }
    for (int i = 0; i < kSBufs; ++i) mbar_init(&s.pv_done[i], 1);
    mbar_init(&s.o_final, 1);
    mbar_init(&s.teardown, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  const Abort ab{&s.abort_flag, p.err};
  bool mma_issued = false;

  if (warp == 0 || warp == kFwdVWarp) {
    // ------------------------------------------------------------ producers
    // Warp 0 loads the K blocks, warp kFwdVWarp the V blocks.  Each walks
    // the whole block sequence (so both agree on every block's slot and
    // phase) and acts on its own kind only: one thread's TMA issue blocks
    // while the copy engine works through its boxes, so with two issuers the
    // engine never idles while the other does its bookkeeping.
    const int my_kind = warp == 0 ? 0 : 1;
    int issued[kFwdSlots];
    for (int i = 0; i < kFwdSlots; ++i) issued[i] = -1;
    if (P > 0) {
      if (lane == 0) {
        if (my_kind == 0) {
          prefetch_tmap(&tmK);
          // the tile's Q: R tokens of one head, or of the gp heads of a group
          mbar_arrive_expect_tx(&s.q_full, NH * kQTile * 128);
          for (int hf = 0; hf < NH; ++hf) tma_load_4d(s.q[hf], gp ? &tmQp : &tmQ, &s.q_full, 64 * hf, h, int(r0), b);
        } else {
          prefetch_tmap(&tmV);
        }
      }
      const uint8_t* base = my_kind ? p.v + (int64_t(b) * p.sv[0] + int64_t(hk) * p.sv[2]) * 2
                                    : p.k + (int64_t(b) * p.sk[0] + int64_t(hk) * p.sk[2]) * 2;
      const int64_t stok = my_kind ? p.sv[1] : p.sk[1];
      const CUtensorMap* tm = my_kind ? &tmV : &tmK;
      int c = 0;
      bool ok = true;
      int e_win = -1, e_pref = 0;  // elist[32 e_win + lane]
      for_each_block(P, [&](int kind, int i) {
        if (!ok) return;
        const int cb = c++;
        if (kind != my_kind) return;
        const int sl = cb % kFwdSlots;
        // first keys of the pair's slash halves (one 32-entry window of the
        // list per lane)
        int key0[2] = {0, 0};
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int u = 2 * i + hh;
          if (u >= nslash) continue;
          if ((u >> 5) != e_win) {
            e_win = u >> 5;
            const int j = 32 * e_win + lane;
            e_pref = j < nslash ? __ldg(elist + j) : 0;
          }
          key0[hh] = int(r0) + R - 64 - __shfl_sync(0xffffffffu, e_pref, u & 31);
        }
        if (cb >= kFwdSlots && !(ok = mbar_wait(&s.slot_empty[sl], ((cb / kFwdSlots) - 1) & 1, ab, VS_ERR_TIMEOUT)))
          return;
        uint32_t tma_bytes = 0;
        bool gath = false;
        for (int hh = 0; hh < 2; ++hh) {
          const int u = 2 * i + hh;
          if (u >= U) continue;
          if (u < nslash) {
            tma_bytes += NH * kKTile * 128;
          } else {
            gather_rows<D>(smem_u32(s.slot[sl][0]) + hh * kKTile * 128, kPairKeys, base, stok,
                           vlist + (u - nslash) * kKTile, kKTile, lane);
            gath = true;
          }
        }
        if (gath)
          asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(&s.slot_full[sl])) : "memory");
        __syncwarp();
        if (lane == 0) {
          if (tma_bytes) {
            mbar_arrive_expect_tx(&s.slot_full[sl], tma_bytes);
            for (int hh = 0; hh < 2; ++hh) {
              const int u = 2 * i + hh;
              if (u >= nslash) continue;
              for (int hf = 0; hf < NH; ++hf)
                tma_load_4d(s.slot[sl][hf] + hh * kKTile * 128, tm, &s.slot_full[sl], 64 * hf, hk, key0[hh], b);
            }
          } else {
            mbar_arrive(&s.slot_full[sl]);
          }
        }
        issued[sl] = cb;
        __syncwarp();
      });
    }
    if (lane == 0 && s.abort_flag && my_kind == 0 && P > 0) {
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(&s.q_full, 0) && global_ns() - t0 < kWaitBudgetNs) {
      }
    }
    if (lane == 0 && s.abort_flag) {
      // drain loads still in flight before the CTA's shared memory is released
      for (int i = 0; i < kFwdSlots; ++i)
        if (issued[i] >= 0) {
          const uint64_t t0 = global_ns();
          while (!mbar_try_wait(&s.slot_full[i], (issued[i] / kFwdSlots) & 1) && global_ns() - t0 < kWaitBudgetNs) {
          }
        }
    }
  } else if (warp == kFwdRecWarp) {
    // ------------------------------------------------------------ mask records
    // Per pair: the bitmap words of its slash tiles (lanes 0-7 for the first
    // unit, 8-15 for the second) and the key positions of its bar chunks are
    // all requested before any is used, so a pair costs one memory round
    // trip; runs as far ahead as the record ring allows.
    const uint64_t* offbits_p = av.offbits + int64_t(bh) * G.WG;
    const uint64_t* colbits_p = av.colbits + int64_t(bh) * G.WG;
    constexpr bool block_cover = BLOCK;
    const uint64_t* bdbits_p = av.bdbits + int64_t(bh) * G.WG;
    int e_win = -1, e_pref = 0;  // elist[32 e_win + lane]
    for (int i = 0; i < P; ++i) {
      const int ri = i % kRecRing;
      if (i >= kRecRing && !mbar_wait(&s.rec_empty[ri], ((i / kRecRing) - 1) & 1, ab, VS_ERR_TIMEOUT)) break;
      int kind[2];
      int64_t cc[2], m0[2], L0a[2], L0b[2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int u = 2 * i + hh;
        kind[hh] = (u >= U) ? 0 : (u < nslash ? 1 : 2);
        cc[hh] = 0;
        if (kind[hh] == 1) {
          if ((u >> 5) != e_win) {
            e_win = u >> 5;
            const int j = 32 * e_win + lane;
            e_pref = j < nslash ? __ldg(elist + j) : 0;
          }
          cc[hh] = r0 + R - 64 - __shfl_sync(0xffffffffu, e_pref, u & 31);
        }
        m0[hh] = (cc[hh] >= 0) ? kpos_g(G, cc[hh]) : cc[hh];  // c < 0 only without striping
        L0a[hh] = qpos_g(G, r0) - m0[hh] - 63;
        L0b[hh] = qpos_g(G, r0 + 64) - m0[hh] - 63;
      }
      // issue every load of the pair
      uint64_t wv = 0;
      {
        const int hh = lane >> 3, j = lane & 7;
        const bool sec = hh == 1;  // lanes 8-15 serve the second unit
        const int kh = sec ? kind[1] : kind[0];
        if (hh < 2 && kh == 1) {
          const int64_t la = sec ? L0a[1] : L0a[0], lb = sec ? L0b[1] : L0b[0], mm = sec ? m0[1] : m0[0];
          const int64_t w = j < 6 ? (((j < 3 ? la : lb) >> 6) + j % 3) : ((mm >> 6) + (j - 6));
          if (block_cover && j < 6) {
            // block cover: the words of "offset >= 0" (the causal entries);
            // the active block diagonals go into the row blocks' keep masks
            const int64_t base = 64 * w;
            wv = base >= 0 ? ~0ull : ~low_bits(-base);
          } else {
            const uint64_t* bm = j < 6 ? offbits_p : colbits_p;
            wv = (w >= 0 && w < G.WG) ? __ldg(bm + w) : 0ull;
          }
        } else if (block_cover && lane >= 16 && lane < 20) {
          // lanes 16 + 2 u + b: unit u, row block b: the diagonals through
          // the unit's two key blocks (bits D2 = I - J - 1 and D2 + 1)
          const int u = (lane - 16) >> 1, rb = lane & 1;
          if (kind[u] == 1) {
            const int64_t D2 = (qpos_g(G, r0 + 64 * rb) >> 6) - (m0[u] >> 6) - 1;
            wv = bits64(bdbits_p, D2, G.WG) & 3ull;
          }
        }
      }
      int key[2][2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int e = 0; e < 2; ++e)
          key[hh][e] = kind[hh] == 2 ? __ldg(vlist + (2 * i + hh - nslash) * kKTile + e * 32 + lane) : -1;
      // publish
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        MaskRec& rc = s.rec[ri][hh];
        if (kind[hh] == 1) {
          const uint64_t c1 = __shfl_sync(0xffffffffu, wv, 8 * hh + 7);
          const uint64_t a0 = __shfl_sync(0xffffffffu, wv, 16 + 2 * hh), a1 = __shfl_sync(0xffffffffu, wv, 17 + 2 * hh);
          if ((lane >> 3) == hh) {
            const int j = lane & 7;
            if (j < 6) rc.W[j] = wv;
            if (j == 6) {
              const int shc = int(m0[hh] & 63);
              const uint64_t colw = shc ? ((wv >> shc) | (c1 << (64 - shc))) : wv;
              // keys that exist: c + k in [0, Nk)
              const uint64_t keep =
                  ~colw & ((cc[hh] < 0) ? ((~0ull) << (-cc[hh])) : ~0ull) & low_bits(int64_t(G.Nk) - cc[hh]);
              if (block_cover) {
                // keys below the split lie in the first key block (diagonal
                // D2 + 1, bit 1), the rest in the next (D2, bit 0)
                const uint64_t lo_keys = low_bits(64 - (m0[hh] & 63));
                rc.keep[0] = keep & (((a0 & 2ull) ? lo_keys : 0ull) | ((a0 & 1ull) ? ~lo_keys : 0ull));
                rc.keep[1] = keep & (((a1 & 2ull) ? lo_keys : 0ull) | ((a1 & 1ull) ? ~lo_keys : 0ull));
              } else {
                rc.keep[0] = rc.keep[1] = keep;
              }
            }
          }
          if (lane == 0) {
            rc.lo6[0] = int(L0a[hh] & 63);
            rc.lo6[1] = int(L0b[hh] & 63);
          }
        } else if (kind[hh] == 2) {
#pragma unroll
          for (int e = 0; e < 2; ++e) rc.kg[e * 32 + lane] = key[hh][e] >= 0 ? kpos_g(G, key[hh][e]) : INT64_MAX;
        }
        if (lane == 0) rc.kind = kind[hh];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.rec_full[ri]);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // S of pair i goes to score buffer i % 3.  Order: S0, S1, S2, then per
    // pair i: PV_i (once its P is in buffer i % 3), S_{i+3} into the same
    // buffer (the tensor pipe runs them in order, so PV_i has read P_i).  The
    // whole warp runs the loop; one elected lane issues.
    if (P > 0) {
      const uint32_t idS = idesc_bf16(128, kPairKeys, 0, 0);
      const uint32_t idO = idesc_bf16(128, D, 0, 1);
      // descriptors of slot 0 as a K block (K-major) and as a V block
      // (MN-major); another slot's and K-chunk's are these plus the offset
      // (shared addresses stay below 256 KB: the 14-bit start field never
      // carries)
      const uint64_t dk0 = sdesc_sw128(smem_u32(s.slot[0][0]), 16, 1024);
      const uint64_t dv0 = sdesc_sw128(smem_u32(s.slot[0][0]), kPairKeys * 128, 1024);
      constexpr uint32_t kSlotDesc = uint32_t(NH * kPairKeys * 128) >> 4;
      const uint64_t dq0 = sdesc_sw128(smem_u32(s.q[0]), 16, 1024);
      bool ok = mbar_wait_warp(&s.q_full, 0, ab, VS_ERR_TIMEOUT);
      int c = 0;
      for_each_block(P, [&](int kind, int i) {
        if (!ok) return;
        const int j = i % kSBufs;
        if (kind) {
          if (!(ok = mbar_wait_warp(&s.p_full[j], (i / kSBufs) & 1, ab, VS_ERR_TIMEOUT))) return;
        }
        const int sl = c % kFwdSlots;
        if (!(ok = mbar_wait_warp(&s.slot_full[sl], (c / kFwdSlots) & 1, ab, VS_ERR_TIMEOUT))) return;
        if (gathered(i)) fence_proxy_async_smem();
        tc_fence_after();
        if (!kind) {
          const uint64_t dks = dk0 + uint64_t(sl) * kSlotDesc;
          // A = Q, B = K, both in shared memory; one K-chunk of 16 per MMA
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t a = dq0 + (uint32_t((kk / 4) * kQTile * 128 + (kk % 4) * 32) >> 4);
            const uint64_t bk = dks + (uint32_t((kk / 4) * kPairKeys * 128 + (kk % 4) * 32) >> 4);
            mma_ss_warp(tmem + kColS + 128 * j, a, bk, idS, kk > 0);
          }
          mma_commit_warp(&s.s_full[j]);
        } else {
          const uint64_t dvs = dv0 + uint64_t(sl) * kSlotDesc;
          // per unit of the pair four K-chunks of 16 keys, one elect; A = P
          // of the unit in TMEM (an odd last unit's second half is left out)
          const int nu = (2 * i + 1 < U) ? 2 : 1;
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            if (u >= nu) break;
            const uint64_t b = dvs + uint32_t(u * 4 * 2048 >> 4);
            const uint32_t a = tmem + kColS + 128 * j + u * 64;
            mma_ts_chain4_warp(tmem + kColO, a, a + 8, a + 16, a + 24, b, b + 128, b + 256, b + 384, idO, i > 0 || u > 0);
          }
          mma_commit_warp(&s.pv_done[j]);
        }
        mma_commit_warp(&s.slot_empty[sl]);
        mma_issued = true;
        ++c;
      });
      mma_commit_warp(&s.o_final);
    }
  } else if (warp >= 2 && warp < 2 + 8) {
    // ------------------------------------------------------------ softmax
    // Every pair goes through all eight warps: the warps of TMEM lane quarter
    // q (warps 2 + q' with q' & 3 == q) hold rows 32 q .. 32 q + 31, one the
    // pair's first unit (keys 0-63), the other its second.  The two threads
    // of a row keep one reference maximum m_run (log2 units) and each its
    // own partial sum; O has one accumulator.
    const int half = (warp - 2) >> 2;        // which unit of each pair
    const int quarter = warp & 3;            // TMEM lane quarter this warp may access
    const int r = quarter * 32 + lane;       // query row within the tile
    const int ti = gp ? r / gp : r;          // its token within the tile
    const int hrow = gp ? h + r % gp : h;    // and its query head
    const uint32_t tl = tmem + (uint32_t(quarter * 32) << 16);
    const int64_t n_loc = r0 + ti;
    const bool row_ok = n_loc < p.Nq;
    const int qbar = 2 + quarter;            // named barrier of the quarter's two warps
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    const int64_t n_g = qpos_g(G, n_loc);
    // A unit's row mask is cut from its record (published well ahead) one
    // pair early: the mask of pair i + 1 while the scores of pair i are on
    // their way from TMEM, so the record's shared-memory latency is hidden.
    bool rec_ok = true;
    auto cut_mask = [&](int i2) {
      const int ri2 = i2 % kRecRing;
      rec_ok = mbar_wait(&s.rec_full[ri2], (i2 / kRecRing) & 1, ab, VS_ERR_TIMEOUT);
      uint64_t m = 0ull;
      if (rec_ok && row_ok) {
        const MaskRec& rc = s.rec[ri2][half];
        m = rec_row_mask<BLOCK>(rc, rc.kind, ti, n_g);
      }
      mbar_arrive(&s.rec_empty[ri2]);
      return m;
    };
    uint64_t mask_nx = 0ull;
    if (P > 0) {
      mask_nx = cut_mask(0);
      ok = __all_sync(0xffffffffu, rec_ok);
    }
    for (int i = 0; ok && i < P; ++i) {
      const int j = i % kSBufs;
      const uint32_t colS = kColS + 128 * j + 64 * half;  // this unit's scores
      const uint64_t mask = mask_nx;
      // the 16-key chunks holding a mask entry of any of the warp's rows
      // (warp-uniform): the others' numerators are zero without arithmetic
      const uint32_t occ = chunk_occupancy16(mask);
      ok = mbar_wait(&s.s_full[j], (i / kSBufs) & 1, ab, VS_ERR_TIMEOUT);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // P against the row's reference maximum m_run.  The reference is lazy:
      // it only moves when a unit's masked sum shows an entry more than 2^64
      // above it (or for the row's first entries); the sum bounds every
      // single entry, so P stays <= 2^64.
      uint32_t pk[32];
      float unit_sum;
      auto make_p = [&](float ref, bool next_mask) {
        // two keys at a time in paired fp32: t = S scale log2(e) - ref, and
        // four pairs of partial row sums
        uint64_t ps2[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) ps2[k] = 0ull;
        const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2), nref2 = f2_pack(-ref, -ref);
        uint32_t sr[64];
        tmem_ld32(tl + colS, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tmem_ld32(tl + colS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        if (next_mask) mask_nx = cut_mask(i + 1);
        tmem_ld_wait_dep(*reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        reg_dep(*reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        const uint32_t mlo = uint32_t(mask), mhi = uint32_t(mask >> 32);
#pragma unroll
        for (int cq = 0; cq < 4; ++cq) {
          if (!((occ >> cq) & 1u)) {
#pragma unroll
            for (int k = 8 * cq; k < 8 * cq + 8; ++k) pk[k] = 0u;
            continue;
          }
#pragma unroll
          for (int k = 8 * cq; k < 8 * cq + 8; ++k) {
            // bits 2k, 2k + 1 of the mask select the numerator or zero
            const uint32_t w = k < 16 ? mlo : mhi;
            float t0, t1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * k]), __uint_as_float(sr[2 * k + 1])), sc2, nref2), t0, t1);
            const float p0 = ((w >> ((2 * k) & 31)) & 1u) ? ex2(t0) : 0.f;
            const float p1 = ((w >> ((2 * k + 1) & 31)) & 1u) ? ex2(t1) : 0.f;
            ps2[k & 3] = f2_add(ps2[k & 3], f2_pack(p0, p1));
            pk[k] = pack_bf16x2(p0, p1);
          }
        }
        float s0, s1, s2, s3, s4, s5, s6, s7;
        f2_unpack(ps2[0], s0, s1);
        f2_unpack(ps2[1], s2, s3);
        f2_unpack(ps2[2], s4, s5);
        f2_unpack(ps2[3], s6, s7);
        unit_sum = ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
      };
      // one copy of the unit body (the hot loops of all warp roles share the
      // SM's instruction cache): a second pass only after a re-basing
#pragma unroll 1
      for (int pass = 0;; ++pass) {
        make_p(m_run == -INFINITY ? 0.f : m_run, pass == 0 && i + 1 < P);
        if (pass) break;
        const bool need = (mask != 0ull) && (m_run == -INFINITY || !(unit_sum <= kRefSlack));
        // both threads of a row see the same decision
        if (!bar_sync_or(qbar, 64, need)) break;
        // re-base: the row's new reference is the masked maximum of the
        // pair (both units); where it grows, O (this thread's half of the
        // columns, once every PV issued so far has completed) and the running
        // sum are rescaled; then P is made again against the new reference
        s.red_m[half][r] = fwd_unit_max(tl + colS, mask, p.scale_log2);
        bar_sync_and(qbar, 64, true);
        const float mt = fmaxf(s.red_m[0][r], s.red_m[1][r]);
        bar_sync_and(qbar, 64, true);  // both have read red_m before the next pair may write it
        const bool grow = (m_run != -INFINITY) && (mt > m_run);
        if (__any_sync(0xffffffffu, grow)) {
          // PV_{i-1} complete implies every earlier PV is (in-order pipe).  S_i
          // having completed implies PV_{i-kSBufs} has, so the barrier of
          // PV_{i-1} is at most one phase behind it and its parity identifies it.
          if (i > 0 && !mbar_wait(&s.pv_done[(i - 1) % kSBufs], ((i - 1) / kSBufs) & 1, ab, VS_ERR_TIMEOUT))
            ok = false;
          if (!__all_sync(0xffffffffu, ok)) break;
          tc_fence_after();
          const float alpha = grow ? ex2(m_run - mt) : 1.f;
          fwd_scale_o(tl + kColO + (D / 2) * half, D / 2, alpha);
          if (grow) l_run *= alpha;
        }
        if (m_run == -INFINITY || grow) m_run = mt;
      }
      if (!__all_sync(0xffffffffu, ok && rec_ok)) {
        ok = false;
        break;
      }
      // P over the first 32 of the unit's own score columns (its scores are
      // in registers; S_{i+2} overwrites the buffer only after PV_i has read
      // P_i, in the pipe's order)
      tmem_st16(tl + colS, *reinterpret_cast<uint32_t(*)[16]>(&pk[0]));
      tmem_st16(tl + colS + 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[16]));
      l_run += unit_sum;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&s.p_full[j]);
    }
    // -------------------------------------------------------------- epilogue
    // Wait for every MMA, add the row's two partial sums; each half writes
    // columns [half d/2, (half + 1) d/2) of the row.
    bool e_ok = ok && (P == 0 || mbar_wait(&s.o_final, 0, ab, VS_ERR_TIMEOUT));
    e_ok = __all_sync(0xffffffffu, e_ok);
    s.red_l[half][r] = l_run;
    e_ok = bar_sync_and(1, kFwdSoftmax, e_ok);
    tc_fence_after();
    if (e_ok) {
      const float l_tot = s.red_l[0][r] + s.red_l[1][r];
      const bool empty = !(l_tot > 0.f);
      const float inv = empty ? 0.f : 1.f / l_tot;
      const float lse_step = empty ? -INFINITY : (m_run + __log2f(l_tot)) * kLn2;
      float* lse_p = p.lse + (int64_t(b) * p.Hq + hrow) * p.Nq + n_loc;
      uint8_t* orow = p.o + (int64_t(b) * p.so[0] + n_loc * p.so[1] + int64_t(hrow) * p.so[2]) * 2;
      float wa = 0.f, wb = 1.f, lse_new = lse_step;
      float* acc = nullptr;
      if (p.o_acc && row_ok) {
        acc = p.o_acc + ((int64_t(b) * p.Nq + n_loc) * p.Hq + hrow) * D;
        const float lse_old = *lse_p;
        if (lse_old == -INFINITY && empty) {
          lse_new = -INFINITY;
          wa = 0.f;
          wb = 0.f;
        } else {
          const float mx = fmaxf(lse_old, lse_step);
          lse_new = mx + __logf(__expf(lse_old - mx) + __expf(lse_step - mx));
          wa = (lse_old == -INFINITY) ? 0.f : __expf(lse_old - lse_new);
          wb = empty ? 0.f : __expf(lse_step - lse_new);
        }
      }
      // both halves have read lse_old before half 0 overwrites it
      bar_sync_and(1, kFwdSoftmax, true);
#pragma unroll 1
      for (int cc = (D / 2) * half; cc < (D / 2) * (half + 1); cc += 16) {
        uint32_t o0[16];
        if (P > 0) {  // warp-collective TMEM reads
          tmem_ld16(tl + kColO + cc, o0);
          tmem_ld_wait();
        }
        if (!row_ok) continue;
        float y[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) y[i] = (empty || P == 0) ? 0.f : __uint_as_float(o0[i]) * inv;
        if (acc) {
#pragma unroll
          for (int i = 0; i < 16; i += 4) {
            float4 a4 = *reinterpret_cast<float4*>(acc + cc + i);
            a4.x = wa * a4.x + wb * y[i];
            a4.y = wa * a4.y + wb * y[i + 1];
            a4.z = wa * a4.z + wb * y[i + 2];
            a4.w = wa * a4.w + wb * y[i + 3];
            *reinterpret_cast<float4*>(acc + cc + i) = a4;
            y[i] = a4.x;
            y[i + 1] = a4.y;
            y[i + 2] = a4.z;
            y[i + 3] = a4.w;
          }
        }
        uint4 w0, w1;
        w0.x = pack_bf16x2(y[0], y[1]);
        w0.y = pack_bf16x2(y[2], y[3]);
        w0.z = pack_bf16x2(y[4], y[5]);
        w0.w = pack_bf16x2(y[6], y[7]);
        w1.x = pack_bf16x2(y[8], y[9]);
        w1.y = pack_bf16x2(y[10], y[11]);
        w1.z = pack_bf16x2(y[12], y[13]);
        w1.w = pack_bf16x2(y[14], y[15]);
        *reinterpret_cast<uint4*>(orow + cc * 2) = w0;
        *reinterpret_cast<uint4*>(orow + cc * 2 + 16) = w1;
      }
      if (row_ok && half == 0) *lse_p = lse_new;
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (lane == 0 && mma_issued && s.abort_flag) {
      // make sure no MMA still writes TMEM before it is released
      mma_commit(&s.teardown);
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(&s.teardown, 0) && global_ns() - t0 < kWaitBudgetNs) {
      }
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
    vs_fwd_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmQp, const FwdParams p) {
  if (arena_view(p.arena).hdr->block_cover) fwd_body<D, true>(tmK, tmV, tmQ, tmQp, p);
  else fwd_body<D, false>(tmK, tmV, tmQ, tmQp, p);
}

template <int D>
vs_status launch_fwd_d(const vs_shape* sh, const void* q, const void* k, const void* v, const void* arena,
                       float scale, void* o, float* lse, float* o_acc, int* err, cudaStream_t st) {
  CUtensorMap tk, tv, tq, tqp;
  vs_status rc;
  if ((rc = make_tmap_bshd(&tk, k, sh->B, sh->Nk, sh->Hkv, D, sh->sk, kKTile)) != VS_OK) return rc;
  if ((rc = make_tmap_bshd(&tv, v, sh->B, sh->Nk, sh->Hkv, D, sh->sv, kKTile)) != VS_OK) return rc;
  // Q tiles: 128 rows of one head, or (GQA packing) 128 / g tokens of the g
  // heads of a KV group, token-major with the heads inside
  const int g = sh->Hq / sh->Hkv, gq = (kQTile % g == 0) ? g : 1;
  if ((rc = make_tmap_bshd(&tq, q, sh->B, sh->Nq, sh->Hq, D, sh->sq, kQTile)) != VS_OK) return rc;
  if ((rc = make_tmap_bshd(&tqp, q, sh->B, sh->Nq, sh->Hq, D, sh->sq, kQTile / gq, gq)) != VS_OK) return rc;
  FwdParams p;
  p.arena = arena;
  p.q = static_cast<const uint8_t*>(q);
  p.k = static_cast<const uint8_t*>(k);
  p.v = static_cast<const uint8_t*>(v);
  for (int i = 0; i < 3; ++i) {
    p.sq[i] = sh->sq[i];
    p.sk[i] = sh->sk[i];
    p.sv[i] = sh->sv[i];
    p.so[i] = sh->so[i];
  }
  p.B = sh->B;
  p.Nq = sh->Nq;
  p.Hq = sh->Hq;
  p.Hkv = sh->Hkv;
  p.scale_log2 = scale * kLog2e;
  p.o = static_cast<uint8_t*>(o);
  p.lse = lse;
  p.o_acc = o_acc;
  p.err = err;
  const size_t smem = sizeof(FwdSmem<D>) + 1024;
  if (cudaFuncSetAttribute(vs_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
    return VS_ERR_CUDA;
  const int T = (sh->Nq + kQTile - 1) / kQTile;
  const dim3 grid(unsigned(T) * sh->B * sh->Hq);
  trace_begin("fwd", st);
  vs_fwd_kernel<D><<<grid, kFwdThreads, smem, st>>>(tk, tv, tq, tqp, p);
  trace_end(st);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? VS_OK : VS_ERR_CUDA;
}

}  // namespace

vs_status launch_fwd(const vs_shape* s, const Geo&, const void* q, const void* k, const void* v, const void* arena,
                     float scale, void* o, float* lse, float* o_acc, int* err, cudaStream_t st) {
  if (s->d == 128) return launch_fwd_d<128>(s, q, k, v, arena, scale, o, lse, o_acc, err, st);
  if (s->d == 64) return launch_fwd_d<64>(s, q, k, v, arena, scale, o, lse, o_acc, err, st);
  return VS_ERR_SHAPE;
}

}  // namespace vs
