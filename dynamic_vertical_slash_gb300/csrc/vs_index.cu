// Sparse index construction (Algorithm 1 `sparseformat`, Algorithm 2
// `convert_index`).
//
// For every (b, h) the arena holds:
//   offbits / colbits  bitmaps of the selected offsets and columns (global);
//   elist / flist      the slash cover.  Unstriped, both hold the starts u of a
//                      greedy cover, by disjoint 64-wide intervals, of
//                      E = {u : some selected o in [u - 127, u]}: a query tile
//                      of 128 rows at r0 reads keys [r0 + 64 - u, r0 + 127 - u]
//                      and a key tile of 128 keys at k0 reads rows
//                      [k0 + u, k0 + u + 63]; together the intervals cover
//                      every entry with a selected offset exactly once.
//                      Striped (local block j = global block world j + rank,
//                      see vs_common.cuh), the cover is block-aligned: elist
//                      holds 64 (D + 1) for each active local block diagonal
//                      D of a (2 row blocks x 1 key block) tile, flist 64 D for
//                      each active D of a (1 row block x 2 key blocks) tile;
//                      D may be negative when the key window lies before the
//                      query window on the sequence;
//   vlist              selected columns that live in this key window, as local
//                      key indices, ascending, padded with -1;
//   vlocbits/vlocpre   the same as a bitmap with word prefix counts;
//   counts             work units of the four attention passes;
//   bdbits             block-cover mode: bit D set iff a selected offset o has
//                      |o - 64 D| <= 63, i.e. a selected slash passes through
//                      the 64 x 64 blocks of block diagonal D; the sheared cover
//                      is then built over the offsets of those blocks.
// GQA packing (pack = g): the g query heads of a KV group share one selection
// and a query-major tile holds R = 128 / g tokens of all g heads, so elist is
// the sheared cover for R-row strips: the greedy 64-wide cover of
// E_R = {u : some selected o in [u - R + 1, u]}; a strip at r0 reads keys
// [r0 + R - 64 - u, r0 + R - 1 - u].  flist stays the 128-key cover.  The
// query-major counts of a group are reported at its first head.
#include "vs_internal.h"

namespace vs {
namespace {

constexpr int kIdxThreads = 256;

struct IndexParams {
  ArenaHeader hdr;
  uint8_t* arena;
  const int32_t* v_idx;
  const int32_t* s_idx;
  int staged;  // the lists walked by thread 0 live in dynamic shared memory
  int sbits;   // the bitmaps are built in dynamic shared memory
};

// Dynamic shared memory of the staged cover: the f- and e-lists (EMAX
// each), the slash list (ks), then either the parallel cover's scratch (4
// (ks + 1) ints) or one flag byte per local block diagonal (striped); 0 when
// that exceeds kIdxStageMax.
constexpr size_t kIdxStageMax = 200 * 1024;
size_t index_stage_bytes(const ArenaHeader& h) {
  size_t b = size_t(4) * (2 * size_t(h.EMAX) + size_t(h.ks)) +
             std::max(size_t(16) * (size_t(h.ks) + 1), size_t(h.EMAX) + 16);
  // block cover: the active block diagonals (at most WG), their words'
  // counts (at most WG) and the cover's scratch instead of the slash list
  if (h.block_cover) b = std::max(b, size_t(4) * (2 * size_t(h.EMAX) + 2 * size_t(h.WG) + 4 * (size_t(h.WG) + 1)));
  return b <= kIdxStageMax ? b : 0;
}
// The offset, column and local-column bitmaps, or 0 when they exceed
// kIdxStageMax.  The same dynamic shared memory serves both, one after the
// other.
size_t index_bits_bytes(const ArenaHeader& h) {
  const size_t b = size_t(8) * (2 * size_t(h.WG) + size_t(h.WL));
  return b <= kIdxStageMax ? b : 0;
}

__device__ __forceinline__ bool block_diag_active(const uint64_t* off, int WG, int64_t x) {
  // some selected offset in [64x - 63, 64x + 63]
  if (x < 0) return false;
  const uint64_t a = bits64(off, 64 * x - 63, WG);
  const uint64_t b = bits64(off, 64 * x + 1, WG) & 0x7FFFFFFFFFFFFFFFull;
  return (a | b) != 0;
}

// Exclusive prefix sum of a[0, n) in shared memory by the whole block;
// returns the total.  part holds kIdxThreads + 1 ints.
__device__ int block_scan_excl(int* a, int n, int* part, int tid) {
  const int per = (n + kIdxThreads - 1) / kIdxThreads;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  int sum = 0;
  for (int i = lo; i < hi; ++i) sum += a[i];
  part[tid] = sum;
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int i = 0; i < kIdxThreads; ++i) {
      const int c = part[i];
      part[i] = run;
      run += c;
    }
    part[kIdxThreads] = run;
  }
  __syncthreads();
  int run = part[tid];
  for (int i = lo; i < hi; ++i) {
    const int v = a[i];
    a[i] = run;
    run += v;
  }
  const int total = part[kIdxThreads];
  __syncthreads();
  return total;
}

// The greedy cover of E = union of the intervals [a_j, b_j] (ascending in
// both ends) by disjoint 64-wide intervals, the starts u <= ulim, at most cap
// of them, written to out; by the whole block, returns their number.  Exact
// offsets (BLK = false): o holds the n ascending selected offsets, [a_j, b_j]
// = [o_j, o_j + dil].  Block cover (BLK = true): o holds the n ascending
// active block diagonals D, whose effective offsets [max(0, 64 D - 63), 64 D
// + 63] are dilated the same way.  Same result as walking the list one by
// one: E falls into segments (runs of intervals that overlap or touch; [A_s,
// B_s]); inside one the walk places starts u_s, u_s + 64, ... while <= B_s,
// with u_s = max(cur, A_s) for the walk's position cur on entry, and leaves
// at u_s + 64 K_s.  The position on entry is at most B_{s-1} + 64, so a
// segment starting that far past its predecessor is entered at A_s whatever
// came before: the walk is split at those segments and the pieces run in
// parallel.  sc holds 4 (n + 1) ints.
template <bool BLK>
__device__ __forceinline__ int64_t cov_a(const int32_t* o, int j) {
  return BLK ? max(int64_t(0), 64 * int64_t(o[j]) - 63) : int64_t(o[j]);
}
template <bool BLK>
__device__ __forceinline__ int64_t cov_b(const int32_t* o, int j, int dil) {
  return BLK ? 64 * int64_t(o[j]) + 63 + dil : int64_t(o[j]) + dil;
}
template <bool BLK>
__device__ int cover_parallel(const int32_t* o, int n, int dil, int64_t ulim, int cap, int32_t* out, int* sc,
                              int* part, int tid) {
  int* first = sc;               // per interval: 1 if it starts a segment, then the segment index
  int* segJ = sc + (n + 1);      // first interval of segment s; segJ[S] = n
  int* segU = segJ + (n + 1);    // the segment's first start
  int* segK = segU + (n + 1);    // its number of starts, then their exclusive prefix
  auto starts_segment = [&](int j) { return j == 0 || cov_a<BLK>(o, j) > cov_b<BLK>(o, j - 1, dil) + 1; };
  for (int j = tid; j < n; j += kIdxThreads) first[j] = starts_segment(j) ? 1 : 0;
  __syncthreads();
  const int S = block_scan_excl(first, n, part, tid);
  for (int j = tid; j < n; j += kIdxThreads)
    if (starts_segment(j)) segJ[first[j]] = j;
  if (tid == 0) segJ[S] = n;
  __syncthreads();
  for (int s = tid; s < S; s += kIdxThreads) {
    const int64_t A = cov_a<BLK>(o, segJ[s]);
    if (s > 0 && A < cov_b<BLK>(o, segJ[s] - 1, dil) + 64) continue;  // not the head of a piece
    int64_t cur = A;
    for (int t = s; t < S; ++t) {
      const int64_t At = cov_a<BLK>(o, segJ[t]), Bt = cov_b<BLK>(o, segJ[t + 1] - 1, dil);
      if (t > s && At >= cov_b<BLK>(o, segJ[t] - 1, dil) + 64) break;  // the next piece's head
      const int64_t u = max(cur, At);
      const int K = u <= Bt ? int((Bt - u) / 64) + 1 : 0;
      segU[t] = int(u);
      segK[t] = K;
      cur = u + 64 * int64_t(K);
    }
  }
  __syncthreads();
  const int T = block_scan_excl(segK, S, part, tid);
  if (tid == 0) segK[S] = T;
  __shared__ int s_cnt;
  if (tid == 0) s_cnt = 0;
  __syncthreads();
  // the starts increase along the walk: those <= ulim are a prefix of it
  int mine = 0;
  for (int s = tid; s < S; s += kIdxThreads) {
    const int p0 = segK[s], K = segK[s + 1] - p0;
    const int64_t u0 = segU[s];
    const int keep = u0 > ulim ? 0 : int(min(int64_t(K), (ulim - u0) / 64 + 1));
    mine += keep;
    for (int k = 0; k < keep && p0 + k < cap; ++k) out[p0 + k] = int32_t(u0 + 64 * k);
  }
  if (mine) atomicAdd(&s_cnt, mine);
  __syncthreads();
  const int cnt = min(s_cnt, cap);
  __syncthreads();
  return cnt;
}

__global__ void __launch_bounds__(kIdxThreads) vs_index_kernel(const IndexParams P) {
  const ArenaHeader& H = P.hdr;
  const int bh = blockIdx.x;
  const int tid = threadIdx.x;
  uint8_t* A = P.arena;
  ArenaHeader* hdr = reinterpret_cast<ArenaHeader*>(A);
  if (bh == 0 && tid == 0) {
    // header (the status word was cleared by the launcher)
    const int32_t* src = reinterpret_cast<const int32_t*>(&H);
    int32_t* dst = reinterpret_cast<int32_t*>(hdr);
    for (int i = 1; i < int(sizeof(ArenaHeader) / 4); ++i) dst[i] = src[i];
  }
  uint64_t* offbits = reinterpret_cast<uint64_t*>(A + H.off_offbits) + int64_t(bh) * H.WG;
  uint64_t* colbits = reinterpret_cast<uint64_t*>(A + H.off_colbits) + int64_t(bh) * H.WG;
  int32_t* elist = reinterpret_cast<int32_t*>(A + H.off_elist) + int64_t(bh) * H.EMAX;
  int32_t* ecount = reinterpret_cast<int32_t*>(A + H.off_ecount) + bh;
  int32_t* flist = reinterpret_cast<int32_t*>(A + H.off_flist) + int64_t(bh) * H.EMAX;
  int32_t* fcount = reinterpret_cast<int32_t*>(A + H.off_fcount) + bh;
  int32_t* vlist = reinterpret_cast<int32_t*>(A + H.off_vlist) + int64_t(bh) * H.KVP;
  int32_t* vcount = reinterpret_cast<int32_t*>(A + H.off_vcount) + bh;
  uint64_t* vloc = reinterpret_cast<uint64_t*>(A + H.off_vlocbits) + int64_t(bh) * H.WL;
  int32_t* vpre = reinterpret_cast<int32_t*>(A + H.off_vlocpre) + int64_t(bh) * H.WL;
  int64_t* counts = reinterpret_cast<int64_t*>(A + H.off_counts) + int64_t(bh) * 4;
  uint64_t* bdbits = reinterpret_cast<uint64_t*>(A + H.off_bdbits) + int64_t(bh) * H.WG;
  const int32_t* iv = P.v_idx + int64_t(bh) * H.kv;
  const int32_t* is = P.s_idx + int64_t(bh) * H.ks;
  const int64_t NG = H.N_global;
  const int W = H.world;

  __shared__ int bad, nks;
  const int gp = H.pack;  // heads per packed tile (0: no packing)
  __shared__ int part[kIdxThreads + 1];
  if (tid == 0) bad = nks = 0;
  __syncthreads();
  // 1. validate: strictly ascending inside [0, N_global), then only -1 (a
  // budget below the list's capacity); nks = the slash entries in use
  for (int i = tid; i < H.kv; i += kIdxThreads) {
    const int x = iv[i];
    if (x < -1 || x >= NG || (x >= 0 && i > 0 && !(iv[i - 1] >= 0 && iv[i - 1] < x))) bad = 1;
  }
  for (int i = tid; i < H.ks; i += kIdxThreads) {
    const int x = is[i];
    if (x < -1 || x >= NG || (x >= 0 && i > 0 && !(is[i - 1] >= 0 && is[i - 1] < x))) bad = 1;
    if (x >= 0) atomicAdd(&nks, 1);
  }
  if (gp) {
    // packing needs one selection per KV group: every head's lists equal its
    // group's first head's
    const int h0 = (bh % H.Hq) / gp * gp, b = bh / H.Hq;
    const int32_t* iv0 = P.v_idx + (int64_t(b) * H.Hq + h0) * H.kv;
    const int32_t* is0 = P.s_idx + (int64_t(b) * H.Hq + h0) * H.ks;
    for (int i = tid; i < H.kv; i += kIdxThreads)
      if (iv[i] != iv0[i]) bad = 1;
    for (int i = tid; i < H.ks; i += kIdxThreads)
      if (is[i] != is0[i]) bad = 1;
  }
  // 2. clear bitmaps
  for (int w = tid; w < H.WG; w += kIdxThreads) offbits[w] = colbits[w] = 0ull;
  for (int w = tid; w < H.WL; w += kIdxThreads) vloc[w] = 0ull;
  for (int w = tid; w < H.WG; w += kIdxThreads) bdbits[w] = 0ull;
  __syncthreads();
  if (bad) {
    if (tid == 0) {
      atomicCAS(&hdr->status, 0, int(VS_ERR_INDEX));
      *ecount = 0;
      *fcount = 0;
      *vcount = 0;
      for (int i = 0; i < 4; ++i) counts[i] = 0;
    }
    for (int i = tid; i < H.KVP; i += kIdxThreads) vlist[i] = -1;
    for (int w = tid; w < H.WL; w += kIdxThreads) vpre[w] = 0;
    return;
  }
  // 3. bitmaps.  Neighbouring entries of a sorted list set bits of the same
  // word; built in shared memory when they fit (cheap same-word atomics),
  // then written out.
  extern __shared__ __align__(16) int32_t stage[];
  uint64_t* ob = offbits;
  uint64_t* cb = colbits;
  uint64_t* vb = vloc;
  if (P.sbits) {
    uint64_t* s64 = reinterpret_cast<uint64_t*>(stage);
    ob = s64;
    cb = s64 + H.WG;
    vb = s64 + 2 * H.WG;
    for (int w = tid; w < 2 * H.WG + H.WL; w += kIdxThreads) s64[w] = 0ull;
    __syncthreads();
  }
  for (int i = tid; i < H.ks; i += kIdxThreads) {
    const int x = is[i];
    if (x >= 0) atomicOr(reinterpret_cast<unsigned long long*>(ob + (x >> 6)), 1ull << (x & 63));
  }
  for (int i = tid; i < H.kv; i += kIdxThreads) {
    const int x = iv[i];
    if (x < 0) continue;
    atomicOr(reinterpret_cast<unsigned long long*>(cb + (x >> 6)), 1ull << (x & 63));
    const int64_t l = local_key_of(W, H.kv_rank, H.Nk, x);
    if (l >= 0) atomicOr(reinterpret_cast<unsigned long long*>(vb + (l >> 6)), 1ull << (l & 63));
  }
  __syncthreads();
  if (P.sbits) {
    for (int w = tid; w < H.WG; w += kIdxThreads) {
      offbits[w] = ob[w];
      colbits[w] = cb[w];
    }
    for (int w = tid; w < H.WL; w += kIdxThreads) vloc[w] = vb[w];
  }
  __threadfence_block();
  __syncthreads();
  // 3b. block cover: the active block diagonals
  const int64_t ndiag = NG / kBlk + 1;
  if (H.block_cover) {
    for (int64_t w = tid; w * 64 < ndiag; w += kIdxThreads) {
      uint64_t word = 0;
      for (int k = 0; k < 64 && w * 64 + k < ndiag; ++k)
        if (block_diag_active(offbits, H.WG, w * 64 + k)) word |= 1ull << k;
      bdbits[w] = word;
    }
    __syncthreads();
  }
  // 4. local vertical list from the local bitmap (ascending by construction)
  const int per = (H.WL + kIdxThreads - 1) / kIdxThreads;
  const int w0 = tid * per, w1 = min(H.WL, w0 + per);
  int mine = 0;
  for (int w = w0; w < w1; ++w) mine += __popcll(vloc[w]);
  part[tid] = mine;
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int i = 0; i < kIdxThreads; ++i) {
      const int c = part[i];
      part[i] = run;
      run += c;
    }
    part[kIdxThreads] = run;
  }
  __syncthreads();
  {
    int run = part[tid];
    for (int w = w0; w < w1; ++w) {
      vpre[w] = run;
      uint64_t x = vloc[w];
      while (x) {
        const int bit = __ffsll(x) - 1;
        x &= x - 1;
        vlist[run++] = w * 64 + bit;
      }
    }
  }
  const int nv = part[kIdxThreads];
  for (int i = nv + tid; i < H.KVP; i += kIdxThreads) vlist[i] = -1;
  __threadfence_block();
  __syncthreads();
  // 5. slash cover.  Staged (the lists fit the dynamic shared memory), the
  // slash list is copied in and the cover lists are built there and copied
  // out afterwards: the exact sheared cover by the whole block
  // (cover_parallel), the striped cover from block-diagonal flags evaluated
  // by all threads, the block-cover walk by thread 0.  Otherwise thread 0
  // walks the lists in global memory.
  __shared__ int s_ne, s_nf;
  const bool staged = P.staged != 0;
  int32_t* fl = staged ? stage : flist;
  int32_t* el = staged ? stage + H.EMAX : elist;
  const int32_t* isr = is;
  uint8_t* dflag = staged ? reinterpret_cast<uint8_t*>(stage + 2 * H.EMAX + H.ks) : nullptr;
  const int64_t rel = int64_t(H.q_rank) - H.kv_rank;
  const int nb = H.Nq / kBlk, nbk = H.Nk / kBlk;
  if (staged) {
    int32_t* s_is = stage + 2 * H.EMAX;
    for (int i = tid; i < H.ks; i += kIdxThreads) s_is[i] = is[i];
    isr = s_is;
    if (!H.sheared) {
      // bit 0: D is active for a (2 row blocks x 1 key block) tile, bit 1:
      // for a (1 row block x 2 key blocks) tile
      for (int D = -nbk + tid; D <= nb; D += kIdxThreads) {
        const bool a = block_diag_active(offbits, H.WG, int64_t(W) * D + rel);
        const bool e = a || block_diag_active(offbits, H.WG, int64_t(W) * D + W + rel);
        const bool f = a || block_diag_active(offbits, H.WG, int64_t(W) * D - W + rel);
        dflag[D + nbk] = uint8_t((e ? 1 : 0) | (f ? 2 : 0));
      }
    }
  }
  __syncthreads();
  // the sheared cover by the whole block: of the exact offsets, or of the
  // active block diagonals (listed first from their bitmap)
  const bool par_cover = staged && H.sheared;
  int pnf = 0, pne = 0;
  if (par_cover) {
    if (H.block_cover) {
      int32_t* dl = stage + 2 * H.EMAX;
      int* wc = dl + H.WG;
      int* sc = wc + H.WG;
      const int nw = int((ndiag + 63) / 64);
      for (int w = tid; w < nw; w += kIdxThreads) wc[w] = __popcll(bdbits[w]);
      __syncthreads();
      const int nd = block_scan_excl(wc, nw, part, tid);
      for (int w = tid; w < nw; w += kIdxThreads) {
        uint64_t x = bdbits[w];
        int at = wc[w];
        while (x) {
          dl[at++] = w * 64 + __ffsll(x) - 1;
          x &= x - 1;
        }
      }
      __syncthreads();
      pnf = cover_parallel<true>(dl, nd, kQTile - 1, int64_t(H.Nq) + kQTile - 2, H.EMAX, fl, sc, part, tid);
      if (gp)
        pne = cover_parallel<true>(dl, nd, kQTile / gp - 1, int64_t(H.Nq) + kQTile / gp - 2, H.EMAX, el, sc, part, tid);
    } else {
      int* sc = stage + 2 * H.EMAX + H.ks;
      pnf = cover_parallel<false>(isr, nks, kQTile - 1, int64_t(H.Nq) + kQTile - 2, H.EMAX, fl, sc, part, tid);
      if (gp)
        pne = cover_parallel<false>(isr, nks, kQTile / gp - 1, int64_t(H.Nq) + kQTile / gp - 2, H.EMAX, el, sc, part,
                                    tid);
    }
    if (!gp) {
      for (int i = tid; i < pnf; i += kIdxThreads) el[i] = fl[i];
      pne = pnf;
    }
    __syncthreads();
  }
  if (tid == 0) {
    int ne = 0, nf = 0;
    // block cover: the smallest offset >= x inside an active block diagonal's
    // offsets [64 D - 63, 64 D + 63], or -1
    auto next_eff = [&](int64_t x) -> int64_t {
      int64_t D = x <= 0 ? 0 : x / kBlk;  // the first D with 64 D + 63 >= x
      while (D < ndiag) {
        const uint64_t wrd = bdbits[D >> 6] & ((~0ull) << (D & 63));
        if (wrd) {
          const int64_t Da = (D >> 6) * 64 + __ffsll(wrd) - 1;  // first active diagonal >= D
          return Da < ndiag ? max(max(x, int64_t(0)), Da * kBlk - 63) : -1;
        }
        D = ((D >> 6) + 1) * 64;
      }
      return -1;
    };
    if (par_cover) {
      nf = pnf;
      ne = pne;
    } else if (H.sheared) {
      // greedy cover by disjoint 64-wide intervals of the selected offsets
      // dilated by `dil` (tile height - 1)
      auto cover = [&](int32_t* list, int64_t dil) {
        int64_t cur = 0;
        int j = 0, n = 0;
        while (true) {
          int64_t o;
          if (H.block_cover) {
            o = next_eff(cur - dil);
            if (o < 0) break;
          } else {
            while (j < nks && isr[j] < cur - dil) ++j;
            if (j == nks) break;
            o = isr[j];
          }
          const int64_t u = max(cur, o);
          if (u > int64_t(H.Nq) + dil - 1 || n >= H.EMAX) break;
          list[n++] = int32_t(u);
          cur = u + 64;
        }
        return n;
      };
      nf = cover(fl, kQTile - 1);
      if (gp) {
        ne = cover(el, kQTile / gp - 1);
      } else {
        for (int i = 0; i < nf; ++i) el[i] = fl[i];
        ne = nf;
      }
    } else {
      // local block diagonals from the key window's end to the query
      // window's end (negative D: keys after the rows locally, which the
      // window offsets may still make causal)
      for (int D = -nbk; D <= nb && ne < H.EMAX; ++D)
        if (staged ? (dflag[D + nbk] & 1)
                   : (block_diag_active(offbits, H.WG, int64_t(W) * D + rel) ||
                      block_diag_active(offbits, H.WG, int64_t(W) * D + W + rel)))
          el[ne++] = 64 * D + 64;
      for (int D = -nbk; D <= nb && nf < H.EMAX; ++D)
        if (staged ? (dflag[D + nbk] & 2)
                   : (block_diag_active(offbits, H.WG, int64_t(W) * D + rel) ||
                      block_diag_active(offbits, H.WG, int64_t(W) * D - W + rel)))
          fl[nf++] = 64 * D;
    }
    *ecount = ne;
    *fcount = nf;
    *vcount = nv;
    s_ne = ne;
    s_nf = nf;
  }
  __syncthreads();
  // 6. work counts of the four passes (every thread a share of the entries;
  // integer sums, so the order does not matter)
  {
    const int ne = s_ne, nf = s_nf;
    const int64_t T = (H.Nq + kQTile - 1) / kQTile;
    const int64_t TK = (H.Nk + kBarK - 1) / kBarK;
    int64_t c[4] = {0, 0, 0, 0};
    // the same unit ranges as the kernels: query tile t takes the entries
    // e in [128 t + 64 - Nk + 1, 128 t + 127] (its 64 keys start before Nk)
    // and the bar chunks whose first column precedes its last row; key tile
    // tau the entries f with rows [128 tau + f, + 64) meeting [0, Nq); a
    // key-major bar chunk runs from the first row block that can attend its
    // first column
    auto ceil_div = [](int64_t a, int64_t b) { return a >= 0 ? (a + b - 1) / b : -((-a) / b); };
    auto floor_div = [](int64_t a, int64_t b) { return a >= 0 ? a / b : -((-a + b - 1) / b); };
    if (!gp) {
      for (int i = tid; i < ne; i += kIdxThreads) {
        const int64_t e = el[i];
        const int64_t tmin = max(int64_t(0), ceil_div(e - 127, kQTile));
        const int64_t tmax = min(T - 1, floor_div(e - 65 + H.Nk, kQTile));
        c[0] += max(int64_t(0), tmax - tmin + 1);
      }
      for (int ch = tid; ch * kKTile < nv; ch += kIdxThreads) {
        const int64_t m_g = (int64_t(W) * (vlist[ch * kKTile] >> 6) + H.kv_rank) * kBlk + (vlist[ch * kKTile] & 63);
        const int64_t tmin = first_causal_row_block(W, H.q_rank, m_g) / 2;
        c[1] += max(int64_t(0), T - tmin);
      }
    } else if ((bh % H.Hq) % gp == 0) {
      // packed strips of R tokens (unstriped): strip s takes the entries e
      // in [R s + R - 63 - Nk, R s + R - 1] and the bar chunks whose first
      // column is at most its last token
      const int64_t R = kQTile / gp, TS = (H.Nq + R - 1) / R;
      for (int i = tid; i < ne; i += kIdxThreads) {
        const int64_t e = el[i];
        const int64_t smin = max(int64_t(0), ceil_div(e - R + 1, R));
        const int64_t smax = min(TS - 1, floor_div(e - R + 63 + H.Nk, R));
        c[0] += max(int64_t(0), smax - smin + 1);
      }
      for (int ch = tid; ch * kKTile < nv; ch += kIdxThreads) {
        const int64_t f = vlist[ch * kKTile];
        c[1] += max(int64_t(0), TS - max(int64_t(0), ceil_div(f - R + 1, R)));
      }
    }
    for (int i = tid; i < nf; i += kIdxThreads) {
      const int64_t f = fl[i];
      const int64_t tmin = max(int64_t(0), ceil_div(-f - 63, kBarK));
      const int64_t tmax = min(TK - 1, floor_div(H.Nq - 1 - f, kBarK));
      c[2] += max(int64_t(0), tmax - tmin + 1);
    }
    for (int ch = tid; ch * kBarK < nv; ch += kIdxThreads) {
      const int64_t m_g = (int64_t(W) * (vlist[ch * kBarK] >> 6) + H.kv_rank) * kBlk + (vlist[ch * kBarK] & 63);
      const int64_t rs = first_causal_row_block(W, H.q_rank, m_g) * kBlk;
      c[3] += max(int64_t(0), (H.Nq - rs + kRowTile - 1) / kRowTile);
    }
    __shared__ unsigned long long s_cnt[4];
    if (tid < 4) s_cnt[tid] = 0ull;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      unsigned long long v = static_cast<unsigned long long>(c[k]);
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if ((tid & 31) == 0 && v) atomicAdd(&s_cnt[k], v);
    }
    __syncthreads();
    if (tid < 4) counts[tid] = static_cast<int64_t>(s_cnt[tid]);
  }
  if (staged) {
    __syncthreads();
    for (int i = tid; i < s_nf; i += kIdxThreads) flist[i] = fl[i];
    for (int i = tid; i < s_ne; i += kIdxThreads) elist[i] = el[i];
  }
}

}  // namespace

size_t index_bytes(const vs_shape* s, int kv, int ks, const vs_stripe* stripe, ArenaHeader* out) {
  ArenaHeader h;
  memset(&h, 0, sizeof(h));
  h.magic = kArenaMagic;
  h.B = s->B;
  h.Hq = s->Hq;
  h.Nq = s->Nq;
  h.Nk = s->Nk;
  h.kv = kv;
  h.ks = ks;
  h.world = stripe ? stripe->world : 1;
  h.stripe = kBlk;
  h.q_rank = stripe ? stripe->q_rank : 0;
  h.kv_rank = stripe ? stripe->kv_rank : 0;
  h.N_global = stripe ? stripe->N_global : s->Nq;
  h.WG = int32_t(h.N_global / 64 + 4);
  h.WL = s->Nk / 64 + 2;
  h.EMAX = (s->Nq + s->Nk) / 64 + 8;
  h.KVP = (kv + kBarK - 1) / kBarK * kBarK;
  h.sheared = stripe ? 0 : 1;
  const int64_t BH = int64_t(s->B) * s->Hq;
  int64_t off = 256;
  auto take = [&](int64_t bytes) {
    const int64_t at = off;
    off += (bytes + 255) / 256 * 256;
    return at;
  };
  h.off_offbits = take(BH * h.WG * 8);
  h.off_colbits = take(BH * h.WG * 8);
  h.off_elist = take(BH * h.EMAX * 4);
  h.off_ecount = take(BH * 4);
  h.off_flist = take(BH * h.EMAX * 4);
  h.off_fcount = take(BH * 4);
  h.off_vlist = take(BH * h.KVP * 4);
  h.off_vcount = take(BH * 4);
  h.off_vlocbits = take(BH * h.WL * 8);
  h.off_vlocpre = take(BH * h.WL * 4);
  h.off_counts = take(BH * 4 * 8);
  h.off_bdbits = take(BH * h.WG * 8);
  h.total_bytes = off;
  if (out) *out = h;
  return size_t(off);
}

vs_status launch_index(const vs_shape* s, const int32_t* v_idx, const int32_t* s_idx, int kv, int ks,
                       const vs_stripe* stripe, int flags, void* arena, size_t, cudaStream_t st) {
  IndexParams P;
  index_bytes(s, kv, ks, stripe, &P.hdr);
  P.hdr.block_cover = (flags & VS_INDEX_BLOCK_COVER) ? 1 : 0;
  P.hdr.pack = (flags & VS_INDEX_PACK_GQA) ? s->Hq / s->Hkv : 0;
  P.arena = static_cast<uint8_t*>(arena);
  P.v_idx = v_idx;
  P.s_idx = s_idx;
  const size_t lists = index_stage_bytes(P.hdr), bits = index_bits_bytes(P.hdr);
  const size_t stage = std::max(lists, bits);
  P.staged = lists > 0;
  P.sbits = bits > 0;
  if (stage > 48 * 1024 &&
      cudaFuncSetAttribute(vs_index_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(stage)) != cudaSuccess)
    return VS_ERR_CUDA;
  if (cudaMemsetAsync(arena, 0, sizeof(int32_t), st) != cudaSuccess) return VS_ERR_CUDA;
  trace_begin("index", st);
  vs_index_kernel<<<s->B * s->Hq, kIdxThreads, stage, st>>>(P);
  trace_end(st);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? VS_OK : VS_ERR_CUDA;
}

}  // namespace vs
