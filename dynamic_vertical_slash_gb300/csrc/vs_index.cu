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
};

__device__ __forceinline__ bool block_diag_active(const uint64_t* off, int WG, int64_t x) {
  // some selected offset in [64x - 63, 64x + 63]
  if (x < 0) return false;
  const uint64_t a = bits64(off, 64 * x - 63, WG);
  const uint64_t b = bits64(off, 64 * x + 1, WG) & 0x7FFFFFFFFFFFFFFFull;
  return (a | b) != 0;
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
  // 3. bitmaps
  for (int i = tid; i < H.ks; i += kIdxThreads) {
    const int x = is[i];
    if (x >= 0) atomicOr(reinterpret_cast<unsigned long long*>(offbits + (x >> 6)), 1ull << (x & 63));
  }
  for (int i = tid; i < H.kv; i += kIdxThreads) {
    const int x = iv[i];
    if (x < 0) continue;
    atomicOr(reinterpret_cast<unsigned long long*>(colbits + (x >> 6)), 1ull << (x & 63));
    const int64_t l = local_key_of(W, H.kv_rank, H.Nk, x);
    if (l >= 0) atomicOr(reinterpret_cast<unsigned long long*>(vloc + (l >> 6)), 1ull << (l & 63));
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
  // 5. slash cover and 6. work counts (sequential; lists are short)
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
    if (H.sheared) {
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
            while (j < nks && is[j] < cur - dil) ++j;
            if (j == nks) break;
            o = is[j];
          }
          const int64_t u = max(cur, o);
          if (u > int64_t(H.Nq) + dil - 1 || n >= H.EMAX) break;
          list[n++] = int32_t(u);
          cur = u + 64;
        }
        return n;
      };
      nf = cover(flist, kQTile - 1);
      if (gp) {
        ne = cover(elist, kQTile / gp - 1);
      } else {
        for (int i = 0; i < nf; ++i) elist[i] = flist[i];
        ne = nf;
      }
    } else {
      // local block diagonals from the key window's end to the query
      // window's end (negative D: keys after the rows locally, which the
      // window offsets may still make causal)
      const int64_t rel = int64_t(H.q_rank) - H.kv_rank;
      const int nb = H.Nq / kBlk, nbk = H.Nk / kBlk;
      for (int D = -nbk; D <= nb && ne < H.EMAX; ++D)
        if (block_diag_active(offbits, H.WG, int64_t(W) * D + rel) ||
            block_diag_active(offbits, H.WG, int64_t(W) * D + W + rel))
          elist[ne++] = 64 * D + 64;
      for (int D = -nbk; D <= nb && nf < H.EMAX; ++D)
        if (block_diag_active(offbits, H.WG, int64_t(W) * D + rel) ||
            block_diag_active(offbits, H.WG, int64_t(W) * D - W + rel))
          flist[nf++] = 64 * D;
    }
    *ecount = ne;
    *fcount = nf;
    *vcount = nv;
    const int64_t T = (H.Nq + kQTile - 1) / kQTile;
    const int64_t TK = (H.Nk + kBarK - 1) / kBarK;
    int64_t c0 = 0, c1 = 0, c2 = 0, c3 = 0;
    // the same unit ranges as the kernels: query tile t takes the entries
    // e in [128 t + 64 - Nk + 1, 128 t + 127] (its 64 keys start before Nk)
    // and the bar chunks whose first column precedes its last row; key tile
    // tau the entries f with rows [128 tau + f, + 64) meeting [0, Nq); a
    // key-major bar chunk runs from the first row block that can attend its
    // first column
    auto ceil_div = [](int64_t a, int64_t b) { return a >= 0 ? (a + b - 1) / b : -((-a) / b); };
    auto floor_div = [](int64_t a, int64_t b) { return a >= 0 ? a / b : -((-a + b - 1) / b); };
    if (!gp) {
      for (int i = 0; i < ne; ++i) {
        const int64_t e = elist[i];
        const int64_t tmin = max(int64_t(0), ceil_div(e - 127, kQTile));
        const int64_t tmax = min(T - 1, floor_div(e - 65 + H.Nk, kQTile));
        c0 += max(int64_t(0), tmax - tmin + 1);
      }
      for (int c = 0; c * kKTile < nv; ++c) {
        const int64_t m_g = (int64_t(W) * (vlist[c * kKTile] >> 6) + H.kv_rank) * kBlk + (vlist[c * kKTile] & 63);
        const int64_t tmin = first_causal_row_block(W, H.q_rank, m_g) / 2;
        c1 += max(int64_t(0), T - tmin);
      }
    } else if ((bh % H.Hq) % gp == 0) {
      // packed strips of R tokens (unstriped): strip s takes the entries e
      // in [R s + R - 63 - Nk, R s + R - 1] and the bar chunks whose first
      // column is at most its last token
      const int64_t R = kQTile / gp, TS = (H.Nq + R - 1) / R;
      for (int i = 0; i < ne; ++i) {
        const int64_t e = elist[i];
        const int64_t smin = max(int64_t(0), ceil_div(e - R + 1, R));
        const int64_t smax = min(TS - 1, floor_div(e - R + 63 + H.Nk, R));
        c0 += max(int64_t(0), smax - smin + 1);
      }
      for (int c = 0; c * kKTile < nv; ++c) {
        const int64_t f = vlist[c * kKTile];
        c1 += max(int64_t(0), TS - max(int64_t(0), ceil_div(f - R + 1, R)));
      }
    }
    for (int i = 0; i < nf; ++i) {
      const int64_t f = flist[i];
      const int64_t tmin = max(int64_t(0), ceil_div(-f - 63, kBarK));
      const int64_t tmax = min(TK - 1, floor_div(H.Nq - 1 - f, kBarK));
      c2 += max(int64_t(0), tmax - tmin + 1);
    }
    for (int c = 0; c * kBarK < nv; ++c) {
      const int64_t m_g = (int64_t(W) * (vlist[c * kBarK] >> 6) + H.kv_rank) * kBlk + (vlist[c * kBarK] & 63);
      const int64_t rs = first_causal_row_block(W, H.q_rank, m_g) * kBlk;
      c3 += max(int64_t(0), (H.Nq - rs + kRowTile - 1) / kRowTile);
    }
    counts[0] = c0;
    counts[1] = c1;
    counts[2] = c2;
    counts[3] = c3;
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
  if (cudaMemsetAsync(arena, 0, sizeof(int32_t), st) != cudaSuccess) return VS_ERR_CUDA;
  trace_begin("index", st);
  vs_index_kernel<<<s->B * s->Hq, kIdxThreads, 0, st>>>(P);
  trace_end(st);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? VS_OK : VS_ERR_CUDA;
}

}  // namespace vs
