// Sparse attention forward on the Vertical-Slash mask (tcgen05 / TMEM / TMA).
//
// One CTA owns one 128-row query tile of one query head and walks its units
//   * slash tiles: 64 keys starting at local key c = 128 t + 64 - e for every
//     entry e <= 128 t + 127 of the head's query-major list, loaded by TMA;
//   * bar chunks: 64 selected columns gathered with cp.async
// two at a time: a pair of units is one 128-key block, so S = Q K^T is one
// M=128, N=128 MMA chain and O += P V one K=128 chain (an odd last unit
// leaves the second half of its pair masked and out of the PV chain).  Per
// pair: fp32 online softmax on the exact token mask in registers (one thread
// per row), P (bf16) back into TMEM.
//
// Warp roles (352 threads): warp 0 issues the loads, warp 10 builds each
// pair's row masks, warp 1 issues MMAs (one lane), warps 2-5 and 6-9 are two
// softmax warpgroups that take alternate pairs (even / odd).  Each group
// keeps its own running maximum, sum and O accumulator, so the groups never
// wait for each other; the epilogue merges the two partial results the way
// merge_out_and_lse of Algorithm 2 merges ring steps.
//
// TMEM columns: O_g [128 g, 128 g + d), S_g [256 + 128 g, +128) for group g.
// P_g overwrites the first 64 columns of S_g once the scores are in
// registers, so the MMA issues S of pair i + 2 into S_g only after the PV of
// pair i; since S of pair i completes after the PV of pair i - 2, a group
// never has to wait for its own PV before it rescales O or writes P.
//
// Shared memory: Q, a ring of slots that each hold K or V of one pair (128
// rows), filled and released in the MMA's order S0 S1 PV0 S2 PV1 S3 ..., and
// a ring of per-pair row masks.
#include "vs_internal.h"
#include "vs_kernel_common.cuh"

namespace vs {
namespace {

constexpr int kFwdThreads = 352;
constexpr int kFwdMaskWarp = 10;
constexpr int kFwdGroup = 128;  // threads per softmax warpgroup
constexpr int kPairKeys = 2 * kKTile;
constexpr int kFwdSlots = 5;
constexpr int kMaskRing = 4;
constexpr uint32_t kColO = 0, kColS = 256, kTmemCols = 512;
constexpr float kRefSlack = 18446744073709551616.0f;  // 2^64: largest masked pair sum accepted against the reference

template <int D>
struct FwdSmem {
  static constexpr int NH = D / 64;
  uint8_t q[NH][kQTile * 128];
  uint8_t slot[kFwdSlots][NH][kPairKeys * 128];  // K or V of one pair, 128B-swizzled, per d-half
  uint64_t mask[kMaskRing][2][kQTile];           // row masks of a pair's two units (mask warp)
  int64_t bar_keys[kKTile];                      // mask warp: global positions of a bar chunk's keys
  int key0[8][2];                                // loader: first key of each slash half, by pair
  uint64_t q_full;
  uint64_t slot_full[kFwdSlots], slot_empty[kFwdSlots];
  uint64_t mask_full[kMaskRing], mask_empty[kMaskRing];
  uint64_t s_full[2], p_full[2];  // per softmax group
  uint64_t o_final, teardown;
  float red_m[2][kQTile];  // per group: reference maximum (log2 units)
  float red_l[2][kQTile];  // per group: row sum
  uint32_t tmem_base;
  int abort_flag;
};

struct FwdParams {
  const void* arena;
  const uint8_t* k;  // K base (bytes)
  const uint8_t* v;
  int64_t sk[3], sv[3], so[3];
  int B, Nq, Hq, Hkv;
  float scale_log2;
  uint8_t* o;
  float* lse;
  float* o_acc;
  int* err;
};

// The order in which the MMA consumes K / V blocks (and the loader fills the
// slot ring): K0, K1, then per pair i: V_i, K_{i+2}.
template <typename F>
__device__ __forceinline__ void for_each_block(int P, F&& f) {
  f(0, 0);
  if (P > 1) f(0, 1);
  for (int i = 0; i < P; ++i) {
    f(1, i);
    if (i + 2 < P) f(0, i + 2);
  }
}

// Moves a row's reference maximum for one pair (the rows with `need` set)
// and writes the pair's P: exact masked maximum from the scores still in
// TMEM, O and the running sum rescaled where the maximum grows, P recomputed
// half by half against the new references and stored as it is made (P half
// hh lands on score columns the recomputation has already read).  Rare (the
// row's first pair, or an entry 2^64 above the reference), so it lives out
// of line and keeps the common path's registers free.  Warp-collective.
struct RowRef {
  float m_run, l_run;
};
template <int D>
__device__ __noinline__ RowRef fwd_rebase_pair(uint32_t tl, uint32_t colS, uint32_t colO, uint64_t mask0,
                                               uint64_t mask1, bool need, float m_run, float l_run,
                                               float scale_log2) {
  float mx[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) mx[k] = -INFINITY;
#pragma unroll 1
  for (int hh = 0; hh < 2; ++hh) {
    const uint64_t mask = hh ? mask1 : mask0;
    uint32_t sr[64];
    tmem_ld32(tl + colS + 64 * hh, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
    tmem_ld32(tl + colS + 64 * hh + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
    tmem_ld_wait();
#pragma unroll
    for (int k = 0; k < 64; ++k)
      if ((mask >> k) & 1ull) mx[k & 7] = fmaxf(mx[k & 7], __uint_as_float(sr[k]) * scale_log2);
  }
  const float mt =
      need ? fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])))
           : -INFINITY;
  const bool grow = need && (m_run != -INFINITY) && (mt > m_run);
  if (need && m_run == -INFINITY) m_run = mt;  // first entries: the O row is still zero
  if (__any_sync(0xffffffffu, grow)) {
    const float alpha = grow ? ex2(m_run - mt) : 1.f;
#pragma unroll 1
    for (int cc = 0; cc < D; cc += 16) {
      uint32_t ov[16];
      tmem_ld16(tl + colO + cc, ov);
      tmem_ld_wait();
#pragma unroll
      for (int k = 0; k < 16; ++k) ov[k] = __float_as_uint(__uint_as_float(ov[k]) * alpha);
      tmem_st16(tl + colO + cc, ov);
    }
    tmem_st_wait();
    if (grow) {
      l_run *= alpha;
      m_run = mt;
    }
  }
  const float nref = (m_run == -INFINITY) ? 0.f : -m_run;
  float ps[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) ps[k] = 0.f;
#pragma unroll 1
  for (int hh = 0; hh < 2; ++hh) {
    const uint64_t mask = hh ? mask1 : mask0;
    uint32_t sr[64], pk[32];
    tmem_ld32(tl + colS + 64 * hh, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
    tmem_ld32(tl + colS + 64 * hh + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
    tmem_ld_wait();
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      float p0 = ex2(fmaf(__uint_as_float(sr[2 * k]), scale_log2, nref));
      float p1 = ex2(fmaf(__uint_as_float(sr[2 * k + 1]), scale_log2, nref));
      p0 = ((mask >> (2 * k)) & 1ull) ? p0 : 0.f;
      p1 = ((mask >> (2 * k + 1)) & 1ull) ? p1 : 0.f;
      ps[k & 7] += p0 + p1;
      pk[k] = pack_bf16x2(p0, p1);
    }
    tmem_st16(tl + colS + 32 * hh, *reinterpret_cast<uint32_t(*)[16]>(&pk[0]));
    tmem_st16(tl + colS + 32 * hh + 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[16]));
  }
  l_run += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
  return RowRef{m_run, l_run};
}

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
    vs_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  constexpr int NH = D / 64;
  extern __shared__ uint8_t smem_raw[];
  FwdSmem<D>& s = *reinterpret_cast<FwdSmem<D>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  const ArenaView av = arena_view(p.arena);
  const Geo G = geo_from(av.hdr, p.Hkv, D);
  const int T = (p.Nq + kQTile - 1) / kQTile;
  const int BH = p.B * p.Hq;
  const int t = T - 1 - int(blockIdx.x) / BH;  // heavy (late) tiles first
  const int bh = int(blockIdx.x) % BH;
  const int b = bh / p.Hq, h = bh % p.Hq, hk = h / G.g;

  // Work list of this tile.
  // a workspace already holding an error makes the call skip its work
  const bool arena_ok = (av.hdr->status == 0) && (av.hdr->magic == kArenaMagic) &&
                        (*reinterpret_cast<volatile int*>(p.err) == 0);
  const int32_t* elist = av.elist + int64_t(bh) * G.EMAX;
  const int32_t* vlist = av.vlist + int64_t(bh) * G.KVP;
  const int64_t last_row = int64_t(t) * kQTile + kQTile - 1;
  int nslash = 0, nbar = 0;
  if (arena_ok) {
    nslash = count_le(elist, __ldg(av.ecount + bh), last_row);
    const int vc = __ldg(av.vcount + bh);
    // chunks whose first column can precede a row of the tile
    int lo = 0, hi = (vc + kKTile - 1) / kKTile;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(vlist + mid * kKTile) <= last_row) lo = mid + 1;
      else hi = mid;
    }
    nbar = lo;
  }
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
    for (int i = 0; i < kMaskRing; ++i) {
      mbar_init(&s.mask_full[i], 1);
      mbar_init(&s.mask_empty[i], kFwdGroup);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], kFwdGroup);
    }
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int issued[kFwdSlots];
    for (int i = 0; i < kFwdSlots; ++i) issued[i] = -1;
    if (P > 0) {
      if (lane == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        mbar_arrive_expect_tx(&s.q_full, NH * kQTile * 128);
        for (int hf = 0; hf < NH; ++hf) tma_load_4d(s.q[hf], &tmQ, &s.q_full, 64 * hf, h, t * kQTile, b);
      }
      const uint8_t* kb = p.k + (int64_t(b) * p.sk[0] + int64_t(hk) * p.sk[2]) * 2;
      const uint8_t* vb = p.v + (int64_t(b) * p.sv[0] + int64_t(hk) * p.sv[2]) * 2;
      int c = 0;
      bool ok = true;
      int e_win = -1, e_pref = 0;  // elist[32 e_win + lane]
      for_each_block(P, [&](int kind, int i) {
        if (!ok) return;
        const int sl = c % kFwdSlots;
        if (!kind) {
          // K blocks come in pair order: read the slash entries of both halves
          // (one 32-entry window per lane) and keep their first keys for V
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int u = 2 * i + hh;
            if (u >= nslash) continue;
            if ((u >> 5) != e_win) {
              e_win = u >> 5;
              const int j = 32 * e_win + lane;
              e_pref = j < nslash ? __ldg(elist + j) : 0;
            }
            const int e = __shfl_sync(0xffffffffu, e_pref, u & 31);
            if (lane == 0) s.key0[i & 7][hh] = t * kQTile + 64 - e;
          }
          __syncwarp();
        }
        if (c >= kFwdSlots && !(ok = mbar_wait(&s.slot_empty[sl], ((c / kFwdSlots) - 1) & 1, ab, VS_ERR_TIMEOUT)))
          return;
        const CUtensorMap* tm = kind ? &tmV : &tmK;
        const uint8_t* base = kind ? vb : kb;
        const int64_t stok = kind ? p.sv[1] : p.sk[1];
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
              const int key0 = s.key0[i & 7][hh];
              for (int hf = 0; hf < NH; ++hf)
                tma_load_4d(s.slot[sl][hf] + hh * kKTile * 128, tm, &s.slot_full[sl], 64 * hf, hk, key0, b);
            }
          } else {
            mbar_arrive(&s.slot_full[sl]);
          }
        }
        issued[sl] = c;
        ++c;
        __syncwarp();
      });
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
  } else if (warp == kFwdMaskWarp) {
    // ------------------------------------------------------------ row masks
    // Builds the 128 row masks of both units of each pair (bitmap reads for
    // slash tiles, position compares for bar chunks, zero for the missing
    // half of an odd last pair); runs as far ahead as the mask ring allows.
    const uint64_t* offbits_p = av.offbits + int64_t(bh) * G.WG;
    const uint64_t* colbits_p = av.colbits + int64_t(bh) * G.WG;
    int e_win = -1, e_pref = 0;  // elist[32 e_win + lane]
    for (int i = 0; i < P; ++i) {
      const int mi = i % kMaskRing;
      if (i >= kMaskRing && !mbar_wait(&s.mask_empty[mi], ((i / kMaskRing) - 1) & 1, ab, VS_ERR_TIMEOUT)) break;
      for (int hh = 0; hh < 2; ++hh) {
        const int u = 2 * i + hh;
        uint64_t* mrow = s.mask[mi][hh];
        uint64_t m[kQTile / 32];
        if (u >= U) {
#pragma unroll
          for (int rr = 0; rr < kQTile / 32; ++rr) m[rr] = 0ull;
        } else if (u < nslash) {
          if ((u >> 5) != e_win) {
            e_win = u >> 5;
            const int j = 32 * e_win + lane;
            e_pref = j < nslash ? __ldg(elist + j) : 0;
          }
          const int e = __shfl_sync(0xffffffffu, e_pref, u & 31);
          slash_tile_masks(G, offbits_p, colbits_p, t, int64_t(t) * kQTile + 64 - e, p.Nq, lane, m);
        } else {
          // bar chunk: ascending keys (padding last), so a row's mask is the
          // prefix of keys at or before the row
          const int32_t* keys = vlist + (u - nslash) * kKTile;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int key = __ldg(keys + e * 32 + lane);
            s.bar_keys[e * 32 + lane] = key >= 0 ? kpos_g(G, key) : INT64_MAX;
          }
          __syncwarp();
#pragma unroll
          for (int rr = 0; rr < kQTile / 32; ++rr) {
            const int64_t nl = int64_t(t) * kQTile + rr * 32 + lane;
            const int64_t ng = qpos_g(G, nl);
            int pos = 0;
#pragma unroll
            for (int step = 32; step > 0; step >>= 1)
              if (s.bar_keys[pos + step - 1] <= ng) pos += step;
            const int cnt = (s.bar_keys[kKTile - 1] <= ng) ? kKTile : pos;
            m[rr] = nl < p.Nq ? (cnt == kKTile ? ~0ull : ((1ull << cnt) - 1)) : 0ull;
          }
          __syncwarp();
        }
#pragma unroll
        for (int rr = 0; rr < kQTile / 32; ++rr) mrow[rr * 32 + lane] = m[rr];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.mask_full[mi]);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Pair i belongs to softmax group g = i & 1.  Order: S0, S1, then per
    // pair i: PV_i (once group g has written P_i), S_{i+2} into the same S_g.
    if (lane == 0 && P > 0) {
      const uint32_t idS = idesc_bf16(128, kPairKeys, 0, 0);
      const uint32_t idO = idesc_bf16(128, D, 0, 1);
      bool ok = mbar_wait(&s.q_full, 0, ab, VS_ERR_TIMEOUT);
      int c = 0;
      for_each_block(P, [&](int kind, int i) {
        if (!ok) return;
        const int g = i & 1;
        if (kind) {
          if (!(ok = mbar_wait(&s.p_full[g], (i >> 1) & 1, ab, VS_ERR_TIMEOUT))) return;
        }
        const int sl = c % kFwdSlots;
        if (!(ok = mbar_wait(&s.slot_full[sl], (c / kFwdSlots) & 1, ab, VS_ERR_TIMEOUT))) return;
        if (gathered(i)) fence_proxy_async_smem();
        tc_fence_after();
        if (!kind) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t da = sdesc_sw128(smem_u32(s.q[kk / 4]) + (kk % 4) * 32, 16, 1024);
            const uint64_t db = sdesc_sw128(smem_u32(s.slot[sl][kk / 4]) + (kk % 4) * 32, 16, 1024);
            mma_ss(tmem + kColS + 128 * g, da, db, idS, kk > 0);
          }
          mma_commit(&s.s_full[g]);
        } else {
          const int nk = (2 * i + 1 < U) ? kPairKeys / 16 : kKTile / 16;
          for (int kk = 0; kk < nk; ++kk) {
            const uint64_t dv = sdesc_sw128(smem_u32(s.slot[sl][0]) + kk * 2048, kPairKeys * 128, 1024);
            mma_ts(tmem + kColO + 128 * g, tmem + kColS + 128 * g + kk * 8, dv, idO, (i >= 2 || kk > 0));
          }
        }
        mma_commit(&s.slot_empty[sl]);
        mma_issued = true;
        ++c;
      });
      mma_commit(&s.o_final);
    }
  } else if (warp >= 2 && warp < 2 + 8) {
    // ------------------------------------------------------------ softmax
    const int grp = (warp - 2) >> 2;         // softmax group: pairs i with i & 1 == grp
    const int quarter = warp & 3;            // TMEM lane quarter this warp may access
    const int r = quarter * 32 + lane;       // query row within the tile
    const uint32_t tl = tmem + (uint32_t(quarter * 32) << 16);
    const int64_t n_loc = int64_t(t) * kQTile + r;
    const bool row_ok = n_loc < p.Nq;
    const uint32_t colO = kColO + 128 * grp, colS = kColS + 128 * grp;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int i = grp; i < P; i += 2) {
      const int mi = i % kMaskRing;
      ok = mbar_wait(&s.s_full[grp], (i >> 1) & 1, ab, VS_ERR_TIMEOUT) &&
           mbar_wait(&s.mask_full[mi], (i / kMaskRing) & 1, ab, VS_ERR_TIMEOUT);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint64_t mask0 = s.mask[mi][0][r], mask1 = s.mask[mi][1][r];
      mbar_arrive(&s.mask_empty[mi]);
      // P against the row's reference maximum m_run (log2 units).  The
      // reference is lazy: it only moves when a pair's masked sum shows an
      // entry more than 2^64 above it (or for the row's first entries); the
      // sum bounds every single entry, so P stays <= 2^64.  S of pair i
      // completing means the group's PV of pair i - 2 has completed too, so
      // O may be rescaled here.
      uint32_t pk[64];
      float pair_sum = 0.f;
      auto make_p = [&](float ref) {
        float ps[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) ps[k] = 0.f;
        const float nref = -ref;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint64_t mask = hh ? mask1 : mask0;
          uint32_t sr[64];
          tmem_ld32(tl + colS + 64 * hh, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
          tmem_ld32(tl + colS + 64 * hh + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            float p0 = ex2(fmaf(__uint_as_float(sr[2 * k]), p.scale_log2, nref));
            float p1 = ex2(fmaf(__uint_as_float(sr[2 * k + 1]), p.scale_log2, nref));
            p0 = ((mask >> (2 * k)) & 1ull) ? p0 : 0.f;
            p1 = ((mask >> (2 * k + 1)) & 1ull) ? p1 : 0.f;
            ps[k & 7] += p0 + p1;
            pk[32 * hh + k] = pack_bf16x2(p0, p1);
          }
        }
        pair_sum = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      };
      make_p(m_run == -INFINITY ? 0.f : m_run);
      const bool need = ((mask0 | mask1) != 0ull) && (m_run == -INFINITY || !(pair_sum <= kRefSlack));
      if (__any_sync(0xffffffffu, need)) {
        const RowRef rr = fwd_rebase_pair<D>(tl, colS, colO, mask0, mask1, need, m_run, l_run, p.scale_log2);
        m_run = rr.m_run;
        l_run = rr.l_run;
      } else {
        l_run += pair_sum;
#pragma unroll
        for (int k = 0; k < 4; ++k) tmem_st16(tl + colS + 16 * k, *reinterpret_cast<uint32_t(*)[16]>(&pk[16 * k]));
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&s.p_full[grp]);
    }
    // -------------------------------------------------------------- epilogue
    // Wait for every MMA, publish this group's (max, sum) per row, and merge
    // the two groups' partial results; group g writes columns [g d/2, (g+1) d/2).
    bool e_ok = ok && (P == 0 || mbar_wait(&s.o_final, 0, ab, VS_ERR_TIMEOUT));
    e_ok = __all_sync(0xffffffffu, e_ok);
    s.red_m[grp][r] = m_run;
    s.red_l[grp][r] = l_run;
    e_ok = bar_sync_and(1, 2 * kFwdGroup, e_ok);
    tc_fence_after();
    if (e_ok) {
      const float m0 = s.red_m[0][r], m1 = s.red_m[1][r];
      const float l0 = s.red_l[0][r], l1 = s.red_l[1][r];
      const bool has0 = P > 0 && l0 > 0.f, has1 = P > 1 && l1 > 0.f;  // group 1 ran only if P > 1
      const float mm = fmaxf(has0 ? m0 : -INFINITY, has1 ? m1 : -INFINITY);
      const float f0 = has0 ? ex2(m0 - mm) : 0.f, f1 = has1 ? ex2(m1 - mm) : 0.f;
      const float l_run2 = l0 * f0 + l1 * f1;
      const bool empty = !(l_run2 > 0.f);
      const float inv = empty ? 0.f : 1.f / l_run2;
      const float lse_step = empty ? -INFINITY : (mm + __log2f(l_run2)) * kLn2;
      float* lse_p = p.lse + (int64_t(b) * p.Hq + h) * p.Nq + n_loc;
      uint8_t* orow = p.o + (int64_t(b) * p.so[0] + n_loc * p.so[1] + int64_t(h) * p.so[2]) * 2;
      float wa = 0.f, wb = 1.f, lse_new = lse_step;
      float* acc = nullptr;
      if (p.o_acc && row_ok) {
        acc = p.o_acc + ((int64_t(b) * p.Nq + n_loc) * p.Hq + h) * D;
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
      // both groups have read lse_old before group 0 overwrites it
      bar_sync_and(1, 2 * kFwdGroup, true);
      const float g0 = f0 * inv, g1 = f1 * inv;
#pragma unroll 1
      for (int cc = (D / 2) * grp; cc < (D / 2) * (grp + 1); cc += 16) {
        uint32_t o0[16], o1[16];
        if (P > 0) {  // warp-collective TMEM reads
          tmem_ld16(tl + kColO + cc, o0);
          if (P > 1) tmem_ld16(tl + kColO + 128 + cc, o1);
          tmem_ld_wait();
        }
        if (!row_ok) continue;
        float y[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a = has0 ? __uint_as_float(o0[i]) * g0 : 0.f;
          const float c = has1 ? __uint_as_float(o1[i]) * g1 : 0.f;
          y[i] = empty ? 0.f : a + c;
        }
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
      if (row_ok && grp == 0) *lse_p = lse_new;
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
vs_status launch_fwd_d(const vs_shape* sh, const void* q, const void* k, const void* v, const void* arena,
                       float scale, void* o, float* lse, float* o_acc, int* err, cudaStream_t st) {
  CUtensorMap tq, tk, tv;
  vs_status rc;
  if ((rc = make_tmap_bshd(&tq, q, sh->B, sh->Nq, sh->Hq, D, sh->sq, kQTile)) != VS_OK) return rc;
  if ((rc = make_tmap_bshd(&tk, k, sh->B, sh->Nk, sh->Hkv, D, sh->sk, kKTile)) != VS_OK) return rc;
  if ((rc = make_tmap_bshd(&tv, v, sh->B, sh->Nk, sh->Hkv, D, sh->sv, kKTile)) != VS_OK) return rc;
  FwdParams p;
  p.arena = arena;
  p.k = static_cast<const uint8_t*>(k);
  p.v = static_cast<const uint8_t*>(v);
  for (int i = 0; i < 3; ++i) {
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
  vs_fwd_kernel<D><<<grid, kFwdThreads, smem, st>>>(tq, tk, tv, p);
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
