// Sparse attention forward on the Vertical-Slash mask (tcgen05 / TMEM / TMA).
//
// One CTA owns one 128-row query tile of one query head and walks its units:
//   * slash tiles: 64 keys starting at local key c = 128 t + 64 - e for every
//     entry e <= 128 t + 127 of the head's query-major list, loaded by TMA;
//   * bar chunks: 64 selected columns gathered with cp.async.
// Per unit: S = Q K^T (M=128, N=64, K=d) into TMEM, fp32 online softmax on
// the exact token mask in registers (one thread per row), P (bf16) back into
// TMEM, O += P V (M=128, N=d, K=64) with A read from TMEM.
//
// Warp roles (352 threads): warp 0 issues the loads, warp 10 builds each
// unit's row masks (both arrive on the stage barrier, so neither waits for
// the other's memory latency), warp 1 issues MMAs (one lane), warps 2-5 and
// 6-9 are two softmax warpgroups that take alternate units (even / odd).  Each group
// keeps its own running maximum, sum and O accumulator, so the groups never
// wait for each other and one group's exp2 phase overlaps the other's
// arithmetic; the epilogue merges the two partial results the way
// merge_out_and_lse of Algorithm 2 merges ring steps.
// TMEM columns: O_g [128 g, 128 g + d), S_g [256 + 64 g, +64),
// P_g [384 + 32 g, +32) for group g.
#include "vs_internal.h"
#include "vs_kernel_common.cuh"

namespace vs {
namespace {

constexpr int kFwdThreads = 352;
constexpr int kFwdMaskWarp = 10;
constexpr int kFwdGroup = 128;  // threads per softmax warpgroup
constexpr int kFwdStages = 5;
constexpr uint32_t kColO = 0, kColS = 256, kColP = 384, kTmemCols = 512;
constexpr float kRefSlack = 18446744073709551616.0f;  // 2^64: largest masked unit sum accepted against the reference

template <int D>
struct FwdSmem {
  static constexpr int NH = D / 64;
  uint8_t q[NH][kQTile * 128];
  uint8_t k[kFwdStages][NH][kKTile * 128];
  uint8_t v[kFwdStages][NH][kKTile * 128];
  uint64_t mask[kFwdStages][kQTile];  // row masks of the unit in stage i (mask warp)
  uint64_t q_full;
  uint64_t kv_full[kFwdStages], kv_empty[kFwdStages];
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];  // per softmax group
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

  if (threadIdx.x == 0) {
    if (!arena_ok && av.hdr->status) raise_error(p.err, av.hdr->status);
    else if (!arena_ok && av.hdr->magic != kArenaMagic) raise_error(p.err, VS_ERR_ARG);
    s.abort_flag = 0;
    mbar_init(&s.q_full, 1);
    for (int i = 0; i < kFwdStages; ++i) {
      mbar_init(&s.kv_full[i], 2);  // loads (producer) + row masks (mask warp)
      mbar_init(&s.kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.s_free[i], kFwdGroup);
      mbar_init(&s.p_full[i], kFwdGroup);
      mbar_init(&s.pv_done[i], 1);
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
    int issued[kFwdStages];
    for (int i = 0; i < kFwdStages; ++i) issued[i] = -1;
    if (U > 0) {
      if (lane == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        mbar_arrive_expect_tx(&s.q_full, NH * kQTile * 128);
        for (int hf = 0; hf < NH; ++hf) tma_load_4d(s.q[hf], &tmQ, &s.q_full, 64 * hf, h, t * kQTile, b);
      }
      const uint8_t* kb = p.k + (int64_t(b) * p.sk[0] + int64_t(hk) * p.sk[2]) * 2;
      const uint8_t* vb = p.v + (int64_t(b) * p.sv[0] + int64_t(hk) * p.sv[2]) * 2;
      int e_pref = 0;  // elist[j0 + lane] for the current 32-unit window
      for (int j = 0; j < U; ++j) {
        const int st = j % kFwdStages;
        if ((j & 31) == 0) e_pref = (j + lane < nslash) ? __ldg(elist + j + lane) : 0;
        const int e_j = __shfl_sync(0xffffffffu, e_pref, j & 31);
        if (j >= kFwdStages && !mbar_wait(&s.kv_empty[st], ((j / kFwdStages) - 1) & 1, ab, VS_ERR_TIMEOUT)) break;
        if (j < nslash) {
          if (lane == 0) {
            const int c = t * kQTile + 64 - e_j;
            mbar_arrive_expect_tx(&s.kv_full[st], 2 * NH * kKTile * 128);
            for (int hf = 0; hf < NH; ++hf) {
              tma_load_4d(s.k[st][hf], &tmK, &s.kv_full[st], 64 * hf, hk, c, b);
              tma_load_4d(s.v[st][hf], &tmV, &s.kv_full[st], 64 * hf, hk, c, b);
            }
          }
        } else {
          const int32_t* keys = vlist + (j - nslash) * kKTile;
          gather_rows<D>(smem_u32(s.k[st][0]), kKTile, kb, p.sk[1], keys, kKTile, lane);
          gather_rows<D>(smem_u32(s.v[st][0]), kKTile, vb, p.sv[1], keys, kKTile, lane);
          asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(&s.kv_full[st])) : "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(&s.kv_full[st]);
        }
        issued[st] = j;
        __syncwarp();
      }
    }
    if (lane == 0 && s.abort_flag) {
      // drain loads still in flight before the CTA's shared memory is released
      for (int i = 0; i < kFwdStages; ++i)
        if (issued[i] >= 0) {
          const uint64_t t0 = global_ns();
          while (!mbar_try_wait(&s.kv_full[i], (issued[i] / kFwdStages) & 1) && global_ns() - t0 < kWaitBudgetNs) {
          }
        }
    }
  } else if (warp == kFwdMaskWarp) {
    // ------------------------------------------------------------ row masks
    // Builds the 128 row masks of each unit into the unit's stage (bitmap
    // reads for slash tiles, position compares for bar chunks) and arrives on
    // the stage barrier; runs as far ahead as the stages allow.
    if (U > 0) {
      const uint64_t* offbits_p = av.offbits + int64_t(bh) * G.WG;
      const uint64_t* colbits_p = av.colbits + int64_t(bh) * G.WG;
      int e_pref = 0;
      for (int j = 0; j < U; ++j) {
        const int st = j % kFwdStages;
        if ((j & 31) == 0) e_pref = (j + lane < nslash) ? __ldg(elist + j + lane) : 0;
        const int e_j = __shfl_sync(0xffffffffu, e_pref, j & 31);
        if (j >= kFwdStages && !mbar_wait(&s.kv_empty[st], ((j / kFwdStages) - 1) & 1, ab, VS_ERR_TIMEOUT)) break;
        if (j < nslash) {
          const int64_t c = int64_t(t) * kQTile + 64 - e_j;
          uint64_t m[kQTile / 32];
#pragma unroll
          for (int rr = 0; rr < kQTile / 32; ++rr) {
            const int64_t nl = int64_t(t) * kQTile + rr * 32 + lane;
            m[rr] = nl < p.Nq ? slash_row_mask(G, offbits_p, colbits_p, qpos_g(G, nl), c) : 0ull;
          }
#pragma unroll
          for (int rr = 0; rr < kQTile / 32; ++rr) s.mask[st][rr * 32 + lane] = m[rr];
        } else {
          const int32_t* keys = vlist + (j - nslash) * kKTile;
          int64_t kg[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int key = __ldg(keys + e * 32 + lane);
            kg[e] = key >= 0 ? kpos_g(G, key) : INT64_MAX;
          }
#pragma unroll
          for (int rr = 0; rr < kQTile / 32; ++rr) {
            const int row = rr * 32 + lane;
            const int64_t nl = int64_t(t) * kQTile + row;
            const int64_t ng = qpos_g(G, nl);
            uint64_t m = 0;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int64_t kge = kg[e];
#pragma unroll 8
              for (int kk = 0; kk < 32; ++kk) {
                const int64_t mg = __shfl_sync(0xffffffffu, kge, kk);
                m |= uint64_t(mg <= ng) << (32 * e + kk);
              }
            }
            s.mask[st][row] = nl < p.Nq ? m : 0ull;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.kv_full[st]);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Unit j belongs to softmax group g = j & 1 (its (j >> 1)-th unit).  S of
    // unit j + 2 is issued as soon as group g has read S of unit j, so a
    // group never waits for its next scores while the other group computes.
    if (lane == 0 && U > 0) {
      const uint32_t idS = idesc_bf16(128, 64, 0, 0);
      const uint32_t idO = idesc_bf16(128, D, 0, 1);
      auto issue_s = [&](int j) {
        const int sk = j % kFwdStages, g = j & 1;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t da = sdesc_sw128(smem_u32(s.q[kk / 4]) + (kk % 4) * 32, 16, 1024);
          const uint64_t db = sdesc_sw128(smem_u32(s.k[sk][kk / 4]) + (kk % 4) * 32, 16, 1024);
          mma_ss(tmem + kColS + 64 * g, da, db, idS, kk > 0);
        }
        mma_commit(&s.s_full[g]);
      };
      bool ok = mbar_wait(&s.q_full, 0, ab, VS_ERR_TIMEOUT);
      for (int j = 0; ok && j < 2 && j < U; ++j) {
        const int sk = j % kFwdStages;
        if (!(ok = mbar_wait(&s.kv_full[sk], (j / kFwdStages) & 1, ab, VS_ERR_TIMEOUT))) break;
        if (j >= nslash) fence_proxy_async_smem();
        tc_fence_after();
        issue_s(j);
        mma_issued = true;
      }
      for (int j = 0; ok && j < U; ++j) {
        const int g = j & 1, k = j >> 1;
        if (j + 2 < U) {
          const int j2 = j + 2, sk2 = j2 % kFwdStages;
          if (!(ok = mbar_wait(&s.s_free[g], k & 1, ab, VS_ERR_TIMEOUT))) break;
          if (!(ok = mbar_wait(&s.kv_full[sk2], (j2 / kFwdStages) & 1, ab, VS_ERR_TIMEOUT))) break;
          if (j2 >= nslash) fence_proxy_async_smem();
          tc_fence_after();
          issue_s(j2);
        }
        const int sv = j % kFwdStages;
        if (!(ok = mbar_wait(&s.p_full[g], k & 1, ab, VS_ERR_TIMEOUT))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kKTile / 16; ++kk) {
          const uint64_t dv = sdesc_sw128(smem_u32(s.v[sv][0]) + kk * 2048, kKTile * 128, 1024);
          mma_ts(tmem + kColO + 128 * g, tmem + kColP + 32 * g + kk * 8, dv, idO, (k > 0 || kk > 0));
        }
        mma_commit(&s.pv_done[g]);
        mma_commit(&s.kv_empty[sv]);
      }
      mma_commit(&s.o_final);
    }
  } else if (warp >= 2 && warp < 2 + 8) {
    // ------------------------------------------------------------ softmax
    const int grp = (warp - 2) >> 2;         // softmax group: units j with j & 1 == grp
    const int quarter = warp & 3;            // TMEM lane quarter this warp may access
    const int r = quarter * 32 + lane;       // query row within the tile
    const uint32_t tl = tmem + (uint32_t(quarter * 32) << 16);
    const int64_t n_loc = int64_t(t) * kQTile + r;
    const bool row_ok = n_loc < p.Nq;
    const uint32_t colO = kColO + 128 * grp, colS = kColS + 64 * grp, colP = kColP + 32 * grp;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = grp; j < U; j += 2) {
      const int k = j >> 1, st = j % kFwdStages;
      ok = mbar_wait(&s.s_full[grp], k & 1, ab, VS_ERR_TIMEOUT);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[64];
      tmem_ld32(tl + colS, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(tl + colS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&s.s_free[grp]);
      // the unit's row masks were written by the producer before it released
      // the stage (acquired here; the phase cannot have moved on, since the
      // stage is recycled only after this unit's P has been consumed)
      ok = mbar_wait(&s.kv_full[st], (j / kFwdStages) & 1, ab, VS_ERR_TIMEOUT);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      const uint64_t mask = s.mask[st][r];
      // The group's previous PV must have landed before O is rescaled or its
      // P buffer is rewritten.
      if (k >= 1) ok = mbar_wait(&s.pv_done[grp], (k - 1) & 1, ab, VS_ERR_TIMEOUT);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // P against the row's reference maximum m_run (log2 units).  The
      // reference is lazy: it only moves when a unit's masked sum shows an
      // entry more than 2^kRefSlack above it (or for the row's first
      // entries); the sum bounds every single entry, so P stays <= 2^64.
      uint32_t pk[32];
      float unit_sum = 0.f;
      auto make_p = [&](float ref) {
        float ps[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) ps[i] = 0.f;
        const float nref = -ref;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float p0 = ex2(fmaf(__uint_as_float(sr[2 * i]), p.scale_log2, nref));
          float p1 = ex2(fmaf(__uint_as_float(sr[2 * i + 1]), p.scale_log2, nref));
          p0 = ((mask >> (2 * i)) & 1ull) ? p0 : 0.f;
          p1 = ((mask >> (2 * i + 1)) & 1ull) ? p1 : 0.f;
          ps[i & 7] += p0 + p1;
          pk[i] = pack_bf16x2(p0, p1);
        }
        unit_sum = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      };
      make_p(m_run == -INFINITY ? 0.f : m_run);
      const bool need = (mask != 0ull) && (m_run == -INFINITY || !(unit_sum <= kRefSlack));
      if (__any_sync(0xffffffffu, need)) {
        // exact masked maximum of this unit (rows that need a new reference)
        float mt = -INFINITY;
        if (need) {
          float mx[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if ((mask >> i) & 1ull) mx[i & 7] = fmaxf(mx[i & 7], __uint_as_float(sr[i]) * p.scale_log2);
          mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        }
        const bool grow = need && (m_run != -INFINITY) && (mt > m_run);
        if (need && m_run == -INFINITY) m_run = mt;  // first entries: the O row is still zero
        if (__any_sync(0xffffffffu, grow)) {
          // tcgen05.ld / st are warp-collective: every lane takes part
          const float alpha = grow ? ex2(m_run - mt) : 1.f;
#pragma unroll 1
          for (int cc = 0; cc < D; cc += 16) {
            uint32_t ov[16];
            tmem_ld16(tl + colO + cc, ov);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st16(tl + colO + cc, ov);
          }
          tmem_st_wait();
          if (grow) {
            l_run *= alpha;
            m_run = mt;
          }
        }
        make_p(m_run == -INFINITY ? 0.f : m_run);
      }
      l_run += unit_sum;
      tmem_st16(tl + colP, *reinterpret_cast<uint32_t(*)[16]>(&pk[0]));
      tmem_st16(tl + colP + 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[16]));
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&s.p_full[grp]);
    }
    // -------------------------------------------------------------- epilogue
    // Wait for every MMA, publish this group's (max, sum) per row, and merge
    // the two groups' partial results; group g writes columns [g d/2, (g+1) d/2).
    bool e_ok = ok && (U == 0 || mbar_wait(&s.o_final, 0, ab, VS_ERR_TIMEOUT));
    e_ok = __all_sync(0xffffffffu, e_ok);
    s.red_m[grp][r] = m_run;
    s.red_l[grp][r] = l_run;
    e_ok = bar_sync_and(1, 2 * kFwdGroup, e_ok);
    tc_fence_after();
    if (e_ok) {
      const float m0 = s.red_m[0][r], m1 = s.red_m[1][r];
      const float l0 = s.red_l[0][r], l1 = s.red_l[1][r];
      const bool has0 = U > 0 && l0 > 0.f, has1 = U > 1 && l1 > 0.f;  // group 1 ran only if U > 1
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
        if (U > 0) {  // warp-collective TMEM reads
          tmem_ld16(tl + kColO + cc, o0);
          if (U > 1) tmem_ld16(tl + kColO + 128 + cc, o1);
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
