// Sparse attention backward on the Vertical-Slash mask (tcgen05 / TMEM / TMA).
//
//   bwd_prep     D_n = rowsum(dO_n * O_n) and LSE in log2 units, per row.
//   dq kernel    query-major, one CTA per (b, h, 128-row tile), the forward's
//                units two at a time: S = Q K^T, dP = dO V^T (N = 128),
//                dS = P (dP - D), dQ += dS K.
//   bar kernel   key-major over gathered selected columns, one CTA per
//                (b, h, 128-column chunk, row split): S^T = K Q^T,
//                dP^T = V dO^T, dV += P^T dO, dK += dS^T Q over 64-row units
//                from the chunk's first column to the end; fp32 partials.
//   dkv kernel   key-major over slash units, one CTA per (b, KV head, 128-key
//                tile), looping over the group's query heads so that the GQA
//                sum happens in TMEM; its epilogue adds the bar partials of
//                the keys that are selected columns, in a fixed order.
// No floating-point atomics: every output element has one writer and a fixed
// summation order.
#include "vs_internal.h"
#include <algorithm>
#include "vs_kernel_common.cuh"

namespace vs {
namespace {

constexpr int kDqThreads = 384;      // + warp 11, the dQ kernel's V loader
// Key-major kernel: 12 warps, one besides the compute warps on each SM
// sub-partition.  A warp that issues MMAs faster than the tensor pipe takes
// them delays the TMEM loads and stores of the compute warps on its
// sub-partition by about the length of its queue, and every unit waits for
// the slowest compute warp; so the two score chains are issued by two warps
// on different sub-partitions (warp 1: S^T, warp 11: dP^T), warp 0 issues
// dV / dK and warp 10 loads.
constexpr int kKvThreads = 384;
constexpr int kKvWarpGrad = 0, kKvWarpS = 1, kKvWarpLoad = 10, kKvWarpDP = 11;
constexpr int kDqVWarp = 11;
constexpr int kBwdCompute = 256;  // two warps per TMEM lane quarter, each owning half the columns
constexpr int kBwdStages = 4;
constexpr int kMaxGroup = 64;  // query heads per KV head supported by the key-major kernel

struct BwdLayout {
  int64_t off_l2, off_d, off_bar_dk, off_bar_dv, total;
  int smax;
};

BwdLayout bwd_layout(int B, int Hq, int Nq, int d, int kv) {
  BwdLayout L;
  const int64_t BH = int64_t(B) * Hq;
  const int64_t KVP = (kv + kBarK - 1) / kBarK * kBarK;
  const int64_t tiles = (Nq + kRowTile - 1) / kRowTile;
  L.smax = int((tiles + kBarSplitTiles - 1) / kBarSplitTiles);
  int64_t off = 256;
  auto take = [&](int64_t bytes) {
    const int64_t at = off;
    off += (bytes + 255) / 256 * 256;
    return at;
  };
  L.off_l2 = take(BH * Nq * 4);
  L.off_d = take(BH * Nq * 4);
  L.off_bar_dk = take(int64_t(L.smax) * BH * KVP * d * 4);
  L.off_bar_dv = take(int64_t(L.smax) * BH * KVP * d * 4);
  L.total = off;
  return L;
}

__device__ __forceinline__ BwdLayout bwd_layout_dev(const ArenaHeader* h, int d) {
  BwdLayout L;
  const int64_t BH = int64_t(h->B) * h->Hq;
  const int64_t KVP = h->KVP;
  const int64_t tiles = (h->Nq + kRowTile - 1) / kRowTile;
  L.smax = int((tiles + kBarSplitTiles - 1) / kBarSplitTiles);
  int64_t off = 256;
  auto take = [&](int64_t bytes) {
    const int64_t at = off;
    off += (bytes + 255) / 256 * 256;
    return at;
  };
  L.off_l2 = take(BH * h->Nq * 4);
  L.off_d = take(BH * h->Nq * 4);
  L.off_bar_dk = take(int64_t(L.smax) * BH * KVP * d * 4);
  L.off_bar_dv = take(int64_t(L.smax) * BH * KVP * d * 4);
  L.total = off;
  return L;
}

struct BwdParams {
  const void* arena;
  const uint8_t* q;
  const uint8_t* k;
  const uint8_t* v;
  const uint8_t* o;
  const uint8_t* dO;
  const float* lse;
  int64_t sq[3], sk[3], sv[3], so[3];
  int B, Nq, Nk, Hq, Hkv;
  float scale, scale_log2;
  uint8_t* dq;
  uint8_t* dk;
  uint8_t* dv;
  float* dq_acc;
  float* dkv_acc;  // NULL, or fp32 [2][B][Nk][Hkv][d]: dK then dV, accumulated
  uint8_t* ws;
  size_t ws_bytes;
  int bar_nchunk;  // chunks per (b, h) in the bar kernel's grid (>= KVP / 128)
  int* err;
};

// Verifies the arena and the workspace size; returns false (and records the
// error once) if the kernel must not run.
__device__ __forceinline__ bool bwd_inputs_ok(const BwdParams& p, const ArenaView& av, int d) {
  const bool arena_ok = (av.hdr->status == 0) && (av.hdr->magic == kArenaMagic) && av.hdr->Nq == p.Nq &&
                        av.hdr->Hq == p.Hq && av.hdr->B == p.B;
  const bool ws_ok = arena_ok && bwd_layout_dev(av.hdr, d).total <= int64_t(p.ws_bytes);
  if (!(arena_ok && ws_ok) && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
    raise_error(p.err, !arena_ok ? (av.hdr->status ? av.hdr->status : int(VS_ERR_ARG)) : int(VS_ERR_WORKSPACE));
  // a workspace already holding an error makes the call skip its work
  return arena_ok && ws_ok && *reinterpret_cast<volatile int*>(p.err) == 0;
}

// ------------------------------------------------------------------ prepass
__global__ void __launch_bounds__(256) bwd_prep(const BwdParams p, int d) {
  const int64_t total = int64_t(p.B) * p.Hq * p.Nq;
  const ArenaView av = arena_view(p.arena);
  if (!bwd_inputs_ok(p, av, d)) return;
  const BwdLayout L = bwd_layout_dev(av.hdr, d);
  float* l2 = reinterpret_cast<float*>(p.ws + L.off_l2);
  float* dd = reinterpret_cast<float*>(p.ws + L.off_d);
  // eight lanes per row, 16-byte pieces (a row's 128 or 256 bytes in one or
  // two coalesced sweeps); a warp takes four consecutive rows and every lane
  // runs the same trip count, so the lane reductions see the whole warp
  const int lane = threadIdx.x & 31, sub = lane & 7;
  const int64_t warps = int64_t(gridDim.x) * (blockDim.x / 32);
  for (int64_t base = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) / 32 * 4; base < total; base += warps * 4) {
    const int64_t i = base + (lane >> 3);
    const bool ok = i < total;
    float acc = 0.f;
    if (ok) {
      const int64_t n = i % p.Nq, bh = i / p.Nq;
      const int64_t b = bh / p.Hq, h = bh % p.Hq;
      const int64_t off = (b * p.so[0] + n * p.so[1] + h * p.so[2]) * 2;
      const uint4* orow = reinterpret_cast<const uint4*>(p.o + off);
      const uint4* grow = reinterpret_cast<const uint4*>(p.dO + off);
      for (int c = sub; c < d / 8; c += 8) {
        const uint4 a = orow[c], g = grow[c];
        const uint32_t av4[4] = {a.x, a.y, a.z, a.w}, gv4[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc = fmaf(__uint_as_float(av4[e] << 16), __uint_as_float(gv4[e] << 16), acc);
          acc = fmaf(__uint_as_float(av4[e] & 0xFFFF0000u), __uint_as_float(gv4[e] & 0xFFFF0000u), acc);
        }
      }
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    if (ok && sub == 0) {
      dd[i] = acc;
      l2[i] = -p.lse[i] * kLog2e;  // stored negated: the kernels add it to the scaled scores
    }
  }
}

// ---------------------------------------------------------------- dQ kernel
// One CTA per (b, h, 128-row query tile) walks the forward's units two at a
// time (a pair: 128 keys, the two units' 64-key blocks stacked):
//   S = Q K^T and dP = dO V^T as M=128, N=128 MMA chains, A (Q, dO) in TMEM;
//   dS = P (dP - D) on the exact mask, written to shared memory (bf16);
//   dQ += dS K over the pair's 128 keys (A = dS, B = K, both in shared memory).
// The compute warps copy S and dP of a pair into registers and release the
// TMEM at once, so the next pair's S / dP run while they compute dS.  Each
// compute thread builds its own row's mask of its unit (slash: a window of
// the offset bitmap; bar: a count of the unit's keys at or before the row).
// Two warps issue MMAs: warp 1 the S / dP chains, warp 10 the dQ chains (the
// two streams touch disjoint TMEM and are ordered by barriers only), so the
// waits of one stream do not leave the tensor pipe idle; two warps load K
// (warp 0) and V (warp 11).
// TMEM: dQ [0, 128), S [128, 256), dP [256, 384), Q [384, 448), dO [448, 512).
constexpr uint32_t kDqColAcc = 0, kDqColS = 128, kDqColDP = 256, kDqColQ = 384, kDqColDO = 448;
constexpr int kDqPairKeys = 2 * kKTile;
constexpr int kDqKSlots = 3, kDqVSlots = 2;

template <int D>
struct DqSmem {
  static constexpr int NH = D / 64;
  uint8_t k[kDqKSlots][NH][kDqPairKeys * 128];  // K of a pair, 128B-swizzled, per d-half
  uint8_t v[kDqVSlots][NH][kDqPairKeys * 128];
  uint8_t ds[2][kQTile * 128];                   // dS of a pair, keys [0, 64) and [64, 128), K-major SW128
  int64_t bar_pos[kDqKSlots][2][kKTile];         // bar units: global key positions (INT64_MAX = none)
  int64_t unit_c[kDqKSlots][2];                  // slash: first local key; bar: kUnitBar; none: kUnitNone
  uint64_t qdo_full;
  uint64_t k_full[kDqKSlots], k_empty[kDqKSlots], v_full[kDqVSlots], v_empty[kDqVSlots];
  uint64_t s_full, s_free, ds_full, ds_done;
  uint64_t fin, teardown, teardown_dq;
  uint32_t tmem_base;
  int abort_flag;
};
constexpr int64_t kUnitBar = INT64_MIN, kUnitNone = INT64_MIN + 1;

// Loads the K (which = 0) or V rows of unit u into half `hf` of a pair slot
// (TMA for slash units, a cp.async gather for bar units); returns the bytes the
// TMA will deliver.  All 32 lanes call it; lane 0 issues the TMA.
template <int D>
__device__ __forceinline__ int dq_load_unit(uint8_t (*slot)[kDqPairKeys * 128], int hf, uint64_t* bar,
                                            const CUtensorMap* tm, const uint8_t* base, int64_t s_tok,
                                            const int32_t* vlist, int u, int nslash, int64_t c, int hk, int b,
                                            int lane) {
  constexpr int NH = D / 64;
  if (u < nslash) {
    if (lane == 0)
      for (int h = 0; h < NH; ++h) tma_load_4d(slot[h] + hf * kKTile * 128, tm, bar, 64 * h, hk, int(c), b);
    return NH * kKTile * 128;
  }
  gather_rows<D>(smem_u32(slot[0]) + hf * kKTile * 128, kDqPairKeys, base, s_tok, vlist + (u - nslash) * kKTile,
                 kKTile, lane);
  return 0;
}

// Kernel body, compiled once per mask reading (BLOCK: block-cover slashes).
template <int D, bool BLOCK>
__device__ __forceinline__ void dq_body(const CUtensorMap& tmK, const CUtensorMap& tmV, const BwdParams& p) {
  extern __shared__ uint8_t smem_raw[];
  DqSmem<D>& s = *reinterpret_cast<DqSmem<D>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const ArenaView av = arena_view(p.arena);
  const bool inputs_ok = bwd_inputs_ok(p, av, D);
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
  const TileWork tw = inputs_ok ? tile_work(av, G, bh, r0, R) : TileWork{0, 0, 0};
  const int32_t* elist = av.elist + int64_t(bh) * G.EMAX + tw.lo;  // this tile's slash units
  const int32_t* vlist = av.vlist + int64_t(bh) * G.KVP;
  const int nslash = tw.nslash, nbar = tw.nbar;
  const int U = nslash + nbar;
  const int P = (U + 1) / 2;  // pairs
  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    mbar_init(&s.qdo_full, kBwdCompute);
    for (int i = 0; i < kDqKSlots; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.k_empty[i], 1);
    }
    for (int i = 0; i < kDqVSlots; ++i) {
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.v_empty[i], 1);
    }
    mbar_init(&s.s_full, 1);
    mbar_init(&s.s_free, kBwdCompute);
    mbar_init(&s.ds_full, kBwdCompute);
    mbar_init(&s.ds_done, 1);
    mbar_init(&s.fin, 1);
    mbar_init(&s.teardown, 1);
    mbar_init(&s.teardown_dq, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  const Abort ab{&s.abort_flag, p.err};
  bool mma_issued = false;
  auto gathered = [&](int i) { return 2 * i + 1 >= nslash; };  // pair i holds a bar unit

  if (warp == 0 || warp == kDqVWarp) {
    // ----------------------------------------------------------- producers
    // Warp 0: per pair the units' descriptions and K into a K slot (kept
    // until the dQ chain of the pair has read it); warp kDqVWarp: V into a V
    // slot.  Both walk the e-list one pair ahead.
    const bool isv = warp == kDqVWarp;
    const int nslot = isv ? kDqVSlots : kDqKSlots;
    uint64_t* full = isv ? s.v_full : s.k_full;
    uint64_t* empty = isv ? s.v_empty : s.k_empty;
    const CUtensorMap* tm = isv ? &tmV : &tmK;
    const uint8_t* base = isv ? p.v + (int64_t(b) * p.sv[0] + int64_t(hk) * p.sv[2]) * 2
                              : p.k + (int64_t(b) * p.sk[0] + int64_t(hk) * p.sk[2]) * 2;
    const int64_t stok = isv ? p.sv[1] : p.sk[1];
    int issued[kDqKSlots];
    for (int i = 0; i < kDqKSlots; ++i) issued[i] = -1;
    int e_cur[2], e_nxt[2];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) e_cur[hf] = hf < nslash ? __ldg(elist + hf) : 0;
    for (int i = 0; i < P; ++i) {
      const int sl = i % nslot;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) e_nxt[hf] = 2 * i + 2 + hf < nslash ? __ldg(elist + 2 * i + 2 + hf) : 0;
      if (i >= nslot && !mbar_wait(&empty[sl], ((i / nslot) - 1) & 1, ab, VS_ERR_TIMEOUT)) break;
      int64_t c[2];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int u = 2 * i + hf;
        c[hf] = u >= U ? kUnitNone : (u < nslash ? r0 + R - 64 - e_cur[hf] : kUnitBar);
        if (!isv) {
          if (c[hf] == kUnitBar) {
            const int32_t* keys = vlist + (u - nslash) * kKTile;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int key = __ldg(keys + e * 32 + lane);
              s.bar_pos[sl][hf][e * 32 + lane] = key >= 0 ? kpos_g(G, key) : INT64_MAX;
            }
          }
          if (lane == 0) s.unit_c[sl][hf] = c[hf];
        }
      }
      // gathers (and their arrivals) first, then the one plain arrival with
      // the TMA byte count, so the phase cannot complete before the gathers
      int bytes = 0;
      uint8_t (*slot)[kDqPairKeys * 128] = isv ? s.v[sl] : s.k[sl];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
        if (2 * i + hf < U)
          bytes += dq_load_unit<D>(slot, hf, &full[sl], tm, base, stok, vlist, 2 * i + hf, nslash, c[hf], hk, b,
                                   lane);
      if (gathered(i))
        asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(&full[sl])) : "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&full[sl], uint32_t(bytes));
      issued[sl] = i;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) e_cur[hf] = e_nxt[hf];
    }
    if (lane == 0 && s.abort_flag) {
      // drain loads still in flight before the CTA's shared memory is released
      for (int i = 0; i < nslot; ++i)
        if (issued[i] >= 0) {
          const uint64_t t0 = global_ns();
          while (!mbar_try_wait(&full[i], (issued[i] / nslot) & 1) && global_ns() - t0 < kWaitBudgetNs) {
          }
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- S / dP issuer
    // Per pair i: S_i, dP_i once the compute warps hold S / dP of pair i - 1
    // in registers.
    // The whole warp runs the loop; one elected lane issues.
    if (P > 0) {
      const uint32_t idS = idesc_bf16(128, kDqPairKeys, 0, 0);
      bool ok = mbar_wait_warp(&s.qdo_full, 0, ab, VS_ERR_TIMEOUT);
      for (int i = 0; ok && i < P; ++i) {
        const int ks = i % kDqKSlots, vsl = i % kDqVSlots;
        if (!(ok = mbar_wait_warp(&s.k_full[ks], (i / kDqKSlots) & 1, ab, VS_ERR_TIMEOUT))) break;
        if (!(ok = mbar_wait_warp(&s.v_full[vsl], (i / kDqVSlots) & 1, ab, VS_ERR_TIMEOUT))) break;
        if (i >= 1 && !(ok = mbar_wait_warp(&s.s_free, (i - 1) & 1, ab, VS_ERR_TIMEOUT))) break;
        if (gathered(i)) fence_proxy_async_smem();
        tc_fence_after();
        // a K-chunk's descriptor is the slot's plus its offset (shared
        // addresses stay below 256 KB: the 14-bit start field never carries)
        const uint64_t dks = sdesc_sw128(smem_u32(s.k[ks][0]), 16, 1024);
        const uint64_t dvs = sdesc_sw128(smem_u32(s.v[vsl][0]), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t dk_ = dks + (uint32_t((kk / 4) * kDqPairKeys * 128 + (kk % 4) * 32) >> 4);
          mma_ts_warp(tmem + kDqColS, tmem + kDqColQ + kk * 8, dk_, idS, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t dv_ = dvs + (uint32_t((kk / 4) * kDqPairKeys * 128 + (kk % 4) * 32) >> 4);
          mma_ts_warp(tmem + kDqColDP, tmem + kDqColDO + kk * 8, dv_, idS, kk > 0);
        }
        mma_commit_warp(&s.s_full);
        mma_commit_warp(&s.v_empty[vsl]);
        mma_issued = true;
      }
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ dQ issuer
    // Per pair i, once its dS is in shared memory: dQ += dS K over the pair's
    // keys (K stays in its slot until then).
    if (P > 0) {
      const uint32_t idQ = idesc_bf16(128, D, 0, 1);
      const uint64_t dds = sdesc_sw128(smem_u32(s.ds[0]), 16, 1024);
      bool ok = true;
      for (int i = 0; ok && i < P; ++i) {
        if (!(ok = mbar_wait_warp(&s.ds_full, i & 1, ab, VS_ERR_TIMEOUT))) break;
        if (gathered(i)) fence_proxy_async_smem();
        tc_fence_after();
        const int ks = i % kDqKSlots;
        const int nk = (2 * i + 1 < U) ? kDqPairKeys / 16 : kKTile / 16;
        const uint64_t dkm = sdesc_sw128(smem_u32(s.k[ks][0]), kDqPairKeys * 128, 1024);
#pragma unroll
        for (int kk = 0; kk < kDqPairKeys / 16; ++kk) {
          if (kk >= nk) break;
          const uint64_t da = dds + (uint32_t((kk / 4) * kQTile * 128 + (kk % 4) * 32) >> 4);
          const uint64_t dk_ = dkm + uint32_t(kk * 2048 >> 4);
          mma_ss_warp(tmem + kDqColAcc, da, dk_, idQ, (i > 0 || kk > 0));
        }
        mma_commit_warp(&s.ds_done);
        mma_commit_warp(&s.k_empty[ks]);
        mma_issued = true;
      }
      mma_commit_warp(&s.fin);
    }
  } else {
    // ------------------------------------------------------------ compute
    // Warp (quarter, half): row quarter * 32 + lane, unit 2 i + half of each
    // pair i (the pair's key columns [64 half, 64 half + 64)).
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const int hrow = gp ? h + r % gp : h;  // the row's query head
    const uint32_t tl = tmem + (uint32_t(quarter * 32) << 16);
    const int64_t n_loc = r0 + (gp ? r / gp : r);
    const bool row_ok = n_loc < p.Nq && inputs_ok;
    const int64_t n_g = qpos_g(G, n_loc);
    const uint64_t* offbits = av.offbits + int64_t(bh) * G.WG;
    const uint64_t* colbits = av.colbits + int64_t(bh) * G.WG;
    // block cover: the row's two candidate block diagonals instead of its
    // offset window
    constexpr bool block_cover = BLOCK;
    const uint64_t* diagbits = block_cover ? av.bdbits + int64_t(bh) * G.WG : offbits;
    float Lr = 0.f, Dr = 0.f;
    if (row_ok) {
      const BwdLayout L = bwd_layout_dev(av.hdr, D);
      const int64_t bhr = int64_t(b) * p.Hq + hrow;
      Lr = reinterpret_cast<const float*>(p.ws + L.off_l2)[bhr * p.Nq + n_loc];
      Dr = reinterpret_cast<const float*>(p.ws + L.off_d)[bhr * p.Nq + n_loc];
    }
    // Q row r and dO row r, d columns [half D/2, (half + 1) D/2), into TMEM
    // as bf16 pairs
#pragma unroll 1
    for (int which = 0; which < 2; ++which) {
      uint32_t w[D / 4];
      const uint8_t* src =
          which ? p.dO + (int64_t(b) * p.so[0] + n_loc * p.so[1] + int64_t(hrow) * p.so[2]) * 2 + half * D
                : p.q + (int64_t(b) * p.sq[0] + n_loc * p.sq[1] + int64_t(hrow) * p.sq[2]) * 2 + half * D;
#pragma unroll
      for (int c = 0; c < D / 16; ++c) {
        const uint4 x = row_ok ? *reinterpret_cast<const uint4*>(src + 16 * c) : make_uint4(0, 0, 0, 0);
        w[4 * c] = x.x;
        w[4 * c + 1] = x.y;
        w[4 * c + 2] = x.z;
        w[4 * c + 3] = x.w;
      }
      const uint32_t col = (which ? kDqColDO : kDqColQ) + half * (D / 4);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tmem_st16(tl + col + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&w[16 * c]));
    }
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(&s.qdo_full);
    uint8_t* ds_row = s.ds[half] + r * 128;
    bool ok = true;
    for (int i = 0; i < P; ++i) {
      const int ks = i % kDqKSlots;
      // the unit's description (written by the producer before K landed)
      ok = mbar_wait(&s.k_full[ks], (i / kDqKSlots) & 1, ab, VS_ERR_TIMEOUT);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      const int64_t c = s.unit_c[ks][half];
      const bool slash = row_ok && c != kUnitNone && c != kUnitBar;
      // slash: bit k of the mask is set iff offset n_g - m_g(c + k) is
      // selected, key c + k exists and is not a selected column (the 64 keys
      // are globally contiguous).  The bitmap words are loaded here and used
      // after the scores arrive.
      const int64_t m0 = slash ? (c >= 0 ? kpos_g(G, c) : c) : 0;
      const int64_t lo = block_cover ? (n_g >> 6) - (m0 >> 6) - 1 : n_g - m0 - 63;
      const int64_t wo = lo >> 6, wc = m0 >> 6;
      const uint64_t oa = (slash && wo >= 0 && wo < G.WG) ? __ldg(diagbits + wo) : 0ull;
      const uint64_t ob = (slash && wo + 1 >= 0 && wo + 1 < G.WG) ? __ldg(diagbits + wo + 1) : 0ull;
      const uint64_t ca = (slash && wc >= 0 && wc < G.WG) ? __ldg(colbits + wc) : 0ull;
      const uint64_t cb = (slash && wc + 1 >= 0 && wc + 1 < G.WG) ? __ldg(colbits + wc + 1) : 0ull;
      uint64_t mask = 0;
      if (slash) {
        const int so = int(lo & 63), sc = int(m0 & 63);
        const uint64_t x = so ? ((oa >> so) | (ob << (64 - so))) : oa;
        const uint64_t cw = sc ? ((ca >> sc) | (cb << (64 - sc))) : ca;
        const uint64_t keep = ~cw & (c < 0 ? ((~0ull) << (-c)) : ~0ull) & low_bits(int64_t(G.Nk) - c);
        if (block_cover) {
          // keys below the split are in the first key block (diagonal bit 1),
          // the rest in the next one (bit 0); causal keys only
          const uint64_t lo_keys = low_bits(64 - (m0 & 63));
          mask = (((x & 2ull) ? lo_keys : 0ull) | ((x & 1ull) ? ~lo_keys : 0ull)) & low_bits(n_g - m0 + 1) & keep;
        } else {
          mask = __brevll(x) & keep;
        }
      } else if (row_ok && c == kUnitBar) {
        const int64_t* pos = s.bar_pos[ks][half];
        int cnt = 0;
#pragma unroll
        for (int step = 32; step > 0; step >>= 1)
          if (pos[cnt + step - 1] <= n_g) cnt += step;
        if (pos[kKTile - 1] <= n_g) cnt = kKTile;
        mask = cnt == kKTile ? ~0ull : ((1ull << cnt) - 1);
      }
      // only the 16-key chunks holding a mask entry of the warp's rows are
      // computed (warp-uniform; on the slash units of sparse selections about
      // half of them are empty); dS of the others is zero.  The row mask is
      // built before the scores arrive.
      const uint32_t occ = chunk_occupancy16(mask);
      ok = mbar_wait(&s.s_full, i & 1, ab, VS_ERR_TIMEOUT);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[64], pr[64];
      tmem_ld32(tl + kDqColS + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(tl + kDqColS + 64 * half + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_ld32(tl + kDqColDP + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&pr[0]));
      tmem_ld32(tl + kDqColDP + 64 * half + 32, *reinterpret_cast<uint32_t(*)[32]>(&pr[32]));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&s.s_free);
      // two keys at a time in paired fp32: P = 2^(S scale log2(e) - LSE log2(e))
      // (Lr = -LSE log2(e)), dS = P (dP - D) on the mask
      uint32_t pk[32];
      const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2), lr2 = f2_pack(Lr, Lr), dr2 = f2_pack(Dr, Dr);
#pragma unroll
      for (int cq = 0; cq < 4; ++cq) {
        if (!((occ >> cq) & 1u)) {
#pragma unroll
          for (int k = 8 * cq; k < 8 * cq + 8; ++k) pk[k] = 0u;
          continue;
        }
#pragma unroll
        for (int k = 8 * cq; k < 8 * cq + 8; ++k) {
          const int col = 2 * k;
          float t0, t1, x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[col]), __uint_as_float(sr[col + 1])), sc2, lr2), t0, t1);
          f2_unpack(f2_mul(f2_pack(ex2(t0), ex2(t1)),
                           f2_sub(f2_pack(__uint_as_float(pr[col]), __uint_as_float(pr[col + 1])), dr2)),
                    x0, x1);
          // after the product: masked scores may be garbage
          pk[k] = pack_bf16x2(((mask >> col) & 1ull) ? x0 : 0.f, ((mask >> (col + 1)) & 1ull) ? x1 : 0.f);
        }
      }
      if (i >= 1) ok = mbar_wait(&s.ds_done, (i - 1) & 1, ab, VS_ERR_TIMEOUT);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      // row r of the unit's 64 keys: eight 16-byte chunks, 128B-swizzled
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint4*>(ds_row + ((j ^ (r & 7)) << 4)) =
            make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
      fence_proxy_async_smem();
      mbar_arrive(&s.ds_full);
    }
    if (ok && P > 0) ok = mbar_wait(&s.fin, 0, ab, VS_ERR_TIMEOUT);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (ok && inputs_ok) {
      // TMEM reads are warp-collective: every lane loads, valid rows store;
      // each half writes its half of the d columns
      const bool store = n_loc < p.Nq;
      uint8_t* drow = p.dq + (int64_t(b) * p.sq[0] + n_loc * p.sq[1] + int64_t(hrow) * p.sq[2]) * 2;
      float* acc = (p.dq_acc && store) ? p.dq_acc + ((int64_t(b) * p.Nq + n_loc) * p.Hq + hrow) * D : nullptr;
#pragma unroll 1
      for (int cc = (D / 2) * half; cc < (D / 2) * (half + 1); cc += 16) {
        uint32_t gv[16];
        if (P > 0) {
          tmem_ld16(tl + kDqColAcc + cc, gv);
          tmem_ld_wait();
        }
        if (!store) continue;
        float y[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) y[i] = P > 0 ? __uint_as_float(gv[i]) * p.scale : 0.f;
        if (acc) {
#pragma unroll
          for (int i = 0; i < 16; i += 4) {
            float4 a4 = *reinterpret_cast<float4*>(acc + cc + i);
            a4.x += y[i];
            a4.y += y[i + 1];
            a4.z += y[i + 2];
            a4.w += y[i + 3];
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
        *reinterpret_cast<uint4*>(drow + cc * 2) = w0;
        *reinterpret_cast<uint4*>(drow + cc * 2 + 16) = w1;
      }
    }
  }
  // an issuer that gave up waits (bounded) for its own MMAs in flight
  if ((warp == 1 || warp == 10) && lane == 0 && mma_issued && s.abort_flag) {
    uint64_t* tb = warp == 1 ? &s.teardown : &s.teardown_dq;
    mma_commit(tb);
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(tb, 0) && global_ns() - t0 < kWaitBudgetNs) {
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
__global__ void __launch_bounds__(kDqThreads, 1)
    vs_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const BwdParams p) {
  if (arena_view(p.arena).hdr->block_cover) dq_body<D, true>(tmK, tmV, p);
  else dq_body<D, false>(tmK, tmV, p);
}

// ------------------------------------------------------ key-major dK / dV
// TMEM: dK [0, 128), dV [128, 256), S^T [256, 320), dP^T [320, 384), P^T (bf16)
// [384, 416), dS^T (bf16) [416, 448), K (bf16, the A operand of S^T = K Q^T,
// loaded once per tile) [448, 512).
constexpr uint32_t kKvColDK = 0, kKvColDV = 128, kKvColS = 256, kKvColDP = 320, kKvColP = 384, kKvColDS = 416,
                   kKvColK = 448;

template <int D>
struct KvSmem {
  static constexpr int NH = D / 64;
  uint8_t v[NH][kBarK * 128];  // A operand of dP^T = V dO^T: 128 keys
  uint8_t q[kBwdStages][NH][kRowTile * 128];  // B operands: 64 rows
  uint8_t g[kBwdStages][NH][kRowTile * 128];
  alignas(16) float l2[kBwdStages][kRowTile];
  alignas(16) float dd[kBwdStages][kRowTile];
  int32_t unit_head[kBwdStages];
  int32_t unit_row[kBwdStages];
  int32_t head_units[kMaxGroup];  // slash: units of each head of the group
  int32_t head_lo[kMaxGroup];     // slash: the head's first f-list entry of this key tile
  uint64_t kv_full, k_tmem;
  uint64_t st_full[kBwdStages], st_empty[kBwdStages];
  uint64_t s_full, sd_full, s_free, p_full, mm_done;
  uint64_t fin, teardown, teardown_g, teardown_d;
  uint32_t tmem_base;
  int abort_flag;
};

// Unit enumeration of a key-major CTA.
//   slash (BAR = false): CTA (b, hk, key tile tau); units run over the query
//     heads h of the group, then the head's flist entries f with
//     128 tau + f <= Nq - 1, rows [128 tau + f, +64).
//   bar (BAR = true): CTA (b, h, chunk c, split sp); units are 64-row tiles
//     from the chunk's first block to the end, split in pieces of
//     kBarSplitTiles tiles.
struct KvWork {
  int n_units;
  int heads;         // slash: number of heads in the group
  int64_t row0;      // bar: first row of the split
};

template <int D, bool BAR, bool BLOCK>
__device__ __forceinline__ void kv_body(const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmQ,
                                        const CUtensorMap& tmG, const BwdParams& p) {
  constexpr int NH = D / 64;
  extern __shared__ uint8_t smem_raw[];
  KvSmem<D>& s = *reinterpret_cast<KvSmem<D>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const ArenaView av = arena_view(p.arena);
  const bool inputs_ok = bwd_inputs_ok(p, av, D);
  const Geo G = geo_from(av.hdr, p.Hkv, D);
  const BwdLayout L = bwd_layout_dev(av.hdr, D);

  // ---- work of this CTA
  int b, hk, h_bar = 0, chunk = 0, split = 0;
  int64_t k0 = 0;
  KvWork w;
  w.n_units = 0;
  w.heads = 0;
  w.row0 = 0;
  bool cta_ok = inputs_ok;
  if (!BAR) {
    // early keys see the most rows: launch them first
    const int BHK = p.B * p.Hkv;
    const int bhk = int(blockIdx.x) % BHK;
    b = bhk / p.Hkv;
    hk = bhk % p.Hkv;
    k0 = int64_t(int(blockIdx.x) / BHK) * kBarK;
    if (cta_ok) {
      w.heads = G.g;
      // the entries f whose rows [k0 + f, + 64) meet [0, Nq)
      for (int hh = 0; hh < G.g; ++hh) {
        const int bh = b * p.Hq + hk * G.g + hh;
        const int32_t* fl = av.flist + int64_t(bh) * G.EMAX;
        const int nf = __ldg(av.fcount + bh);
        const int lo = count_le(fl, nf, -k0 - 64);
        const int c = count_le(fl, nf, int64_t(p.Nq) - 1 - k0) - lo;
        if (threadIdx.x == 0) {
          s.head_units[hh] = c;
          s.head_lo[hh] = lo;
        }
        w.n_units += c;
      }
    }
  } else {
    split = int(blockIdx.x) % L.smax;
    const int rest = int(blockIdx.x) / L.smax;
    chunk = rest % p.bar_nchunk;
    const int bh = rest / p.bar_nchunk;
    b = bh / p.Hq;
    h_bar = bh % p.Hq;
    hk = h_bar / G.g;
    k0 = int64_t(chunk) * kBarK;  // position in the vertical list
    if (cta_ok) {
      const int vc = __ldg(av.vcount + bh);
      if (chunk * kBarK < vc && chunk * kBarK < G.KVP) {
        const int64_t rs =
            first_causal_row_block(G.world, G.q_rank, kpos_g(G, __ldg(av.vlist + int64_t(bh) * G.KVP + chunk * kBarK))) *
            kBlk;
        const int64_t tiles = (p.Nq - rs + kRowTile - 1) / kRowTile;
        const int64_t first = int64_t(split) * kBarSplitTiles;
        if (first < tiles) {
          w.row0 = rs + first * kRowTile;
          w.n_units = int(min(int64_t(kBarSplitTiles), tiles - first));
        }
      }
    }
  }
  const int U = w.n_units;
  const bool run = cta_ok && U > 0;
  if (BAR && !run) return;  // nothing to write for this split

  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    mbar_init(&s.kv_full, 1);
    mbar_init(&s.k_tmem, kBwdCompute);
    for (int i = 0; i < kBwdStages; ++i) {
      mbar_init(&s.st_full[i], 1);
      mbar_init(&s.st_empty[i], 1);
    }
    mbar_init(&s.s_full, 1);
    mbar_init(&s.sd_full, 1);
    mbar_init(&s.s_free, kBwdCompute);
    mbar_init(&s.p_full, kBwdCompute);
    mbar_init(&s.mm_done, 1);
    mbar_init(&s.fin, 1);
    mbar_init(&s.teardown, 1);
    mbar_init(&s.teardown_g, 1);
    mbar_init(&s.teardown_d, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  const Abort ab{&s.abort_flag, p.err};
  bool mma_issued = false;
  const int32_t* bar_keys = BAR ? av.vlist + (int64_t(b) * p.Hq + h_bar) * G.KVP + k0 : nullptr;

  if (warp == kKvWarpLoad) {
    // ------------------------------------------------------------ producer
    int issued[kBwdStages];
    for (int i = 0; i < kBwdStages; ++i) issued[i] = -1;
    bool kv_issued = false;
    if (run) {
      if (!BAR) {
        if (lane == 0) {
          mbar_arrive_expect_tx(&s.kv_full, NH * kBarK * 128);
          for (int hf = 0; hf < NH; ++hf) tma_load_4d(s.v[hf], &tmV, &s.kv_full, 64 * hf, hk, int(k0), b);
        }
      } else {
        const uint8_t* vb = p.v + (int64_t(b) * p.sv[0] + int64_t(hk) * p.sv[2]) * 2;
        gather_rows<D>(smem_u32(s.v[0]), kBarK, vb, p.sv[1], bar_keys, kBarK, lane);
        asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(&s.kv_full)) : "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.kv_full);
      }
      kv_issued = true;
      const float* l2g = reinterpret_cast<const float*>(p.ws + L.off_l2);
      const float* ddg = reinterpret_cast<const float*>(p.ws + L.off_d);
      // slash: the group's head of a unit and its f-list entry, read one unit
      // ahead so that the load overlaps the previous unit's issue
      int cur_h = 0, cur_j = 0, h_nxt = 0;
      int32_t f_nxt = 0;
      auto next_unit = [&]() {
        while (cur_h < w.heads - 1 && cur_j >= s.head_units[cur_h]) {
          cur_j = 0;
          ++cur_h;
        }
        h_nxt = hk * G.g + cur_h;
        f_nxt = __ldg(av.flist + (int64_t(b) * G.Hq + h_nxt) * G.EMAX + s.head_lo[cur_h] + cur_j);
        ++cur_j;
      };
      if (!BAR && U > 0) next_unit();
      for (int j = 0; j < U; ++j) {
        const int st = j % kBwdStages;
        if (j >= kBwdStages && !mbar_wait(&s.st_empty[st], ((j / kBwdStages) - 1) & 1, ab, VS_ERR_TIMEOUT)) break;
        int h;
        int64_t r0;
        if (BAR) {
          h = h_bar;
          r0 = w.row0 + int64_t(j) * kRowTile;
        } else {
          h = h_nxt;
          r0 = k0 + f_nxt;
          if (j + 1 < U) next_unit();
        }
        // the rows' LSE and D by asynchronous copies (zero past the end),
        // tracked by the stage's barrier like the TMA loads
        const float* l2r = l2g + (int64_t(b) * p.Hq + h) * p.Nq;
        const float* ddr = ddg + (int64_t(b) * p.Hq + h) * p.Nq;
        for (int i = lane; i < kRowTile; i += 32) {
          const int64_t n = r0 + i;
          const bool in = n >= 0 && n < p.Nq;
          cp_async_4(smem_u32(&s.l2[st][i]), in ? l2r + n : l2r, in ? 4u : 0u);
          cp_async_4(smem_u32(&s.dd[st][i]), in ? ddr + n : ddr, in ? 4u : 0u);
        }
        asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(&s.st_full[st])) : "memory");
        if (lane == 0) {
          s.unit_head[st] = h;
          s.unit_row[st] = int32_t(r0);
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(&s.st_full[st], 2 * NH * kRowTile * 128);
          for (int hf = 0; hf < NH; ++hf) {
            tma_load_4d(s.q[st][hf], &tmQ, &s.st_full[st], 64 * hf, h, int(r0), b);
            tma_load_4d(s.g[st][hf], &tmG, &s.st_full[st], 64 * hf, h, int(r0), b);
          }
        }
        issued[st] = j;
        __syncwarp();
      }
    }
    if (lane == 0 && s.abort_flag) {
      const uint64_t t0 = global_ns();
      if (kv_issued)
        while (!mbar_try_wait(&s.kv_full, 0) && global_ns() - t0 < kWaitBudgetNs) {
        }
      for (int i = 0; i < kBwdStages; ++i)
        if (issued[i] >= 0) {
          const uint64_t t1 = global_ns();
          while (!mbar_try_wait(&s.st_full[i], (issued[i] / kBwdStages) & 1) && global_ns() - t1 < kWaitBudgetNs) {
          }
        }
    }
  } else if (warp == kKvWarpS || warp == kKvWarpDP) {
    // ------------------------------------------ S^T issuer, dP^T issuer
    // Unit j once the compute warps hold S^T / dP^T of unit j - 1: warp
    // kKvWarpS issues S^T = K Q^T (A = K in TMEM), warp kKvWarpDP issues
    // dP^T = V dO^T (A = V in shared memory).  Each whole warp runs its
    // loop; one elected lane issues.
    if (run) {
      const bool is_s = warp == kKvWarpS;
      const uint32_t idS = idesc_bf16(128, kRowTile, 0, 0);
      const uint64_t dv0 = sdesc_sw128(smem_u32(s.v[0]), 16, 1024);
      bool ok = is_s ? mbar_wait_warp(&s.k_tmem, 0, ab, VS_ERR_TIMEOUT) : mbar_wait_warp(&s.kv_full, 0, ab, VS_ERR_TIMEOUT);
      if (ok && BAR && !is_s) fence_proxy_async_smem();
      for (int j = 0; ok && j < U; ++j) {
        const int st = j % kBwdStages;
        if (!(ok = mbar_wait_warp(&s.st_full[st], (j / kBwdStages) & 1, ab, VS_ERR_TIMEOUT))) break;
        if (j >= 1 && !(ok = mbar_wait_warp(&s.s_free, (j - 1) & 1, ab, VS_ERR_TIMEOUT))) break;
        tc_fence_after();
        // a K-chunk's descriptor is the stage's plus its offset (shared
        // addresses stay below 256 KB: the 14-bit start field never carries)
        if (is_s) {
          const uint64_t dqs = sdesc_sw128(smem_u32(s.q[st][0]), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t dq_ = dqs + (uint32_t((kk / 4) * kRowTile * 128 + (kk % 4) * 32) >> 4);
            mma_ts_warp(tmem + kKvColS, tmem + kKvColK + kk * 8, dq_, idS, kk > 0);
          }
          mma_commit_warp(&s.s_full);
        } else {
          const uint64_t dgs = sdesc_sw128(smem_u32(s.g[st][0]), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t dva = dv0 + (uint32_t((kk / 4) * kBarK * 128 + (kk % 4) * 32) >> 4);
            const uint64_t dg_ = dgs + (uint32_t((kk / 4) * kRowTile * 128 + (kk % 4) * 32) >> 4);
            mma_ss_warp(tmem + kKvColDP, dva, dg_, idS, kk > 0);
          }
          mma_commit_warp(&s.sd_full);
        }
        mma_issued = true;
      }
    }
  } else if (warp == kKvWarpGrad) {
    // ------------------------------------------------------- dV / dK issuer
    // Unit j once its P^T / dS^T are in TMEM; the unit's stage is released
    // after these MMAs (the S^T / dP^T MMAs that read it completed before the
    // compute warps saw the scores).
    if (run) {
      const uint32_t idG = idesc_bf16(128, D, 0, 1);
      bool ok = true;
      for (int j = 0; ok && j < U; ++j) {
        const int st = j % kBwdStages;
        if (!(ok = mbar_wait_warp(&s.p_full, j & 1, ab, VS_ERR_TIMEOUT))) break;
        tc_fence_after();
        const uint64_t dgm = sdesc_sw128(smem_u32(s.g[st][0]), kRowTile * 128, 1024);
        const uint64_t dqm = sdesc_sw128(smem_u32(s.q[st][0]), kRowTile * 128, 1024);
#pragma unroll
        for (int kk = 0; kk < kRowTile / 16; ++kk) {
          const uint64_t dg_ = dgm + uint32_t(kk * 2048 >> 4);
          const uint64_t dq_ = dqm + uint32_t(kk * 2048 >> 4);
          mma_ts_warp(tmem + kKvColDV, tmem + kKvColP + kk * 8, dg_, idG, (j > 0 || kk > 0));
          mma_ts_warp(tmem + kKvColDK, tmem + kKvColDS + kk * 8, dq_, idG, (j > 0 || kk > 0));
        }
        mma_issued = true;
        mma_commit_warp(&s.mm_done);
        mma_commit_warp(&s.st_empty[st]);
      }
      mma_commit_warp(&s.fin);
    }
  } else {
    // ------------------------------------------------------------ compute
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;   // which 32 of the unit's 64 rows
    const int r = quarter * 32 + lane;  // key row of the tile
    const uint32_t tl = tmem + (uint32_t(quarter * 32) << 16);
    int64_t kl;                          // local key index
    if (BAR) kl = __ldg(bar_keys + r);
    else kl = k0 + r;
    const bool key_ok = run && kl >= 0 && kl < p.Nk;
    const int64_t m_g = key_ok ? kpos_g(G, kl) : 0;
    constexpr bool block_cover = BLOCK;
    // slash: bit hh set iff head hk g + hh selected the key as a column (its
    // rows are the bar kernel's); read once, the key is fixed per thread
    uint64_t vsel = 0;
    if (!BAR && key_ok)
      for (int hh = 0; hh < G.g; ++hh) {
        const int64_t bh = int64_t(b) * p.Hq + hk * G.g + hh;
        vsel |= ((__ldg(av.vlocbits + bh * G.WL + (kl >> 6)) >> (kl & 63)) & 1ull) << hh;
      }
    if (run) {
      // K row of key r, d columns [half D/2, (half + 1) D/2), into TMEM
      uint32_t w[D / 4];
      const uint8_t* src = p.k + (int64_t(b) * p.sk[0] + kl * p.sk[1] + int64_t(hk) * p.sk[2]) * 2 + half * D;
#pragma unroll
      for (int c = 0; c < D / 16; ++c) {
        const uint4 x = key_ok ? *reinterpret_cast<const uint4*>(src + 16 * c) : make_uint4(0, 0, 0, 0);
        w[4 * c] = x.x;
        w[4 * c + 1] = x.y;
        w[4 * c + 2] = x.z;
        w[4 * c + 3] = x.w;
      }
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tmem_st16(tl + kKvColK + half * (D / 4) + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&w[16 * c]));
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&s.k_tmem);
    }
    bool ok = true;
    for (int j = 0; run && j < U; ++j) {
      const int st = j % kBwdStages;
      ok = mbar_wait(&s.s_full, j & 1, ab, VS_ERR_TIMEOUT) && mbar_wait(&s.sd_full, j & 1, ab, VS_ERR_TIMEOUT) &&
           mbar_wait(&s.st_full[st], (j / kBwdStages) & 1, ab, VS_ERR_TIMEOUT);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[32], pr[32];
      tmem_ld32(tl + kKvColS + 32 * half, sr);
      tmem_ld32(tl + kKvColDP + 32 * half, pr);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&s.s_free);
      const int h = s.unit_head[st];
      const int64_t r0 = s.unit_row[st];
      const int64_t bh = int64_t(b) * p.Hq + h;
      uint64_t mask = 0;
      if (key_ok) {
        if (BAR) {
          const int64_t n_g0 = qpos_g(G, r0);  // rows of a unit are one aligned block
          const int64_t rows = int64_t(p.Nq) - r0;
          const int64_t lim = m_g - n_g0;    // rows i >= lim are causal
          uint64_t valid = rows >= 64 ? ~0ull : (rows <= 0 ? 0ull : ((1ull << rows) - 1));
          if (lim >= 64) valid = 0;
          else if (lim > 0) valid &= (~0ull) << lim;
          mask = valid;
        } else {
          if (!((vsel >> (h - hk * G.g)) & 1ull))
            mask = block_cover ? block_col_mask(G, av.bdbits + bh * G.WG, kl, r0)
                               : slash_col_mask(G, av.offbits + bh * G.WG, kl, r0);
        }
      }
      const uint32_t hm = uint32_t(mask >> (32 * half));
      // the rows' -LSE log2(e) and D, read pair by pair inside the loop
      // (broadcast shared-memory reads; fewer registers live at once)
      const float2* l2p = reinterpret_cast<const float2*>(&s.l2[st][32 * half]);
      const float2* ddp = reinterpret_cast<const float2*>(&s.dd[st][32 * half]);
      // two rows at a time in paired fp32: t = S^T scale log2(e) - LSE log2(e)
      // (the workspace holds -LSE log2(e)), P = 2^t on the mask, dS = P (dP - D)
      uint32_t pk[16], dk[16];
      const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int c = 2 * i;
        float t0, t1;
        const float2 lv = l2p[i], dv2 = ddp[i];
        f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sc2, f2_pack(lv.x, lv.y)), t0,
                  t1);
        const float x0 = ((hm >> c) & 1u) ? ex2(t0) : 0.f;  // one select: dS inherits the zero
        const float x1 = ((hm >> (c + 1)) & 1u) ? ex2(t1) : 0.f;
        float d0, d1;
        f2_unpack(f2_mul(f2_pack(x0, x1), f2_sub(f2_pack(__uint_as_float(pr[c]), __uint_as_float(pr[c + 1])),
                                                  f2_pack(dv2.x, dv2.y))),
                  d0, d1);
        pk[i] = pack_bf16x2(x0, x1);
        dk[i] = pack_bf16x2(d0, d1);
      }
      if (j >= 1) ok = mbar_wait(&s.mm_done, (j - 1) & 1, ab, VS_ERR_TIMEOUT);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_st16(tl + kKvColP + 16 * half, pk);
      tmem_st16(tl + kKvColDS + 16 * half, dk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&s.p_full);
    }
    if (ok && run) ok = mbar_wait(&s.fin, 0, ab, VS_ERR_TIMEOUT);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    // ------------------------------------------------------------ epilogue
    if (ok && cta_ok) {
      if (BAR) {
        {
          // TMEM reads are warp-collective: every lane loads, valid keys store
          const int64_t bh = int64_t(b) * p.Hq + h_bar;
          const int64_t rank = k0 + r;  // position in the vertical list
          float* pdk = reinterpret_cast<float*>(p.ws + L.off_bar_dk) + ((int64_t(split) * p.B * p.Hq + bh) * G.KVP + rank) * D;
          float* pdv = reinterpret_cast<float*>(p.ws + L.off_bar_dv) + ((int64_t(split) * p.B * p.Hq + bh) * G.KVP + rank) * D;
#pragma unroll 1
          for (int cc = (D / 2) * half; cc < (D / 2) * (half + 1); cc += 16) {
            uint32_t a[16], c2[16];
            tmem_ld16(tl + kKvColDK + cc, a);
            tmem_ld16(tl + kKvColDV + cc, c2);
            tmem_ld_wait();
            if (!key_ok) continue;
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
              *reinterpret_cast<float4*>(pdk + cc + i) =
                  make_float4(__uint_as_float(a[i]) * p.scale, __uint_as_float(a[i + 1]) * p.scale,
                              __uint_as_float(a[i + 2]) * p.scale, __uint_as_float(a[i + 3]) * p.scale);
              *reinterpret_cast<float4*>(pdv + cc + i) = make_float4(
                  __uint_as_float(c2[i]), __uint_as_float(c2[i + 1]), __uint_as_float(c2[i + 2]), __uint_as_float(c2[i + 3]));
            }
          }
        }
      } else {
        // slash part (TMEM) + the bar partials of every head that selected this key
        uint8_t* okr = p.dk + (int64_t(b) * p.sk[0] + kl * p.sk[1] + int64_t(hk) * p.sk[2]) * 2;
        uint8_t* ovr = p.dv + (int64_t(b) * p.sv[0] + kl * p.sv[1] + int64_t(hk) * p.sv[2]) * 2;
        const float* bdk = reinterpret_cast<const float*>(p.ws + L.off_bar_dk);
        const float* bdv = reinterpret_cast<const float*>(p.ws + L.off_bar_dv);
#pragma unroll 1
        for (int cc = (D / 2) * half; cc < (D / 2) * (half + 1); cc += 16) {
          float yk[16], yv[16];
          if (U > 0) {
            uint32_t a[16], c2[16];
            tmem_ld16(tl + kKvColDK + cc, a);
            tmem_ld16(tl + kKvColDV + cc, c2);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              yk[i] = __uint_as_float(a[i]) * p.scale;
              yv[i] = __uint_as_float(c2[i]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) yk[i] = yv[i] = 0.f;
          }
          if (kl >= p.Nk) continue;  // past the end of the keys: load only
          for (int hh = 0; hh < G.g; ++hh) {
            const int64_t bh = int64_t(b) * p.Hq + hk * G.g + hh;
            const uint64_t vw = __ldg(av.vlocbits + bh * G.WL + (kl >> 6));
            if (!((vw >> (kl & 63)) & 1ull)) continue;
            // this head selected the key as a column: add its bar partials
            const int64_t rank =
                __ldg(av.vlocpre + bh * G.WL + (kl >> 6)) + __popcll(vw & ((1ull << (kl & 63)) - 1));
            const int64_t first = __ldg(av.vlist + bh * G.KVP + (rank / kBarK) * kBarK);
            const int64_t rs = first_causal_row_block(G.world, G.q_rank, kpos_g(G, first)) * kBlk;
            const int64_t tiles = (p.Nq - rs + kRowTile - 1) / kRowTile;
            const int nsplit = int((tiles + kBarSplitTiles - 1) / kBarSplitTiles);
            for (int sp = 0; sp < nsplit; ++sp) {
              const int64_t base = ((int64_t(sp) * p.B * p.Hq + bh) * G.KVP + rank) * D + cc;
#pragma unroll
              for (int i = 0; i < 16; i += 4) {
                const float4 a4 = *reinterpret_cast<const float4*>(bdk + base + i);
                const float4 c4 = *reinterpret_cast<const float4*>(bdv + base + i);
                yk[i] += a4.x;
                yk[i + 1] += a4.y;
                yk[i + 2] += a4.z;
                yk[i + 3] += a4.w;
                yv[i] += c4.x;
                yv[i + 1] += c4.y;
                yv[i + 2] += c4.z;
                yv[i + 3] += c4.w;
              }
            }
          }
          if (p.dkv_acc) {
            // accumulate mode: acc += this call's dK / dV; the outputs are the sums
            float* ak = p.dkv_acc + ((int64_t(b) * p.Nk + kl) * p.Hkv + hk) * D + cc;
            float* avv = ak + int64_t(p.B) * p.Nk * p.Hkv * D;
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
              float4 a4 = *reinterpret_cast<float4*>(ak + i);
              float4 c4 = *reinterpret_cast<float4*>(avv + i);
              a4.x += yk[i];
              a4.y += yk[i + 1];
              a4.z += yk[i + 2];
              a4.w += yk[i + 3];
              c4.x += yv[i];
              c4.y += yv[i + 1];
              c4.z += yv[i + 2];
              c4.w += yv[i + 3];
              *reinterpret_cast<float4*>(ak + i) = a4;
              *reinterpret_cast<float4*>(avv + i) = c4;
              yk[i] = a4.x;
              yk[i + 1] = a4.y;
              yk[i + 2] = a4.z;
              yk[i + 3] = a4.w;
              yv[i] = c4.x;
              yv[i + 1] = c4.y;
              yv[i + 2] = c4.z;
              yv[i + 3] = c4.w;
            }
          }
          uint4 k0w, k1w, v0w, v1w;
          k0w.x = pack_bf16x2(yk[0], yk[1]);
          k0w.y = pack_bf16x2(yk[2], yk[3]);
          k0w.z = pack_bf16x2(yk[4], yk[5]);
          k0w.w = pack_bf16x2(yk[6], yk[7]);
          k1w.x = pack_bf16x2(yk[8], yk[9]);
          k1w.y = pack_bf16x2(yk[10], yk[11]);
          k1w.z = pack_bf16x2(yk[12], yk[13]);
          k1w.w = pack_bf16x2(yk[14], yk[15]);
          v0w.x = pack_bf16x2(yv[0], yv[1]);
          v0w.y = pack_bf16x2(yv[2], yv[3]);
          v0w.z = pack_bf16x2(yv[4], yv[5]);
          v0w.w = pack_bf16x2(yv[6], yv[7]);
          v1w.x = pack_bf16x2(yv[8], yv[9]);
          v1w.y = pack_bf16x2(yv[10], yv[11]);
          v1w.z = pack_bf16x2(yv[12], yv[13]);
          v1w.w = pack_bf16x2(yv[14], yv[15]);
          *reinterpret_cast<uint4*>(okr + cc * 2) = k0w;
          *reinterpret_cast<uint4*>(okr + cc * 2 + 16) = k1w;
          *reinterpret_cast<uint4*>(ovr + cc * 2) = v0w;
          *reinterpret_cast<uint4*>(ovr + cc * 2 + 16) = v1w;
        }
      }
    }
  }
  // an issuer that gave up waits (bounded) for its own MMAs in flight
  if ((warp == kKvWarpS || warp == kKvWarpGrad || warp == kKvWarpDP) && lane == 0 && mma_issued && s.abort_flag) {
    uint64_t* tb = warp == kKvWarpS ? &s.teardown : (warp == kKvWarpGrad ? &s.teardown_g : &s.teardown_d);
    mma_commit(tb);
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(tb, 0) && global_ns() - t0 < kWaitBudgetNs) {
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Bars hold whole columns: only the slash kernel depends on the reading.
template <int D, bool BAR>
__global__ void __launch_bounds__(kKvThreads, 1)
    vs_bwd_kv_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmG,
                     const BwdParams p) {
  if (!BAR && arena_view(p.arena).hdr->block_cover) kv_body<D, BAR, true>(tmK, tmV, tmQ, tmG, p);
  else kv_body<D, BAR, false>(tmK, tmV, tmQ, tmG, p);
}

BwdParams make_params(const vs_shape* sh, const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dO, const void* arena, float scale, void* dq, void* dk, void* dv,
                      float* dq_acc, float* dkv_acc, void* ws, size_t ws_bytes) {
  BwdParams p;
  p.arena = arena;
  p.q = static_cast<const uint8_t*>(q);
  p.k = static_cast<const uint8_t*>(k);
  p.v = static_cast<const uint8_t*>(v);
  p.o = static_cast<const uint8_t*>(o);
  p.dO = static_cast<const uint8_t*>(dO);
  p.lse = lse;
  for (int i = 0; i < 3; ++i) {
    p.sq[i] = sh->sq[i];
    p.sk[i] = sh->sk[i];
    p.sv[i] = sh->sv[i];
    p.so[i] = sh->so[i];
  }
  p.B = sh->B;
  p.Nq = sh->Nq;
  p.Nk = sh->Nk;
  p.Hq = sh->Hq;
  p.Hkv = sh->Hkv;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  p.dq = static_cast<uint8_t*>(dq);
  p.dk = static_cast<uint8_t*>(dk);
  p.dv = static_cast<uint8_t*>(dv);
  p.dq_acc = dq_acc;
  p.dkv_acc = dkv_acc;
  p.ws = static_cast<uint8_t*>(ws);
  p.ws_bytes = ws_bytes;
  p.err = static_cast<int*>(ws);
  return p;
}

template <int D>
vs_status launch_bwd_d(const vs_shape* sh, const BwdParams& p, int grid_per_bh, cudaStream_t st) {
  CUtensorMap tk64, tv64, tk128, tv128, tq64, tg64;
  vs_status rc;
  if ((rc = make_tmap_bshd(&tk64, p.k, sh->B, sh->Nk, sh->Hkv, D, sh->sk, kKTile)) != VS_OK) return rc;
  if ((rc = make_tmap_bshd(&tv64, p.v, sh->B, sh->Nk, sh->Hkv, D, sh->sv, kKTile)) != VS_OK) return rc;
  if ((rc = make_tmap_bshd(&tk128, p.k, sh->B, sh->Nk, sh->Hkv, D, sh->sk, kBarK)) != VS_OK) return rc;
  if ((rc = make_tmap_bshd(&tv128, p.v, sh->B, sh->Nk, sh->Hkv, D, sh->sv, kBarK)) != VS_OK) return rc;
  if ((rc = make_tmap_bshd(&tq64, p.q, sh->B, sh->Nq, sh->Hq, D, sh->sq, kRowTile)) != VS_OK) return rc;
  if ((rc = make_tmap_bshd(&tg64, p.dO, sh->B, sh->Nq, sh->Hq, D, sh->so, kRowTile)) != VS_OK) return rc;
  const size_t sm_dq = sizeof(DqSmem<D>) + 1024;
  const size_t sm_kv = sizeof(KvSmem<D>) + 1024;
  if (cudaFuncSetAttribute(vs_bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm_dq)) !=
          cudaSuccess ||
      cudaFuncSetAttribute(vs_bwd_kv_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm_kv)) !=
          cudaSuccess ||
      cudaFuncSetAttribute(vs_bwd_kv_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm_kv)) !=
          cudaSuccess)
    return VS_ERR_CUDA;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t rows = int64_t(sh->B) * sh->Hq * sh->Nq;
  const int prep_grid = int(std::min<int64_t>((rows + 255) / 256, int64_t(sms) * 8));
  trace_begin("bwd_prep", st);
  bwd_prep<<<prep_grid, 256, 0, st>>>(p, D);
  trace_end(st);
  // bar partials first: the slash kernel's epilogue reads them
  trace_begin("bwd_dkv_bar", st);
  vs_bwd_kv_kernel<D, true><<<unsigned(int64_t(sh->B) * sh->Hq * grid_per_bh), kKvThreads, sm_kv, st>>>(
      tk128, tv128, tq64, tg64, p);
  trace_end(st);
  const int TK = (sh->Nk + kBarK - 1) / kBarK;
  trace_begin("bwd_dkv_slash", st);
  vs_bwd_kv_kernel<D, false><<<unsigned(int64_t(sh->B) * sh->Hkv * TK), kKvThreads, sm_kv, st>>>(
      tk128, tv128, tq64, tg64, p);
  trace_end(st);
  const int T = (sh->Nq + kQTile - 1) / kQTile;
  trace_begin("bwd_dq", st);
  vs_bwd_dq_kernel<D><<<unsigned(int64_t(T) * sh->B * sh->Hq), kDqThreads, sm_dq, st>>>(tk64, tv64, p);
  trace_end(st);
  note_launch(4);
  return cudaGetLastError() == cudaSuccess ? VS_OK : VS_ERR_CUDA;
}

}  // namespace

size_t bwd_workspace_bytes(const vs_shape* s, int kv) {
  return size_t(bwd_layout(s->B, s->Hq, s->Nq, s->d, kv).total);
}

vs_status launch_bwd(const vs_shape* s, const Geo&, const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const void* dO, const void* arena, float scale, void* dq, void* dk, void* dv,
                     float* dq_acc, float* dkv_acc, void* ws, size_t ws_bytes, cudaStream_t st) {
  BwdParams p = make_params(s, q, k, v, o, lse, dO, arena, scale, dq, dk, dv, dq_acc, dkv_acc, ws, ws_bytes);
  // Grid of the bar kernel: (KVP / 128) chunks x splits per (b, h).  KVP
  // lives in the arena header on the device; the largest value the
  // workspace can hold bounds it, and CTAs beyond the real count exit.
  const BwdLayout L1 = bwd_layout(s->B, s->Hq, s->Nq, s->d, kBarK);
  const int64_t per_chunk = int64_t(L1.smax) * s->B * s->Hq * kBarK * s->d * 4 * 2;
  const int64_t room = int64_t(ws_bytes) - L1.off_bar_dk;
  int64_t nchunk = room > 0 ? room / per_chunk : 1;
  const int64_t cap = (int64_t(s->Nk) + kBarK - 1) / kBarK;
  if (nchunk > cap) nchunk = cap;
  if (nchunk < 1) nchunk = 1;
  p.bar_nchunk = int(nchunk);
  const int grid_per_bh = int(nchunk * L1.smax);
  if (s->d == 128) return launch_bwd_d<128>(s, p, grid_per_bh, st);
  if (s->d == 64) return launch_bwd_d<64>(s, p, grid_per_bh, st);
  return VS_ERR_SHAPE;
}

}  // namespace vs
