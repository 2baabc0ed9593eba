// Online Vertical-Slash estimation (Algorithm 1, first four lines), with the
// last-64-row logits on the tensor cores.
//
// The g query heads of a KV head share its keys, so their last-64 query rows
// are stacked two heads per 128-row tile (M = 128) and multiplied by
// 128-key tiles of K (N = 128, K = d) with tcgen05.mma into TMEM:
//   pass 1  est_rowstats : per (b, KV head, row tile, key split) partial
//                          (max, sum exp) of every row's causal logits
//   est_lse              : LSE of every row from its key-split partials
//   pass 2  est_scores   : per (b, KV head, 128-key tile) A_hat = exp(S - LSE)
//                          staged in shared memory: column sums -> v[m]
//                          (complete per tile), diagonal sums -> 191 partial
//                          slash sums per head and tile
//   pass 3  est_scombine : s[o] = the (at most two) tile partials of o, added
//                          in a fixed order (deterministic, no float atomics)
//   pass 4  est_topk     : radix select of the k-th largest score, then an
//                          index-ordered compaction; ties go to the lower index
//                          (one thread-block cluster of 8 CTAs per list)
// Warp roles in passes 1 and 2: warp 0 issues TMA loads, warp 1 the MMAs
// (the whole warp runs the loop, an elected lane issues), warps 2-9 read the scores (one thread per TMEM lane, two warps
// per lane quarter, each on half the columns).  Waits are bounded.
#include <cooperative_groups.h>

#include "vs_internal.h"
#include "vs_kernel_common.cuh"

namespace cg = cooperative_groups;

namespace vs {
namespace {

constexpr int kLastQ = 64;
constexpr int kSplits = 64;        // key splits per row tile in pass 1
constexpr int kEstKeys = 128;      // keys per tile (MMA N)
constexpr int kEstThreads = 320;   // warp 0 TMA, warp 1 MMA, warps 2-9 compute
constexpr int kEstCompute = 256;
constexpr int kEstDiag = 192;      // 191 diagonals (row - key in [-127, 63]) per head and key tile, padded
constexpr int kTopkThreads = 1024;
constexpr size_t kToppMaxSmem = size_t(192) << 10;  // pooled slash units: N <= 1,572,864

struct EstLayout {
  int64_t off_part, off_lse, off_vbuf, off_spart, off_sbuf, off_gv, off_gs, total;
};

EstLayout est_layout(const vs_shape* s) {
  EstLayout L;
  const int64_t BH = int64_t(s->B) * s->Hq, N = s->Nk, NT = (N + kEstKeys - 1) / kEstKeys;
  int64_t off = 256;
  auto take = [&](int64_t bytes) {
    const int64_t at = off;
    off += (bytes + 255) / 256 * 256;
    return at;
  };
  L.off_part = take(BH * kSplits * kLastQ * 8);
  L.off_lse = take(BH * kLastQ * 4);
  L.off_vbuf = take(BH * N * 4);
  L.off_spart = take(BH * NT * kEstDiag * 4);
  L.off_sbuf = take(BH * N * 4);
  const int64_t BHK = int64_t(s->B) * s->Hkv;
  L.off_gv = take(BHK * N * 4);  // per-KV-group score sums (shared selection)
  L.off_gs = take(BHK * N * 4);
  L.total = off;
  return L;
}

struct EstParams {
  int B, N, Hq, Hkv, d, g, MT;  // MT: 128-row tiles per KV head = ceil(g / 2)
  float scale_log2;
  float2* part;   // [BH][kSplits][64] (max, sum) in log2 units
  float* lse;     // [BH][64] log2 units
  float* v;       // [BH][N]
  float* spart;   // [BH][NT][kEstDiag]
  float* s;       // [BH][N]
  float* gv;      // shared selection: [BHK][N] group sums (null: per-head selection)
  float* gs;
  int* err;
};

// Shared memory of both tensor-core passes: one 128-row Q tile (two heads'
// last 64 rows) per buffer, 128-key K tiles, the staged A_hat tile.
template <int D>
struct EstSmem {
  static constexpr int NH = D / 64;
  uint8_t q[2][NH][128 * 128];
  uint8_t k[2][NH][kEstKeys * 128];
  float stage[128][kEstKeys + 1];  // pass 2: A_hat of the row tile (pitch 129: conflict-free rows and columns)
  float lse[128];
  float red_m[128], red_l[128];    // pass 1: the second column half's (max, sum)
  uint64_t q_full[2], q_empty[2], k_full[2], k_empty[2], s_full[2], s_free[2], teardown;
  uint32_t tmem_base;
  int abort_flag;
  int skip;  // the status word already held a failure when the CTA started
};

// A failure recorded earlier in this call (or left in the status word by an
// earlier call) makes the estimator's later kernels skip their work, so that
// no kernel reads scratch a failed kernel left unwritten.  VS_ERR_SCORE is a
// per-list outcome of the top-p step, not a failure of the scores.
__device__ __forceinline__ bool est_failed(const int* err) {
  const int w = *reinterpret_cast<const volatile int*>(err);
  return w != 0 && w != VS_ERR_SCORE;
}

// First query head (within the group) of row tile mt's two heads; a tile's
// second head may not exist (odd g): its rows load the first head again and
// are ignored.
__device__ __forceinline__ int est_tile_head(int hk, int g, int mt, int hh) {
  return hk * g + min(2 * mt + hh, g - 1);
}

template <int D>
__device__ __forceinline__ void est_load_q(EstSmem<D>& s, int buf, const CUtensorMap* tmQ, int hk, int g, int mt,
                                           int N, int b) {
  constexpr int NH = D / 64;
  mbar_arrive_expect_tx(&s.q_full[buf], 2 * NH * 64 * 128);
  for (int hh = 0; hh < 2; ++hh)
    for (int hf = 0; hf < NH; ++hf)
      tma_load_4d(s.q[buf][hf] + hh * 64 * 128, tmQ, &s.q_full[buf], 64 * hf, est_tile_head(hk, g, mt, hh),
                  N - kLastQ, b);
}

// S = Q K^T of one row tile and one key tile into TMEM columns [col, col + 128).
// Warp-collective: an elected lane issues.
template <int D>
__device__ __forceinline__ void est_mma(EstSmem<D>& s, int qb, int kb, uint32_t dst) {
  const uint32_t idS = idesc_bf16(128, kEstKeys, 0, 0);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t da = sdesc_sw128(smem_u32(s.q[qb][kk / 4]) + (kk % 4) * 32, 16, 1024);
    const uint64_t db = sdesc_sw128(smem_u32(s.k[kb][kk / 4]) + (kk % 4) * 32, 16, 1024);
    mma_ss_warp(dst, da, db, idS, kk > 0);
  }
}

template <int D>
__device__ __forceinline__ void est_init(EstSmem<D>& s, int ncols, const int* err) {
  const int warp = threadIdx.x / 32;
  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    s.skip = est_failed(err) ? 1 : 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.q_full[i], 1);
      mbar_init(&s.q_empty[i], 1);
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.k_empty[i], 1);
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.s_free[i], kEstCompute);
    }
    mbar_init(&s.teardown, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

template <int D>
__device__ __forceinline__ void est_teardown(EstSmem<D>& s, bool mma_issued, int ncols) {
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x / 32 == 1) {
    if (threadIdx.x % 32 == 0 && mma_issued && s.abort_flag) {
      // make sure no MMA still writes TMEM before it is released
      mma_commit(&s.teardown);
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(&s.teardown, 0) && global_ns() - t0 < kWaitBudgetNs) {
      }
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(s.tmem_base, ncols);
  }
}

// Pass 1: grid (B * Hkv * MT, kSplits).  Keys of split sp: 128-key chunks
// [c * 128, c * 128 + 128) with c = sp, sp + kSplits, ... (interleaved so that
// every split sees the same share of the causal edge).
template <int D>
__global__ void __launch_bounds__(kEstThreads, 1)
    est_rowstats(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const EstParams p) {
  constexpr int NH = D / 64;
  extern __shared__ uint8_t smem_raw[];
  EstSmem<D>& s = *reinterpret_cast<EstSmem<D>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int mt = int(blockIdx.x) % p.MT, bhk = int(blockIdx.x) / p.MT;
  const int b = bhk / p.Hkv, hk = bhk % p.Hkv, sp = blockIdx.y;
  const int N = p.N, NT = (N + kEstKeys - 1) / kEstKeys;
  est_init<D>(s, 256, p.err);
  const int nchunk = (NT > sp && !s.skip) ? (NT - sp + kSplits - 1) / kSplits : 0;
  const uint32_t tmem = s.tmem_base;
  const Abort ab{&s.abort_flag, p.err};
  bool mma_issued = false;
  if (warp == 0) {
    if (lane == 0 && nchunk > 0) {
      est_load_q<D>(s, 0, &tmQ, hk, p.g, mt, N, b);
      for (int c = 0; c < nchunk; ++c) {
        const int kb = c & 1;
        if (c >= 2 && !mbar_wait(&s.k_empty[kb], ((c >> 1) - 1) & 1, ab, VS_ERR_TIMEOUT)) break;
        mbar_arrive_expect_tx(&s.k_full[kb], NH * kEstKeys * 128);
        for (int hf = 0; hf < NH; ++hf)
          tma_load_4d(s.k[kb][hf], &tmK, &s.k_full[kb], 64 * hf, hk, (sp + c * kSplits) * kEstKeys, b);
      }
    }
  } else if (warp == 1) {
    if (nchunk > 0) {
      bool ok = mbar_wait_warp(&s.q_full[0], 0, ab, VS_ERR_TIMEOUT);
      for (int c = 0; ok && c < nchunk; ++c) {
        const int kb = c & 1;
        if (!(ok = mbar_wait_warp(&s.k_full[kb], (c >> 1) & 1, ab, VS_ERR_TIMEOUT))) break;
        if (c >= 2 && !(ok = mbar_wait_warp(&s.s_free[kb], ((c >> 1) - 1) & 1, ab, VS_ERR_TIMEOUT))) break;
        tc_fence_after();
        est_mma<D>(s, 0, kb, tmem + 128 * kb);
        mma_commit_warp(&s.s_full[kb]);
        mma_commit_warp(&s.k_empty[kb]);
        mma_issued = true;
      }
    }
  } else {
    const int quarter = warp & 3, half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane, i = r & 63;
    const int64_t n_i = int64_t(N) - kLastQ + i;
    const uint32_t tl = tmem + (uint32_t(quarter * 32) << 16);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int c = 0; c < nchunk; ++c) {
      const int kb = c & 1;
      ok = mbar_wait(&s.s_full[kb], (c >> 1) & 1, ab, VS_ERR_TIMEOUT);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      uint32_t x[64];
      tmem_ld32(tl + 128 * kb + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
      tmem_ld32(tl + 128 * kb + 64 * half + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&s.s_free[kb]);
      const int64_t key0 = int64_t(sp + c * kSplits) * kEstKeys + 64 * half;
      const int nvalid = int(max(int64_t(0), min(int64_t(64), n_i - key0 + 1)));  // keys <= n_i (N - 1 at most)
      float mx = -INFINITY;
#pragma unroll
      for (int k = 0; k < 64; ++k)
        if (k < nvalid) mx = fmaxf(mx, __uint_as_float(x[k]) * p.scale_log2);
      if (mx == -INFINITY) continue;
      if (mx > m) {
        l = (m == -INFINITY) ? 0.f : l * ex2(m - mx);
        m = mx;
      }
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < 64; ++k)
        if (k < nvalid) acc[k & 3] += ex2(fmaf(__uint_as_float(x[k]), p.scale_log2, -m));
      l += (acc[0] + acc[1]) + (acc[2] + acc[3]);
    }
    // merge the two column halves of each row
    if (half == 1) {
      s.red_m[r] = m;
      s.red_l[r] = l;
    }
    bar_sync_and(1, kEstCompute, true);
    if (half == 0 && ok && !s.skip) {
      const float mo = s.red_m[r], lo = s.red_l[r];
      const float mn = fmaxf(m, mo);
      const float ln = (mn == -INFINITY) ? 0.f
                                         : ((m == -INFINITY ? 0.f : l * ex2(m - mn)) +
                                            (mo == -INFINITY ? 0.f : lo * ex2(mo - mn)));
      const int hh = r >> 6;
      if (2 * mt + hh < p.g) {
        const int64_t bh = int64_t(b) * p.Hq + hk * p.g + 2 * mt + hh;
        p.part[(bh * kSplits + sp) * kLastQ + i] = make_float2(mn, ln);
      }
    }
  }
  est_teardown<D>(s, mma_issued, 256);
}

// LSE (log2 units) of every (b, h, last-64 row) from its key-split partials.
__global__ void est_lse(const EstParams p) {
  if (est_failed(p.err)) return;
  const int bh = blockIdx.x, i = threadIdx.x;
  const float2* pp = p.part + int64_t(bh) * kSplits * kLastQ + i;
  float m = -INFINITY, l = 0.f;
  for (int sp = 0; sp < kSplits; ++sp) {  // fixed order
    const float2 x = pp[sp * kLastQ];
    if (x.x == -INFINITY) continue;
    const float mn = fmaxf(m, x.x);
    l = (m == -INFINITY ? 0.f : l * exp2f(m - mn)) + x.y * exp2f(x.x - mn);
    m = mn;
  }
  p.lse[int64_t(bh) * kLastQ + i] = m + log2f(l);
}

// Pass 2: grid (B * Hkv, NT).  One key tile; its row tiles one after another.
template <int D>
__global__ void __launch_bounds__(kEstThreads, 1)
    est_scores(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const EstParams p) {
  constexpr int NH = D / 64;
  extern __shared__ uint8_t smem_raw[];
  EstSmem<D>& s = *reinterpret_cast<EstSmem<D>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int bhk = blockIdx.x, tile = blockIdx.y;
  const int b = bhk / p.Hkv, hk = bhk % p.Hkv;
  const int N = p.N, NT = (N + kEstKeys - 1) / kEstKeys;
  const int64_t m0 = int64_t(tile) * kEstKeys;
  est_init<D>(s, 256, p.err);
  const int MT = s.skip ? 0 : p.MT;
  const uint32_t tmem = s.tmem_base;
  const Abort ab{&s.abort_flag, p.err};
  bool mma_issued = false;
  if (warp == 0) {
    if (lane == 0 && MT > 0) {
      mbar_arrive_expect_tx(&s.k_full[0], NH * kEstKeys * 128);
      for (int hf = 0; hf < NH; ++hf) tma_load_4d(s.k[0][hf], &tmK, &s.k_full[0], 64 * hf, hk, int(m0), b);
      for (int mt = 0; mt < MT; ++mt) {
        const int qb = mt & 1;
        if (mt >= 2 && !mbar_wait(&s.q_empty[qb], ((mt >> 1) - 1) & 1, ab, VS_ERR_TIMEOUT)) break;
        est_load_q<D>(s, qb, &tmQ, hk, p.g, mt, N, b);
      }
    }
  } else if (warp == 1) {
    if (MT > 0) {
      bool ok = mbar_wait_warp(&s.k_full[0], 0, ab, VS_ERR_TIMEOUT);
      for (int mt = 0; ok && mt < MT; ++mt) {
        const int qb = mt & 1;
        if (!(ok = mbar_wait_warp(&s.q_full[qb], (mt >> 1) & 1, ab, VS_ERR_TIMEOUT))) break;
        if (mt >= 2 && !(ok = mbar_wait_warp(&s.s_free[qb], ((mt >> 1) - 1) & 1, ab, VS_ERR_TIMEOUT))) break;
        tc_fence_after();
        est_mma<D>(s, qb, 0, tmem + 128 * qb);
        mma_commit_warp(&s.s_full[qb]);
        mma_commit_warp(&s.q_empty[qb]);
        mma_issued = true;
      }
    }
  } else {
    const int t = threadIdx.x - 64;  // 0..255
    const int quarter = warp & 3, half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane, i = r & 63;
    const int64_t n_i = int64_t(N) - kLastQ + i;
    const uint32_t tl = tmem + (uint32_t(quarter * 32) << 16);
    bool ok = true;
    for (int mt = 0; mt < MT; ++mt) {
      const int qb = mt & 1;
      if (half == 0) {
        const int hh = r >> 6;
        const int64_t bh = int64_t(b) * p.Hq + est_tile_head(hk, p.g, mt, hh);
        s.lse[r] = p.lse[bh * kLastQ + i];
      }
      ok = mbar_wait(&s.s_full[qb], (mt >> 1) & 1, ab, VS_ERR_TIMEOUT);
      // every compute warp takes the same decision (and the tile's lse is visible)
      ok = bar_sync_and(1, kEstCompute, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t x[64];
      tmem_ld32(tl + 128 * qb + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
      tmem_ld32(tl + 128 * qb + 64 * half + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&s.s_free[qb]);
      const float L = s.lse[r];
      const int64_t key0 = m0 + 64 * half;
      const int nvalid = int(max(int64_t(0), min(int64_t(64), n_i - key0 + 1)));
      float* row = &s.stage[r][64 * half];
#pragma unroll
      for (int k = 0; k < 64; ++k)
        row[k] = (k < nvalid) ? ex2(fmaf(__uint_as_float(x[k]), p.scale_log2, -L)) : 0.f;
      bar_sync_and(1, kEstCompute, true);  // tile staged
      // vertical: column sums of each head's 64 rows
      {
        const int j = t & 127, hh = t >> 7;
        if (2 * mt + hh < p.g && m0 + j < N) {
          float a0 = 0.f, a1 = 0.f;
#pragma unroll 8
          for (int ii = 0; ii < 64; ii += 2) {
            a0 += s.stage[64 * hh + ii][j];
            a1 += s.stage[64 * hh + ii + 1][j];
          }
          const int64_t bh = int64_t(b) * p.Hq + hk * p.g + 2 * mt + hh;
          p.v[bh * N + m0 + j] = a0 + a1;
        }
      }
      // slash: diagonal delta = row - key in [-127, 63] of each head
      for (int w = t; w < 2 * kEstDiag; w += kEstCompute) {
        const int hh = w / kEstDiag, dgi = w % kEstDiag;
        if (2 * mt + hh >= p.g) continue;
        float sum = 0.f;
        if (dgi < 191) {
          const int delta = dgi - 127;
          const int lo = max(0, delta), hi = min(63, 127 + delta);
          for (int ii = lo; ii <= hi; ++ii) sum += s.stage[64 * hh + ii][ii - delta];
        }
        const int64_t bh = int64_t(b) * p.Hq + hk * p.g + 2 * mt + hh;
        p.spart[(bh * NT + tile) * kEstDiag + dgi] = sum;
      }
      bar_sync_and(1, kEstCompute, true);  // stage and lse free for the next row tile
    }
  }
  est_teardown<D>(s, mma_issued, 256);
}

__global__ void est_scombine(const EstParams p) {
  if (est_failed(p.err)) return;
  const int bh = blockIdx.y;
  const int N = p.N, NT = (N + kEstKeys - 1) / kEstKeys;
  const int o = blockIdx.x * blockDim.x + threadIdx.x;
  if (o >= N) return;
  const float* sp = p.spart + int64_t(bh) * NT * kEstDiag;
  const int x = N - kLastQ - o;  // tile T holds o at delta = 128 T - x in [-127, 63]
  const int Thi = (x + 63 >= 0) ? (x + 63) / kEstKeys : -1;
  float sum = 0.f;
  for (int T = Thi - 1; T <= Thi; ++T) {  // fixed order
    if (T < 0 || T >= NT) continue;
    const int delta = kEstKeys * T - x;
    if (delta >= -127 && delta <= 63) sum += sp[int64_t(T) * kEstDiag + delta + 127];
  }
  p.s[int64_t(bh) * N + o] = sum;
}

// Inclusive block scan of one int per thread (1024 threads); returns the
// inclusive prefix and writes the block total to *total.
__device__ __forceinline__ int block_scan(int x, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int v = x;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += y;
  }
  if (lane == 31) wsum[w] = v;
  __syncthreads();
  if (w == 0) {
    int s = wsum[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += y;
    }
    wsum[lane] = s;
  }
  __syncthreads();
  const int res = v + (w > 0 ? wsum[w - 1] : 0);
  *total = wsum[31];
  __syncthreads();
  return res;
}

// Selection on a thread-block cluster: the kSelCluster CTAs of a cluster
// share one list, each holding a contiguous chunk of it (whole 64-token
// blocks).  Per radix digit every CTA histograms its chunk; after a cluster
// barrier each CTA adds the kSelCluster histograms in rank order from the
// peers' shared memory (integer counts: the same in every CTA) and takes the
// same decision, so no CTA waits for another's broadcast.  Histograms are
// double-buffered across digits: the buffer of digit p is zeroed again at
// digit p + 2, after every peer has passed the barrier of digit p + 1 and
// hence finished reading it.  The compaction places each CTA's chunk after
// the counts of the lower ranks.  Every CTA of a cluster takes the same
// branches and passes the same barriers; the last one keeps a CTA's shared
// memory alive until its peers have read it.
constexpr int kSelCluster = 8;

struct SelShared {
  int cnt[2][256];                // digit counts of this CTA's chunk, per digit parity
  unsigned long long sum[2][256]; // top-p: digit mass of this CTA's chunk
  int mcnt[256];                  // the cluster's counts of the current digit
  unsigned long long msum[256];
  int wsum[32];
  uint64_t red[32];
  uint64_t part;                  // published: this chunk's saturated mass
  int bad, skip, n_gt, n_eq;      // published: validation, skip flag, compaction counts
  uint64_t prefix, want;
  int above;
};

// The chunk [lo, hi) of an N-token list that cluster rank `rank` holds.
__device__ __forceinline__ void sel_chunk(int N, int rank, int& lo, int& hi) {
  const int nb = (N + 63) / 64, per = (nb + kSelCluster - 1) / kSelCluster;
  lo = min(N, 64 * per * rank);
  hi = min(N, 64 * per * (rank + 1));
}

// True in every CTA of the cluster if the status word holds a failure when
// any of them looked (read before any CTA of this launch may raise one).
__device__ bool sel_skip(const int* err, SelShared& S) {
  cg::cluster_group cl = cg::this_cluster();
  if (threadIdx.x == 0) S.skip = est_failed(err);
  cl.sync();
  int any = 0;
  for (int r = 0; r < kSelCluster; ++r) any |= *cl.map_shared_rank(&S.skip, r);
  cl.sync();
  return any != 0;
}

// The k-th largest key (k >= 1) of the cluster's list and how many of its
// copies belong to the k largest (ties to the lower index).
__device__ void sel_kth(const uint32_t* x, int lo, int hi, int k, SelShared& S, uint32_t& kth, int& take) {
  cg::cluster_group cl = cg::this_cluster();
  uint32_t prefix = 0;
  int want = k;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass, b = pass & 1;
    for (int i = threadIdx.x; i < 256; i += blockDim.x) S.cnt[b][i] = 0;
    __syncthreads();
    const uint32_t hi_mask = pass == 0 ? 0u : (0xFFFFFFFFu << (shift + 8));
    for (int i = lo + threadIdx.x; i < hi; i += blockDim.x) {
      const uint32_t v = x[i];
      if ((v & hi_mask) == prefix) atomicAdd(&S.cnt[b][(v >> shift) & 255], 1);
    }
    cl.sync();
    if (threadIdx.x < 256) {
      int m = 0;
      for (int r = 0; r < kSelCluster; ++r) m += cl.map_shared_rank(&S.cnt[b][0], r)[threadIdx.x];
      S.mcnt[threadIdx.x] = m;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int cum = 0, sel = 0;
      for (int bin = 255; bin >= 0; --bin) {
        if (cum + S.mcnt[bin] >= want) {
          sel = bin;
          break;
        }
        cum += S.mcnt[bin];
      }
      S.want = uint64_t(want - cum);
      S.prefix = prefix | (uint32_t(sel) << shift);
    }
    __syncthreads();
    prefix = uint32_t(S.prefix);
    want = int(S.want);
    __syncthreads();
  }
  kth = prefix;
  take = want;
}

// Index-ordered compaction of the k largest (keys above kth, then the first
// `take` copies of kth): out[j * stride + i] for every copy j < rep.
__device__ void sel_compact(const uint32_t* x, int lo, int hi, uint32_t kth, int take, int k, int32_t* out,
                            int rep, int stride, SelShared& S) {
  cg::cluster_group cl = cg::this_cluster();
  const int rank = int(cl.block_rank());
  if (threadIdx.x == 0) S.n_gt = S.n_eq = 0;
  __syncthreads();
  int gt = 0, eq = 0;
  for (int i = lo + threadIdx.x; i < hi; i += blockDim.x) {
    const uint32_t v = x[i];
    gt += v > kth;
    eq += v == kth;
  }
  gt = __reduce_add_sync(0xffffffffu, gt);
  eq = __reduce_add_sync(0xffffffffu, eq);
  if ((threadIdx.x & 31) == 0) {
    atomicAdd(&S.n_gt, gt);
    atomicAdd(&S.n_eq, eq);
  }
  cl.sync();
  int gt_before = 0, eq_before = 0;
  for (int r = 0; r < rank; ++r) {
    gt_before += *cl.map_shared_rank(&S.n_gt, r);
    eq_before += *cl.map_shared_rank(&S.n_eq, r);
  }
  int eq_base = eq_before, out_base = gt_before + min(eq_before, take);
  for (int i0 = lo; i0 < hi; i0 += blockDim.x) {
    const int i = i0 + threadIdx.x;
    const uint32_t v = (i < hi) ? x[i] : 0u;
    const int is_eq = (i < hi && v == kth) ? 1 : 0;
    int tot;
    const int eq_incl = block_scan(is_eq, S.wsum, &tot);
    const int sel = (i < hi) && (v > kth || (is_eq && eq_base + eq_incl - 1 < take));
    eq_base += tot;
    int tot2;
    const int pos = block_scan(sel, S.wsum, &tot2);
    if (sel && out_base + pos - 1 < k)
      for (int j = 0; j < rep; ++j) out[int64_t(j) * stride + out_base + pos - 1] = i;
    out_base += tot2;
  }
}

struct TopkParams {
  const float* score;  // [L][N] score lists for v, then s
  const float* score2;
  int32_t* out;        // [L * rep][k]: list l is written to rows l * rep .. l * rep + rep - 1
  int32_t* out2;
  int N, k, k2;
  int rep;             // copies of each list (the heads of a group sharing it)
  const int* err;      // status word: a recorded failure skips the selection
};

// Grid (lists x kSelCluster, 2): one cluster per list; y = 0 the vertical
// lists, y = 1 the slash lists.  Radix select of the k-th largest score (the
// bit patterns of nonnegative floats order like their values), then the
// index-ordered compaction: the k largest scores' indices, ties to the lower
// index, ascending.
__global__ void __cluster_dims__(kSelCluster, 1, 1) __launch_bounds__(kTopkThreads) est_topk(const TopkParams p) {
  __shared__ SelShared S;
  if (sel_skip(p.err, S)) return;
  cg::cluster_group cl = cg::this_cluster();
  const int l = int(blockIdx.x) / kSelCluster, which = blockIdx.y;
  const uint32_t* x = reinterpret_cast<const uint32_t*>(which == 0 ? p.score : p.score2) + int64_t(l) * p.N;
  const int k = which == 0 ? p.k : p.k2;
  int32_t* out = (which == 0 ? p.out : p.out2) + int64_t(l) * p.rep * k;
  int lo, hi;
  sel_chunk(p.N, int(cl.block_rank()), lo, hi);
  if (k > 0) {
    uint32_t kth;
    int take;
    sel_kth(x, lo, hi, k, S, kth, take);
    sel_compact(x, lo, hi, kth, take, k, out, p.rep, k, S);
  }
  cl.sync();  // peers may still read this CTA's counts
}

// Per-KV-group sums of the heads' scores, added in head order (fp32), for
// the shared selection: gv[b, hk, m] = sum_j v[b, hk g + j, m].
__global__ void __launch_bounds__(256) est_group_sum(const float* v, const float* s, float* gv, float* gs, int N,
                                                     int g, const int* err) {
  if (est_failed(err)) return;
  const int l = blockIdx.y;  // b * Hkv + hk
  const int64_t m = int64_t(blockIdx.x) * 256 + threadIdx.x;
  if (m >= N) return;
  const float* pv = v + int64_t(l) * g * N + m;
  const float* ps = s + int64_t(l) * g * N + m;
  float a = pv[0], c = ps[0];
  for (int j = 1; j < g; ++j) {
    a += pv[int64_t(j) * N];
    c += ps[int64_t(j) * N];
  }
  gv[int64_t(l) * N + m] = a;
  gs[int64_t(l) * N + m] = c;
}

// ---------------------------------------------------------------- top-p
// Top-p budgets (Algorithm 1, `topp` and `Pool`): the budget is the smallest
// k whose k largest scores carry at least a fraction p of the list's mass.
// The decision is taken exactly: a score x counts floor(x * 2^40) mass units
// (integers; their sums do not depend on the order of addition), the target
// is t = ceil(p * T) for the total T (one rounded double product), and the
// k-th largest is found by a radix select that tracks unit sums per digit.
// Scores must be finite and nonnegative with a total below 2^13 (the
// estimator's total is last_q); otherwise VS_ERR_SCORE and empty lists.
constexpr double kUnitScale = 1099511627776.0;   // 2^40
constexpr uint64_t kUnitTotalMax = 1ull << 53;  // totals stay exact as doubles
constexpr uint64_t kSat = 1ull << 62;

__device__ __forceinline__ uint64_t mass_unit(float x) { return __double2ull_rz(double(x) * kUnitScale); }
__device__ __forceinline__ uint64_t sat_add(uint64_t a, uint64_t b) {
  const uint64_t c = a + b;  // a, b <= 2^62: no wrap
  return c > kSat ? kSat : c;
}

struct ToppParams {
  const float* v;  // [BH][N]
  const float* s;
  int32_t* v_idx;  // [BH][kv_max]
  int32_t* s_idx;  // [BH][ks_max]
  int32_t* kv;     // [BH] budgets (out)
  int32_t* ks;
  int* err;
  int N, kv_max, ks_max;
  double pv, ps;
};

// Saturating block sum of one value per thread (values <= 2^62).
__device__ uint64_t block_sum_sat(uint64_t x, SelShared& S) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x = sat_add(x, __shfl_xor_sync(0xffffffffu, x, off));
  if (lane == 0) S.red[w] = x;
  __syncthreads();
  uint64_t t = 0;
  for (int i = 0; i < int(blockDim.x >> 5); ++i) t = sat_add(t, S.red[i]);
  __syncthreads();
  return t;
}

// Smallest k in [0, n] with (sum of the k largest units of the cluster's
// list) >= t, for t >= 1 and t <= total.  This CTA holds keys [lo, hi) of
// x (fp32 score bits) or, POOLED, pooled[0, hi - lo) (the units, < 2^53,
// themselves); keys order the elements like their units.
template <bool POOLED>
__device__ int topp_count(const uint32_t* x, const uint64_t* pooled, int lo, int hi, int n, uint64_t t,
                          SelShared& S) {
  cg::cluster_group cl = cg::this_cluster();
  uint64_t prefix = 0, want = t;
  int above = 0;
  for (int pass = 0, shift = POOLED ? 48 : 24; shift >= 0; ++pass, shift -= 8) {
    const int b = pass & 1;
    for (int i = threadIdx.x; i < 256; i += blockDim.x) {
      S.cnt[b][i] = 0;
      S.sum[b][i] = 0;
    }
    __syncthreads();
    const uint64_t hi_key = prefix >> (shift + 8);
    for (int i = threadIdx.x; i < hi - lo; i += blockDim.x) {
      const uint64_t key = POOLED ? pooled[i] : uint64_t(x[lo + i]);
      if ((key >> (shift + 8)) == hi_key) {
        const int dgt = int((key >> shift) & 255);
        atomicAdd(&S.cnt[b][dgt], 1);
        atomicAdd(&S.sum[b][dgt], static_cast<unsigned long long>(POOLED ? key : mass_unit(__uint_as_float(uint32_t(key)))));
      }
    }
    cl.sync();
    if (threadIdx.x < 256) {
      int m = 0;
      unsigned long long u = 0;  // below 2^53: the list's total is
      for (int r = 0; r < kSelCluster; ++r) {
        m += cl.map_shared_rank(&S.cnt[b][0], r)[threadIdx.x];
        u += cl.map_shared_rank(&S.sum[b][0], r)[threadIdx.x];
      }
      S.mcnt[threadIdx.x] = m;
      S.msum[threadIdx.x] = u;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      uint64_t cum = 0;
      int ab = 0, sel = 0;
      for (int bin = 255; bin >= 0; --bin) {
        if (cum + S.msum[bin] >= want) {
          sel = bin;
          break;
        }
        cum += S.msum[bin];
        ab += S.mcnt[bin];
      }
      S.want = want - cum;  // > 0: the bins above sum to less than want
      S.above = above + ab;
      S.prefix = prefix | (uint64_t(sel) << shift);
    }
    __syncthreads();
    prefix = S.prefix;
    want = S.want;
    above = S.above;
    __syncthreads();
  }
  // the k-th largest has key `prefix`; the smallest j with j * u >= want of
  // its copies completes the budget
  const uint64_t u = POOLED ? prefix : mass_unit(__uint_as_float(uint32_t(prefix)));
  const int k = above + (u ? int((want + u - 1) / u) : 0);
  return k < n ? k : n;
}

// Grid (BH x kSelCluster, 2): one cluster per list; y = 0 the vertical list,
// y = 1 the slash list.  Dynamic shared memory: the pooled slash units of
// this CTA's chunk, one per 64-offset block.
__global__ void __cluster_dims__(kSelCluster, 1, 1) __launch_bounds__(kTopkThreads) est_topp(const ToppParams p) {
  extern __shared__ __align__(16) uint64_t pooled[];
  __shared__ SelShared S;
  if (sel_skip(p.err, S)) return;
  cg::cluster_group cl = cg::this_cluster();
  const int rank = int(cl.block_rank());
  const int bh = int(blockIdx.x) / kSelCluster, which = blockIdx.y;
  const int N = p.N;
  const float* xf = (which == 0 ? p.v : p.s) + int64_t(bh) * N;
  const uint32_t* x = reinterpret_cast<const uint32_t*>(xf);
  int lo, hi;
  sel_chunk(N, rank, lo, hi);
  if (threadIdx.x == 0) S.bad = 0;
  __syncthreads();
  // 1. validate, total mass; the slash list is pooled per 64-offset block
  uint64_t mine = 0;
  int bad = 0;
  if (which == 0) {
    for (int i = lo + threadIdx.x; i < hi; i += blockDim.x) {
      const float f = xf[i];
      if (!(f >= 0.f && f < 8192.f)) bad = 1;
      else mine = sat_add(mine, mass_unit(f));
    }
  } else {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int b = lo / 64 + w; b < hi / 64; b += nw) {
      uint64_t u = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float f = xf[64 * b + 32 * h + lane];
        if (!(f >= 0.f && f < 8192.f)) bad = 1;
        else u += mass_unit(f);  // < 2^54 for two scores below 2^13
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) u = sat_add(u, __shfl_xor_sync(0xffffffffu, u, off));
      if (lane == 0) pooled[b - lo / 64] = u;
      mine = sat_add(mine, lane == 0 ? u : 0ull);
    }
  }
  if (bad) S.bad = 1;
  const uint64_t part = block_sum_sat(mine, S);  // its syncs also publish S.bad and pooled[]
  if (threadIdx.x == 0) S.part = part;
  cl.sync();
  uint64_t T = 0;
  int any_bad = 0;
  for (int r = 0; r < kSelCluster; ++r) {
    T = sat_add(T, *cl.map_shared_rank(&S.part, r));
    any_bad |= *cl.map_shared_rank(&S.bad, r);
  }
  const bool ok = !any_bad && T < kUnitTotalMax;
  // 2. budget (the same in every CTA of the cluster)
  int k = 0;
  if (ok) {
    const double prod = (which == 0 ? p.pv : p.ps) * double(T);
    const uint64_t t = uint64_t(ceil(prod));
    if (t > 0)
      k = which == 0 ? topp_count<false>(x, nullptr, lo, hi, N, t, S)
                     : topp_count<true>(nullptr, pooled, lo / 64, hi / 64, N / 64, t, S);
  } else if (rank == 0 && threadIdx.x == 0) {
    raise_error(p.err, VS_ERR_SCORE);
  }
  const int cap = which == 0 ? p.kv_max : p.ks_max;
  if (which == 1) k = min(64 * k, N);
  k = min(k, cap);
  if (rank == 0 && threadIdx.x == 0) (which == 0 ? p.kv : p.ks)[bh] = k;
  // 3. the k largest at token level, padded to the list capacity
  int32_t* out = (which == 0 ? p.v_idx : p.s_idx) + int64_t(bh) * cap;
  for (int i = k + rank * int(blockDim.x) + threadIdx.x; i < cap; i += kSelCluster * int(blockDim.x)) out[i] = -1;
  if (k > 0) {
    uint32_t kth;
    int take;
    sel_kth(x, lo, hi, k, S, kth, take);
    sel_compact(x, lo, hi, kth, take, k, out, 1, cap, S);
  }
  cl.sync();  // peers may still read this CTA's counts
}

// Pooled slash units of one CTA's chunk.
size_t topp_smem_bytes(int N) {
  const int nb = N / 64;
  return size_t((nb + kSelCluster - 1) / kSelCluster) * sizeof(uint64_t);
}

vs_status launch_topp(const ToppParams& tp, int BH, cudaStream_t st) {
  const size_t sm = topp_smem_bytes(tp.N);
  if (sm > kToppMaxSmem) return VS_ERR_SHAPE;
  if (cudaFuncSetAttribute(est_topp, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm)) != cudaSuccess)
    return VS_ERR_CUDA;
  trace_begin("est_topp", st);
  est_topp<<<dim3(BH * kSelCluster, 2), kTopkThreads, sm, st>>>(tp);
  trace_end(st);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? VS_OK : VS_ERR_CUDA;
}

// The estimator's kernels on the given scratch (p.part / lse / spart and the
// score outputs set by the caller).
template <int D>
vs_status launch_est_kernels(const vs_shape* s, const void* q, const void* k, EstParams& p, int kv, int ks,
                             int32_t* v_idx, int32_t* s_idx, ToppParams* topp, cudaStream_t st) {
  CUtensorMap tq, tk;
  vs_status rc;
  if ((rc = make_tmap_bshd(&tq, q, s->B, s->Nq, s->Hq, D, s->sq, kLastQ)) != VS_OK) return rc;
  if ((rc = make_tmap_bshd(&tk, k, s->B, s->Nk, s->Hkv, D, s->sk, kEstKeys)) != VS_OK) return rc;
  const size_t sm = sizeof(EstSmem<D>) + 1024;
  if (cudaFuncSetAttribute(est_rowstats<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm)) != cudaSuccess ||
      cudaFuncSetAttribute(est_scores<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm)) != cudaSuccess)
    return VS_ERR_CUDA;
  const int BH = s->B * s->Hq, BHK = s->B * s->Hkv;
  const int NT = (s->Nk + kEstKeys - 1) / kEstKeys;
  trace_begin("est_rowstats", st);
  est_rowstats<D><<<dim3(BHK * p.MT, kSplits), kEstThreads, sm, st>>>(tq, tk, p);
  trace_end(st);
  trace_begin("est_lse", st);
  est_lse<<<BH, kLastQ, 0, st>>>(p);
  trace_end(st);
  trace_begin("est_scores", st);
  est_scores<D><<<dim3(BHK, NT), kEstThreads, sm, st>>>(tq, tk, p);
  trace_end(st);
  trace_begin("est_scombine", st);
  est_scombine<<<dim3((s->Nk + 255) / 256, BH), 256, 0, st>>>(p);
  trace_end(st);
  if (topp) {
    topp->v = p.v;
    topp->s = p.s;
    topp->err = p.err;
    note_launch(4);
    return launch_topp(*topp, BH, st);
  }
  TopkParams tp;
  tp.score = p.v;
  tp.score2 = p.s;
  tp.out = v_idx;
  tp.out2 = s_idx;
  tp.N = s->Nk;
  tp.k = kv;
  tp.k2 = ks;
  tp.rep = 1;
  tp.err = p.err;
  int lists = BH;
  if (p.gv) {
    trace_begin("est_group_sum", st);
    est_group_sum<<<dim3((s->Nk + 255) / 256, BHK), 256, 0, st>>>(p.v, p.s, p.gv, p.gs, s->Nk, p.g, p.err);
    trace_end(st);
    note_launch();
    tp.score = p.gv;
    tp.score2 = p.gs;
    tp.rep = p.g;
    lists = BHK;
  }
  trace_begin("est_topk", st);
  est_topk<<<dim3(lists * kSelCluster, 2), kTopkThreads, 0, st>>>(tp);
  trace_end(st);
  note_launch(5);
  return cudaGetLastError() == cudaSuccess ? VS_OK : VS_ERR_CUDA;
}

EstParams est_params(const vs_shape* s, float scale, int* err) {
  EstParams p;
  p.B = s->B;
  p.N = s->Nk;
  p.Hq = s->Hq;
  p.Hkv = s->Hkv;
  p.d = s->d;
  p.g = s->Hq / s->Hkv;
  p.MT = (p.g + 1) / 2;
  p.scale_log2 = scale * kLog2e;
  p.err = err;
  p.gv = p.gs = nullptr;
  return p;
}

vs_status launch_est(const vs_shape* s, const void* q, const void* k, EstParams& p, int kv, int ks, int32_t* v_idx,
                     int32_t* s_idx, cudaStream_t st, ToppParams* topp = nullptr) {
  if (topp && size_t(s->Nk) > topp_max_n()) return VS_ERR_SHAPE;
  if (s->d == 128) return launch_est_kernels<128>(s, q, k, p, kv, ks, v_idx, s_idx, topp, st);
  if (s->d == 64) return launch_est_kernels<64>(s, q, k, p, kv, ks, v_idx, s_idx, topp, st);
  return VS_ERR_SHAPE;
}

}  // namespace

size_t estimate_workspace_bytes(const vs_shape* s, int) { return size_t(est_layout(s).total); }

size_t topp_max_n() { return kToppMaxSmem / sizeof(uint64_t) * 64; }

vs_status launch_estimate_topp(const vs_shape* s, const void* q, const void* k, double pv, double ps, int kv_max,
                               int ks_max, float scale, int32_t* v_idx, int32_t* s_idx, int32_t* kv, int32_t* ks,
                               float* v_score, float* s_score, void* ws, cudaStream_t st) {
  const EstLayout L = est_layout(s);
  uint8_t* W = static_cast<uint8_t*>(ws);
  EstParams p = est_params(s, scale, static_cast<int*>(ws));
  p.part = reinterpret_cast<float2*>(W + L.off_part);
  p.lse = reinterpret_cast<float*>(W + L.off_lse);
  p.v = v_score ? v_score : reinterpret_cast<float*>(W + L.off_vbuf);
  p.spart = reinterpret_cast<float*>(W + L.off_spart);
  p.s = s_score ? s_score : reinterpret_cast<float*>(W + L.off_sbuf);
  ToppParams tp{};
  tp.v_idx = v_idx;
  tp.s_idx = s_idx;
  tp.kv = kv;
  tp.ks = ks;
  tp.N = s->Nk;
  tp.kv_max = kv_max;
  tp.ks_max = ks_max;
  tp.pv = pv;
  tp.ps = ps;
  return launch_est(s, q, k, p, kv_max, ks_max, v_idx, s_idx, st, &tp);
}

vs_status launch_select_topp(int B, int H, int N, const float* v_score, const float* s_score, double pv, double ps,
                             int kv_max, int ks_max, int32_t* v_idx, int32_t* s_idx, int32_t* kv, int32_t* ks,
                             int* err, cudaStream_t st) {
  ToppParams tp{};
  tp.v = v_score;
  tp.s = s_score;
  tp.v_idx = v_idx;
  tp.s_idx = s_idx;
  tp.kv = kv;
  tp.ks = ks;
  tp.err = err;
  tp.N = N;
  tp.kv_max = kv_max;
  tp.ks_max = ks_max;
  tp.pv = pv;
  tp.ps = ps;
  return launch_topp(tp, B * H, st);
}

vs_status launch_estimate(const vs_shape* s, const void* q, const void* k, int, int kv, int ks, float scale,
                          int32_t* v_idx, int32_t* s_idx, float* v_score, float* s_score, void* ws, int shared,
                          cudaStream_t st) {
  const EstLayout L = est_layout(s);
  uint8_t* W = static_cast<uint8_t*>(ws);
  EstParams p = est_params(s, scale, static_cast<int*>(ws));
  if (shared) {
    p.gv = reinterpret_cast<float*>(W + L.off_gv);
    p.gs = reinterpret_cast<float*>(W + L.off_gs);
  }
  p.part = reinterpret_cast<float2*>(W + L.off_part);
  p.lse = reinterpret_cast<float*>(W + L.off_lse);
  p.v = v_score ? v_score : reinterpret_cast<float*>(W + L.off_vbuf);
  p.spart = reinterpret_cast<float*>(W + L.off_spart);
  p.s = s_score ? s_score : reinterpret_cast<float*>(W + L.off_sbuf);
  return launch_est(s, q, k, p, kv, ks, v_idx, s_idx, st);
}

}  // namespace vs

// ===========================================================================
// vs_estimate_noalloc: the estimator for callers that cannot allocate device
// memory while they run (see include/vs.h).  Its scratch is a fixed array in
// the module's static device memory, shared by every call on a device.
// ===========================================================================
#include <mutex>

static constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the static scratch on the current device (host code may
// not use the array's name as a device address), looked up once per device.
// The look-up may load the module onto the device, which must not happen
// inside a stream capture: while `stream` is capturing and the address is not
// known yet, the call is refused with VS_ERR_ARG.
vs_status noalloc_scratch_address(cudaStream_t stream, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return VS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return VS_ERR_CUDA;
    if (cap != cudaStreamCaptureStatusNone) return VS_ERR_ARG;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return VS_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return VS_OK;
}

// The scratch address of the current device if a call has looked it up.
void* noalloc_known_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  return g_noalloc_ptr[dev];
}

// Scratch layout: 256-byte status header, per-split row statistics, row
// LSEs, per-tile slash partials.  Returns the bytes needed.
int64_t noalloc_layout(const vs_shape* s, int64_t* off_part, int64_t* off_lse, int64_t* off_spart) {
  const int64_t BH = int64_t(s->B) * s->Hq, N = s->Nk, NT = (N + vs::kEstKeys - 1) / vs::kEstKeys;
  int64_t off = 256;
  *off_part = off;
  off += (BH * vs::kSplits * vs::kLastQ * 8 + 255) / 256 * 256;
  *off_lse = off;
  off += (BH * vs::kLastQ * 4 + 255) / 256 * 256;
  *off_spart = off;
  off += (BH * NT * vs::kEstDiag * 4 + 255) / 256 * 256;
  return off;
}

}  // namespace

extern "C" vs_status vs_estimate_noalloc(const vs_shape* s, const void* q, const void* k, int last_q, int kv, int ks,
                                         float scale, int32_t* v_idx, int32_t* s_idx, float* v_score, float* s_score,
                                         cudaStream_t stream) {
  using namespace vs;
  // every argument check happens on the host, before any CUDA call, and
  // refuses exactly what vs_estimate refuses (plus missing score buffers)
  if (!v_score || !s_score) return VS_ERR_ARG;
  vs_status rc = check_estimate_args(s, q, k, last_q, kv, ks, scale, v_idx, s_idx);
  if (rc != VS_OK) return rc;
  int64_t off_part = 0, off_lse = 0, off_spart = 0;
  if (size_t(noalloc_layout(s, &off_part, &off_lse, &off_spart)) > kNoAllocScratchBytes) return VS_ERR_WORKSPACE;
  void* base = nullptr;
  if ((rc = noalloc_scratch_address(stream, &base)) != VS_OK) return rc;
  uint8_t* W = static_cast<uint8_t*>(base);
  // The kernels write every scratch element they later read within the
  // call, unless a kernel records a failure in the status word, after which
  // the later kernels skip their work; only the status header is cleared.
  if (cudaMemsetAsync(W, 0, 256, stream) != cudaSuccess) return VS_ERR_CUDA;
  EstParams p = est_params(s, scale, reinterpret_cast<int*>(W));
  p.part = reinterpret_cast<float2*>(W + off_part);
  p.lse = reinterpret_cast<float*>(W + off_lse);
  p.v = v_score;
  p.spart = reinterpret_cast<float*>(W + off_spart);
  p.s = s_score;
  return launch_est(s, q, k, p, kv, ks, v_idx, s_idx, stream);
}

extern "C" vs_status vs_estimate_noalloc_status(cudaStream_t stream) {
  void* W = noalloc_known_address();
  if (!W) return VS_OK;  // no call has run on this device
  return vs_check_status(W, stream);
}

extern "C" vs_status vs_estimate_noalloc_selftest_plant(int code, cudaStream_t stream) {
  void* W = nullptr;
  vs_status rc = noalloc_scratch_address(stream, &W);
  if (rc != VS_OK) return rc;
  const int32_t word = code;
  if (cudaMemcpyAsync(W, &word, sizeof(word), cudaMemcpyHostToDevice, stream) != cudaSuccess) return VS_ERR_CUDA;
  return cudaStreamSynchronize(stream) == cudaSuccess ? VS_OK : VS_ERR_CUDA;
}
