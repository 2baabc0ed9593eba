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
// Warp roles (192 threads): warp 0 loads, warp 1 issues MMAs (one lane),
// warps 2-5 run the softmax (thread <-> TMEM lane <-> query row).
// TMEM columns: O [0, d), S double buffer [128, 256), P double buffer [256, 320).
#include "vs_internal.h"
#include "vs_kernel_common.cuh"

namespace vs {
namespace {

constexpr int kFwdThreads = 192;
constexpr int kFwdStages = 3;
constexpr uint32_t kColO = 0, kColS = 128, kColP = 256, kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays <= 2^8 between rescales

template <int D>
struct FwdSmem {
  static constexpr int NH = D / 64;
  uint8_t q[NH][kQTile * 128];
  uint8_t k[kFwdStages][NH][kKTile * 128];
  uint8_t v[kFwdStages][NH][kKTile * 128];
  uint64_t q_full;
  uint64_t kv_full[kFwdStages], kv_empty[kFwdStages];
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
  uint64_t o_final, teardown;
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
      mbar_init(&s.kv_full[i], 1);
      mbar_init(&s.kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.s_free[i], 128);
      mbar_init(&s.p_full[i], 128);
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
      for (int j = 0; j < U; ++j) {
        const int st = j % kFwdStages;
        if (j >= kFwdStages && !mbar_wait(&s.kv_empty[st], ((j / kFwdStages) - 1) & 1, ab, VS_ERR_TIMEOUT)) break;
        if (j < nslash) {
          if (lane == 0) {
            const int c = t * kQTile + 64 - __ldg(elist + j);
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
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && U > 0) {
      const uint32_t idS = idesc_bf16(128, 64, 0, 0);
      const uint32_t idO = idesc_bf16(128, D, 0, 1);
      bool ok = mbar_wait(&s.q_full, 0, ab, VS_ERR_TIMEOUT);
      for (int j = 0; ok && j <= U; ++j) {
        if (j < U) {
          const int st = j % kFwdStages;
          if (!(ok = mbar_wait(&s.kv_full[st], (j / kFwdStages) & 1, ab, VS_ERR_TIMEOUT))) break;
          if (j >= nslash) fence_proxy_async_smem();
          if (j >= 2 && !(ok = mbar_wait(&s.s_free[j & 1], ((j - 2) >> 1) & 1, ab, VS_ERR_TIMEOUT))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t da = sdesc_sw128(smem_u32(s.q[kk / 4]) + (kk % 4) * 32, 16, 1024);
            const uint64_t db = sdesc_sw128(smem_u32(s.k[st][kk / 4]) + (kk % 4) * 32, 16, 1024);
            mma_ss(tmem + kColS + (j & 1) * 64, da, db, idS, kk > 0);
          }
          mma_issued = true;
          mma_commit(&s.s_full[j & 1]);
        }
        if (j >= 1) {
          const int jj = j - 1, st = jj % kFwdStages;
          if (!(ok = mbar_wait(&s.p_full[jj & 1], (jj >> 1) & 1, ab, VS_ERR_TIMEOUT))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kKTile / 16; ++kk) {
            const uint64_t dv = sdesc_sw128(smem_u32(s.v[st][0]) + kk * 2048, kKTile * 128, 1024);
            mma_ts(tmem + kColO, tmem + kColP + (jj & 1) * 32 + kk * 8, dv, idO, (jj > 0 || kk > 0));
          }
          mma_commit(&s.pv_done[jj & 1]);
          mma_commit(&s.kv_empty[st]);
        }
      }
      mma_commit(&s.o_final);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;            // TMEM lane quarter this warp may access
    const int r = quarter * 32 + lane;       // query row within the tile
    const uint32_t tl = tmem + (uint32_t(quarter * 32) << 16);
    const int64_t n_loc = int64_t(t) * kQTile + r;
    const bool row_ok = n_loc < p.Nq;
    const int64_t n_g = qpos_g(G, n_loc);
    const uint64_t* offbits = av.offbits + int64_t(bh) * G.WG;
    const uint64_t* colbits = av.colbits + int64_t(bh) * G.WG;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < U; ++j) {
      ok = mbar_wait(&s.s_full[j & 1], (j >> 1) & 1, ab, VS_ERR_TIMEOUT);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[64];
      tmem_ld32(tl + kColS + (j & 1) * 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(tl + kColS + (j & 1) * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&s.s_free[j & 1]);

      uint64_t mask = 0;
      if (row_ok) {
        if (j < nslash) {
          const int64_t c = int64_t(t) * kQTile + 64 - __ldg(elist + j);
          mask = slash_row_mask(G, offbits, colbits, n_g, c);
        } else {
          const int4* kq = reinterpret_cast<const int4*>(vlist + (j - nslash) * kKTile);
#pragma unroll
          for (int q4 = 0; q4 < 16; ++q4) {
            const int4 kk4 = __ldg(kq + q4);
            const int kk[4] = {kk4.x, kk4.y, kk4.z, kk4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (kk[e] >= 0 && kpos_g(G, kk[e]) <= n_g) mask |= 1ull << (q4 * 4 + e);
          }
        }
      }
      float x[64];
      float mt = -INFINITY;
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        x[i] = ((mask >> i) & 1ull) ? __uint_as_float(sr[i]) * p.scale_log2 : -INFINITY;
        mt = fmaxf(mt, x[i]);
      }
      // Lazy rescale: O and l are rescaled only when the row maximum grows by
      // more than the threshold.  tcgen05.ld / st are warp-collective, so the
      // decision is voted per warp and every lane takes part (alpha = 1 for
      // rows that keep their reference maximum).
      const bool grow = (m_run != -INFINITY) && (mt > m_run + kRescaleThreshold);
      if (m_run == -INFINITY && mt > -INFINITY) m_run = mt;  // first entries: O row is still zero
      if (__any_sync(0xffffffffu, grow)) {
        const float alpha = grow ? ex2(m_run - mt) : 1.f;
        ok = mbar_wait(&s.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, ab, VS_ERR_TIMEOUT);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 16) {
          uint32_t ov[16];
          tmem_ld16(tl + kColO + cc, ov);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
          tmem_st16(tl + kColO + cc, ov);
        }
        tmem_st_wait();
        if (grow) {
          l_run *= alpha;
          m_run = mt;
        }
      }
      uint32_t pk[32];
      float rs = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float p0 = ((mask >> (2 * i)) & 1ull) ? ex2(x[2 * i] - m_run) : 0.f;
        const float p1 = ((mask >> (2 * i + 1)) & 1ull) ? ex2(x[2 * i + 1] - m_run) : 0.f;
        rs += p0 + p1;
        pk[i] = pack_bf16x2(p0, p1);
      }
      l_run += rs;
      if (j >= 2) ok = mbar_wait(&s.pv_done[j & 1], ((j - 2) >> 1) & 1, ab, VS_ERR_TIMEOUT);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_st16(tl + kColP + (j & 1) * 32, *reinterpret_cast<uint32_t(*)[16]>(&pk[0]));
      tmem_st16(tl + kColP + (j & 1) * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[16]));
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&s.p_full[j & 1]);
    }
    // -------------------------------------------------------------- epilogue
    if (ok && U > 0) ok = mbar_wait(&s.o_final, 0, ab, VS_ERR_TIMEOUT);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (ok) {
      // every lane of the warp reads TMEM (warp-collective); only valid rows store
      const bool empty = (U == 0) || !(l_run > 0.f);
      const float inv = empty ? 0.f : 1.f / l_run;
      const float lse_step = empty ? -INFINITY : (m_run + __log2f(l_run)) * kLn2;
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
#pragma unroll 1
      for (int cc = 0; cc < D; cc += 16) {
        uint32_t ov[16];
        if (U > 0) {
          tmem_ld16(tl + kColO + cc, ov);
          tmem_ld_wait();
        }
        if (!row_ok) continue;
        float y[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) y[i] = empty ? 0.f : __uint_as_float(ov[i]) * inv;
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
      if (row_ok) *lse_p = lse_new;
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
