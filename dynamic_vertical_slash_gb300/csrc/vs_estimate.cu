// Online Vertical-Slash estimation (Algorithm 1, first four lines).
//
//   pass 1  est_rowstats : per (b, h, key split) partial (max, sum exp) of the
//                          last 64 query rows' causal logits
//   pass 2  est_scores   : per (b, h, 64-key tile) A_hat = exp(S - LSE):
//                          column sums -> v[m] (complete per tile), diagonal
//                          sums -> 127 partial slash sums per tile
//   pass 3  est_scombine : s[o] = the (at most two) tile partials of o, added
//                          in a fixed order (deterministic, no float atomics)
//   pass 4  est_topk     : radix select of the k-th largest score, then an
//                          index-ordered compaction; ties go to the lower index
#include "vs_internal.h"

namespace vs {
namespace {

constexpr int kEstThreads = 256;
constexpr int kLastQ = 64;
constexpr int kChunk = 32;     // keys per chunk in pass 1
constexpr int kSplits = 64;    // key splits per head in pass 1
constexpr int kTopkThreads = 1024;

struct EstLayout {
  int64_t off_part, off_vbuf, off_spart, off_sbuf, total;
};

EstLayout est_layout(const vs_shape* s) {
  EstLayout L;
  const int64_t BH = int64_t(s->B) * s->Hq, N = s->Nk, NT = N / 64;
  int64_t off = 256;
  auto take = [&](int64_t bytes) {
    const int64_t at = off;
    off += (bytes + 255) / 256 * 256;
    return at;
  };
  L.off_part = take(BH * kSplits * kLastQ * 8);
  L.off_vbuf = take(BH * N * 4);
  L.off_spart = take(BH * NT * 128 * 4);
  L.off_sbuf = take(BH * N * 4);
  L.total = off;
  return L;
}

// Loads `rows` rows of d bf16 values (token stride s_tok elements) into a
// float tile with row pitch `pitch`.
__device__ __forceinline__ void load_rows_f32(float* dst, int pitch, const uint16_t* src, int64_t s_tok, int rows,
                                              int d, int row0, int row_limit) {
  for (int i = threadIdx.x; i < rows * (d / 8); i += blockDim.x) {
    const int r = i / (d / 8), c8 = (i % (d / 8)) * 8;
    float* o = dst + r * pitch + c8;
    if (row0 + r < row_limit) {
      const uint4 w = *reinterpret_cast<const uint4*>(src + int64_t(row0 + r) * s_tok + c8);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        o[2 * e] = __uint_as_float(ws[e] << 16);
        o[2 * e + 1] = __uint_as_float(ws[e] & 0xFFFF0000u);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = 0.f;
    }
  }
}

struct EstParams {
  const uint16_t* q;
  const uint16_t* k;
  int64_t sq[3], sk[3];
  int B, N, Hq, Hkv, d;
  float scale_log2;
  float2* part;   // [BH][kSplits][64] (max, sum) in log2 units
  float* v;       // [BH][N]
  float* spart;   // [BH][NT][128]
  float* s;       // [BH][N]
};

__global__ void __launch_bounds__(kEstThreads) est_rowstats(const EstParams p) {
  extern __shared__ float sm[];
  const int d = p.d, pitch = d + 4;
  float* qs = sm;                      // [64][pitch]
  float* ks = sm + kLastQ * pitch;     // [kChunk][pitch]
  const int bh = blockIdx.x, sp = blockIdx.y;
  const int b = bh / p.Hq, h = bh % p.Hq, hk = h / (p.Hq / p.Hkv);
  const int N = p.N;
  const int per = ((N + kSplits - 1) / kSplits + kChunk - 1) / kChunk * kChunk;
  const int k0 = sp * per, k1 = min(N, k0 + per);
  const uint16_t* qb = p.q + int64_t(b) * p.sq[0] + int64_t(h) * p.sq[2];
  const uint16_t* kb = p.k + int64_t(b) * p.sk[0] + int64_t(hk) * p.sk[2];
  load_rows_f32(qs, pitch, qb, p.sq[1], kLastQ, d, N - kLastQ, N);
  const int r = threadIdx.x / 4, kl = threadIdx.x % 4;
  const int n = N - kLastQ + r;
  float m = -INFINITY, l = 0.f;
  for (int c0 = k0; c0 < k1; c0 += kChunk) {
    __syncthreads();
    load_rows_f32(ks, pitch, kb, p.sk[1], kChunk, d, c0, k1);
    __syncthreads();
    float acc[kChunk / 4];
#pragma unroll
    for (int i = 0; i < kChunk / 4; ++i) acc[i] = 0.f;
    for (int c = 0; c < d; c += 4) {
      const float4 qv = *reinterpret_cast<const float4*>(qs + r * pitch + c);
#pragma unroll
      for (int i = 0; i < kChunk / 4; ++i) {
        const float4 kv = *reinterpret_cast<const float4*>(ks + (kl + 4 * i) * pitch + c);
        acc[i] += qv.x * kv.x + qv.y * kv.y + qv.z * kv.z + qv.w * kv.w;
      }
    }
#pragma unroll
    for (int i = 0; i < kChunk / 4; ++i) {
      const int key = c0 + kl + 4 * i;
      if (key < k1 && key <= n) {
        const float x = acc[i] * p.scale_log2;
        if (x > m) {
          l = l * exp2f(m - x) + 1.f;
          m = x;
        } else {
          l += exp2f(x - m);
        }
      }
    }
  }
  // merge the four key lanes of the row
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, off);
    const float lo = __shfl_xor_sync(0xffffffffu, l, off);
    const float mn = fmaxf(m, mo);
    if (mn == -INFINITY) continue;
    l = (m == -INFINITY ? 0.f : l * exp2f(m - mn)) + (mo == -INFINITY ? 0.f : lo * exp2f(mo - mn));
    m = mn;
  }
  if (kl == 0) p.part[(int64_t(bh) * kSplits + sp) * kLastQ + r] = make_float2(m, l);
}

__global__ void __launch_bounds__(kEstThreads) est_scores(const EstParams p) {
  extern __shared__ float sm[];
  const int d = p.d, pitch = d + 4;
  float* qs = sm;                        // [64][pitch]
  float* ks = qs + kLastQ * pitch;       // [64][pitch]
  float* at = ks + 64 * pitch;           // [64][65]  A_hat tile
  float* lse = at + 64 * 65;             // [64]
  const int bh = blockIdx.x, tile = blockIdx.y;
  const int b = bh / p.Hq, h = bh % p.Hq, hk = h / (p.Hq / p.Hkv);
  const int N = p.N, m0 = tile * 64;
  if (threadIdx.x < kLastQ) {
    const float2* pp = p.part + int64_t(bh) * kSplits * kLastQ + threadIdx.x;
    float m = -INFINITY, l = 0.f;
    for (int sp = 0; sp < kSplits; ++sp) {
      const float2 x = pp[sp * kLastQ];
      if (x.x == -INFINITY) continue;
      const float mn = fmaxf(m, x.x);
      l = (m == -INFINITY ? 0.f : l * exp2f(m - mn)) + x.y * exp2f(x.x - mn);
      m = mn;
    }
    lse[threadIdx.x] = m + log2f(l);
  }
  const uint16_t* qb = p.q + int64_t(b) * p.sq[0] + int64_t(h) * p.sq[2];
  const uint16_t* kb = p.k + int64_t(b) * p.sk[0] + int64_t(hk) * p.sk[2];
  load_rows_f32(qs, pitch, qb, p.sq[1], kLastQ, d, N - kLastQ, N);
  load_rows_f32(ks, pitch, kb, p.sk[1], 64, d, m0, N);
  __syncthreads();
  const int r = threadIdx.x / 4, kl = threadIdx.x % 4;
  const int n = N - kLastQ + r;
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  for (int c = 0; c < d; c += 4) {
    const float4 qv = *reinterpret_cast<const float4*>(qs + r * pitch + c);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float4 kv = *reinterpret_cast<const float4*>(ks + (kl + 4 * i) * pitch + c);
      acc[i] += qv.x * kv.x + qv.y * kv.y + qv.z * kv.z + qv.w * kv.w;
    }
  }
  const float L = lse[r];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int j = kl + 4 * i, key = m0 + j;
    at[r * 65 + j] = (key <= n) ? exp2f(acc[i] * p.scale_log2 - L) : 0.f;
  }
  __syncthreads();
  // vertical: column sums (4 threads per key, 16 rows each)
  {
    const int j = threadIdx.x / 4, part = threadIdx.x % 4;
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) sum += at[(part * 16 + i) * 65 + j];
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    if (part == 0) p.v[int64_t(bh) * N + m0 + j] = sum;
  }
  // slash: diagonal delta = r - j in [-63, 63] <-> offset o = N - 64 - m0 + delta
  if (threadIdx.x < 128) {
    const int t = threadIdx.x;
    float sum = 0.f;
    if (t < 127) {
      const int delta = t - 63;
      const int rlo = max(0, delta), rhi = min(63, 63 + delta);
      for (int rr = rlo; rr <= rhi; ++rr) sum += at[rr * 65 + (rr - delta)];
    }
    p.spart[(int64_t(bh) * (N / 64) + tile) * 128 + t] = sum;
  }
}

__global__ void est_scombine(const EstParams p) {
  const int bh = blockIdx.y;
  const int N = p.N, NT = N / 64;
  const int o = blockIdx.x * blockDim.x + threadIdx.x;
  if (o >= N) return;
  const float* sp = p.spart + int64_t(bh) * NT * 128;
  const int x = N - 64 - o;
  const int Tc = (x >= 0) ? x / 64 : -1;
  float sum = 0.f;
  for (int T = Tc; T <= Tc + 1; ++T) {  // fixed order
    if (T < 0 || T >= NT) continue;
    const int delta = o - (N - 64 - 64 * T);
    if (delta >= -63 && delta <= 63) sum += sp[int64_t(T) * 128 + delta + 63];
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

struct TopkParams {
  const float* score;  // [BH][N] for v, then s
  const float* score2;
  int32_t* out;        // [BH][k]
  int32_t* out2;
  int N, k, k2;
};

__global__ void __launch_bounds__(kTopkThreads) est_topk(const TopkParams p) {
  const int bh = blockIdx.x, which = blockIdx.y;
  const uint32_t* x = reinterpret_cast<const uint32_t*>(which == 0 ? p.score : p.score2) + int64_t(bh) * p.N;
  const int k = which == 0 ? p.k : p.k2;
  int32_t* out = (which == 0 ? p.out : p.out2) + int64_t(bh) * k;
  __shared__ int hist[256];
  __shared__ uint32_t s_prefix;
  __shared__ int s_want;
  __shared__ int wsum[32];
  if (threadIdx.x == 0) {
    s_prefix = 0;
    s_want = k;
  }
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix;
    const uint32_t hi_mask = (shift == 24) ? 0u : (0xFFFFFFFFu << (shift + 8));
    for (int i = threadIdx.x; i < p.N; i += blockDim.x) {
      const uint32_t v = x[i];
      if ((v & hi_mask) == prefix) atomicAdd(&hist[(v >> shift) & 255], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int want = s_want, cum = 0, sel = 0;
      for (int bin = 255; bin >= 0; --bin) {
        if (cum + hist[bin] >= want) {
          sel = bin;
          break;
        }
        cum += hist[bin];
      }
      s_want = want - cum;
      s_prefix = prefix | (uint32_t(sel) << shift);
    }
    __syncthreads();
  }
  const uint32_t kth = s_prefix;
  const int take_eq = s_want;
  int eq_base = 0, out_base = 0;
  for (int i0 = 0; i0 < p.N; i0 += blockDim.x) {
    const int i = i0 + threadIdx.x;
    const uint32_t v = (i < p.N) ? x[i] : 0u;
    const int is_eq = (i < p.N && v == kth) ? 1 : 0;
    int tot;
    const int eq_incl = block_scan(is_eq, wsum, &tot);
    const int sel = (i < p.N) && (v > kth || (is_eq && eq_base + eq_incl - 1 < take_eq));
    eq_base += tot;
    int tot2;
    const int pos = block_scan(sel, wsum, &tot2);
    if (sel && out_base + pos - 1 < k) out[out_base + pos - 1] = i;
    out_base += tot2;
  }
}

}  // namespace

size_t estimate_workspace_bytes(const vs_shape* s, int) { return size_t(est_layout(s).total); }

vs_status launch_estimate(const vs_shape* s, const void* q, const void* k, int, int kv, int ks, float scale,
                          int32_t* v_idx, int32_t* s_idx, float* v_score, float* s_score, void* ws,
                          cudaStream_t st) {
  const EstLayout L = est_layout(s);
  uint8_t* W = static_cast<uint8_t*>(ws);
  EstParams p;
  p.q = static_cast<const uint16_t*>(q);
  p.k = static_cast<const uint16_t*>(k);
  for (int i = 0; i < 3; ++i) {
    p.sq[i] = s->sq[i];
    p.sk[i] = s->sk[i];
  }
  p.B = s->B;
  p.N = s->Nk;
  p.Hq = s->Hq;
  p.Hkv = s->Hkv;
  p.d = s->d;
  p.scale_log2 = scale * kLog2e;
  p.part = reinterpret_cast<float2*>(W + L.off_part);
  p.v = v_score ? v_score : reinterpret_cast<float*>(W + L.off_vbuf);
  p.spart = reinterpret_cast<float*>(W + L.off_spart);
  p.s = s_score ? s_score : reinterpret_cast<float*>(W + L.off_sbuf);
  const int BH = s->B * s->Hq;
  const int pitch = s->d + 4;
  const size_t sm1 = size_t(kLastQ + kChunk) * pitch * 4;
  const size_t sm2 = (size_t(kLastQ + 64) * pitch + 64 * 65 + 64) * 4;
  if (cudaFuncSetAttribute(est_rowstats, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm1)) != cudaSuccess ||
      cudaFuncSetAttribute(est_scores, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm2)) != cudaSuccess)
    return VS_ERR_CUDA;
  trace_begin("est_rowstats", st);
  est_rowstats<<<dim3(BH, kSplits), kEstThreads, sm1, st>>>(p);
  trace_end(st);
  trace_begin("est_scores", st);
  est_scores<<<dim3(BH, s->Nk / 64), kEstThreads, sm2, st>>>(p);
  trace_end(st);
  trace_begin("est_scombine", st);
  est_scombine<<<dim3((s->Nk + 255) / 256, BH), 256, 0, st>>>(p);
  trace_end(st);
  TopkParams tp;
  tp.score = p.v;
  tp.score2 = p.s;
  tp.out = v_idx;
  tp.out2 = s_idx;
  tp.N = s->Nk;
  tp.k = kv;
  tp.k2 = ks;
  trace_begin("est_topk", st);
  est_topk<<<dim3(BH, 2), kTopkThreads, 0, st>>>(tp);
  trace_end(st);
  note_launch(4);
  return cudaGetLastError() == cudaSuccess ? VS_OK : VS_ERR_CUDA;
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

// Device address of the static scratch on the current device, looked up once
// per device (host code may not use the array's name as a device address).
void* noalloc_scratch_address(int dev) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    g_noalloc_ptr[dev] = p;
  }
  return g_noalloc_ptr[dev];
}

// Scratch layout: 256-byte status header, per-split row statistics,
// per-tile slash partials.  Returns the bytes needed.
int64_t noalloc_layout(const vs_shape* s, int64_t* off_part, int64_t* off_spart) {
  const int64_t BH = int64_t(s->B) * s->Hq, N = s->Nk, NT = N / 64;
  int64_t off = 256;
  *off_part = off;
  off += (BH * vs::kSplits * vs::kLastQ * 8 + 255) / 256 * 256;
  *off_spart = off;
  off += (BH * NT * 128 * 4 + 255) / 256 * 256;
  return off;
}

}  // namespace

extern "C" vs_status vs_estimate_noalloc(const vs_shape* s, const void* q, const void* k, int last_q, int kv, int ks,
                                         float scale, int32_t* v_idx, int32_t* s_idx, float* v_score, float* s_score,
                                         cudaStream_t stream) {
  using namespace vs;
  // every check happens on the host, before any CUDA call
  if (!s || !q || !k || !v_idx || !s_idx || !v_score || !s_score) return VS_ERR_ARG;
  if (s->B < 1 || s->Nk < 64 || s->Hq < 1 || s->Hkv < 1 || (s->d != 64 && s->d != 128)) return VS_ERR_SHAPE;
  if (s->Nq != s->Nk || s->Nk % 64 || s->Hq % s->Hkv) return VS_ERR_SHAPE;
  for (int i = 0; i < 3; ++i)
    if (s->sq[i] <= 0 || s->sk[i] <= 0 || s->sq[i] % 8 || s->sk[i] % 8) return VS_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k)) & 15u) return VS_ERR_SHAPE;
  if (last_q != 64) return VS_ERR_ARG;
  if (kv < 1 || ks < 1 || kv > s->Nk || ks > s->Nk || !(scale > 0.f)) return VS_ERR_ARG;
  int64_t off_part = 0, off_spart = 0;
  if (size_t(noalloc_layout(s, &off_part, &off_spart)) > kNoAllocScratchBytes) return VS_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return VS_ERR_CUDA;
  uint8_t* W = static_cast<uint8_t*>(noalloc_scratch_address(dev));
  if (!W) return VS_ERR_CUDA;
  // The kernels write every scratch element they later read within the
  // call; only the status header is cleared.
  if (cudaMemsetAsync(W, 0, 256, stream) != cudaSuccess) return VS_ERR_CUDA;
  EstParams p;
  p.q = static_cast<const uint16_t*>(q);
  p.k = static_cast<const uint16_t*>(k);
  for (int i = 0; i < 3; ++i) {
    p.sq[i] = s->sq[i];
    p.sk[i] = s->sk[i];
  }
  p.B = s->B;
  p.N = s->Nk;
  p.Hq = s->Hq;
  p.Hkv = s->Hkv;
  p.d = s->d;
  p.scale_log2 = scale * kLog2e;
  p.part = reinterpret_cast<float2*>(W + off_part);
  p.v = v_score;
  p.spart = reinterpret_cast<float*>(W + off_spart);
  p.s = s_score;
  const int BH = s->B * s->Hq;
  const int pitch = s->d + 4;
  const size_t sm1 = size_t(kLastQ + kChunk) * pitch * 4;
  const size_t sm2 = (size_t(kLastQ + 64) * pitch + 64 * 65 + 64) * 4;
  if (cudaFuncSetAttribute(est_rowstats, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm1)) != cudaSuccess ||
      cudaFuncSetAttribute(est_scores, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm2)) != cudaSuccess)
    return VS_ERR_CUDA;
  est_rowstats<<<dim3(BH, kSplits), kEstThreads, sm1, stream>>>(p);
  est_scores<<<dim3(BH, s->Nk / 64), kEstThreads, sm2, stream>>>(p);
  est_scombine<<<dim3((s->Nk + 255) / 256, BH), 256, 0, stream>>>(p);
  TopkParams tp;
  tp.score = p.v;
  tp.score2 = p.s;
  tp.out = v_idx;
  tp.out2 = s_idx;
  tp.N = s->Nk;
  tp.k = kv;
  tp.k2 = ks;
  est_topk<<<dim3(BH, 2), kTopkThreads, 0, stream>>>(tp);
  note_launch(4);
  return cudaGetLastError() == cudaSuccess ? VS_OK : VS_ERR_CUDA;
}
