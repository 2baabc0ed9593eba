// Work of a context-parallel ring under the VS mask (MTraining, section 3.3
// worker- and step-level imbalance; section 4.2 Balanced Sparse Ring
// Attention; section 2 Striped vs ZigZag Ring Attention).
//
// out[r][q] = number of entries M[n, m] of the mask on the global sequence,
//   M[n, m] = (m <= n) and (m in iv or n - m in is),
// whose query n lives on worker r and key m on worker q, summed over (b, h).
// Layouts: striped (64-token block j on worker j mod W) and ZigZag (2W chunks
// of C = N / (2W) tokens; worker r holds chunks r and 2W - 1 - r).
//
// Counting, per (b, h), with owner-constant segments instead of entries:
//   vertical: every selected column m owns all rows n in [m, N); the rows of
//     worker r in [m, N) are F_r(N) - F_r(m), F_r(x) = tokens of worker r
//     below x (closed form);
//   slash: a selected offset o covers (n, n - o) for n in [o, N); the keys
//     run over [0, N - o) in owner segments (one per key block, split where
//     the query n = m + o crosses a query block), and the keys of a segment
//     that are selected columns are left out (already counted as vertical),
//     using prefix counts of the column bitmap.
// Integer atomics only: the result does not depend on the order of work.
#include "vs_internal.h"

namespace vs {
namespace {

constexpr int kRwThreads = 512;
constexpr int kRwSplits = 16;  // CTAs per (b, h)

struct RwParams {
  const int32_t* iv;
  const int32_t* is;
  int kv, ks;
  int64_t N;
  int W, zigzag;
  int64_t unit;     // block (striped: 64) or chunk (zigzag: N / (2W)) length
  int nwords;       // N / 64 rounded up
  unsigned long long* out;  // [W][W]
  int* err;
};

__device__ __forceinline__ int owner_of(const RwParams& p, int64_t n) {
  const int64_t c = n / p.unit;
  if (!p.zigzag) return int(c % p.W);
  return int(c < p.W ? c : 2 * p.W - 1 - c);
}

// Tokens of worker r below x.
__device__ __forceinline__ int64_t tokens_below(const RwParams& p, int r, int64_t x) {
  const int64_t U = p.unit;
  if (!p.zigzag) {
    const int64_t period = U * p.W;
    const int64_t full = x / period, rem = x - full * period;
    return full * U + min(max(rem - int64_t(r) * U, int64_t(0)), U);
  }
  const int64_t a = int64_t(r) * U, b = int64_t(2 * p.W - 1 - r) * U;
  return min(max(x - a, int64_t(0)), U) + min(max(x - b, int64_t(0)), U);
}

// Grid (B * H, kRwSplits).  Dynamic shared memory: the column bitmap, its
// word prefix counts and the W x W accumulator.
__global__ void __launch_bounds__(kRwThreads) ring_work_kernel(const RwParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint64_t* colw = reinterpret_cast<uint64_t*>(smem);
  int32_t* pre = reinterpret_cast<int32_t*>(colw + p.nwords);
  unsigned long long* acc = reinterpret_cast<unsigned long long*>(pre + ((p.nwords + 1 + 1) & ~1));
  __shared__ int bad;
  __shared__ int wsum[kRwThreads / 32];
  const int bh = blockIdx.x, split = blockIdx.y, tid = threadIdx.x;
  const int32_t* iv = p.iv + int64_t(bh) * p.kv;
  const int32_t* is = p.is + int64_t(bh) * p.ks;
  if (tid == 0) bad = 0;
  for (int i = tid; i < p.nwords; i += kRwThreads) colw[i] = 0ull;
  for (int i = tid; i < p.W * p.W; i += kRwThreads) acc[i] = 0ull;
  __syncthreads();
  // lists: ascending entries in [0, N), then only -1
  for (int i = tid; i < p.kv; i += kRwThreads) {
    const int x = iv[i];
    if (x < -1 || x >= p.N || (x >= 0 && i > 0 && !(iv[i - 1] >= 0 && iv[i - 1] < x))) bad = 1;
    else if (x >= 0) atomicOr(reinterpret_cast<unsigned long long*>(colw + (x >> 6)), 1ull << (x & 63));
  }
  for (int i = tid; i < p.ks; i += kRwThreads) {
    const int x = is[i];
    if (x < -1 || x >= p.N || (x >= 0 && i > 0 && !(is[i - 1] >= 0 && is[i - 1] < x))) bad = 1;
  }
  __syncthreads();
  if (bad) {
    if (tid == 0 && split == 0) atomicCAS(p.err, 0, int(VS_ERR_INDEX));
    return;
  }
  // exclusive prefix counts of the column words (chunk per thread, then a
  // scan of the thread totals)
  {
    const int per = (p.nwords + kRwThreads - 1) / kRwThreads;
    const int w0 = tid * per, w1 = min(p.nwords, w0 + per);
    int mine = 0;
    for (int w = w0; w < w1; ++w) mine += __popcll(colw[w]);
    const int lane = tid & 31, wp = tid >> 5;
    int v = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += y;
    }
    if (lane == 31) wsum[wp] = v;
    __syncthreads();
    if (tid < 32) {
      int t = tid < kRwThreads / 32 ? wsum[tid] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, t, off);
        if (tid >= off) t += y;
      }
      if (tid < kRwThreads / 32) wsum[tid] = t;
    }
    __syncthreads();
    int run = v - mine + (wp > 0 ? wsum[wp - 1] : 0);
    for (int w = w0; w < w1; ++w) {
      pre[w] = run;
      run += __popcll(colw[w]);
    }
    if (tid == kRwThreads - 1) pre[p.nwords] = run;
  }
  __syncthreads();
  auto cols_below = [&](int64_t x) -> int64_t {  // selected columns < x (0 <= x <= N)
    const int64_t w = x >> 6;
    if (w >= p.nwords) return pre[p.nwords];
    const int b = int(x & 63);
    return pre[w] + (b ? __popcll(colw[w] & ((1ull << b) - 1)) : 0);
  };
  const int W = p.W;
  // vertical: columns of this split
  for (int i = split * kRwThreads + tid; i < p.kv; i += kRwSplits * kRwThreads) {
    const int64_t m = iv[i];
    if (m < 0) break;
    const int q = owner_of(p, m);
    for (int r = 0; r < W; ++r) {
      const int64_t c = tokens_below(p, r, p.N) - tokens_below(p, r, m);
      if (c) atomicAdd(acc + r * W + q, static_cast<unsigned long long>(c));
    }
  }
  // slash: key segments of every offset; item = (offset, key block)
  const int64_t U = p.unit;
  const int64_t nkb = (p.N + U - 1) / U;  // key blocks
  const int64_t items = int64_t(p.ks) * nkb;
  for (int64_t it = int64_t(split) * kRwThreads + tid; it < items; it += int64_t(kRwSplits) * kRwThreads) {
    const int j = int(it / nkb);
    const int64_t kb = it - int64_t(j) * nkb;
    const int64_t o = is[j];
    if (o < 0) continue;
    const int64_t m_lo = kb * U, m_end = min(p.N - o, (kb + 1) * U);  // keys [m_lo, m_end)
    if (m_lo >= m_end) continue;
    const int q = owner_of(p, m_lo);
    // the queries n = m + o cross at most one query-block boundary
    const int64_t n_lo = m_lo + o, n_hi = m_end + o;  // [n_lo, n_hi)
    const int64_t cut = min(n_hi, (n_lo / U + 1) * U);
    const int64_t segs[3] = {n_lo, cut, n_hi};
#pragma unroll
    for (int sgi = 0; sgi < 2; ++sgi) {
      const int64_t a = segs[sgi], b = segs[sgi + 1];
      if (a >= b) continue;
      const int64_t cnt = (b - a) - (cols_below(b - o) - cols_below(a - o));
      if (cnt) atomicAdd(acc + owner_of(p, a) * W + q, static_cast<unsigned long long>(cnt));
    }
  }
  __syncthreads();
  for (int i = tid; i < W * W; i += kRwThreads)
    if (acc[i]) atomicAdd(p.out + i, acc[i]);
}

}  // namespace

size_t ring_work_smem(int64_t N, int W) {
  const int64_t nwords = (N + 63) / 64;
  return size_t(nwords * 8 + ((nwords + 2) & ~int64_t(1)) * 4 + int64_t(W) * W * 8);
}

vs_status launch_ring_work(int B, int H, int64_t N, const int32_t* v_idx, int kv, const int32_t* s_idx, int ks,
                           int world, int layout, int64_t* out, int* err, cudaStream_t st) {
  RwParams p;
  p.iv = v_idx;
  p.is = s_idx;
  p.kv = kv;
  p.ks = ks;
  p.N = N;
  p.W = world;
  p.zigzag = layout == 1;
  p.unit = layout == 1 ? N / (2 * world) : int64_t(kBlk);
  p.nwords = int((N + 63) / 64);
  p.out = reinterpret_cast<unsigned long long*>(out);
  p.err = err;
  const size_t sm = ring_work_smem(N, world);
  if (cudaFuncSetAttribute(ring_work_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm)) != cudaSuccess)
    return VS_ERR_CUDA;
  if (cudaMemsetAsync(out, 0, size_t(world) * world * sizeof(int64_t), st) != cudaSuccess) return VS_ERR_CUDA;
  trace_begin("ring_work", st);
  ring_work_kernel<<<dim3(unsigned(B * H), kRwSplits), kRwThreads, sm, st>>>(p);
  trace_end(st);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? VS_OK : VS_ERR_CUDA;
}

}  // namespace vs
