// Token layouts of a context-parallel ring, as permutations of 64-token
// blocks (a block is one contiguous run of 64*H*d elements in the
// token-major layout, so the kernel streams 16-byte vectors and only remaps
// the block index):
//   striped (section 4.2 (ii)): global block j goes to worker j mod W at local
//     block j / W;
//   zigzag (section 2, Figure 1): the sequence is cut into 2W chunks of
//     N / (2W) tokens and worker r holds chunks r and 2W - 1 - r, in that
//     order (chunks of whole 64-token blocks).
#include "vs_internal.h"

namespace vs {
namespace {

struct PermParams {
  const uint4* x;
  uint4* y;
  int64_t B, N, W, vec_per_tok, total_vec;  // total over the written output
  int layout, inverse, only_rank;
};

// Global block of local block lb of worker r.
__device__ __forceinline__ int64_t global_block(const PermParams& p, int64_t r, int64_t lb) {
  if (p.layout == VS_LAYOUT_STRIPED) return lb * p.W + r;
  const int64_t cb = p.N / (2 * p.W * kBlk);  // blocks per chunk
  return lb < cb ? r * cb + lb : (2 * p.W - 1 - r) * cb + (lb - cb);
}

// Worker and local block of global block j.
__device__ __forceinline__ void owner_block(const PermParams& p, int64_t j, int64_t& r, int64_t& lb) {
  if (p.layout == VS_LAYOUT_STRIPED) {
    r = j % p.W;
    lb = j / p.W;
    return;
  }
  const int64_t cb = p.N / (2 * p.W * kBlk);
  const int64_t a = j / cb;
  r = a < p.W ? a : 2 * p.W - 1 - a;
  lb = (a < p.W ? 0 : cb) + (j - a * cb);
}

__global__ void __launch_bounds__(256) vs_permute_kernel(const PermParams p) {
  const int64_t nlb = p.N / p.W / kBlk;  // local blocks per worker
  const int64_t vpb = kBlk * p.vec_per_tok;  // vectors per 64-token block
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < p.total_vec;
       i += int64_t(gridDim.x) * blockDim.x) {
    if (!p.inverse) {
      // i indexes the output: [r][b][local block][vpb] (or one shard)
      const int64_t within = i % vpb;
      int64_t t = i / vpb;
      const int64_t lb = t % nlb;
      t /= nlb;
      const int64_t b = t % p.B;
      const int64_t r = (p.only_rank >= 0) ? p.only_rank : t / p.B;
      p.y[i] = p.x[(b * (p.N / kBlk) + global_block(p, r, lb)) * vpb + within];
    } else {
      // i indexes the output [b][global block][vpb]
      const int64_t within = i % vpb;
      const int64_t t = i / vpb;
      const int64_t j = t % (p.N / kBlk);
      const int64_t b = t / (p.N / kBlk);
      int64_t r, lb;
      owner_block(p, j, r, lb);
      p.y[i] = p.x[((r * p.B + b) * nlb + lb) * vpb + within];
    }
  }
}

}  // namespace

vs_status launch_permute(const void* x, void* y, int B, int64_t N, int H, int d, int world, int layout, int inverse,
                         int only_rank, cudaStream_t st) {
  PermParams p;
  p.x = static_cast<const uint4*>(x);
  p.y = static_cast<uint4*>(y);
  p.B = B;
  p.N = N;
  p.W = world;
  p.vec_per_tok = int64_t(H) * d / 8;
  p.layout = layout;
  p.inverse = inverse;
  p.only_rank = only_rank;
  const int64_t toks = (only_rank >= 0) ? N / world : N;
  p.total_vec = int64_t(B) * toks * p.vec_per_tok;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (p.total_vec + 255) / 256;
  const int grid = int(want < int64_t(sms) * 16 ? (want > 0 ? want : 1) : int64_t(sms) * 16);
  trace_begin(layout == VS_LAYOUT_STRIPED ? "striped_permute" : "zigzag_permute", st);
  vs_permute_kernel<<<grid, 256, 0, st>>>(p);
  trace_end(st);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? VS_OK : VS_ERR_CUDA;
}

}  // namespace vs
