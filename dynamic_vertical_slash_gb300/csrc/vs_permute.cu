// Block-level striping (section 4.2 (ii)): global 64-token block j of
// x [B, N, H, d] goes to shard j mod W at local block j / W.  A 64-token block
// is one contiguous run of 64*H*d elements in the token-major layout, so the
// kernel streams 16-byte vectors and only remaps the block index.
#include "vs_internal.h"

namespace vs {
namespace {

struct PermParams {
  const uint4* x;
  uint4* y;
  int64_t B, N, W, stripe, vec_per_tok, total_vec;  // total over the written output
  int inverse, only_rank;
};

__global__ void __launch_bounds__(256) vs_permute_kernel(const PermParams p) {
  const int64_t nloc = p.N / p.W;
  const int64_t vpb = p.stripe * p.vec_per_tok;  // vectors per 64-token block
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < p.total_vec;
       i += int64_t(gridDim.x) * blockDim.x) {
    if (!p.inverse) {
      // i indexes the output: [r][b][local block][vpb] (or one shard)
      const int64_t within = i % vpb;
      int64_t t = i / vpb;
      const int64_t lb = t % (nloc / p.stripe);
      t /= (nloc / p.stripe);
      const int64_t b = t % p.B;
      const int64_t r = (p.only_rank >= 0) ? p.only_rank : t / p.B;
      const int64_t j = lb * p.W + r;  // global block
      p.y[i] = p.x[(b * (p.N / p.stripe) + j) * vpb + within];
    } else {
      // i indexes the output [b][global block][vpb]
      const int64_t within = i % vpb;
      const int64_t t = i / vpb;
      const int64_t j = t % (p.N / p.stripe);
      const int64_t b = t / (p.N / p.stripe);
      const int64_t r = j % p.W, lb = j / p.W;
      p.y[i] = p.x[((r * p.B + b) * (nloc / p.stripe) + lb) * vpb + within];
    }
  }
}

}  // namespace

vs_status launch_permute(const void* x, void* y, int B, int64_t N, int H, int d, int world, int stripe, int inverse,
                         int only_rank, cudaStream_t st) {
  PermParams p;
  p.x = static_cast<const uint4*>(x);
  p.y = static_cast<uint4*>(y);
  p.B = B;
  p.N = N;
  p.W = world;
  p.stripe = stripe;
  p.vec_per_tok = int64_t(H) * d / 8;
  p.inverse = inverse;
  p.only_rank = only_rank;
  const int64_t toks = (only_rank >= 0) ? N / world : N;
  p.total_vec = int64_t(B) * toks * p.vec_per_tok;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (p.total_vec + 255) / 256;
  const int grid = int(want < int64_t(sms) * 16 ? (want > 0 ? want : 1) : int64_t(sms) * 16);
  trace_begin("striped_permute", st);
  vs_permute_kernel<<<grid, 256, 0, st>>>(p);
  trace_end(st);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? VS_OK : VS_ERR_CUDA;
}

}  // namespace vs
