// Internal declarations shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include "vs_common.cuh"

namespace vs {

// Launch counter (all kernels launched by the library).
void note_launch(int n = 1);

// Tracing: brackets one kernel launch with CUDA events when tracing is on.
void trace_begin(const char* name, cudaStream_t st);
void trace_end(cudaStream_t st);

// Encodes a 4-D BSHD bf16 tensor map: dims {d, H, N, B}, box
// {64, box_heads, box_rows, 1} (rows land in smem in (token, head) order),
// 128-byte swizzle.  Returns VS_OK or VS_ERR_CUDA / VS_ERR_SHAPE.
vs_status make_tmap_bshd(CUtensorMap* m, const void* base, int B, int N, int H, int d, const int64_t s[3],
                         int box_rows, int box_heads = 1);

Geo make_geo(const vs_shape* s, const ArenaHeader& h);

// Host-side argument checks shared by the estimator entry points.
vs_status check_estimate_args(const vs_shape* s, const void* q, const void* k, int last_q, int kv, int ks,
                              float scale, const int32_t* v_idx, const int32_t* s_idx);

// Kernel launchers (one per translation unit).
vs_status launch_fwd(const vs_shape* s, const Geo& G, const void* q, const void* k, const void* v,
                     const void* arena, float scale, void* o, float* lse, float* o_acc, int* err,
                     cudaStream_t st);
vs_status launch_bwd(const vs_shape* s, const Geo& G, const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const void* dO, const void* arena, float scale, void* dq, void* dk, void* dv,
                     float* dq_acc, float* dkv_acc, void* ws, size_t ws_bytes, cudaStream_t st);
size_t bwd_workspace_bytes(const vs_shape* s, int kv);
vs_status launch_estimate(const vs_shape* s, const void* q, const void* k, int last_q, int kv, int ks, float scale,
                          int32_t* v_idx, int32_t* s_idx, float* v_score, float* s_score, void* ws, int shared,
                          cudaStream_t st);
size_t estimate_workspace_bytes(const vs_shape* s, int last_q);
vs_status launch_estimate_topp(const vs_shape* s, const void* q, const void* k, double pv, double ps, int kv_max,
                               int ks_max, float scale, int32_t* v_idx, int32_t* s_idx, int32_t* kv, int32_t* ks,
                               float* v_score, float* s_score, void* ws, cudaStream_t st);
vs_status launch_select_topp(int B, int H, int N, const float* v_score, const float* s_score, double pv, double ps,
                             int kv_max, int ks_max, int32_t* v_idx, int32_t* s_idx, int32_t* kv, int32_t* ks,
                             int* err, cudaStream_t st);
size_t topp_max_n();
size_t ring_work_smem(int64_t N, int W);
vs_status launch_ring_work(int B, int H, int64_t N, const int32_t* v_idx, int kv, const int32_t* s_idx, int ks,
                           int world, int layout, int64_t* out, int* err, cudaStream_t st);
vs_status launch_index(const vs_shape* s, const int32_t* v_idx, const int32_t* s_idx, int kv, int ks,
                       const vs_stripe* stripe, int flags, void* arena, size_t arena_bytes, cudaStream_t st);
size_t index_bytes(const vs_shape* s, int kv, int ks, const vs_stripe* stripe, ArenaHeader* hdr_out);
vs_status launch_permute(const void* x, void* y, int B, int64_t N, int H, int d, int world, int layout,
                         int inverse, int only_rank, cudaStream_t st);

}  // namespace vs
