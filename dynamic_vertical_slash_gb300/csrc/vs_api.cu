// Host side of the C ABI: argument validation, tensor-map encoding, status
// handling and dispatch to the kernels.
#include <atomic>
#include <cstring>
#include <string>
#include <vector>
#include "vs_internal.h"

namespace vs {

static std::atomic<int64_t> g_launches{0};
void note_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

// ------------------------------------------------------------------ tracing
struct TraceRec {
  const char* name;
  cudaEvent_t a, b;
};
static bool g_trace = false;
static std::vector<TraceRec> g_recs;
static cudaEvent_t g_open = nullptr;
static const char* g_open_name = nullptr;

void trace_begin(const char* name, cudaStream_t st) {
  if (!g_trace) return;
  if (cudaEventCreate(&g_open) != cudaSuccess) {
    g_open = nullptr;
    return;
  }
  g_open_name = name;
  cudaEventRecord(g_open, st);
}

void trace_end(cudaStream_t st) {
  if (!g_trace || !g_open) return;
  cudaEvent_t e;
  if (cudaEventCreate(&e) != cudaSuccess) return;
  cudaEventRecord(e, st);
  g_recs.push_back({g_open_name, g_open, e});
  g_open = nullptr;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

vs_status make_tmap_bshd(CUtensorMap* m, const void* base, int B, int N, int H, int d, const int64_t s[3],
                         int box_rows, int box_heads) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return VS_ERR_CUDA;
  cuuint64_t dims[4] = {cuuint64_t(d), cuuint64_t(H), cuuint64_t(N), cuuint64_t(B)};
  cuuint64_t strides[3] = {cuuint64_t(s[2]) * 2, cuuint64_t(s[1]) * 2, cuuint64_t(s[0]) * 2};
  cuuint32_t box[4] = {64, cuuint32_t(box_heads), cuuint32_t(box_rows), 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? VS_OK : VS_ERR_SHAPE;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static bool strides_ok(const int64_t s[3]) {
  for (int i = 0; i < 3; ++i)
    if (s[i] <= 0 || (s[i] % 8) != 0) return false;
  return true;
}

// Shape checks common to every attention entry point.
static vs_status check_shape(const vs_shape* s) {
  if (!s) return VS_ERR_ARG;
  if (s->B < 1 || s->Nq < 1 || s->Nk < 1 || s->Hq < 1 || s->Hkv < 1) return VS_ERR_SHAPE;
  if (s->d != 64 && s->d != 128) return VS_ERR_SHAPE;
  if (s->Hq % s->Hkv || s->Hq / s->Hkv > 64) return VS_ERR_SHAPE;
  if (s->Nq % kBlk || s->Nk % kBlk) return VS_ERR_SHAPE;
  if (int64_t(s->Nq) > (int64_t(1) << 30) || int64_t(s->Nk) > (int64_t(1) << 30)) return VS_ERR_SHAPE;
  if (!strides_ok(s->sq) || !strides_ok(s->sk) || !strides_ok(s->sv) || !strides_ok(s->so)) return VS_ERR_SHAPE;
  if (s->sq[2] < s->d || s->sk[2] < s->d || s->sv[2] < s->d || s->so[2] < s->d) return VS_ERR_SHAPE;
  return VS_OK;
}

// Argument checks of the estimator entry points (vs_estimate,
// vs_estimate_group, vs_estimate_noalloc), all on the host before any CUDA
// call: the shape checks of every entry point plus the estimator's own.
vs_status check_estimate_args(const vs_shape* s, const void* q, const void* k, int last_q, int kv, int ks,
                              float scale, const int32_t* v_idx, const int32_t* s_idx) {
  vs_status rc = check_shape(s);
  if (rc != VS_OK) return rc;
  if (!q || !k || !v_idx || !s_idx) return VS_ERR_ARG;
  if (s->Nq != s->Nk) return VS_ERR_SHAPE;
  if (last_q != 64) return VS_ERR_ARG;
  if (kv < 1 || ks < 1 || kv > s->Nk || ks > s->Nk) return VS_ERR_ARG;
  if (!(scale > 0.f)) return VS_ERR_ARG;
  if (!aligned16(q) || !aligned16(k)) return VS_ERR_SHAPE;
  return VS_OK;
}

}  // namespace vs

using namespace vs;

extern "C" {

const char* vs_status_string(vs_status st) {
  switch (st) {
    case VS_OK: return "VS_OK";
    case VS_ERR_ARG: return "VS_ERR_ARG: null pointer or bad scalar argument";
    case VS_ERR_SHAPE: return "VS_ERR_SHAPE: unsupported shape, stride or alignment";
    case VS_ERR_WORKSPACE: return "VS_ERR_WORKSPACE: workspace or index arena too small";
    case VS_ERR_INDEX: return "VS_ERR_INDEX: index list out of range, unsorted or duplicated";
    case VS_ERR_TIMEOUT: return "VS_ERR_TIMEOUT: a bounded device wait ran out";
    case VS_ERR_CUDA: return "VS_ERR_CUDA: CUDA runtime error";
    case VS_ERR_SCORE: return "VS_ERR_SCORE: a score is negative or not finite, or a list's total is too large";
  }
  return "unknown vs_status";
}

int64_t vs_launch_count(void) { return g_launches.load(); }

void vs_trace_enable(int on) { g_trace = on != 0; }

void vs_trace_reset(void) {
  for (auto& r : g_recs) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  g_recs.clear();
}

int vs_trace_report(char* names, int names_len, int64_t* counts, double* ms, int max_kernels) {
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  std::vector<std::string> keys;
  std::vector<int64_t> cnt;
  std::vector<double> tot;
  for (auto& r : g_recs) {
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return -1;
    size_t i = 0;
    while (i < keys.size() && keys[i] != r.name) ++i;
    if (i == keys.size()) {
      keys.push_back(r.name);
      cnt.push_back(0);
      tot.push_back(0.0);
    }
    cnt[i] += 1;
    tot[i] += t;
  }
  int pos = 0;
  for (size_t i = 0; i < keys.size() && int(i) < max_kernels; ++i) {
    if (counts) counts[i] = cnt[i];
    if (ms) ms[i] = tot[i];
    if (names) {
      const int len = int(keys[i].size()) + 1;
      if (pos + len <= names_len) {
        memcpy(names + pos, keys[i].c_str(), size_t(len));
        pos += len;
      }
    }
  }
  return int(keys.size());
}

vs_status vs_check_status(void* ws, cudaStream_t stream) {
  if (!ws) return VS_ERR_ARG;
  int32_t code = 0;
  if (cudaMemcpyAsync(&code, ws, sizeof(code), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return VS_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return VS_ERR_CUDA;
  if (code != 0) {
    const int32_t zero = 0;
    if (cudaMemcpyAsync(ws, &zero, sizeof(zero), cudaMemcpyHostToDevice, stream) != cudaSuccess) return VS_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return VS_ERR_CUDA;
  }
  return static_cast<vs_status>(code);
}

// ------------------------------------------------------------------ estimate
size_t vs_estimate_workspace(const vs_shape* s, int last_q) {
  if (!s) return 0;
  return estimate_workspace_bytes(s, last_q);
}

static vs_status estimate_any(const vs_shape* s, const void* q, const void* k, int last_q, int kv, int ks,
                              float scale, int32_t* v_idx, int32_t* s_idx, float* v_score, float* s_score, void* ws,
                              size_t ws_bytes, int shared, cudaStream_t stream);

vs_status vs_estimate(const vs_shape* s, const void* q, const void* k, int last_q, int kv, int ks, float scale,
                      int32_t* v_idx, int32_t* s_idx, float* v_score, float* s_score, void* ws, size_t ws_bytes,
                      cudaStream_t stream) {
  return estimate_any(s, q, k, last_q, kv, ks, scale, v_idx, s_idx, v_score, s_score, ws, ws_bytes, 0, stream);
}

vs_status vs_estimate_group(const vs_shape* s, const void* q, const void* k, int last_q, int kv, int ks, float scale,
                            int32_t* v_idx, int32_t* s_idx, float* v_score, float* s_score, void* ws,
                            size_t ws_bytes, cudaStream_t stream) {
  return estimate_any(s, q, k, last_q, kv, ks, scale, v_idx, s_idx, v_score, s_score, ws, ws_bytes, 1, stream);
}

static vs_status estimate_any(const vs_shape* s, const void* q, const void* k, int last_q, int kv, int ks,
                              float scale, int32_t* v_idx, int32_t* s_idx, float* v_score, float* s_score, void* ws,
                              size_t ws_bytes, int shared, cudaStream_t stream) {
  vs_status rc = check_estimate_args(s, q, k, last_q, kv, ks, scale, v_idx, s_idx);
  if (rc != VS_OK) return rc;
  if (!ws) return VS_ERR_ARG;
  if (ws_bytes < estimate_workspace_bytes(s, last_q)) return VS_ERR_WORKSPACE;
  return launch_estimate(s, q, k, last_q, kv, ks, scale, v_idx, s_idx, v_score, s_score, ws, shared, stream);
}

vs_status vs_estimate_topp(const vs_shape* s, const void* q, const void* k, int last_q, double pv, double ps,
                           int kv_max, int ks_max, float scale, int32_t* v_idx, int32_t* s_idx, int32_t* kv,
                           int32_t* ks, float* v_score, float* s_score, void* ws, size_t ws_bytes,
                           cudaStream_t stream) {
  vs_status rc = check_shape(s);
  if (rc != VS_OK) return rc;
  if (!q || !k || !v_idx || !s_idx || !kv || !ks || !ws) return VS_ERR_ARG;
  if (s->Nq != s->Nk || size_t(s->Nk) > topp_max_n()) return VS_ERR_SHAPE;
  if (last_q != 64) return VS_ERR_ARG;
  if (!(pv >= 0.0 && pv <= 1.0) || !(ps >= 0.0 && ps <= 1.0)) return VS_ERR_ARG;
  if (kv_max < 1 || ks_max < 1 || kv_max > s->Nk || ks_max > s->Nk) return VS_ERR_ARG;
  if (!(scale > 0.f)) return VS_ERR_ARG;
  if (!aligned16(q) || !aligned16(k)) return VS_ERR_SHAPE;
  if (ws_bytes < estimate_workspace_bytes(s, last_q)) return VS_ERR_WORKSPACE;
  return launch_estimate_topp(s, q, k, pv, ps, kv_max, ks_max, scale, v_idx, s_idx, kv, ks, v_score, s_score, ws,
                              stream);
}

vs_status vs_select_topp(int B, int H, int N, const float* v_score, const float* s_score, double pv, double ps,
                         int kv_max, int ks_max, int32_t* v_idx, int32_t* s_idx, int32_t* kv, int32_t* ks, void* ws,
                         size_t ws_bytes, cudaStream_t stream) {
  if (!v_score || !s_score || !v_idx || !s_idx || !kv || !ks || !ws) return VS_ERR_ARG;
  if (B < 1 || H < 1 || N < 64 || N % 64 || size_t(N) > topp_max_n()) return VS_ERR_SHAPE;
  if (int64_t(B) * H > (int64_t(1) << 31) - 1 || int64_t(B) * H > 65535 * 1024) return VS_ERR_SHAPE;
  if (!(pv >= 0.0 && pv <= 1.0) || !(ps >= 0.0 && ps <= 1.0)) return VS_ERR_ARG;
  if (kv_max < 1 || ks_max < 1 || kv_max > N || ks_max > N) return VS_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(v_score) | reinterpret_cast<uintptr_t>(s_score)) & 3u) return VS_ERR_SHAPE;
  if (ws_bytes < 256) return VS_ERR_WORKSPACE;
  return launch_select_topp(B, H, N, v_score, s_score, pv, ps, kv_max, ks_max, v_idx, s_idx, kv, ks,
                            static_cast<int*>(ws), stream);
}

// --------------------------------------------------------------------- index
size_t vs_block_index_bytes(const vs_shape* s, int kv, int ks, const vs_stripe* stripe) {
  if (check_shape(s) != VS_OK) return 0;
  return index_bytes(s, kv, ks, stripe, nullptr);
}

vs_status vs_build_block_index(const vs_shape* s, const int32_t* v_idx, const int32_t* s_idx, int kv, int ks,
                               const vs_stripe* stripe, void* arena, size_t arena_bytes, cudaStream_t stream) {
  return vs_build_block_index_ex(s, v_idx, s_idx, kv, ks, stripe, 0, arena, arena_bytes, stream);
}

vs_status vs_build_block_index_ex(const vs_shape* s, const int32_t* v_idx, const int32_t* s_idx, int kv, int ks,
                                  const vs_stripe* stripe, int flags, void* arena, size_t arena_bytes,
                                  cudaStream_t stream) {
  if (flags & ~int(VS_INDEX_BLOCK_COVER | VS_INDEX_PACK_GQA)) return VS_ERR_ARG;
  vs_status rc = check_shape(s);
  if (rc != VS_OK) return rc;
  if (flags & VS_INDEX_PACK_GQA) {
    // one head-packed tile is 128 / g tokens of the g heads of a KV group
    // (unstriped, exact token mask)
    const int g = s->Hq / s->Hkv;
    if (stripe || (flags & VS_INDEX_BLOCK_COVER)) return VS_ERR_ARG;
    if (g < 2 || kQTile % g) return VS_ERR_SHAPE;
  }
  if (!v_idx || !s_idx || !arena) return VS_ERR_ARG;
  if (stripe) {
    if (stripe->world < 1 || stripe->stripe != kBlk) return VS_ERR_ARG;
    if (stripe->q_rank < 0 || stripe->kv_rank < 0) return VS_ERR_ARG;
    if (s->Nq != s->Nk || stripe->N_global % kBlk || stripe->N_global > (int64_t(1) << 31) - 1) return VS_ERR_SHAPE;
    // every local block must map inside the global sequence
    const int64_t nbg = stripe->N_global / kBlk;
    if (int64_t(stripe->world) * (s->Nq / kBlk - 1) + stripe->q_rank >= nbg ||
        int64_t(stripe->world) * (s->Nk / kBlk - 1) + stripe->kv_rank >= nbg)
      return VS_ERR_SHAPE;
  } else if (s->Nq != s->Nk) {
    return VS_ERR_SHAPE;
  }
  const int64_t NG = stripe ? stripe->N_global : s->Nq;
  if (kv < 1 || ks < 1 || kv > NG || ks > NG) return VS_ERR_ARG;
  if (!aligned16(arena)) return VS_ERR_ARG;
  if (arena_bytes < index_bytes(s, kv, ks, stripe, nullptr)) return VS_ERR_WORKSPACE;
  return launch_index(s, v_idx, s_idx, kv, ks, stripe, flags, arena, arena_bytes, stream);
}

vs_status vs_index_counts(const void* arena, int64_t* out, cudaStream_t stream) {
  if (!arena || !out) return VS_ERR_ARG;
  ArenaHeader h;
  if (cudaMemcpyAsync(&h, arena, sizeof(h), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return VS_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return VS_ERR_CUDA;
  if (h.magic != kArenaMagic) return VS_ERR_ARG;
  const size_t n = size_t(h.B) * h.Hq * 4;
  if (cudaMemcpyAsync(out, static_cast<const uint8_t*>(arena) + h.off_counts, n * sizeof(int64_t),
                      cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return VS_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return VS_ERR_CUDA;
  return VS_OK;
}

// ----------------------------------------------------------------- attention
size_t vs_attn_fwd_workspace(const vs_shape*) { return 256; }

vs_status vs_attn_fwd(const vs_shape* s, const void* q, const void* k, const void* v, const void* arena, float scale,
                      void* o, float* lse, float* o_acc, void* ws, size_t ws_bytes, cudaStream_t stream) {
  vs_status rc = check_shape(s);
  if (rc != VS_OK) return rc;
  if (!q || !k || !v || !arena || !o || !lse || !ws) return VS_ERR_ARG;
  if (!(scale > 0.f)) return VS_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(arena) ||
      (o_acc && !aligned16(o_acc)))
    return VS_ERR_SHAPE;
  if (ws_bytes < 256) return VS_ERR_WORKSPACE;
  Geo G{};
  return launch_fwd(s, G, q, k, v, arena, scale, o, lse, o_acc, static_cast<int*>(ws), stream);
}

size_t vs_attn_bwd_workspace(const vs_shape* s, int kv) {
  if (check_shape(s) != VS_OK) return 0;
  return bwd_workspace_bytes(s, kv);
}

vs_status vs_attn_bwd(const vs_shape* s, const void* q, const void* k, const void* v, const void* o, const float* lse,
                      const void* dO, const void* arena, float scale, void* dq, void* dk, void* dv, float* dq_acc,
                      void* ws, size_t ws_bytes, cudaStream_t stream) {
  return vs_attn_bwd_ex(s, q, k, v, o, lse, dO, arena, scale, dq, dk, dv, dq_acc, nullptr, ws, ws_bytes, stream);
}

vs_status vs_attn_bwd_ex(const vs_shape* s, const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dO, const void* arena, float scale, void* dq, void* dk,
                         void* dv, float* dq_acc, float* dkv_acc, void* ws, size_t ws_bytes, cudaStream_t stream) {
  vs_status rc = check_shape(s);
  if (rc != VS_OK) return rc;
  if (!q || !k || !v || !o || !lse || !dO || !arena || !dq || !dk || !dv || !ws) return VS_ERR_ARG;
  if (!(scale > 0.f)) return VS_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || !aligned16(arena) || (dq_acc && !aligned16(dq_acc)) ||
      (dkv_acc && !aligned16(dkv_acc)))
    return VS_ERR_SHAPE;
  if (ws_bytes < bwd_workspace_bytes(s, 1)) return VS_ERR_WORKSPACE;
  // The bar-partial region grows with kv, which the arena header holds on the
  // device; the kernels compare it with ws_bytes and record VS_ERR_WORKSPACE.
  Geo G{};
  return launch_bwd(s, G, q, k, v, o, lse, dO, arena, scale, dq, dk, dv, dq_acc, dkv_acc, ws, ws_bytes, stream);
}

vs_status vs_ring_work(int B, int H, int64_t N, const int32_t* v_idx, int kv, const int32_t* s_idx, int ks,
                       int world, int layout, int64_t* out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!v_idx || !s_idx || !out || !ws) return VS_ERR_ARG;
  if (B < 1 || H < 1 || N < 1 || N > (int64_t(1) << 31) - 1 || world < 1 || world > 64) return VS_ERR_SHAPE;
  if (layout != VS_LAYOUT_STRIPED && layout != VS_LAYOUT_ZIGZAG) return VS_ERR_ARG;
  if (layout == VS_LAYOUT_STRIPED && N % (int64_t(kBlk) * world)) return VS_ERR_SHAPE;
  if (layout == VS_LAYOUT_ZIGZAG && N % (2 * int64_t(world))) return VS_ERR_SHAPE;
  if (kv < 1 || ks < 1) return VS_ERR_ARG;
  if (int64_t(B) * H > 65535) return VS_ERR_SHAPE;
  if (ring_work_smem(N, world) > size_t(200) << 10) return VS_ERR_SHAPE;
  if (ws_bytes < 256) return VS_ERR_WORKSPACE;
  return launch_ring_work(B, H, N, v_idx, kv, s_idx, ks, world, layout, out, static_cast<int*>(ws), stream);
}

vs_status striped_permute(const void* x, void* y, int B, int64_t N, int H, int d, int world, int stripe, int inverse,
                          int only_rank, cudaStream_t stream) {
  if (!x || !y) return VS_ERR_ARG;
  if (B < 1 || N < 1 || H < 1 || (d != 64 && d != 128) || world < 1 || stripe != kBlk) return VS_ERR_SHAPE;
  if (N % (int64_t(world) * stripe)) return VS_ERR_SHAPE;
  if (only_rank < -1 || only_rank >= world) return VS_ERR_ARG;
  if (inverse && only_rank != -1) return VS_ERR_ARG;
  if (!aligned16(x) || !aligned16(y)) return VS_ERR_SHAPE;
  return launch_permute(x, y, B, N, H, d, world, VS_LAYOUT_STRIPED, inverse, only_rank, stream);
}

vs_status vs_ring_permute(const void* x, void* y, int B, int64_t N, int H, int d, int world, int layout, int inverse,
                          int only_rank, cudaStream_t stream) {
  if (!x || !y) return VS_ERR_ARG;
  if (layout != VS_LAYOUT_STRIPED && layout != VS_LAYOUT_ZIGZAG) return VS_ERR_ARG;
  if (B < 1 || N < 1 || H < 1 || (d != 64 && d != 128) || world < 1) return VS_ERR_SHAPE;
  if (N % (int64_t(world) * kBlk * (layout == VS_LAYOUT_ZIGZAG ? 2 : 1))) return VS_ERR_SHAPE;
  if (only_rank < -1 || only_rank >= world) return VS_ERR_ARG;
  if (inverse && only_rank != -1) return VS_ERR_ARG;
  if (!aligned16(x) || !aligned16(y)) return VS_ERR_SHAPE;
  return launch_permute(x, y, B, N, H, d, world, layout, inverse, only_rank, stream);
}

}  // extern "C"
