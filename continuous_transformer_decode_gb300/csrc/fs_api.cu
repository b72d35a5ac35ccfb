// Host side of the C ABI (include/fs.h): descriptor validation, weight
// upload and re-layout, the paged KV arena and its page allocator, and the
// orchestration of one decode_step_batch call as a sequence of kernels on
// the handle's stream.
//
// The step follows "Fat-station continuous batching" ("The capture"): the
// caller passes, per lane, its position and the token it consumes; the call
// appends that token's K/V to the lane's cache, returns its logits and
// advances the position. Validation and page allocation happen before any
// launch, so an invalid call changes nothing.

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <map>
#include <set>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/fs.h"
#include "fs_internal.h"

using namespace fsk;

namespace {

thread_local std::string g_create_error;

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// tcgen05 operand map and the fixed K split of one weight matrix.
struct TcW {
  int m_tiles = 0, P = 1;  // row tiles, stream-K width
  int8_t* q8_tiles = nullptr;  // Q8_0 tiles (see launch_tile_q8)
  // bf16 copy of a Q8_0 matrix, bf16(q * d) (see launch_dequant_q8_bf16):
  // kept where the handle's lane capacity splits the matrix's Q8_0 GEMM into
  // at least q8_copy_groups lane groups
  __nv_bfloat16* q8_bf16 = nullptr;
};

struct LayerW {
  Mat qkv, o, gateup, down;
  TcW qkv_tc, o_tc, gateup_tc, down_tc;
  float* g_attn = nullptr;
  float* g_ffn = nullptr;
};

// Stream-K width P of a weight matrix (blocks per lane group), from event
// timings of this kernel on the decode step's matrix shapes at 1, 32 and 128
// lanes:
//  * at least as many 128-row tiles as SMs: one whole tile per block
//    (P = m_tiles), no partial sums;
//  * lane capacity <= 8 and at least 4 k-blocks per block at P = 2 x SMs:
//    P = 2 x SMs, ranges crossing tile boundaries (partials are tiny);
//  * otherwise s equal K splits of every tile, P = m_tiles * s: about
//    1.3 x SMs blocks with splits of >= 8 k-blocks up to 32 lanes, about
//    0.85 x SMs blocks with splits of >= 32 k-blocks beyond (lane groups then
//    bring the launch to about two blocks per SM), s <= 8.
// P depends on the matrix, the handle's lane capacity and the device only,
// never on a call's lane count.
// Kernel timeline tracing is process-wide (a device pointer in every kernel
// translation unit); one handle at a time owns the buffer.
TraceBuf* g_trace_buf = nullptr;
int64_t g_trace_cap = 0;
const fs_handle* g_trace_owner = nullptr;

bool trace_install_all(TraceBuf* b) {
  return trace_install_misc(b) && trace_install_gemm(b) && trace_install_gemv(b) &&
         trace_install_attn(b) && trace_install_attn_mma(b) && trace_install_attn_tma(b) &&
         trace_install_attn_warp(b) &&
         trace_install_attn_tiled(b);
}

// Uninstalls and frees the trace buffer if h owns it (the stream has been
// synchronised by the caller).
int trace_release(const fs_handle* h) {
  if (g_trace_owner != h) return FS_OK;
  const bool ok = trace_install_all(nullptr);
  cudaFree(g_trace_buf);
  g_trace_buf = nullptr;
  g_trace_cap = 0;
  g_trace_owner = nullptr;
  return ok ? FS_OK : FS_ERR_CUDA;
}

int choose_width(int m_tiles, int kb_total, int max_lanes, int sms) {
  const int64_t T = (int64_t)m_tiles * kb_total;
  if (m_tiles >= sms) return m_tiles;
  // FS_TC_SPLIT_KB=r (a tuning knob, read once): matrices with fewer row
  // tiles than SMs take ceil(kb_total / r) equal K splits of every tile
  static const int split_kb = [] {
    const char* e = getenv("FS_TC_SPLIT_KB");
    return e ? std::max(0, atoi(e)) : 0;
  }();
  if (split_kb > 0) return m_tiles * std::min(kb_total, (kb_total + split_kb - 1) / split_kb);
  // small handles, large matrices: about two blocks per SM, a whole number
  // of splits per row tile so that no block's range crosses a tile
  if (max_lanes <= 8 && T >= (int64_t)8 * sms)
    return m_tiles * std::max(1, std::min(kb_total, 2 * sms / m_tiles));
  const bool narrow = max_lanes <= 32;
  int s = narrow ? (13 * sms + 5 * m_tiles) / (10 * m_tiles) : (85 * sms) / (100 * m_tiles);
  // short K (fewer than 32 k-blocks, e.g. a 576- or 1536-wide input): no
  // splits, as the multi-k-block stages bring a whole tile's K in two or
  // three copies and a cluster reduction would cost more (SmolLM2 bf16, ms
  // per step on handles of 1 / 4 / 16 / 64 lanes: 0.929 / 0.968 / 1.000 /
  // 1.175 with splits of 3 k-blocks, 0.887 / 0.886 / 0.903 / 0.921
  // without); long K: splits of at least 32 k-blocks (8 on handles of at
  // most 32 lanes)
  const int cap = kb_total < 32 ? 1 : kb_total / (narrow ? 8 : 32);
  s = std::min(s, std::min(8, cap));
  return m_tiles * std::max(1, s);
}

// FS_Q8_BF16_GROUPS (read at create): the lane-group count from which a Q8_0
// GEMM call multiplies the matrix's bf16 copy (default 2; 0: no copies).
int q8_copy_groups_env() {
  const char* e = getenv("FS_Q8_BF16_GROUPS");
  return e ? std::max(0, atoi(e)) : 2;
}

// Every lane group of a Q8_0 GEMM dequantises each weight tile it
// multiplies, so a call of g groups converts the matrix g times. A Q8_0
// handle of B lanes keeps a bf16 copy of a matrix of stream-K width P when a
// call of all B lanes would run copy_groups or more Q8_0 lane groups.
bool q8_keeps_copy(int B, int P, int sms, int copy_groups) {
  int lg = 0, groups = 1;
  tc_lane_groups(B, P, sms, &lg, &groups, 32);
  return copy_groups > 0 && groups >= copy_groups;
}

// Lane groups of one GEMM call of n lanes. Q8_0 groups take at least 32
// lanes; a Q8_0 call that would run copy_groups or more of them multiplies
// the matrix's bf16 copy when it has one (*use_copy) and is then grouped as a
// bf16 call (the same operand bits either way).
void gemm_call_groups(int n, int P, int sms, bool q8, bool has_copy, int copy_groups, int* lg,
                      int* groups, bool* use_copy) {
  tc_lane_groups(n, P, sms, lg, groups, q8 ? 32 : 16);
  *use_copy = q8 && has_copy && *groups >= copy_groups;
  if (*use_copy) tc_lane_groups(n, P, sms, lg, groups, 16);
}
}  // namespace

struct fs_handle {
  fs_model_desc d{};
  int wtype = W_BF16;
  int xtype = X_BF16;
  int Kp_d = 0, Kp_q = 0, Kp_f = 0;
  int Nq = 0, Nkv = 0, Nqkv = 0;
  int G = 1;
  int sms = 1;  // SMs of the handle's device
  int split_len = 256, max_splits = 1;
  int max_pages_per_lane = 0;

  std::vector<LayerW> layers;
  Mat embed, head;
  TcW head_tc;
  bool use_tc = false;
  int act_split = 0;
  // Q8_0: a GEMM call whose lane groups would number at least this many
  // multiplies the matrix's bf16 copy instead (0: no copies)
  int q8_copy_groups = 2;
  bool map_fail = false;  // a GEMM launch could not encode its tensor maps
  int64_t lo_h = 0, lo_o = 0, lo_a = 0;  // remainder offsets (elements; 0: none)
  float* ws = nullptr;
  int* counters = nullptr;
  int* err_flag = nullptr;  // mapped pinned host memory
  int* d_err_flag = nullptr;
  float* g_final = nullptr;
  std::vector<void*> allocs;  // every cudaMalloc of the handle

  KV kv;
  std::vector<std::vector<int32_t>> pt;  // host page tables
  std::vector<int32_t> len;              // lane lengths
  std::set<int32_t> free_pages;
  std::vector<int32_t> page_ref;     // lanes holding each page (0: free)
  int32_t* d_reloc_pt = nullptr;     // [max_pages_per_lane]: a table before a move

  float* rope_cos = nullptr;
  float* rope_sin = nullptr;

  float* x = nullptr;
  float* y = nullptr;  // projection output added to x by the next norm
  void* hpanel = nullptr;
  void* opanel = nullptr;
  void* apanel = nullptr;
  float* qkv = nullptr;
  float* q = nullptr;
  float* logits = nullptr;
  float* part_ml = nullptr;
  float* part_acc = nullptr;
  int* attn_counters = nullptr;  // [max_lanes * Hkv], zero between steps
  bool attn_tiled = false;
  bool attn_mma = false;
  bool attn_tma = false;         // KV tiles by TMA (k_attn_tma.cu)
  // one warp per (lane, KV head) on handles of <= 64 positions, for calls of
  // at least attn_warp_rows rows (the cp.async kernel serves smaller calls)
  bool attn_warp = false;
  int attn_warp_rows = 0;
  CUtensorMap tm_kv_k, tm_kv_v;  // KV arenas as [rows][hd] bf16 for that kernel

  int32_t* d_args = nullptr;  // [7 * max_lanes + 1]
  int32_t* h_args = nullptr;  // pinned staging
  StepArgs args{};
  cudaEvent_t args_done = nullptr;

  float* d_temps = nullptr;
  uint64_t* d_seeds = nullptr;
  uint64_t* d_counters = nullptr;
  int32_t* d_tokens = nullptr;
  // greedy steps: tile maxima of the LM head's argmax epilogue, the step's
  // tokens, and zero temperatures / seeds / counters for the sampler fallback
  bool greedy_fused = false;
  float* am_val = nullptr;
  int* am_idx = nullptr;
  int32_t* d_greedy = nullptr;
  float* d_zero_temps = nullptr;
  uint64_t* d_zero_u64 = nullptr;
  unsigned char* h_samp = nullptr;  // pinned staging for sampler I/O

  cudaStream_t own_stream = nullptr;
  cudaStream_t stream = nullptr;

  int last_n = -1;
  const float* last_logits = nullptr;
  // one CUDA graph per lane count n (steps whose logits stay internal)
  struct Graph {
    cudaGraphExec_t exec = nullptr;
    int64_t kernels = 0;
  };
  std::map<int, Graph> graphs;
  bool graphs_on = true;
  int64_t launches = 0;
  std::string err;

  // event profiler (fs_profile_enable / fs_profile_read)
  struct ProfRec {
    int cls;
    cudaEvent_t a, b;
    double bytes;
  };
  bool prof_on = false;
  std::vector<ProfRec> prof_pending;
  std::vector<cudaEvent_t> prof_pool;
  double prof_ms[FS_PROF_CLASSES] = {0, 0, 0};
  double prof_bytes[FS_PROF_CLASSES] = {0, 0, 0};
  int64_t prof_n[FS_PROF_CLASSES] = {0, 0, 0};

  cudaEvent_t prof_event() {
    if (!prof_pool.empty()) {
      cudaEvent_t e = prof_pool.back();
      prof_pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
  // Launches through `fn` (returns the kernel count) with optional timing.
  template <typename Fn>
  void launch(int cls, double bytes, Fn fn) {
    if (!prof_on) {
      launches += fn();
      return;
    }
    cudaEvent_t a = prof_event(), b = prof_event();
    cudaEventRecord(a, stream);
    launches += fn();
    cudaEventRecord(b, stream);
    prof_pending.push_back({cls, a, b, bytes});
  }

  int fail(int code, const std::string& msg) {
    err = msg;
    return code;
  }
  int cuda_fail(cudaError_t e, const char* what) {
    err = std::string(what) + ": " + cudaGetErrorString(e);
    return FS_ERR_CUDA;
  }
  void release(void* p) {
    for (size_t i = 0; i < allocs.size(); ++i)
      if (allocs[i] == p) {
        cudaFree(p);
        allocs.erase(allocs.begin() + i);
        return;
      }
  }
  template <typename T>
  cudaError_t alloc(T** p, size_t bytes) {
    void* v = nullptr;
    cudaError_t e = cudaMalloc(&v, bytes ? bytes : 16);
    if (e == cudaSuccess) {
      allocs.push_back(v);
      *p = static_cast<T*>(v);
    }
    return e;
  }
};

#define FS_CK(h, call)                                   \
  do {                                                   \
    cudaError_t e_ = (call);                             \
    if (e_ != cudaSuccess) return (h)->cuda_fail(e_, #call); \
  } while (0)

namespace {

size_t elem_bytes(int wtype) { return wtype == W_F32 ? 4 : (wtype == W_BF16 ? 2 : 1); }

// Allocates a device matrix of N rows in the library layout.
int alloc_mat(fs_handle* h, Mat* m, int N, int K) {
  m->N = N;
  m->K = K;
  m->Kp = (int)round_up(K, 64);
  m->wtype = h->wtype;
  void* w = nullptr;
  const size_t bytes = (size_t)N * m->Kp * elem_bytes(h->wtype);
  if (h->alloc(&w, bytes) != cudaSuccess)
    return h->fail(FS_ERR_OOM, "weight allocation failed");
  FS_CK(h, cudaMemset(w, 0, bytes));
  m->w = w;
  if (h->wtype == W_Q8) {
    __half* s = nullptr;
    const size_t sb = (size_t)N * (m->Kp / 32) * sizeof(__half);
    if (h->alloc(&s, sb) != cudaSuccess)
      return h->fail(FS_ERR_OOM, "scale allocation failed");
    FS_CK(h, cudaMemset(s, 0, sb));
    m->scales = s;
  }
  return FS_OK;
}

// Copies a [rows, cols] source matrix (host or device, caller layout) into
// rows [row_offset, row_offset + rows) of m.
int upload_rows(fs_handle* h, Mat* m, const void* src, int rows, int cols,
                int row_offset, uint8_t* staging) {
  if (!src) return h->fail(FS_ERR_ARG, "missing weight pointer");
  if (h->wtype == W_Q8) {
    const size_t bytes = (size_t)rows * (cols / 32) * 34;
    FS_CK(h, cudaMemcpy(staging, src, bytes, cudaMemcpyDefault));
    h->launches += launch_repack_q8(staging, rows, cols, m->Kp,
                                    (int8_t*)m->w, (__half*)m->scales,
                                    row_offset, h->stream);
    FS_CK(h, cudaGetLastError());
    FS_CK(h, cudaStreamSynchronize(h->stream));
    return FS_OK;
  }
  const size_t es = elem_bytes(h->wtype);
  char* dst = (char*)m->w + (size_t)row_offset * m->Kp * es;
  FS_CK(h, cudaMemcpy2D(dst, (size_t)m->Kp * es, src, (size_t)cols * es,
                        (size_t)cols * es, rows, cudaMemcpyDefault));
  return FS_OK;
}

int validate_desc(const fs_model_desc* d, std::string* why) {
  auto bad = [&](const char* m) {
    *why = m;
    return FS_ERR_ARG;
  };
  if (d->n_layers < 1 || d->d_model < 1 || d->n_heads < 1 ||
      d->n_kv_heads < 1 || d->head_dim < 2 || d->d_ffn < 1 || d->vocab < 1)
    return bad("model dimensions must be positive");
  if (d->n_heads % d->n_kv_heads) return bad("n_heads must be a multiple of n_kv_heads");
  if (d->n_heads / d->n_kv_heads > 8) return bad("at most 8 query heads per KV head");
  if (d->head_dim % 2 || d->head_dim > 256) return bad("head_dim must be even and <= 256");
  if (d->weight_dtype < 0 || d->weight_dtype > 2) return bad("unknown weight_dtype");
  if (d->kv_dtype != FS_DTYPE_F32 && d->kv_dtype != FS_DTYPE_BF16)
    return bad("kv_dtype must be F32 or BF16");
  if (d->weight_dtype == FS_DTYPE_Q8_0 &&
      (d->d_model % 32 || d->d_ffn % 32 || (d->n_heads * d->head_dim) % 32))
    return bad("Q8_0 needs every input width to be a multiple of 32");
  if (d->max_lanes < 1 || d->page_size < 1 || d->n_pages < 1 || d->max_pos < 1)
    return bad("max_lanes, page_size, n_pages and max_pos must be positive");
  if (!(d->rms_eps >= 0.0f) || !(d->rope_theta > 0.0)) return bad("bad rms_eps or rope_theta");
  if (d->d_model > 8192 || d->d_model % 4) return bad("d_model must be a multiple of 4, <= 8192");
  return FS_OK;
}

int create_impl(fs_handle* h, const fs_weights* W) {
  const fs_model_desc& d = h->d;
  h->wtype = d.weight_dtype == FS_DTYPE_F32 ? W_F32
             : d.weight_dtype == FS_DTYPE_BF16 ? W_BF16 : W_Q8;
  h->xtype = h->wtype == W_F32 ? X_F32 : X_BF16;
  h->Nq = d.n_heads * d.head_dim;
  h->Nkv = d.n_kv_heads * d.head_dim;
  h->Nqkv = h->Nq + 2 * h->Nkv;
  h->G = d.n_heads / d.n_kv_heads;
  h->Kp_d = (int)round_up(d.d_model, 64);
  h->Kp_q = (int)round_up(h->Nq, 64);
  h->Kp_f = (int)round_up(d.d_ffn, 64);
  {
    int dev = 0;
    FS_CK(h, cudaGetDevice(&dev));
    FS_CK(h, cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, dev));
  }
  // attention split length: a handle constant (it fixes the merge order).
  // Long splits amortise each block's fixed cost (page indices, q rotation,
  // the first copies' latency, merges); the longest of 1024 / 512 / 256 whose
  // (lane, KV head, split) blocks of a full handle still number three per SM
  // is taken, else 128 for the parallelism (measured on the Mistral-7B shape,
  // contexts U[128, 4096]: B = 8 is fastest at 512, B = 32 and up at 1024,
  // B = 1 at 128).
  {
    auto blocks = [&](int len) {
      return (int64_t)d.max_lanes * d.n_kv_heads * ((d.max_pos + len - 1) / len);
    };
    const int64_t want = 3 * (int64_t)h->sms;
    h->split_len = !attn_tiled_supports(d.head_dim, d.n_heads / d.n_kv_heads, d.page_size, 128)
                       ? 256
                   : blocks(1024) >= want ? 1024
                   : blocks(512) >= want  ? 512
                   : blocks(256) >= want  ? 256
                                          : 128;
    // FS_SPLIT_LEN=128|256|512|1024 overrides the rule (a tuning knob)
    const char* e = getenv("FS_SPLIT_LEN");
    const int v = e ? atoi(e) : 0;
    if ((v == 128 || v == 256 || v == 512 || v == 1024) && h->split_len != 256) h->split_len = v;
  }
  h->max_splits = (d.max_pos + h->split_len - 1) / h->split_len;
  h->max_pages_per_lane = (d.max_pos + d.page_size - 1) / d.page_size;
  {
    h->use_tc = (h->wtype == W_BF16 || h->wtype == W_Q8) && d.d_ffn % 64 == 0 &&
                tc_available();
    if (d.act_split != 0 && d.act_split != 1) return h->fail(FS_ERR_ARG, "act_split must be 0 or 1");
    if (d.act_split && !h->use_tc)
      return h->fail(FS_ERR_ARG, "act_split needs the tensor-core path (bf16 or Q8_0 weights, "
                                 "d_ffn a multiple of 64)");
    h->act_split = d.act_split;
    const char* genv = getenv("FS_GRAPHS");
    h->graphs_on = !(genv && std::string(genv) == "0");
    h->q8_copy_groups = q8_copy_groups_env();
  }

  FS_CK(h, cudaStreamCreateWithFlags(&h->own_stream, cudaStreamDefault));
  h->stream = h->own_stream;
  FS_CK(h, cudaEventCreateWithFlags(&h->args_done, cudaEventDisableTiming));

  // ---- weights
  size_t stage = 0;
  if (h->wtype == W_Q8) {
    auto blk = [](int64_t r, int64_t c) { return (size_t)(r * (c / 32) * 34); };
    stage = std::max({blk(d.vocab, d.d_model), blk(d.d_ffn, d.d_model),
                      blk(d.d_model, d.d_ffn), blk(h->Nq, d.d_model),
                      blk(d.d_model, h->Nq)});
  }
  uint8_t* staging = nullptr;
  if (stage) {
    if (cudaMalloc(&staging, stage) != cudaSuccess)
      return h->fail(FS_ERR_OOM, "staging allocation failed");
  }
  struct StageFree {
    uint8_t* p;
    ~StageFree() { if (p) cudaFree(p); }
  } sf{staging};

  if (!W || !W->embed || !W->final_norm || !W->layers)
    return h->fail(FS_ERR_ARG, "missing weights");
  if (!d.tied_embeddings && !W->lm_head)
    return h->fail(FS_ERR_ARG, "lm_head is NULL but tied_embeddings == 0");
  int rc;
  if ((rc = alloc_mat(h, &h->embed, d.vocab, d.d_model))) return rc;
  if ((rc = upload_rows(h, &h->embed, W->embed, d.vocab, d.d_model, 0, staging))) return rc;
  if (d.tied_embeddings) {
    h->head = h->embed;
  } else {
    if ((rc = alloc_mat(h, &h->head, d.vocab, d.d_model))) return rc;
    if ((rc = upload_rows(h, &h->head, W->lm_head, d.vocab, d.d_model, 0, staging))) return rc;
  }
  auto upload_vec = [&](float** dst, const float* src, int n) -> int {
    if (!src) return h->fail(FS_ERR_ARG, "missing norm gain");
    if (h->alloc(dst, (size_t)n * 4) != cudaSuccess)
      return h->fail(FS_ERR_OOM, "norm allocation failed");
    FS_CK(h, cudaMemcpy(*dst, src, (size_t)n * 4, cudaMemcpyDefault));
    return FS_OK;
  };
  if ((rc = upload_vec(&h->g_final, W->final_norm, d.d_model))) return rc;
  h->layers.resize(d.n_layers);
  for (int l = 0; l < d.n_layers; ++l) {
    const fs_layer_weights& s = W->layers[l];
    LayerW& L = h->layers[l];
    if ((rc = alloc_mat(h, &L.qkv, h->Nqkv, d.d_model))) return rc;
    if ((rc = upload_rows(h, &L.qkv, s.wq, h->Nq, d.d_model, 0, staging))) return rc;
    if ((rc = upload_rows(h, &L.qkv, s.wk, h->Nkv, d.d_model, h->Nq, staging))) return rc;
    if ((rc = upload_rows(h, &L.qkv, s.wv, h->Nkv, d.d_model, h->Nq + h->Nkv, staging))) return rc;
    if ((rc = alloc_mat(h, &L.o, d.d_model, h->Nq))) return rc;
    if ((rc = upload_rows(h, &L.o, s.wo, d.d_model, h->Nq, 0, staging))) return rc;
    if ((rc = alloc_mat(h, &L.gateup, 2 * d.d_ffn, d.d_model))) return rc;
    if (h->use_tc) {
      // 128-row tiles of 64 gate rows then the 64 matching up rows
      const size_t rb = h->wtype == W_Q8 ? (size_t)d.d_model / 32 * 34
                                         : (size_t)d.d_model * elem_bytes(h->wtype);
      for (int t = 0; t < d.d_ffn / 64; ++t) {
        if ((rc = upload_rows(h, &L.gateup, (const char*)s.w_gate + (size_t)t * 64 * rb, 64,
                              d.d_model, 128 * t, staging)))
          return rc;
        if ((rc = upload_rows(h, &L.gateup, (const char*)s.w_up + (size_t)t * 64 * rb, 64,
                              d.d_model, 128 * t + 64, staging)))
          return rc;
      }
    } else {
      if ((rc = upload_rows(h, &L.gateup, s.w_gate, d.d_ffn, d.d_model, 0, staging))) return rc;
      if ((rc = upload_rows(h, &L.gateup, s.w_up, d.d_ffn, d.d_model, d.d_ffn, staging)))
        return rc;
    }
    if ((rc = alloc_mat(h, &L.down, d.d_model, d.d_ffn))) return rc;
    if ((rc = upload_rows(h, &L.down, s.w_down, d.d_model, d.d_ffn, 0, staging))) return rc;
    if ((rc = upload_vec(&L.g_attn, s.attn_norm, d.d_model))) return rc;
    if ((rc = upload_vec(&L.g_ffn, s.ffn_norm, d.d_model))) return rc;
  }

  // ---- KV arena
  KV& kv = h->kv;
  kv.kv_f32 = d.kv_dtype == FS_DTYPE_F32;
  kv.Hkv = d.n_kv_heads;
  kv.hd = d.head_dim;
  kv.page_size = d.page_size;
  kv.max_pages = h->max_pages_per_lane;
  kv.layer_stride = (int64_t)d.n_pages * kv.Hkv * kv.page_size * kv.hd;
  const size_t kv_bytes = (size_t)d.n_layers * kv.layer_stride * (kv.kv_f32 ? 4 : 2);
  if (h->alloc(&kv.k, kv_bytes) != cudaSuccess || h->alloc(&kv.v, kv_bytes) != cudaSuccess)
    return h->fail(FS_ERR_OOM, "KV arena allocation failed");
  if (h->alloc(&kv.pt, (size_t)d.max_lanes * kv.max_pages * 4) != cudaSuccess)
    return h->fail(FS_ERR_OOM, "page table allocation failed");
  FS_CK(h, cudaMemset(kv.pt, 0, (size_t)d.max_lanes * kv.max_pages * 4));
  h->pt.assign(d.max_lanes, {});
  h->len.assign(d.max_lanes, 0);
  for (int p = 0; p < d.n_pages; ++p) h->free_pages.insert(p);
  h->page_ref.assign(d.n_pages, 0);
  if (h->alloc(&h->d_reloc_pt, (size_t)kv.max_pages * 4) != cudaSuccess)
    return h->fail(FS_ERR_OOM, "page table scratch allocation failed");

  // ---- RoPE tables: cos/sin of pos * theta^(-2i/hd), in double, to f32
  {
    const int half = d.head_dim / 2;
    std::vector<float> c((size_t)d.max_pos * half), s((size_t)d.max_pos * half);
    for (int i = 0; i < half; ++i) {
      const double inv = std::pow(d.rope_theta, -2.0 * (double)i / (double)d.head_dim);
      for (int p = 0; p < d.max_pos; ++p) {
        const double a = (double)p * inv;
        c[(size_t)p * half + i] = (float)std::cos(a);
        s[(size_t)p * half + i] = (float)std::sin(a);
      }
    }
    if (h->alloc(&h->rope_cos, c.size() * 4) != cudaSuccess ||
        h->alloc(&h->rope_sin, s.size() * 4) != cudaSuccess)
      return h->fail(FS_ERR_OOM, "rope table allocation failed");
    FS_CK(h, cudaMemcpy(h->rope_cos, c.data(), c.size() * 4, cudaMemcpyHostToDevice));
    FS_CK(h, cudaMemcpy(h->rope_sin, s.data(), s.size() * 4, cudaMemcpyHostToDevice));
  }

  // ---- scratch panels
  const int B = d.max_lanes;
  const size_t xs = h->xtype == X_F32 ? 4 : 2;
  bool ok = h->alloc(&h->x, (size_t)B * d.d_model * 4) == cudaSuccess &&
            h->alloc(&h->y, (size_t)B * d.d_model * 4) == cudaSuccess &&
            h->alloc(&h->hpanel, (size_t)(1 + h->act_split) * B * h->Kp_d * xs) == cudaSuccess &&
            h->alloc(&h->opanel, (size_t)(1 + h->act_split) * B * h->Kp_q * xs) == cudaSuccess &&
            h->alloc(&h->apanel, (size_t)(1 + h->act_split) * B * h->Kp_f * xs) == cudaSuccess &&
            h->alloc(&h->qkv, (size_t)B * h->Nqkv * 4) == cudaSuccess &&
            h->alloc(&h->q, (size_t)B * h->Nq * 4) == cudaSuccess &&
            h->alloc(&h->logits, (size_t)B * d.vocab * 4) == cudaSuccess &&
            h->alloc(&h->part_ml, (size_t)B * h->max_splits * d.n_heads * 2 * 4) == cudaSuccess &&
            h->alloc(&h->part_acc, (size_t)B * h->max_splits * h->Nq * 4) == cudaSuccess &&
            h->alloc(&h->attn_counters, (size_t)B * d.n_kv_heads * 4) == cudaSuccess &&
            h->alloc(&h->d_args, (size_t)(7 * B + 1) * 4) == cudaSuccess &&
            h->alloc(&h->d_temps, (size_t)B * 4) == cudaSuccess &&
            h->alloc(&h->d_seeds, (size_t)B * 8) == cudaSuccess &&
            h->alloc(&h->d_counters, (size_t)B * 8) == cudaSuccess &&
            h->alloc(&h->d_tokens, (size_t)B * 4) == cudaSuccess &&
            h->alloc(&h->d_greedy, (size_t)B * 4) == cudaSuccess &&
            h->alloc(&h->d_zero_temps, (size_t)B * 4) == cudaSuccess &&
            h->alloc(&h->d_zero_u64, (size_t)B * 8) == cudaSuccess;
  if (!ok) return h->fail(FS_ERR_OOM, "scratch allocation failed");
  FS_CK(h, cudaMemset(h->attn_counters, 0, (size_t)B * d.n_kv_heads * 4));
  FS_CK(h, cudaMemset(h->d_zero_temps, 0, (size_t)B * 4));
  FS_CK(h, cudaMemset(h->d_zero_u64, 0, (size_t)B * 8));
  {
    // FS_ATTN=mma / warp (comparison knobs read at create) keep the cp.async
    // kernel on every handle / the one-warp kernel for every call of a
    // short-context handle; the kernels give the same bits
    const char* e = getenv("FS_ATTN");
    const bool force_mma = e && std::string(e) == "mma";
    const bool force_warp = e && std::string(e) == "warp";
    h->attn_mma = attn_mma_supports(d.head_dim, h->G, d.kv_dtype == FS_DTYPE_F32, h->split_len,
                                    h->max_splits);
    // the TMA kernel's producer warp and barrier set-up pay off on long
    // contexts; a handle whose lanes stay short keeps the cp.async kernel
    h->attn_tma = !force_mma && d.max_pos > 256 &&
                  attn_tma_supports(d.head_dim, h->G, d.kv_dtype == FS_DTYPE_F32, d.page_size,
                                    h->split_len, h->max_splits);
    if (h->attn_tma) {
      const int64_t rows = (int64_t)d.n_layers * (h->kv.layer_stride / d.head_dim);
      if (attn_tma_make_map(h->kv.k, rows, d.head_dim, d.page_size, &h->tm_kv_k) ||
          attn_tma_make_map(h->kv.v, rows, d.head_dim, d.page_size, &h->tm_kv_v))
        h->attn_tma = false;  // arena too large for 32-bit rows: the cp.async kernel serves
    }
    // lanes of at most 64 positions: one warp per (lane, KV head), the
    // cp.async kernel's bits. It holds ten pairs an SM against the cp.async
    // kernel's six of four warps each, so it pays once a call fills the SMs
    // ten times over (SmolLM2 shape: 8.0 vs 5.8 us per layer at 256 lanes,
    // faster at 960); smaller calls keep the cp.async kernel.
    h->attn_warp = !force_mma && h->attn_mma &&
                   attn_warp_supports(d.head_dim, h->G, d.kv_dtype == FS_DTYPE_F32, d.max_pos);
    h->attn_warp_rows = force_warp ? 0 : (10 * h->sms + d.n_kv_heads - 1) / d.n_kv_heads;
    // f32 KV and head dims below 64: the tiled kernel
    h->attn_tiled = !h->attn_tma && !h->attn_mma &&
                    attn_tiled_supports(d.head_dim, h->G, d.page_size, h->split_len);
    if (!h->attn_tma && !h->attn_mma && !h->attn_tiled)
      return h->fail(FS_ERR_ARG,
                     "no attention kernel for this shape: head_dim must be 16, 32, 64, 128 or "
                     "256, and page_size 16, 32 or 64 for f32 KV or head_dim < 64");
  }
  FS_CK(h, cudaMemset(h->hpanel, 0, (size_t)(1 + h->act_split) * B * h->Kp_d * xs));
  FS_CK(h, cudaMemset(h->opanel, 0, (size_t)(1 + h->act_split) * B * h->Kp_q * xs));
  FS_CK(h, cudaMemset(h->apanel, 0, (size_t)(1 + h->act_split) * B * h->Kp_f * xs));
  // remainder parts follow their panels (act_split)
  if (h->act_split) {
    h->lo_h = (int64_t)B * h->Kp_d;
    h->lo_o = (int64_t)B * h->Kp_q;
    h->lo_a = (int64_t)B * h->Kp_f;
  }
  FS_CK(h, cudaHostAlloc((void**)&h->h_args, (size_t)(7 * B + 1) * 4, cudaHostAllocDefault));
  FS_CK(h, cudaHostAlloc((void**)&h->err_flag, 16, cudaHostAllocMapped));
  *h->err_flag = 0;
  FS_CK(h, cudaHostGetDevicePointer((void**)&h->d_err_flag, h->err_flag, 0));
  if (h->use_tc) {
    size_t ws_elems = 0;
    int max_tiles = 1;
    auto setup = [&](const Mat& m, TcW* t) -> int {
      t->m_tiles = (m.N + 127) / 128;
      t->P = choose_width(t->m_tiles, m.Kp / 64, B, h->sms);
      if (!tc_width_ok(t->m_tiles, m.Kp / 64, t->P))
        return h->fail(FS_ERR_ARG, "weight matrix too large for the tcgen05 GEMM");
      max_tiles = std::max(max_tiles, t->m_tiles);
      ws_elems = std::max(ws_elems, tc_ws_floats(t->P, B));
      if (h->wtype == W_Q8) {
        const size_t tiles = (size_t)t->m_tiles * (m.Kp / 64);
        if (h->alloc(&t->q8_tiles, tiles * (8192 + 512)) != cudaSuccess)
          return h->fail(FS_ERR_OOM, "Q8_0 tile allocation failed");
        h->launches += launch_tile_q8((const int8_t*)m.w, m.scales, m.N, m.Kp, t->q8_tiles,
                                      h->stream);
        FS_CK(h, cudaGetLastError());
        // where the lane capacity reaches q8_copy_groups lane groups the
        // handle also keeps the matrix in bf16, converted once here: such
        // calls stream 16 instead of 8.5 KB per tile and convert nothing
        if (q8_keeps_copy(B, t->P, h->sms, h->q8_copy_groups)) {
          if (h->alloc(&t->q8_bf16, (size_t)m.N * m.Kp * 2) != cudaSuccess)
            return h->fail(FS_ERR_OOM, "Q8_0 bf16 copy allocation failed");
          h->launches += launch_dequant_q8_bf16((const int8_t*)m.w, m.scales, m.N, m.Kp,
                                                t->q8_bf16, h->stream);
          FS_CK(h, cudaGetLastError());
          CUtensorMap tm;
          if (tc_make_map(t->q8_bf16, m.N, m.Kp, 128, 1, &tm))
            return h->fail(FS_ERR_CUDA, "tensor map");
        }
        FS_CK(h, cudaStreamSynchronize(h->stream));
        return FS_OK;
      }
      CUtensorMap tm;  // the launches encode (and keep) their maps; this checks the shape
      if (tc_make_map(m.w, m.N, m.Kp, 128, 1, &tm)) return h->fail(FS_ERR_CUDA, "tensor map");
      return FS_OK;
    };
    for (auto& L : h->layers) {
      if ((rc = setup(L.qkv, &L.qkv_tc)) || (rc = setup(L.o, &L.o_tc)) ||
          (rc = setup(L.gateup, &L.gateup_tc)) || (rc = setup(L.down, &L.down_tc)))
        return rc;
    }
    if ((rc = setup(h->head, &h->head_tc))) return rc;
    // the argmax epilogue needs every head tile whole in one block
    h->greedy_fused = h->head_tc.P == h->head_tc.m_tiles;
    if (h->greedy_fused &&
        (h->alloc(&h->am_val, (size_t)B * h->head_tc.m_tiles * 4) != cudaSuccess ||
         h->alloc(&h->am_idx, (size_t)B * h->head_tc.m_tiles * 4) != cudaSuccess))
      return h->fail(FS_ERR_OOM, "argmax buffer allocation failed");
    if (h->wtype == W_Q8) {  // only the embedding gather still reads row-major codes
      for (auto& L : h->layers) {
        for (Mat* m : {&L.qkv, &L.o, &L.gateup, &L.down}) {
          h->release((void*)m->w);
          h->release((void*)m->scales);
          m->w = nullptr;
          m->scales = nullptr;
        }
      }
      if (!d.tied_embeddings) {
        h->release((void*)h->head.w);
        h->release((void*)h->head.scales);
      }
    }
    auto maps = [&](const void* panel, int Kp, int64_t lo) {
      CUtensorMap tm;
      return tc_make_map(panel, B, Kp, 16, 1, &tm) ||
             (lo && tc_make_map(static_cast<const __nv_bfloat16*>(panel) + lo, B, Kp, 16, 1, &tm));
    };
    if (maps(h->hpanel, h->Kp_d, h->lo_h) || maps(h->opanel, h->Kp_q, h->lo_o) ||
        maps(h->apanel, h->Kp_f, h->lo_a))
      return h->fail(FS_ERR_CUDA, "panel tensor map");
    const size_t n_counters = (size_t)max_tiles * ((B + 15) / 16);
    if (h->alloc(&h->ws, std::max<size_t>(ws_elems, 1) * 4) != cudaSuccess ||
        h->alloc(&h->counters, n_counters * 4) != cudaSuccess)
      return h->fail(FS_ERR_OOM, "GEMM workspace allocation failed");
    FS_CK(h, cudaMemset(h->counters, 0, n_counters * 4));

  }
  FS_CK(h, cudaHostAlloc((void**)&h->h_samp, (size_t)B * 24, cudaHostAllocDefault));
  int32_t* a = h->d_args;
  h->args.lane = a;
  h->args.pos = a + B;
  h->args.tok = a + 2 * B;
  h->args.upd_lane = a + 3 * B;
  h->args.upd_slot = a + 4 * B;
  h->args.upd_page = a + 5 * B;
  h->args.n_upd = a + 7 * B;
  FS_CK(h, cudaDeviceSynchronize());
  return FS_OK;
}

void destroy_impl(fs_handle* h) {
  if (h->stream) cudaStreamSynchronize(h->stream);
  trace_release(h);
  for (void* p : h->allocs) cudaFree(p);
  h->allocs.clear();
  if (h->h_args) cudaFreeHost(h->h_args);
  if (h->h_samp) cudaFreeHost(h->h_samp);
  if (h->err_flag) cudaFreeHost(h->err_flag);
  if (h->args_done) cudaEventDestroy(h->args_done);
  for (auto& r : h->prof_pending) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (cudaEvent_t e : h->prof_pool) cudaEventDestroy(e);
  for (auto& g : h->graphs) cudaGraphExecDestroy(g.second.exec);
  h->graphs.clear();
  if (h->own_stream) cudaStreamDestroy(h->own_stream);
}

// The lowest free page, now held by one lane.
int32_t take_page(fs_handle* h) {
  const int32_t p = *h->free_pages.begin();
  h->free_pages.erase(h->free_pages.begin());
  h->page_ref[p] = 1;
  return p;
}

// One lane lets go of page p; the page is free once no lane holds it.
void release_page(fs_handle* h, int32_t p) {
  if (--h->page_ref[p] == 0) h->free_pages.insert(p);
}

// Allocates pages for `n` more tokens of lane k starting at its current
// length (lowest free index first). Caller has checked capacity.
void take_pages(fs_handle* h, int k, int n_tokens_after) {
  const int ps = h->d.page_size;
  const int need = (n_tokens_after + ps - 1) / ps;
  while ((int)h->pt[k].size() < need) {
    h->pt[k].push_back(take_page(h));
  }
}

int seed_lane_pages(fs_handle* h, int lane, int n) {
  if (lane < 0 || lane >= h->d.max_lanes) return h->fail(FS_ERR_LANE, "lane out of range");
  if (n < 0) return h->fail(FS_ERR_ARG, "negative token count");
  if (h->len[lane] != 0) return h->fail(FS_ERR_STATE, "lane is not empty");
  if (n > h->d.max_pos) return h->fail(FS_ERR_KV_FULL, "n exceeds max_pos");
  const int need = (n + h->d.page_size - 1) / h->d.page_size;
  if (need > (int)h->free_pages.size()) return h->fail(FS_ERR_KV_FULL, "page pool exhausted");
  take_pages(h, lane, n);
  h->len[lane] = n;
  if (need)
    FS_CK(h, cudaMemcpyAsync(h->kv.pt + (size_t)lane * h->kv.max_pages, h->pt[lane].data(),
                             (size_t)need * 4, cudaMemcpyHostToDevice, h->stream));
  return FS_OK;
}

// Enqueues every kernel of one step for the n panel rows on h->stream (the
// per-step arguments are read from device memory, so the sequence can be
// captured once per n and replayed).
void enqueue_step(fs_handle* h, int n, float* out, double kv_read, bool chunked,
                  int32_t* greedy) {
  const fs_model_desc& d = h->d;
  cudaStream_t s = h->stream;
  const StepArgs& args = h->args;
  const double xs = h->xtype == X_F32 ? 4.0 : 2.0;
  const double kvs = h->kv.kv_f32 ? 4.0 : 2.0;
  auto wbytes = [&](const Mat& m) {
    double b = (double)m.N * m.K * (m.wtype == W_F32 ? 4 : (m.wtype == W_BF16 ? 2 : 1));
    if (m.wtype == W_Q8) b += (double)m.N * (m.K / 32) * 2;
    return b;
  };
  // algorithmic bytes: weights once, activations in, outputs out
  auto gemm = [&](const Mat& W, const TcW& T, const void* X, int64_t x_lo, int epi, float* of,
                  void* ox, int ldo, int n_out) {
    double bytes = wbytes(W) + (double)n * W.K * xs;
    bytes += epi == EPI_ARGMAX ? (double)n * T.m_tiles * 8.0
             : epi == EPI_SWIGLU ? (double)n * n_out * xs
             : (double)n * n_out * 4.0 * (epi == EPI_RESID ? 2 : 1);
    if (!h->use_tc) {
      GemmArgs g{};
      g.W = W; g.X = X; g.x_type = h->xtype; g.B = n; g.epi = epi;
      g.out_f32 = of; g.out_x = ox; g.ldo = ldo; g.n_out = n_out;
      h->launch(FS_PROF_GEMM, bytes, [&] { return launch_gemv(g, s); });
      return;
    }
    TcParams p{};
    p.m_tiles = T.m_tiles; p.P = T.P; p.kb_total = W.Kp / 64;
    p.lanes_total = n; p.sms = h->sms;
    const bool q8 = h->wtype == W_Q8;
    bool q8_copy = false;  // the bf16 copy serves this call
    gemm_call_groups(n, T.P, h->sms, q8, T.q8_bf16 != nullptr, h->q8_copy_groups, &p.lg,
                     &p.groups, &q8_copy);
    p.tmem_cols = tc_tmem_cols(p.lg);
    // the cluster reduction pays where partial tiles are large or K short;
    // long-K splits of small lane groups sum through the workspace
    p.cs_off = (p.kb_total >= 32 && p.lg < 32) ? 1 : 0;
    p.epi = epi; p.out_f32 = of; p.out_x = ox; p.ldo = ldo; p.n_out = n_out;
    p.ws = h->ws; p.counters = h->counters; p.err = h->d_err_flag;
    p.q8_tiles = T.q8_tiles;
    p.am_val = h->am_val; p.am_idx = h->am_idx;
    p.split = h->act_split;
    p.lo_off = epi == EPI_SWIGLU ? h->lo_a : 0;
    const TcOperands o{q8_copy ? T.q8_bf16 : W.w, W.N, X, d.max_lanes, W.Kp, x_lo};
    h->launch(FS_PROF_GEMM, bytes, [&] {
      const int r = q8 && !q8_copy ? launch_gemm_tc_q8(o, p, s) : launch_gemm_tc(o, p, s);
      if (r < 0) h->map_fail = true;
      return std::max(r, 0);
    });
  };
  const double norm_bytes = (double)n * d.d_model * (4.0 * 3 + xs);
  // embedding gather + the first layer's input norm
  h->launch(FS_PROF_OTHER, (double)n * d.d_model * (4.0 * 2 + xs), [&] {
    return launch_embed(h->embed, args, n, h->kv, h->x, d.d_model, h->layers[0].g_attn,
                        d.rms_eps, h->hpanel, h->xtype, h->Kp_d, h->lo_h, s);
  });
  for (int l = 0; l < d.n_layers; ++l) {
    const LayerW& W = h->layers[l];
    if (l > 0)
      h->launch(FS_PROF_OTHER, norm_bytes, [&] {
        return launch_rmsnorm(h->x, h->y, W.g_attn, n, d.d_model, d.rms_eps, h->hpanel,
                              h->xtype, h->Kp_d, h->lo_h, s);
      });
    gemm(W.qkv, W.qkv_tc, h->hpanel, h->lo_h, EPI_STORE, h->qkv, nullptr, h->Nqkv, h->Nqkv);
    // a chunked step first appends every row's k, v (rows of one lane at
    // consecutive positions see each other's keys); the MMA attention kernels
    // then only read, the other kernels give way to the three-kernel path
    if (chunked)
      h->launch(FS_PROF_OTHER, (double)n * (h->Nqkv * 4.0 + h->Nq * 4.0 + 2.0 * h->Nkv * kvs),
                [&] {
                  return launch_rope_append(h->qkv, n, d.n_heads, d.n_kv_heads, d.head_dim,
                                            h->rope_cos, h->rope_sin, args, h->kv, l, h->q, s);
                });
    {
      AttnParams ap{};
      ap.kv_written = chunked ? 1 : 0;
      ap.qkv = h->qkv; ap.H = d.n_heads; ap.rc = h->rope_cos; ap.rs = h->rope_sin;
      ap.args = args; ap.kv = h->kv; ap.layer = l; ap.split_len = h->split_len;
      ap.max_splits = h->max_splits; ap.part_ml = h->part_ml; ap.part_acc = h->part_acc;
      ap.counters = h->attn_counters; ap.o = h->opanel; ap.ld_o = h->Kp_q; ap.err = h->d_err_flag;
      ap.o_lo = h->lo_o;
      h->launch(FS_PROF_ATTN,
                kv_read + (double)n * (h->Nqkv * 4.0 + h->Nq * xs + 2.0 * h->Nkv * kvs),
                [&] {
                  if (h->attn_warp && n >= h->attn_warp_rows)
                    return launch_attention_warp(ap, n, h->xtype, s);
                  if (h->attn_tma)
                    return launch_attention_tma(h->tm_kv_k, h->tm_kv_v, ap, n, h->xtype, s);
                  return h->attn_mma ? launch_attention_mma(ap, n, h->xtype, s)
                                     : launch_attention_tiled(ap, n, h->xtype, s);
                });
    }
    gemm(W.o, W.o_tc, h->opanel, h->lo_o, EPI_STORE, h->y, nullptr, d.d_model,
         d.d_model);
    h->launch(FS_PROF_OTHER, norm_bytes, [&] {
        return launch_rmsnorm(h->x, h->y, W.g_ffn, n, d.d_model, d.rms_eps, h->hpanel,
                              h->xtype, h->Kp_d, h->lo_h, s);
      });
    gemm(W.gateup, W.gateup_tc, h->hpanel, h->lo_h, EPI_SWIGLU, nullptr, h->apanel, h->Kp_f,
         d.d_ffn);
    gemm(W.down, W.down_tc, h->apanel, h->lo_a, EPI_STORE, h->y, nullptr, d.d_model,
         d.d_model);
  }
  h->launch(FS_PROF_OTHER, norm_bytes, [&] {
      return launch_rmsnorm(h->x, h->y, h->g_final, n, d.d_model, d.rms_eps, h->hpanel, h->xtype,
                            h->Kp_d, h->lo_h, s);
    });
  if (greedy && h->greedy_fused) {  // greedy tokens straight from the head's epilogue
    gemm(h->head, h->head_tc, h->hpanel, h->lo_h, EPI_ARGMAX, nullptr, nullptr,
         d.vocab, d.vocab);
    h->launch(FS_PROF_OTHER, (double)n * (h->head_tc.m_tiles * 8.0 + 4.0), [&] {
      return launch_argmax_tiles(h->am_val, h->am_idx, n, h->head_tc.m_tiles, greedy, s);
    });
    return;
  }
  gemm(h->head, h->head_tc, h->hpanel, h->lo_h, EPI_STORE, out, nullptr, d.vocab, d.vocab);
  if (greedy)
    h->launch(FS_PROF_OTHER, (double)n * d.vocab * 4.0, [&] {
      return launch_sample(out, n, d.vocab, h->d_zero_temps, h->d_zero_u64, h->d_zero_u64,
                           greedy, s);
    });
}

}  // namespace

extern "C" {

int fs_create(const fs_model_desc* desc, const fs_weights* weights, fs_handle** out) {
  if (!desc || !out) {
    g_create_error = "NULL descriptor or output pointer";
    return FS_ERR_ARG;
  }
  *out = nullptr;
  std::string why;
  if (validate_desc(desc, &why)) {
    g_create_error = why;
    return FS_ERR_ARG;
  }
  fs_handle* h = new fs_handle();
  h->d = *desc;
  int rc = create_impl(h, weights);
  if (rc) {
    g_create_error = h->err;
    destroy_impl(h);
    delete h;
    return rc;
  }
  *out = h;
  return FS_OK;
}

int fs_destroy(fs_handle* h) {
  if (!h) return FS_OK;
  destroy_impl(h);
  delete h;
  return FS_OK;
}

const char* fs_last_error(const fs_handle* h) {
  return h ? h->err.c_str() : g_create_error.c_str();
}

int fs_set_stream(fs_handle* h, void* stream) {
  if (!h) return FS_ERR_ARG;
  FS_CK(h, cudaStreamSynchronize(h->stream));
  h->stream = stream ? (cudaStream_t)stream : h->own_stream;
  return FS_OK;
}

int fs_lane_reset(fs_handle* h, int32_t lane) {
  if (!h) return FS_ERR_ARG;
  if (lane < 0 || lane >= h->d.max_lanes) return h->fail(FS_ERR_LANE, "lane out of range");
  for (int32_t p : h->pt[lane]) release_page(h, p);
  h->pt[lane].clear();
  h->len[lane] = 0;
  return FS_OK;
}

int fs_lane_clone(fs_handle* h, int32_t src, int32_t dst) {
  if (!h) return FS_ERR_ARG;
  const int B = h->d.max_lanes, ps = h->d.page_size;
  if (src < 0 || src >= B || dst < 0 || dst >= B) return h->fail(FS_ERR_LANE, "lane out of range");
  if (src == dst) return h->fail(FS_ERR_ARG, "src and dst are the same lane");
  if (h->len[dst] != 0 || !h->pt[dst].empty()) return h->fail(FS_ERR_STATE, "dst lane is not empty");
  const int n = h->len[src], full = n / ps;
  const bool partial = n % ps != 0;
  if (partial && h->free_pages.empty()) return h->fail(FS_ERR_KV_FULL, "page pool exhausted");
  // full pages are shared (never written again: later tokens go to later
  // pages); the partial last page, which both lanes go on writing, is copied
  // to the lowest free page. Device work first, host state after it, so a
  // failed call leaves the lanes as they were (dst's row is unused while
  // dst is empty).
  std::vector<int32_t> t(h->pt[src].begin(), h->pt[src].begin() + full);
  if (partial) t.push_back(*h->free_pages.begin());
  if (!t.empty()) {
    int32_t* dst_row = h->kv.pt + (size_t)dst * h->kv.max_pages;
    FS_CK(h, cudaMemcpyAsync(dst_row, t.data(), t.size() * 4, cudaMemcpyHostToDevice, h->stream));
    if (partial) {
      h->launches += launch_kv_relocate(h->kv, h->d.n_layers,
                                        h->kv.pt + (size_t)src * h->kv.max_pages, dst_row,
                                        full * ps, n, n, 0, h->rope_cos, h->rope_sin, h->stream);
      FS_CK(h, cudaGetLastError());
    }
  }
  for (int x = 0; x < full; ++x) ++h->page_ref[t[x]];
  if (partial) take_page(h);  // the page chosen above: the lowest free one
  h->pt[dst] = std::move(t);
  h->len[dst] = n;
  return FS_OK;
}

int fs_lane_evict(fs_handle* h, int32_t lane, int32_t start, int32_t end) {
  if (!h) return FS_ERR_ARG;
  if (lane < 0 || lane >= h->d.max_lanes) return h->fail(FS_ERR_LANE, "lane out of range");
  const int n = h->len[lane], ps = h->d.page_size;
  if (start < 0 || start > end || end > n) return h->fail(FS_ERR_ARG, "span outside [0, length]");
  if (start == end) return FS_OK;
  const int delta = end - start, nl = n - delta;
  const int keep = (nl + ps - 1) / ps, first = start / ps;
  const std::vector<int32_t>& old = h->pt[lane];
  // pages [first, keep) are written (moved rows now, the next token later):
  // a page another lane still holds is replaced by a private copy, the
  // lowest free pages in ascending index order
  std::vector<int32_t> t(old.begin(), old.begin() + keep);
  auto fresh = h->free_pages.begin();
  for (int x = first; x < keep; ++x)
    if (h->page_ref[old[x]] > 1) {
      if (fresh == h->free_pages.end()) return h->fail(FS_ERR_KV_FULL, "page pool exhausted");
      t[x] = *fresh++;
    }
  // rows [start, nl) move down by delta; a replaced first page also takes
  // its rows below start. Device work first, host state after it.
  const int q_begin = (first < keep && t[first] != old[first]) ? first * ps : start;
  if (q_begin < nl) {
    int32_t* row = h->kv.pt + (size_t)lane * h->kv.max_pages;
    FS_CK(h, cudaMemcpyAsync(h->d_reloc_pt, row, old.size() * 4, cudaMemcpyDeviceToDevice,
                             h->stream));
    cudaError_t e = cudaMemcpyAsync(row, t.data(), t.size() * 4, cudaMemcpyHostToDevice, h->stream);
    if (e == cudaSuccess) {
      h->launches += launch_kv_relocate(h->kv, h->d.n_layers, h->d_reloc_pt, row, q_begin, nl,
                                        start, delta, h->rope_cos, h->rope_sin, h->stream);
      e = cudaGetLastError();
    }
    if (e != cudaSuccess) {  // put the lane's device row back (best effort)
      cudaMemcpyAsync(row, old.data(), old.size() * 4, cudaMemcpyHostToDevice, h->stream);
      return h->cuda_fail(e, "evict");
    }
  }
  for (int x = first; x < keep; ++x)
    if (t[x] != old[x]) {
      --h->page_ref[old[x]];
      take_page(h);  // == t[x]: the same lowest-first order
    }
  // pages past the new end are let go (stream order keeps them unwritten
  // until the move above has read them)
  for (int x = keep; x < (int)old.size(); ++x) release_page(h, old[x]);
  h->pt[lane] = std::move(t);
  h->len[lane] = nl;
  return FS_OK;
}

}  // extern "C"

namespace {
// Commit and launch of a validated step: page allocation (per lane in
// position order, lowest free index first), the argument block, then the
// kernels (one graph replay per (n, mode)).
int decode_step(fs_handle* h, const int32_t* lanes, int32_t* positions, const int32_t* tokens,
                int32_t n, float* logits_out, int32_t* greedy_out);

// An NVTX range around each step (no cost unless a tool is attached; a
// profiler can then select a step's kernels by range).
struct StepRange {
  explicit StepRange(const char* name) { nvtxRangePushA(name); }
  ~StepRange() { nvtxRangePop(); }
};

int run_step(fs_handle* h, const int32_t* lanes, int32_t* positions, const int32_t* tokens,
             int n, float* logits_out, bool chunked, int32_t* greedy_out = nullptr) {
  const StepRange range(chunked ? "fs_step_batch_chunked"
                                : greedy_out ? "fs_decode_step_greedy" : "fs_decode_step_batch");
  const fs_model_desc& d = h->d;
  FS_CK(h, cudaEventSynchronize(h->args_done));  // staging no longer in use
  const int B = d.max_lanes;
  int32_t* A = h->h_args;
  int n_upd = 0;
  // lanes in order of first appearance; a lane's positions (its length on
  // up, one per row of this step) in ascending order
  std::vector<int32_t> rows(d.max_lanes, 0);
  for (int i = 0; i < n; ++i) {
    A[i] = lanes[i];
    A[B + i] = positions[i];
    A[2 * B + i] = tokens[i];
    rows[lanes[i]] += 1;
  }
  for (int i = 0; i < n; ++i) {
    const int k = lanes[i];
    if (rows[k] == 0) continue;  // this lane's pages are already taken
    for (int p = h->len[k]; p < h->len[k] + rows[k]; ++p) {
      if (p % d.page_size) continue;
      take_pages(h, k, p + 1);
      A[3 * B + n_upd] = k;
      A[4 * B + n_upd] = p / d.page_size;
      A[5 * B + n_upd] = h->pt[k].back();
      ++n_upd;
    }
    rows[k] = 0;
  }
  A[7 * B] = n_upd;
  // one copy of the whole block keeps this to a single H2D transfer per step
  FS_CK(h, cudaMemcpyAsync(h->d_args, h->h_args, (size_t)(7 * B + 1) * 4,
                           cudaMemcpyHostToDevice, h->stream));
  FS_CK(h, cudaEventRecord(h->args_done, h->stream));

  // ---- the step: one graph replay, or the kernels one by one
  double kv_read = 0.0;  // K and V bytes attention reads per layer
  for (int i = 0; i < n; ++i)
    kv_read += (double)(positions[i] + 1) * h->Nkv * 2.0 * (h->kv.kv_f32 ? 4.0 : 2.0);
  float* out = logits_out ? logits_out : h->logits;
  int32_t* greedy = greedy_out ? h->d_greedy : nullptr;
  if (!logits_out && !h->prof_on && h->graphs_on) {
    const int key = n + (chunked ? (1 << 20) : 0) + (greedy ? (2 << 20) : 0);
    auto it = h->graphs.find(key);
    if (it == h->graphs.end()) {
      const int64_t before = h->launches;
      cudaGraph_t g = nullptr;
      FS_CK(h, cudaStreamBeginCapture(h->stream, cudaStreamCaptureModeThreadLocal));
      h->map_fail = false;
      enqueue_step(h, n, out, kv_read, chunked, greedy);
      cudaError_t e = cudaStreamEndCapture(h->stream, &g);
      if (e != cudaSuccess) return h->cuda_fail(e, "cudaStreamEndCapture");
      if (h->map_fail) {
        cudaGraphDestroy(g);
        return h->fail(FS_ERR_CUDA, "GEMM tensor map encoding failed");
      }
      fs_handle::Graph G;
      e = cudaGraphInstantiate(&G.exec, g, 0);
      cudaGraphDestroy(g);
      if (e != cudaSuccess) return h->cuda_fail(e, "cudaGraphInstantiate");
      G.kernels = h->launches - before;
      h->launches = before;
      it = h->graphs.emplace(key, G).first;
    }
    FS_CK(h, cudaGraphLaunch(it->second.exec, h->stream));
    h->launches += it->second.kernels;
  } else {
    h->map_fail = false;
    enqueue_step(h, n, out, kv_read, chunked, greedy);
    if (h->map_fail) return h->fail(FS_ERR_CUDA, "GEMM tensor map encoding failed");
  }
  FS_CK(h, cudaGetLastError());
  if (greedy_out)
    FS_CK(h, cudaMemcpyAsync(greedy_out, h->d_greedy, (size_t)n * 4, cudaMemcpyDefault,
                             h->stream));

  for (int i = 0; i < n; ++i) {
    h->len[lanes[i]] += 1;
    positions[i] += 1;
  }
  h->last_n = greedy_out ? -1 : n;  // a greedy step leaves no logits to sample
  h->last_logits = greedy_out ? nullptr : out;
  return FS_OK;
}
}  // namespace

extern "C" {

int fs_decode_step_greedy(fs_handle* h, const int32_t* lanes, int32_t* positions,
                          const int32_t* tokens, int32_t n, int32_t* tokens_out) {
  if (!h) return FS_ERR_ARG;
  if (n > 0 && !tokens_out) return h->fail(FS_ERR_ARG, "NULL tokens_out");
  const int rc = decode_step(h, lanes, positions, tokens, n, nullptr, tokens_out);
  if (rc != FS_OK || n == 0) return rc;
  cudaPointerAttributes at{};
  const bool dev = cudaPointerGetAttributes(&at, tokens_out) == cudaSuccess &&
                   (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged);
  cudaGetLastError();  // a plain host pointer may leave an error behind
  if (!dev) FS_CK(h, cudaStreamSynchronize(h->stream));  // host tokens written on return
  return FS_OK;
}

int fs_decode_step_batch(fs_handle* h, const int32_t* lanes, int32_t* positions,
                         const int32_t* tokens, int32_t n, float* logits_out) {
  return decode_step(h, lanes, positions, tokens, n, logits_out, nullptr);
}

}  // extern "C"

namespace {
int decode_step(fs_handle* h, const int32_t* lanes, int32_t* positions, const int32_t* tokens,
                int32_t n, float* logits_out, int32_t* greedy_out) {
  if (!h) return FS_ERR_ARG;
  if (n == 0) return FS_OK;
  if (n < 0 || n > h->d.max_lanes) return h->fail(FS_ERR_ARG, "n outside [0, max_lanes]");
  if (!lanes || !positions || !tokens) return h->fail(FS_ERR_ARG, "NULL argument array");
  const fs_model_desc& d = h->d;
  // ---- validate (no state change)
  std::vector<char> seen(d.max_lanes, 0);
  int need = 0;
  for (int i = 0; i < n; ++i) {
    const int k = lanes[i];
    if (k < 0 || k >= d.max_lanes) return h->fail(FS_ERR_LANE, "lane out of range");
    if (seen[k]) return h->fail(FS_ERR_DUP_LANE, "lane appears twice in one step");
    seen[k] = 1;
    if (positions[i] != h->len[k]) return h->fail(FS_ERR_POSITION, "position differs from lane length");
    if (tokens[i] < 0 || tokens[i] >= d.vocab) return h->fail(FS_ERR_TOKEN, "token outside [0, vocab)");
    if (h->len[k] >= d.max_pos) return h->fail(FS_ERR_KV_FULL, "lane is at max_pos");
    if (h->len[k] % d.page_size == 0) ++need;
  }
  if (need > (int)h->free_pages.size()) return h->fail(FS_ERR_KV_FULL, "page pool exhausted");
  return run_step(h, lanes, positions, tokens, n, logits_out, false, greedy_out);
}
}  // namespace

extern "C" {

int fs_step_batch_chunked(fs_handle* h, const int32_t* lanes, int32_t* positions,
                          const int32_t* tokens, int32_t n, float* logits_out) {
  if (!h) return FS_ERR_ARG;
  if (n == 0) return FS_OK;
  if (n < 0 || n > h->d.max_lanes) return h->fail(FS_ERR_ARG, "n outside [0, max_lanes]");
  if (!lanes || !positions || !tokens) return h->fail(FS_ERR_ARG, "NULL argument array");
  const fs_model_desc& d = h->d;
  // ---- validate (no state change): per lane, its rows' positions are
  // exactly len, len + 1, ..., len + rows - 1 (in any order)
  std::vector<int32_t> rows(d.max_lanes, 0);
  for (int i = 0; i < n; ++i) {
    const int k = lanes[i];
    if (k < 0 || k >= d.max_lanes) return h->fail(FS_ERR_LANE, "lane out of range");
    if (tokens[i] < 0 || tokens[i] >= d.vocab) return h->fail(FS_ERR_TOKEN, "token outside [0, vocab)");
    rows[k] += 1;
  }
  std::vector<std::vector<char>> hit;  // per lane with rows: which offsets are present
  std::vector<int> idx(d.max_lanes, -1);
  int need = 0;
  for (int i = 0; i < n; ++i) {
    const int k = lanes[i];
    const int64_t off = (int64_t)positions[i] - h->len[k];
    if (off < 0 || off >= rows[k]) return h->fail(FS_ERR_POSITION, "positions of a lane must be its next consecutive ones");
    if (idx[k] < 0) {
      if ((int64_t)h->len[k] + rows[k] > d.max_pos) return h->fail(FS_ERR_KV_FULL, "lane would pass max_pos");
      idx[k] = (int)hit.size();
      hit.emplace_back(rows[k], 0);
    }
    if (hit[idx[k]][off]) return h->fail(FS_ERR_POSITION, "a position appears twice");
    hit[idx[k]][off] = 1;
    if (positions[i] % d.page_size == 0) ++need;
  }
  if (need > (int)h->free_pages.size()) return h->fail(FS_ERR_KV_FULL, "page pool exhausted");
  return run_step(h, lanes, positions, tokens, n, logits_out, true);
}

int fs_sample(fs_handle* h, int32_t n, const float* temps, const uint64_t* seeds,
              const uint64_t* counters, int32_t* tokens_out) {
  if (!h) return FS_ERR_ARG;
  if (h->last_n < 0) return h->fail(FS_ERR_STATE, "no decode step to sample from");
  if (n != h->last_n) return h->fail(FS_ERR_STATE, "n differs from the last step's n");
  if (!temps || !seeds || !counters || !tokens_out) return h->fail(FS_ERR_ARG, "NULL argument array");
  for (int i = 0; i < n; ++i)
    if (!(temps[i] >= 0.0f)) return h->fail(FS_ERR_ARG, "temperature must be >= 0");
  const int B = h->d.max_lanes;
  unsigned char* st = h->h_samp;
  float* ht = (float*)st;
  uint64_t* hs = (uint64_t*)(st + (size_t)B * 8);
  uint64_t* hc = (uint64_t*)(st + (size_t)B * 16);
  std::memcpy(ht, temps, (size_t)n * 4);
  std::memcpy(hs, seeds, (size_t)n * 8);
  std::memcpy(hc, counters, (size_t)n * 8);
  cudaStream_t s = h->stream;
  FS_CK(h, cudaMemcpyAsync(h->d_temps, ht, (size_t)n * 4, cudaMemcpyHostToDevice, s));
  FS_CK(h, cudaMemcpyAsync(h->d_seeds, hs, (size_t)n * 8, cudaMemcpyHostToDevice, s));
  FS_CK(h, cudaMemcpyAsync(h->d_counters, hc, (size_t)n * 8, cudaMemcpyHostToDevice, s));
  h->launch(FS_PROF_OTHER, (double)n * h->d.vocab * 4.0, [&] {
    return launch_sample(h->last_logits, n, h->d.vocab, h->d_temps, h->d_seeds,
                         h->d_counters, h->d_tokens, s);
  });
  FS_CK(h, cudaGetLastError());
  int32_t* ho = (int32_t*)(st);  // temps are consumed by now: reuse after sync
  FS_CK(h, cudaStreamSynchronize(s));
  FS_CK(h, cudaMemcpyAsync(ho, h->d_tokens, (size_t)n * 4, cudaMemcpyDeviceToHost, s));
  FS_CK(h, cudaStreamSynchronize(s));
  std::memcpy(tokens_out, ho, (size_t)n * 4);
  if (*(volatile int*)h->err_flag)
    return h->fail(FS_ERR_DEVICE, "a GEMM block timed out waiting on a barrier (code " +
                                      std::to_string(*(volatile int*)h->err_flag) + ")");
  return FS_OK;
}

int fs_sample_device(fs_handle* h, int32_t n, const float* temps, const uint64_t* seeds,
                     const uint64_t* counters, int32_t* tokens_out) {
  if (!h) return FS_ERR_ARG;
  if (h->last_n < 0) return h->fail(FS_ERR_STATE, "no decode step to sample from");
  if (n != h->last_n) return h->fail(FS_ERR_STATE, "n differs from the last step's n");
  if (!temps || !seeds || !counters || !tokens_out) return h->fail(FS_ERR_ARG, "NULL argument array");
  cudaStream_t s = h->stream;
  h->launch(FS_PROF_OTHER, (double)n * h->d.vocab * 4.0, [&] {
    return launch_sample(h->last_logits, n, h->d.vocab, temps, seeds, counters, tokens_out, s);
  });
  FS_CK(h, cudaGetLastError());
  return FS_OK;
}

int fs_profile_enable(fs_handle* h, int32_t enable) {
  if (!h) return FS_ERR_ARG;
  h->prof_on = enable != 0;
  return FS_OK;
}

int fs_profile_read(fs_handle* h, int32_t cls, double* ms_out, int64_t* launches_out,
                    double* bytes_out) {
  if (!h || cls < 0 || cls >= FS_PROF_CLASSES) return FS_ERR_ARG;
  FS_CK(h, cudaStreamSynchronize(h->stream));
  for (auto& r : h->prof_pending) {
    float ms = 0.0f;
    FS_CK(h, cudaEventElapsedTime(&ms, r.a, r.b));
    h->prof_ms[r.cls] += ms;
    h->prof_n[r.cls] += 1;
    h->prof_bytes[r.cls] += r.bytes;
    h->prof_pool.push_back(r.a);
    h->prof_pool.push_back(r.b);
  }
  h->prof_pending.clear();
  if (ms_out) *ms_out = h->prof_ms[cls];
  if (launches_out) *launches_out = h->prof_n[cls];
  if (bytes_out) *bytes_out = h->prof_bytes[cls];
  h->prof_ms[cls] = 0.0;
  h->prof_n[cls] = 0;
  h->prof_bytes[cls] = 0.0;
  return FS_OK;
}

int fs_copy_logits(fs_handle* h, float* dst) {
  if (!h || !dst) return FS_ERR_ARG;
  if (h->last_n < 0) return h->fail(FS_ERR_STATE, "no decode step yet");
  FS_CK(h, cudaMemcpyAsync(dst, h->last_logits, (size_t)h->last_n * h->d.vocab * 4,
                           cudaMemcpyDefault, h->stream));
  FS_CK(h, cudaStreamSynchronize(h->stream));
  return FS_OK;
}

int fs_lane_length(const fs_handle* h, int32_t lane, int32_t* length_out) {
  if (!h || !length_out) return FS_ERR_ARG;
  if (lane < 0 || lane >= h->d.max_lanes) return FS_ERR_LANE;
  *length_out = h->len[lane];
  return FS_OK;
}

int fs_lane_pages(const fs_handle* h, int32_t lane, int32_t* pages_out, int32_t cap,
                  int32_t* n_out) {
  if (!h || !n_out || cap < 0 || (cap > 0 && !pages_out)) return FS_ERR_ARG;
  if (lane < 0 || lane >= h->d.max_lanes) return FS_ERR_LANE;
  const auto& t = h->pt[lane];
  for (int i = 0; i < (int)t.size() && i < cap; ++i) pages_out[i] = t[i];
  *n_out = (int32_t)t.size();
  return FS_OK;
}

int fs_lane_export_kv(fs_handle* h, int32_t lane, int32_t layer, float* k_out, float* v_out) {
  if (!h || !k_out || !v_out) return FS_ERR_ARG;
  if (lane < 0 || lane >= h->d.max_lanes) return h->fail(FS_ERR_LANE, "lane out of range");
  if (layer < 0 || layer >= h->d.n_layers) return h->fail(FS_ERR_ARG, "layer out of range");
  const int n = h->len[lane];
  if (n == 0) return FS_OK;
  const size_t cnt = (size_t)n * h->kv.Hkv * h->kv.hd;
  int32_t* dp = nullptr;
  float *dk = nullptr, *dv = nullptr;
  int rc = FS_OK;
  if (cudaMalloc(&dp, h->pt[lane].size() * 4) != cudaSuccess ||
      cudaMalloc(&dk, cnt * 4) != cudaSuccess || cudaMalloc(&dv, cnt * 4) != cudaSuccess) {
    rc = h->fail(FS_ERR_OOM, "export buffers");
  } else {
    cudaError_t e = cudaMemcpyAsync(dp, h->pt[lane].data(), h->pt[lane].size() * 4,
                                    cudaMemcpyHostToDevice, h->stream);
    if (e == cudaSuccess) {
      h->launches += launch_export_kv(h->kv, layer, dp, n, dk, dv, h->stream);
      e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaMemcpyAsync(k_out, dk, cnt * 4, cudaMemcpyDeviceToHost, h->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(v_out, dv, cnt * 4, cudaMemcpyDeviceToHost, h->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
    if (e != cudaSuccess) rc = h->cuda_fail(e, "export_kv");
  }
  cudaFree(dp);
  cudaFree(dk);
  cudaFree(dv);
  return rc;
}

int fs_lane_import_kv(fs_handle* h, int32_t lane, const float* k, const float* v, int32_t n) {
  if (!h || (n > 0 && (!k || !v))) return FS_ERR_ARG;
  int rc = seed_lane_pages(h, lane, n);
  if (rc) return rc;
  if (n == 0) return FS_OK;
  const size_t cnt = (size_t)n * h->kv.Hkv * h->kv.hd;
  int32_t* dp = nullptr;
  float *dk = nullptr, *dv = nullptr;
  if (cudaMalloc(&dp, h->pt[lane].size() * 4) != cudaSuccess ||
      cudaMalloc(&dk, cnt * 4) != cudaSuccess || cudaMalloc(&dv, cnt * 4) != cudaSuccess) {
    rc = h->fail(FS_ERR_OOM, "import buffers");
  } else {
    cudaError_t e = cudaMemcpyAsync(dp, h->pt[lane].data(), h->pt[lane].size() * 4,
                                    cudaMemcpyHostToDevice, h->stream);
    for (int l = 0; l < h->d.n_layers && e == cudaSuccess; ++l) {
      e = cudaMemcpyAsync(dk, k + (size_t)l * cnt, cnt * 4, cudaMemcpyHostToDevice, h->stream);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(dv, v + (size_t)l * cnt, cnt * 4, cudaMemcpyHostToDevice, h->stream);
      if (e == cudaSuccess) {
        h->launches += launch_import_kv(h->kv, l, dp, n, dk, dv, h->stream);
        e = cudaGetLastError();
      }
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
    if (e != cudaSuccess) rc = h->cuda_fail(e, "import_kv");
  }
  cudaFree(dp);
  cudaFree(dk);
  cudaFree(dv);
  return rc;
}

int fs_lane_fill_random_kv(fs_handle* h, int32_t lane, int32_t n, uint64_t seed) {
  if (!h) return FS_ERR_ARG;
  int rc = seed_lane_pages(h, lane, n);
  if (rc || n == 0) return rc;
  int32_t* dp = nullptr;
  const size_t np = h->pt[lane].size();
  if (cudaMalloc(&dp, np * 4) != cudaSuccess) return h->fail(FS_ERR_OOM, "fill buffers");
  cudaError_t e = cudaMemcpyAsync(dp, h->pt[lane].data(), np * 4, cudaMemcpyHostToDevice, h->stream);
  if (e == cudaSuccess) {
    h->launches += launch_fill_random_kv(h->kv, h->d.n_layers, dp, (int)np, seed, h->stream);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
  cudaFree(dp);
  if (e != cudaSuccess) return h->cuda_fail(e, "fill_random_kv");
  return FS_OK;
}

int fs_quantize_q8_0(const float* src, int64_t n, uint8_t* blocks_out, void* stream) {
  if (!src || !blocks_out || n < 0 || n % 32) return FS_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  launch_quantize_q8_0(src, n, blocks_out, s);
  if (cudaGetLastError() != cudaSuccess) return FS_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FS_ERR_CUDA;
  return FS_OK;
}

int fs_trace_enable(fs_handle* h, int64_t capacity) {
  if (!h || capacity < 0) return FS_ERR_ARG;
  if (capacity > 0 && g_trace_owner && g_trace_owner != h)
    return h->fail(FS_ERR_STATE, "another handle is tracing");
  FS_CK(h, cudaStreamSynchronize(h->stream));
  const int rc = trace_release(h);
  if (rc != FS_OK || capacity == 0) return rc;
  TraceBuf* b = nullptr;
  const size_t bytes = 16 + (size_t)capacity * sizeof(TraceRec);
  if (cudaMalloc(&b, bytes) != cudaSuccess) return h->fail(FS_ERR_OOM, "trace buffer");
  const unsigned long long head[2] = {0ull, (unsigned long long)capacity};
  cudaError_t e = cudaMemcpy(b, head, sizeof head, cudaMemcpyHostToDevice);
  if (e != cudaSuccess || !trace_install_all(b)) {
    cudaFree(b);
    trace_install_all(nullptr);
    return e != cudaSuccess ? h->cuda_fail(e, "trace buffer") : h->fail(FS_ERR_CUDA, "trace install");
  }
  g_trace_buf = b;
  g_trace_cap = capacity;
  g_trace_owner = h;
  return FS_OK;
}

int fs_trace_read(fs_handle* h, uint64_t* records_out, int64_t cap, int64_t* appended_out,
                  int reset) {
  if (!h || !appended_out || cap < 0 || (cap > 0 && !records_out)) return FS_ERR_ARG;
  if (g_trace_owner != h || !g_trace_buf) return h->fail(FS_ERR_STATE, "tracing is not enabled on this handle");
  FS_CK(h, cudaStreamSynchronize(h->stream));
  unsigned long long n = 0;
  FS_CK(h, cudaMemcpy(&n, g_trace_buf, 8, cudaMemcpyDeviceToHost));
  const int64_t m = std::min<int64_t>(std::min<int64_t>((int64_t)n, g_trace_cap), cap);
  if (m > 0)
    FS_CK(h, cudaMemcpy(records_out, g_trace_buf->rec, (size_t)m * sizeof(TraceRec),
                        cudaMemcpyDeviceToHost));
  *appended_out = (int64_t)n;
  if (reset) FS_CK(h, cudaMemset(g_trace_buf, 0, 8));
  return FS_OK;
}

int fs_kernel_launches(const fs_handle* h, int64_t* count_out) {
  if (!h || !count_out) return FS_ERR_ARG;
  *count_out = h->launches;
  return FS_OK;
}

const char* fs_gemm_path(const fs_handle* h) {
  if (!h) return "";
  if (!h->use_tc) return "warp-gemv";
  if (h->wtype != W_Q8) return "tcgen05";
  return h->head_tc.q8_bf16 || (!h->layers.empty() && (h->layers[0].qkv_tc.q8_bf16 ||
                                                       h->layers[0].gateup_tc.q8_bf16))
             ? "tcgen05-q8_0+bf16"
             : "tcgen05-q8_0";
}

int fs_gemm_plan(int64_t n_rows, int64_t k_inputs, int max_lanes, int n, int sms,
                 int weight_dtype, int32_t* out) {
  if (!out || n_rows < 1 || k_inputs < 1 || k_inputs % 32 || max_lanes < 1 || n < 1 ||
      n > max_lanes || sms < 1 || weight_dtype < FS_DTYPE_BF16 ||
      weight_dtype > FS_DTYPE_Q8_0 || n_rows > ((int64_t)1 << 30) ||
      k_inputs > ((int64_t)1 << 30))
    return FS_ERR_ARG;
  const int m_tiles = (int)((n_rows + 127) / 128);
  const int kb_total = (int)(round_up(k_inputs, 64) / 64);
  const int P = choose_width(m_tiles, kb_total, max_lanes, sms);
  if (!tc_width_ok(m_tiles, kb_total, P)) return FS_ERR_ARG;
  const bool q8 = weight_dtype == FS_DTYPE_Q8_0;
  const int copy_groups = q8_copy_groups_env();
  const bool kept = q8 && q8_keeps_copy(max_lanes, P, sms, copy_groups);
  int lg = 0, groups = 1;
  bool use_copy = false;
  gemm_call_groups(n, P, sms, q8, kept, copy_groups, &lg, &groups, &use_copy);
  out[0] = P;
  out[1] = lg;
  out[2] = groups;
  out[3] = tc_tmem_cols(lg);
  out[4] = kept ? 1 : 0;
  out[5] = use_copy ? 1 : 0;
  out[6] = m_tiles;
  out[7] = kb_total;
  return FS_OK;
}

const char* fs_attention_path(const fs_handle* h) {
  if (!h) return "";
  if (h->attn_warp) return "warp-mma";
  if (h->attn_tma) return "tma-mma";
  if (h->attn_mma) return "cp.async-mma";
  if (h->attn_tiled) return "tiled";
  return "three-kernel";
}

int fs_lane_capacity(const fs_handle* h, int32_t* tokens_out) {
  if (!h || !tokens_out) return FS_ERR_ARG;
  *tokens_out = h->d.max_pos;
  return FS_OK;
}

int fs_selftest_bounded_wait(fs_handle* h, int32_t timeout_us, int32_t* code_out) {
  if (!h || !code_out || timeout_us < 1 || timeout_us > 1000000) return FS_ERR_ARG;
  h->launches += launch_wait_selftest((uint64_t)timeout_us * 1000ull, h->d_err_flag, h->stream);
  FS_CK(h, cudaGetLastError());
  return fs_device_error(h, code_out);
}

int fs_device_error(fs_handle* h, int32_t* code_out) {
  if (!h || !code_out) return FS_ERR_ARG;
  FS_CK(h, cudaStreamSynchronize(h->stream));
  *code_out = *(volatile int*)h->err_flag;
  *(volatile int*)h->err_flag = 0;
  return FS_OK;
}

}  // extern "C"

namespace {
// tcgen05 GEMM of the test hooks with stream-K width P and its own workspace.
int gemm_tc_hook(const uint16_t* W, int N, int K, const uint16_t* X, int B, float* Y, int P,
                 int reps, double* ms_out, cudaStream_t s, int cs_off = 0) {
  using namespace fsk;
  const TcOperands o{W, N, X, B, K, 0};
  const int m_tiles = (N + 127) / 128;
  if (!tc_width_ok(m_tiles, K / 64, P)) return FS_ERR_ARG;
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FS_ERR_CUDA;
  float* ws = nullptr;
  int *cnt = nullptr, *err = nullptr;
  const int max_groups = (B + 15) / 16;
  int rc = FS_OK;
  if (cudaMalloc(&ws, tc_ws_floats(P, B) * 4) != cudaSuccess ||
      cudaMalloc(&cnt, (size_t)m_tiles * max_groups * 4) != cudaSuccess ||
      cudaMalloc(&err, 4) != cudaSuccess) {
    rc = FS_ERR_OOM;
  } else {
    cudaMemsetAsync(cnt, 0, (size_t)m_tiles * max_groups * 4, s);
    cudaMemsetAsync(err, 0, 4, s);
    TcParams p{};
    p.m_tiles = m_tiles; p.P = P; p.kb_total = K / 64;
    p.lanes_total = B; p.sms = sms;
    tc_lane_groups(B, P, sms, &p.lg, &p.groups);
    p.tmem_cols = tc_tmem_cols(p.lg);
    p.epi = EPI_STORE; p.out_f32 = Y; p.ldo = N; p.n_out = N;
    p.ws = ws; p.counters = cnt; p.err = err;
    p.cs_off = cs_off;
    if (launch_gemm_tc(o, p, s) < 0) rc = FS_ERR_CUDA;
    if (rc == FS_OK && reps > 0 && ms_out) {
      // each launch between two events, after a 256 MiB memset that evicts
      // the operands from L2 and keeps the GPU busy (clocks up)
      const size_t flush_bytes = (size_t)256 << 20;
      void* flush = nullptr;
      std::vector<cudaEvent_t> ev(2 * (size_t)reps);
      for (auto& e : ev) cudaEventCreate(&e);
      if (cudaMalloc(&flush, flush_bytes) == cudaSuccess) {
        for (int r = 0; r < reps; ++r) {
          cudaMemsetAsync(flush, r & 0xff, flush_bytes, s);
          cudaEventRecord(ev[2 * r], s);
          launch_gemm_tc(o, p, s);
          cudaEventRecord(ev[2 * r + 1], s);
        }
        double sum = 0.0;
        bool ok = cudaEventSynchronize(ev.back()) == cudaSuccess;
        for (int r = 0; ok && r < reps; ++r) {
          float ms = 0.0f;
          ok = cudaEventElapsedTime(&ms, ev[2 * r], ev[2 * r + 1]) == cudaSuccess;
          sum += ms;
        }
        if (ok) *ms_out = sum / reps;
        cudaFree(flush);
      }
      for (auto& e : ev) cudaEventDestroy(e);
    }
    int herr = 0;
    if (rc != FS_OK) {
    } else if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemcpy(&herr, err, 4, cudaMemcpyDeviceToHost) != cudaSuccess)
      rc = FS_ERR_CUDA;
    else if (herr)
      rc = FS_ERR_DEVICE;
  }
  cudaFree(ws);
  cudaFree(cnt);
  cudaFree(err);
  return rc;
}
}  // namespace

extern "C" {

int fs_gemm_bf16(const uint16_t* W, int32_t N, int32_t K, const uint16_t* X, int32_t B,
                 float* Y, int32_t splits, int32_t path, void* stream) {
  using namespace fsk;
  if (!W || !X || !Y || N < 1 || K < 64 || K % 64 || B < 1 || splits < 1 ||
      splits > K / 64 || splits > 8 || path < 0 || path > 2)
    return FS_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (path == 0) {
    Mat m;
    m.w = W; m.N = N; m.K = K; m.Kp = K; m.wtype = W_BF16;
    GemmArgs g{};
    g.W = m; g.X = X; g.x_type = X_BF16; g.B = B; g.epi = EPI_STORE;
    g.out_f32 = Y; g.ldo = N; g.n_out = N;
    launch_gemv(g, s);
    if (cudaGetLastError() != cudaSuccess) return FS_ERR_CUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? FS_OK : FS_ERR_CUDA;
  }
  // stream-K width m_tiles * splits: every block's range is the K split of
  // one tile, so the pieces are exactly the `splits` K splits
  const int m_tiles = (N + 127) / 128;
  return gemm_tc_hook(W, N, K, X, B, Y, m_tiles * splits, 0, nullptr, s, path == 2 ? 1 : 0);
}

int fs_gemm_bf16_width(const uint16_t* W, int32_t N, int32_t K, const uint16_t* X, int32_t B,
                       float* Y, int32_t width, void* stream) {
  if (!W || !X || !Y || N < 1 || K < 64 || K % 64 || B < 1 || width < 1 ||
      (int64_t)width > (int64_t)((N + 127) / 128) * (K / 64))
    return FS_ERR_ARG;
  return gemm_tc_hook(W, N, K, X, B, Y, width, 0, nullptr, (cudaStream_t)stream);
}

int fs_gemm_bf16_time(const uint16_t* W, int32_t N, int32_t K, const uint16_t* X, int32_t B,
                      float* Y, int32_t width, int32_t reps, double* ms_out, void* stream) {
  if (!W || !X || !Y || !ms_out || N < 1 || K < 64 || K % 64 || B < 1 || width < 1 ||
      (int64_t)width > (int64_t)((N + 127) / 128) * (K / 64) || reps < 1)
    return FS_ERR_ARG;
  *ms_out = 0.0;
  return gemm_tc_hook(W, N, K, X, B, Y, width, reps, ms_out, (cudaStream_t)stream);
}

}  // extern "C"
