// Internal interfaces between the host orchestrator (fs_api.cu) and the
// kernel translation units. Not installed; not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cstdlib>
#include <utility>

namespace fsk {

// Programmatic dependent launch: a kernel waits for its predecessor in the
// stream (griddepcontrol.wait) before touching memory the predecessor may
// write or read, and immediately allows its successor to be scheduled, so
// a successor's launch and prologue overlap this kernel's tail. Without the
// launch attribute both instructions are no-ops.
__device__ __forceinline__ void pdl_wait() {
#if defined(__CUDA_ARCH__)
  asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}
__device__ __forceinline__ void pdl_trigger() {
#if defined(__CUDA_ARCH__)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}
bool pdl_enabled();  // FS_PDL=0 in the environment turns the attribute off

// ---- kernel timeline tracing. Off unless a buffer is installed: thread 0
// of every block of a traced kernel then appends one record with the
// %globaltimer time at entry, after its dependency wait, and at its end.
// The buffer pointer is a __constant__ of each translation unit (the
// library is built without relocatable device code; a constant-cache read
// keeps the untraced path free of a memory round trip at every block's
// start); fs_trace_enable installs it in all of them.
struct TraceRec {
  // tag << 40 | waited << 39 | smid << 24 | linear block index; waited: the
  // block passed its wait for the preceding kernel (a block that leaves
  // early, e.g. an attention split past the lane's length, does not wait)
  unsigned long long tag_sm_block;
  unsigned long long t_entry, t_ready, t_exit;  // ns
};
struct TraceBuf {
  unsigned long long count, cap;  // records appended (may exceed cap), capacity
  TraceRec rec[1];
};
// record tags
enum TraceTag {
  TR_EMBED = 1, TR_RMSNORM = 2, TR_SAMPLE = 3, TR_ARGMAX = 4,
  TR_ATTN_MMA = 5, TR_ATTN_TMA = 6, TR_ATTN_TILED = 7, TR_ATTN_WARP = 8,
  TR_ROPE_APPEND = 9, TR_GEMV = 10, TR_ATTN_PARTIAL = 11, TR_ATTN_COMBINE = 12,
  TR_GEMV_SWIGLU = 13,
  TR_GEMM = 16  // + the epilogue kind (Epi)
};

__device__ __forceinline__ unsigned long long gtime() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void trace_write(TraceBuf* b, unsigned tag, bool waited,
                                            unsigned long long t0, unsigned long long t1) {
  const unsigned long long i = atomicAdd(&b->count, 1ull);
  if (i >= b->cap) return;
  unsigned sm;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
  const unsigned long long blk =
      ((unsigned long long)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
  TraceRec r;
  r.tag_sm_block = ((unsigned long long)tag << 40) | ((unsigned long long)waited << 39) |
                   ((unsigned long long)(sm & 0x7fff) << 24) | (blk & 0xffffff);
  r.t_entry = t0;
  r.t_ready = t1;
  r.t_exit = gtime();
  b->rec[i] = r;
}

// Thread 0's marks kept in registers.
struct TraceMark {
  TraceBuf* b = nullptr;
  unsigned long long t0 = 0, t1 = 0;
  bool waited = false;
  __device__ __forceinline__ void begin(TraceBuf* buf) {
    if (threadIdx.x == 0 && threadIdx.y == 0 && threadIdx.z == 0 && buf) {
      b = buf;
      t0 = t1 = gtime();
    }
  }
  __device__ __forceinline__ void ready() {
    if (b) {
      t1 = gtime();
      waited = true;
    }
  }
  __device__ __forceinline__ void end(unsigned tag) {
    if (!b) return;
    trace_write(b, tag, waited, t0, t1);
    b = nullptr;
  }
};

// Thread 0's marks kept in a __shared__ unsigned long long[4] (buffer, entry,
// ready, waited), for kernels that have no registers to spare.
struct TraceSmem {
  static __device__ __forceinline__ void begin(unsigned long long* sm, TraceBuf* buf) {
    if (threadIdx.x == 0) {
      sm[0] = reinterpret_cast<unsigned long long>(buf);
      sm[3] = 0;
      if (buf) sm[1] = sm[2] = gtime();
    }
  }
  static __device__ __forceinline__ void ready(unsigned long long* sm) {
    if (threadIdx.x == 0 && sm[0]) {
      sm[2] = gtime();
      sm[3] = 1;
    }
  }
  static __device__ __forceinline__ void end(unsigned long long* sm, unsigned tag) {
    if (threadIdx.x == 0 && sm[0])
      trace_write(reinterpret_cast<TraceBuf*>(sm[0]), tag, sm[3] != 0, sm[1], sm[2]);
  }
};

// A TraceMark that writes its record when the kernel leaves its scope (for
// kernels with several exits).
struct TraceScope : TraceMark {
  unsigned tag;
  __device__ __forceinline__ TraceScope(TraceBuf* buf, unsigned t) : tag(t) { begin(buf); }
  __device__ __forceinline__ ~TraceScope() { end(tag); }
};

// Defines this translation unit's trace pointer and its host installer.
#define FS_TRACE_TU(name)                                                     \
  static __constant__ TraceBuf* g_trace = nullptr;                            \
  int trace_install_##name(TraceBuf* p) {                                     \
    return cudaMemcpyToSymbol(g_trace, &p, sizeof(p)) == cudaSuccess ? 1 : 0; \
  }
int trace_install_misc(TraceBuf* p);
int trace_install_gemm(TraceBuf* p);
int trace_install_gemv(TraceBuf* p);
int trace_install_attn(TraceBuf* p);
int trace_install_attn_mma(TraceBuf* p);
int trace_install_attn_warp(TraceBuf* p);
int trace_install_attn_tma(TraceBuf* p);
int trace_install_attn_tiled(TraceBuf* p);

// Kernel launch with the programmatic-stream-serialization attribute.
template <typename... K, typename... A>
inline cudaError_t launch_k(void (*kern)(K...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t s, A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<K>(args)...);
}
// The same with thread-block clusters of cluster_x blocks along x (grid.x a
// multiple of cluster_x).
template <typename... K, typename... A>
inline cudaError_t launch_k_cluster(void (*kern)(K...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t s, int cluster_x, A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cluster_x;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<K>(args)...);
}

enum WType { W_F32 = 0, W_BF16 = 1, W_Q8 = 2 };
enum XType { X_F32 = 0, X_BF16 = 1 };

// A weight matrix in the library's device layout: rows of Kp elements
// (K rounded up to 64, zero padded). Q8_0 is split into int8 codes [N][Kp]
// and fp16 scales [N][Kp/32] so that both are read with aligned vector loads.
struct Mat {
  const void* w = nullptr;
  const __half* scales = nullptr;
  int N = 0, K = 0, Kp = 0;
  int wtype = W_BF16;
};

// Device copy of one step's arguments (written by one H2D copy per step).
// Arrays have max_lanes entries; row b of every panel belongs to lane[b].
struct StepArgs {
  const int32_t* lane;
  const int32_t* pos;   // position of the token consumed (length before step)
  const int32_t* tok;
  const int32_t* upd_lane;  // page-table updates for this step
  const int32_t* upd_slot;
  const int32_t* upd_page;
  const int32_t* n_upd;
};

struct KV {
  void* k = nullptr;  // [L][n_pages][Hkv][page_size][hd] in kv dtype
  void* v = nullptr;
  int kv_f32 = 0;     // 1: f32, 0: bf16
  int64_t layer_stride = 0;  // elements per layer
  int Hkv = 0, hd = 0, page_size = 0;
  int32_t* pt = nullptr;     // [max_lanes][max_pages_per_lane]
  int max_pages = 0;
};

// RoPE of one rotate-half pair (x0 = element i, x1 = element i + hd/2) with
// cos c and sin s: (x0 c - x1 s, x1 c + x0 s), every product and sum rounded
// on its own (no contraction into fused multiply-adds). Every kernel that
// rotates q or k calls this, so a key written by one kernel has the same bits
// as the key another kernel would write.
__device__ __forceinline__ void rope_pair(float x0, float x1, float c, float s, float& y0,
                                          float& y1) {
  y0 = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
  y1 = __fadd_rn(__fmul_rn(x1, c), __fmul_rn(x0, s));
}

enum Epi {
  EPI_STORE = 0,
  EPI_RESID = 1,
  EPI_SWIGLU = 2,
  // per (lane, 128-row tile): the largest output and its lowest row index
  // (greedy sampling without writing the outputs; whole-tile pieces only)
  EPI_ARGMAX = 3
};

// Y = X * W^T over B panel rows with a fused epilogue:
//   EPI_STORE : out_f32[b * ldo + n] = y
//   EPI_RESID : out_f32[b * ldo + n] += y       (residual stream)
//   EPI_SWIGLU: W holds gate rows [0, F) then up rows [F, 2F);
//               out_x[b * ldo + f] = silu(gate) * up  (x_type panel)
// X is a panel [B][W.Kp] of x_type (zero padded beyond K).
struct GemmArgs {
  Mat W;
  const void* X;
  int x_type;
  int B;
  int epi;
  float* out_f32;
  void* out_x;
  int ldo;
  int n_out;  // output rows (W.N, or F for SwiGLU)
};

// Launchers (each returns the number of kernels launched).
int launch_gemv(const GemmArgs& a, cudaStream_t s);

// tcgen05 GEMM (bf16 weights and panels). Stream-K: the m_tiles * kb_total
// k-blocks are cut into P equal ranges; grid = P * groups, the lane groups
// of one range adjacent so they share its weight tiles through L2.
struct TcParams {
  int m_tiles, kb_total;
  int P;           // stream-K blocks per lane group (1 <= P <= m_tiles * kb_total)
  int groups;      // lane groups
  int lg;          // lanes per group (multiple of 16, <= 256)
  int lanes_total; // lanes of the step (panel rows 0 .. lanes_total-1)
  int tmem_cols;   // power of two >= max(32, lg)
  int sms;         // SMs of the device (stage budget: one or two blocks per SM)
  int stages, stage_bytes;  // set by the launcher
  int kq;          // k-blocks per stage (set by the launcher)
  int xh;          // panel rows per k-block of a stage: lg rounded up to 16 (set by the launcher)
  int prod_warps;  // TMA-issuing warps of single-piece blocks (set by the launcher)
  int epi;
  float* out_f32;
  void* out_x;
  int ldo;
  int n_out;       // output rows (W rows, or F for SwiGLU)
  float* ws;       // partial pieces [2][P][lanes_total][128] f32
  int* counters;   // [m_tiles * groups], zero between launches
  int* err;        // device-visible error flag
  // Q8_0 weights in tiles [m_tiles][kb], each its codes [128][64] int8 then
  // its scales [128][2] fp16 (one per 32 inputs): 8704 bytes
  const int8_t* q8_tiles;
  float* am_val;   // EPI_ARGMAX: [lanes_total][m_tiles] tile maxima
  int* am_idx;     //             and their row indices
  // 1: the panel has a remainder part (map tmX*lo): two MMAs per k-step,
  // W x hi then W x lo, into the one accumulator
  int split;
  int64_t lo_off;  // EPI_SWIGLU with split: remainders at out_x + lo_off
  // cluster reduction (set by the launcher): 0, or the number of K splits
  // of every row tile (P = m_tiles * cs, 2 <= cs <= 8) when the splits of
  // one (row tile, lane group) run as one thread-block cluster and sum their
  // partial tiles through distributed shared memory, in split order (the
  // order of the workspace reduction, so the bits are the same)
  int cs;
  int cs_off;      // 1: never the cluster reduction (the caller's workspace serves)
};
// Per lane, the argmax over the tiles' (max, index) pairs of an EPI_ARGMAX
// launch (lowest index on ties): tokens_out[b] for b < B.
int launch_argmax_tiles(const float* am_val, const int* am_idx, int B, int m_tiles,
                        int32_t* tokens_out, cudaStream_t s);
// Lanes per group of one tcgen05 GEMM call: at most tc_lg_max(); a matrix
// with fewer stream-K blocks than SMs is spread over more groups to fill
// about two blocks per SM, groups of at least lg_min lanes and of at least
// n/16 (rounded up to 16: at most about 16 groups per row tile; SmolLM2 at
// 960 lanes measured 1.70 ms per step with 64-lane groups against 1.84 with
// 32 and 1.90 with 128; up to 256 lanes this leaves lg_min). Groups split
// N only, so this may depend on the call's lane count.
// FS_TC_LG_MIN (16..256, a tuning knob read once) overrides the smallest
// lane group the fill rule may cut (0: the caller's value).
inline int tc_lg_min(int dflt) {
  static const int v = [] {
    const char* e = getenv("FS_TC_LG_MIN");
    const int x = e ? atoi(e) : 0;
    return x ? std::max(16, std::min(256, x)) : 0;
  }();
  return v ? v : dflt;
}
// Lanes of a group are at most 128 (the MMA's N could take 256, but a
// 256-lane group's stage holds 32 KB of panel next to 16 KB of weights, so
// only two stages fit the ring: the LM heads of SmolLM2 at 256 lanes and of
// its Q8_0 form at 960 lanes measured 40.3 -> 38.7 us and 216 -> 179 us).
// FS_TC_LG_MAX (16..256) overrides it, a tuning knob read once.
inline int tc_lg_max() {
  static const int v = [] {
    const char* e = getenv("FS_TC_LG_MAX");
    const int x = e ? atoi(e) : 128;
    return std::max(16, std::min(256, x / 16 * 16));
  }();
  return v;
}
// Blocks per SM the fill rule aims at (FS_TC_FILL=1 or 2, a tuning knob
// read once; default 2).
inline int tc_fill_per_sm() {
  static const int v = [] {
    const char* e = getenv("FS_TC_FILL");
    const int x = e ? atoi(e) : 2;
    return std::max(1, std::min(2, x));
  }();
  return v;
}
// lg_min: the smallest group the fill rule may cut (16 for bf16 weights;
// Q8_0 takes 32, as every group dequantises its weight tiles itself).
inline void tc_lane_groups(int n, int P, int sms, int* lg, int* groups, int lg_min = 16) {
  const int cap = tc_lg_max();
  int g = (n + cap - 1) / cap;
  if (P < sms) {
    const int fill = std::max(1, tc_fill_per_sm() * sms / P);
    const int m = std::max(tc_lg_min(lg_min), (n + 255) / 256 * 16);
    g = std::max(g, std::min(fill, std::max(1, (n + m - 1) / m)));
  }
  const int l = ((n + g - 1) / g + 15) / 16 * 16;
  *lg = l;
  *groups = (n + l - 1) / l;
}
// The kernel's stream-K index arithmetic is 32-bit: (P + 1) * T < 2^31 with
// T = m_tiles * kb_total.
inline bool tc_width_ok(int m_tiles, int kb_total, int P) {
  const int64_t T = (int64_t)m_tiles * kb_total;
  return P >= 1 && P <= T && (int64_t)(P + 1) * T < ((int64_t)1 << 31);
}
// Workspace floats of a launch: two slots per block and lane, 128 rows each.
inline size_t tc_ws_floats(int P, int lanes) { return (size_t)2 * P * lanes * 128; }
// TMEM columns of a block: a power of two >= max(32, lg).
inline int tc_tmem_cols(int lg) {
  int c = 32;
  while (c < lg) c *= 2;
  return c;
}
bool tc_available();
// K splits of a row tile may sum through a thread-block cluster (see
// TcParams::cs); FS_TC_CLUSTER=0, a comparison knob read once, keeps the
// workspace reduction everywhere.
bool tc_cluster_reduce();
// Tensor map of a bf16 [rows][Kp] matrix (Kp a multiple of 64) whose copies
// bring kq consecutive 64-wide k-blocks of box_rows rows; 0 on success.
int tc_make_map(const void* base, int64_t rows, int Kp, int box_rows, int kq, CUtensorMap* out);
// Operands of one tcgen05 GEMM launch: bf16 weights w [w_rows][Kp] (unused
// for Q8_0, whose tiles are in TcParams), the bf16 panel x [x_rows][Kp]
// and, with TcParams::split, its remainder panel at x + x_lo elements. All
// base addresses 16-byte aligned, Kp a multiple of 64.
struct TcOperands {
  const void* w;
  int64_t w_rows;
  const void* x;
  int64_t x_rows;
  int Kp;
  int64_t x_lo;
};
// Launches the GEMM; returns the number of launches (1), or -1 when a tensor
// map cannot be encoded (nothing launched).
int launch_gemm_tc(const TcOperands& o, const TcParams& p, cudaStream_t s);
// Same GEMM over Q8_0 tiles (p.q8_tiles), dequantised to bf16
// in shared memory inside the kernel.
int launch_gemm_tc_q8(const TcOperands& o, const TcParams& p, cudaStream_t s);
// Row-major Q8_0 codes [N][Kp] / scales [N][Kp/32] -> the tiled layout above
// (rows beyond N are zero).
int launch_tile_q8(const int8_t* codes, const __half* scales, int N, int Kp, int8_t* tiles,
                   cudaStream_t s);
// Row-major Q8_0 codes [N][Kp] / scales [N][Kp/32] -> bf16 [N][Kp] holding
// bf16(q * d), the operand value the Q8_0 GEMM dequantises in shared memory.
int launch_dequant_q8_bf16(const int8_t* codes, const __half* scales, int N, int Kp,
                           __nv_bfloat16* out, cudaStream_t s);

// x = E[tok]; if g is given also h = RMSNorm(x) * g (x_type panel).
// lo_off (elements, bf16 panels only; 0: none): the row's rounding
// remainders bf16(v - hi) are stored lo_off elements after its bf16 values.
int launch_embed(const Mat& E, const StepArgs& args, int B, const KV& kv, float* x, int d,
                 const float* g, float eps, void* h, int x_type, int ld_h, int64_t lo_off,
                 cudaStream_t s);
// x += resid (if resid is given), out = RMSNorm(x) * g (and its remainders
// at out + lo_off when lo_off > 0).
int launch_rmsnorm(float* x, const float* resid, const float* g, int B, int d, float eps,
                   void* out, int x_type, int ld_out, int64_t lo_off, cudaStream_t s);
int launch_rope_append(const float* qkv, int B, int H, int Hkv, int hd,
                       const float* rope_cos, const float* rope_sin,
                       const StepArgs& args, const KV& kv, int layer,
                       float* q_out, cudaStream_t s);
// Arguments of the tiled attention kernel (k_attn_tiled.cu).
struct AttnParams {
  const float* qkv;  // [B][(H + 2 Hkv) hd] projection output
  int H;
  const float* rc;   // RoPE cos [max_pos][hd/2]
  const float* rs;   // RoPE sin
  StepArgs args;
  KV kv;
  int layer;
  int split_len, max_splits;
  float* part_ml;    // [B][max_splits][H][2]
  float* part_acc;   // [B][max_splits][H][hd]
  int* counters;     // [B][Hkv]
  void* o;           // output panel
  int ld_o;
  int64_t o_lo;      // bf16 panel: remainders bf16(v - hi) at o + o_lo (0: none)
  int* err;          // device-visible error flag
  // 0: the block holding a row's position rotates k and appends k, v there;
  // 1: every row's k, v were appended by a preceding kernel of the step (rows
  //    of one lane at consecutive positions, chunked prefill), so the kernel
  //    appends nothing and reads no KV before its predecessor has finished
  int kv_written;
  int n_rows;        // panel rows of the step (set by the one-warp kernel's launcher)
};
bool attn_tiled_supports(int hd, int G, int page_size, int split_len);
bool attn_mma_supports(int hd, int G, int kv_f32, int split_len, int max_splits);
// One warp per (lane, KV head) for handles whose lanes hold at most 64
// positions (k_attn_warp.cu): the bits of k_attn_mma.
bool attn_warp_supports(int hd, int G, int kv_f32, int max_pos);
int launch_attention_warp(const AttnParams& a, int B, int x_type, cudaStream_t s);
// Same attention with the KV tiles fetched by TMA (k_attn_tma.cu): bf16 KV,
// page_size a multiple of 8 that divides or is a multiple of 64.
bool attn_tma_supports(int hd, int G, int kv_f32, int page_size, int split_len,
                       int max_splits);
int attn_tma_make_map(const void* arena, int64_t rows, int hd, int page_size, CUtensorMap* out);
int launch_attention_tma(const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnParams& a,
                         int B, int x_type, cudaStream_t s);
int launch_attention_mma(const AttnParams& a, int B, int x_type, cudaStream_t s);
int launch_attention_tiled(const AttnParams& a, int B, int x_type, cudaStream_t s);

int launch_sample(const float* logits, int B, int V, const float* temps,
                  const uint64_t* seeds, const uint64_t* counters,
                  int32_t* out, cudaStream_t s);
int launch_quantize_q8_0(const float* src, int64_t n, uint8_t* blocks,
                         cudaStream_t s);
int launch_repack_q8(const uint8_t* blocks, int N, int K, int Kp,
                     int8_t* qs, __half* scales, int row_offset,
                     cudaStream_t s);
int launch_fill_random_kv(const KV& kv, int L, const int32_t* pages,
                          int n_pages, uint64_t seed, cudaStream_t s);
int launch_import_kv(const KV& kv, int layer, const int32_t* pages, int n,
                     const float* k, const float* v, cudaStream_t s);
int launch_export_kv(const KV& kv, int layer, const int32_t* pages, int n,
                     float* k, float* v, cudaStream_t s);
// The failure-detection check's kernel (k_misc.cu): a bounded wait on a
// barrier nothing arrives on; sets *err to kErrSelftest when it gives up.
constexpr int kErrSelftest = 99;
int launch_wait_selftest(uint64_t timeout_ns, int* err, cudaStream_t s);
// Rows [q_begin, q_end) of one lane into the pages of dst_pt: row q from row
// q (q < a) or q + delta (q >= a) of src_pt's pages, keys moved down by delta
// turned back delta positions (k_misc.cu). Every layer, K and V.
int launch_kv_relocate(const KV& kv, int L, const int32_t* src_pt, const int32_t* dst_pt,
                       int q_begin, int q_end, int a, int delta, const float* rc,
                       const float* rs, cudaStream_t s);

}  // namespace fsk
