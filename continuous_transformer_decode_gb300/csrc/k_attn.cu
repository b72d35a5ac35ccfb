// RoPE + paged KV append, and per-lane split-K GQA decode attention.
//
// Per-user attention: lane b's query attends only to lane b's own keys
// 0..pos_b ("MODEL-BATCHING-RESULTS", "The lever": attention is per-user,
// zero cross-user mixing). The KV lives in fixed-size pages of a shared
// arena (mlx-bun "Parallel slots", "KV memory", rung 3); lane b's page j
// holds its tokens [j*P, (j+1)*P). The position is read once per lane and
// used for both Q and K ("S1b decode: design traps", trap 2).
//
// Attention is split along the lane's keys into fixed chunks of split_len
// tokens (flash-decode); the number of splits depends only on the lane's
// own length, and the combine runs the splits in ascending order, so the
// result does not depend on B or on the other lanes.

#include <math_constants.h>

#include "fs_internal.h"

namespace fsk {
FS_TRACE_TU(attn)
namespace {

template <typename T>
__device__ __forceinline__ float ld_f(const T* p, int64_t i);
template <>
__device__ __forceinline__ float ld_f<float>(const float* p, int64_t i) {
  return p[i];
}
template <>
__device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16* p,
                                                     int64_t i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void st_f(float* p, int64_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st_f(__nv_bfloat16* p, int64_t i, float v) {
  p[i] = __float2bfloat16_rn(v);
}

// Offset (elements) of token `t` of KV head `g` in layer `layer` for a lane
// whose page-table row is `ptrow`.
__device__ __forceinline__ int64_t kv_off(const KV& kv, const int32_t* ptrow,
                                          int layer, int g, int t) {
  const int page = ptrow[t / kv.page_size];
  const int slot = t - (t / kv.page_size) * kv.page_size;
  return (int64_t)layer * kv.layer_stride +
         (((int64_t)page * kv.Hkv + g) * kv.page_size + slot) * kv.hd;
}

template <typename KVT>
__global__ void k_rope_append(const float* __restrict__ qkv, int H, int Hkv,
                              int hd, const float* __restrict__ rc,
                              const float* __restrict__ rs, StepArgs args,
                              KV kv, int layer, float* __restrict__ q_out) {
  TraceScope tr(g_trace, TR_ROPE_APPEND);
  pdl_wait();
  tr.ready();
  pdl_trigger();
  const int b = blockIdx.x;
  const int lane = args.lane[b];
  const int pos = args.pos[b];
  const int half = hd / 2;
  const int nq = H * hd, nk = Hkv * hd;
  const float* row = qkv + (int64_t)b * (nq + 2 * nk);
  const float* c = rc + (int64_t)pos * half;
  const float* s = rs + (int64_t)pos * half;
  const int32_t* ptrow = kv.pt + (int64_t)lane * kv.max_pages;
  KVT* K = static_cast<KVT*>(kv.k);
  KVT* V = static_cast<KVT*>(kv.v);
  for (int idx = threadIdx.x; idx < H * half; idx += blockDim.x) {
    const int h = idx / half, i = idx - h * half;
    const float a = row[h * hd + i], e = row[h * hd + i + half];
    float* qo = q_out + (int64_t)b * nq + h * hd;
    rope_pair(a, e, c[i], s[i], qo[i], qo[i + half]);
  }
  for (int idx = threadIdx.x; idx < Hkv * half; idx += blockDim.x) {
    const int g = idx / half, i = idx - g * half;
    const float a = row[nq + g * hd + i], e = row[nq + g * hd + i + half];
    const int64_t off = kv_off(kv, ptrow, layer, g, pos);
    float k0, k1;
    rope_pair(a, e, c[i], s[i], k0, k1);
    st_f(K, off + i, k0);
    st_f(K, off + i + half, k1);
  }
  for (int idx = threadIdx.x; idx < Hkv * hd; idx += blockDim.x) {
    const int g = idx / hd, i = idx - g * hd;
    st_f(V, kv_off(kv, ptrow, layer, g, pos) + i, row[nq + nk + idx]);
  }
}

constexpr int kCh = 128;     // tokens per chunk = threads per block
constexpr int kMaxG = 8;     // query heads per KV head
constexpr int kMaxHd = 256;

__device__ __forceinline__ float block_reduce(float v, bool is_max,
                                              float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float u = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, u) : v + u;
  }
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float r = red[0];
  for (int i = 1; i < kCh / 32; ++i) r = is_max ? fmaxf(r, red[i]) : r + red[i];
  return r;
}

// One block = (split s, KV head g, panel row b). Writes the split's running
// max m, sum l and unnormalised output acc for the G query heads of g.
template <typename KVT>
__global__ void __launch_bounds__(kCh)
    k_attn_partial(const float* __restrict__ q, int H, StepArgs args, KV kv,
                   int layer, int split_len, int max_splits,
                   float* __restrict__ part_ml, float* __restrict__ part_acc) {
  TraceScope tr(g_trace, TR_ATTN_PARTIAL);
  pdl_wait();
  tr.ready();
  pdl_trigger();
  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int len = args.pos[b] + 1;
  const int start = s * split_len;
  if (start >= len) return;
  const int end = min(len, start + split_len);
  const int hd = kv.hd;
  const int G = H / kv.Hkv;
  const int lane = args.lane[b];
  const int32_t* ptrow = kv.pt + (int64_t)lane * kv.max_pages;
  const KVT* K = static_cast<const KVT*>(kv.k);
  const KVT* V = static_cast<const KVT*>(kv.v);

  __shared__ float qs[kMaxG * kMaxHd];
  __shared__ float ps[kMaxG][kCh];
  __shared__ int64_t voff[kCh];
  __shared__ float red[kCh / 32];

  for (int i = threadIdx.x; i < G * hd; i += kCh)
    qs[i] = q[((int64_t)b * H + g * G) * hd + i];
  __syncthreads();

  const float scale = 1.0f / sqrtf((float)hd);
  float m[kMaxG], l[kMaxG];
  for (int h = 0; h < G; ++h) {
    m[h] = -CUDART_INF_F;
    l[h] = 0.0f;
  }
  constexpr int kOut = kMaxG * kMaxHd / kCh;  // outputs owned per thread
  float acc[kOut];
#pragma unroll
  for (int j = 0; j < kOut; ++j) acc[j] = 0.0f;
  const int n_out = G * hd;

  for (int c0 = start; c0 < end; c0 += kCh) {
    const int t = c0 + threadIdx.x;
    const bool valid = t < end;
    float sc[kMaxG];
    if (valid) {
      const int64_t ko = kv_off(kv, ptrow, layer, g, t);
      voff[threadIdx.x] = ko;
      for (int h = 0; h < G; ++h) sc[h] = 0.0f;
      for (int i = 0; i < hd; ++i) {
        const float kk = ld_f(K, ko + i);
        for (int h = 0; h < G; ++h) sc[h] = fmaf(qs[h * hd + i], kk, sc[h]);
      }
      for (int h = 0; h < G; ++h) sc[h] *= scale;
    } else {
      for (int h = 0; h < G; ++h) sc[h] = -CUDART_INF_F;
    }
    float alpha[kMaxG];
    for (int h = 0; h < G; ++h) {
      const float cmax = block_reduce(sc[h], true, red);
      const float mnew = fmaxf(m[h], cmax);
      const float p = valid ? expf(sc[h] - mnew) : 0.0f;
      ps[h][threadIdx.x] = p;
      const float csum = block_reduce(p, false, red);
      alpha[h] = (m[h] == -CUDART_INF_F) ? 0.0f : expf(m[h] - mnew);
      l[h] = l[h] * alpha[h] + csum;
      m[h] = mnew;
    }
    __syncthreads();
    const int cnt = min(kCh, end - c0);
#pragma unroll
    for (int j = 0; j < kOut; ++j) {
      const int o = threadIdx.x + j * kCh;
      if (o < n_out) {
        const int h = o / hd, i = o - h * hd;
        float a = acc[j] * alpha[h];
        for (int u = 0; u < cnt; ++u) a = fmaf(ps[h][u], ld_f(V, voff[u] + i), a);
        acc[j] = a;
      }
    }
    __syncthreads();
  }
  const int64_t base = ((int64_t)b * max_splits + s) * H + g * G;
  if (threadIdx.x < G) {
    part_ml[2 * (base + threadIdx.x)] = m[threadIdx.x];
    part_ml[2 * (base + threadIdx.x) + 1] = l[threadIdx.x];
  }
#pragma unroll
  for (int j = 0; j < kOut; ++j) {
    const int o = threadIdx.x + j * kCh;
    if (o < n_out) part_acc[base * hd + o] = acc[j];
  }
}

// Merges a lane's splits in ascending order and writes o = acc / l.
template <typename OT>
__global__ void k_attn_combine(int H, int hd, StepArgs args, int split_len,
                               int max_splits, const float* __restrict__ part_ml,
                               const float* __restrict__ part_acc, OT* o,
                               int ld_o) {
  TraceScope tr(g_trace, TR_ATTN_COMBINE);
  pdl_wait();
  tr.ready();
  pdl_trigger();
  const int b = blockIdx.x;
  const int len = args.pos[b] + 1;
  const int ns = (len + split_len - 1) / split_len;
  for (int idx = threadIdx.x; idx < H * hd; idx += blockDim.x) {
    const int h = idx / hd, i = idx - h * hd;
    float mx = -CUDART_INF_F;
    for (int s = 0; s < ns; ++s)
      mx = fmaxf(mx, part_ml[2 * (((int64_t)b * max_splits + s) * H + h)]);
    float L = 0.0f, A = 0.0f;
    for (int s = 0; s < ns; ++s) {
      const int64_t base = ((int64_t)b * max_splits + s) * H + h;
      const float w = expf(part_ml[2 * base] - mx);
      L = fmaf(part_ml[2 * base + 1], w, L);
      A = fmaf(part_acc[base * hd + i], w, A);
    }
    st_f(o, (int64_t)b * ld_o + idx, A / L);
  }
}

}  // namespace

int launch_rope_append(const float* qkv, int B, int H, int Hkv, int hd,
                       const float* rope_cos, const float* rope_sin,
                       const StepArgs& args, const KV& kv, int layer,
                       float* q_out, cudaStream_t s) {
  if (B <= 0) return 0;
  if (kv.kv_f32)
    launch_k(k_rope_append<float>, B, 256, 0, s, qkv, H, Hkv, hd, rope_cos, rope_sin,
                                           args, kv, layer, q_out);
  else
    launch_k(k_rope_append<__nv_bfloat16>, B, 256, 0, s, 
        qkv, H, Hkv, hd, rope_cos, rope_sin, args, kv, layer, q_out);
  return 1;
}

int launch_attention(const float* q, int B, int H, const StepArgs& args,
                     const KV& kv, int layer, int max_splits, int split_len,
                     float* part_ml, float* part_acc, void* o_panel,
                     int x_type, int ld_o, cudaStream_t s) {
  if (B <= 0) return 0;
  dim3 grid(max_splits, kv.Hkv, B);
  if (kv.kv_f32)
    launch_k(k_attn_partial<float>, grid, kCh, 0, s, q, H, args, kv, layer,
                                               split_len, max_splits, part_ml,
                                               part_acc);
  else
    launch_k(k_attn_partial<__nv_bfloat16>, grid, kCh, 0, s, 
        q, H, args, kv, layer, split_len, max_splits, part_ml, part_acc);
  if (x_type == X_BF16)
    launch_k(k_attn_combine<__nv_bfloat16>, B, 256, 0, s, 
        H, kv.hd, args, split_len, max_splits, part_ml, part_acc,
        static_cast<__nv_bfloat16*>(o_panel), ld_o);
  else
    launch_k(k_attn_combine<float>, B, 256, 0, s, H, kv.hd, args, split_len,
                                            max_splits, part_ml, part_acc,
                                            static_cast<float*>(o_panel), ld_o);
  return 2;
}

}  // namespace fsk
