// Fused RoPE + paged KV append + per-lane split-K GQA decode attention.
//
// One block per (split s, KV head g, panel row b). Lane b's query heads
// g*G .. g*G+G-1 attend over the lane's own keys 0..pos_b ("MODEL-BATCHING-
// RESULTS", "The lever": per-user attention, no cross-user mixing), read from
// the lane's pages of the shared KV arena (mlx-bun "Parallel slots", "KV
// memory", rung 3). The block rotates its q heads itself from the QKV
// projection output; the block whose split holds position pos_b also rotates
// k and appends k and v at pos_b ("S1b decode: design traps", trap 2: the
// position is read once and used for both Q and K).
//
// Keys are split into fixed chunks of split_len positions (flash-decode);
// the number of splits of a lane depends only on its length. A lane with one
// split writes its output directly; otherwise every split writes (m, l, acc)
// and the last block of (b, g) to finish merges the splits in ascending
// order. Either way the result does not depend on B or on the other lanes.

#include <math_constants.h>

#include "fs_internal.h"

namespace fsk {
FS_TRACE_TU(attn_fused)
namespace {

constexpr int kT = 128;   // threads = keys per chunk
constexpr int kG = 8;     // max query heads per KV head

template <typename T>
struct KVIO;
template <>
struct KVIO<float> {
  static constexpr int kVec = 4;  // elements per 16-byte load
  __device__ static void load(const float* p, float* out) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
  }
  __device__ static float ld(const float* p) { return *p; }
  __device__ static void st(float* p, float v) { *p = v; }
};
template <>
struct KVIO<__nv_bfloat16> {
  static constexpr int kVec = 8;
  __device__ static void load(const __nv_bfloat16* p, float* out) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      out[2 * e] = f.x;
      out[2 * e + 1] = f.y;
    }
  }
  __device__ static float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  __device__ static void st(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};

__device__ __forceinline__ void st_out(float* p, float v) { *p = v; }
__device__ __forceinline__ void st_out(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);
}

__device__ __forceinline__ int64_t kv_base(const KV& kv, const int32_t* ptrow, int layer,
                                           int g, int t) {
  const int pi = t / kv.page_size;
  const int slot = t - pi * kv.page_size;
  return (int64_t)layer * kv.layer_stride +
         (((int64_t)ptrow[pi] * kv.Hkv + g) * kv.page_size + slot) * kv.hd;
}

template <typename KVT, typename OT, int HD>
__global__ void __launch_bounds__(kT)
    k_attn_fused(const float* __restrict__ qkv, int H, const float* __restrict__ rc,
                 const float* __restrict__ rs, StepArgs args, KV kv, int layer,
                 int split_len, int max_splits, float* __restrict__ part_ml,
                 float* __restrict__ part_acc, int* __restrict__ counters, OT* o_panel,
                 int ld_o, int kv_written) {
  TraceScope tr(g_trace, TR_ATTN_FUSED);
  pdl_wait();
  tr.ready();
  pdl_trigger();
  constexpr int kHalf = HD / 2;
  constexpr int kVec = KVIO<KVT>::kVec;
  constexpr int kOut = (kG * HD + kT - 1) / kT;  // outputs per thread (max)
  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int pos = args.pos[b];
  const int len = pos + 1;
  const int start = s * split_len;
  if (start >= len) return;
  const int end = min(len, start + split_len);
  const int ns = (len + split_len - 1) / split_len;
  const int Hkv = kv.Hkv;
  const int G = H / Hkv;
  const int tid = threadIdx.x;
  const int32_t* ptrow = kv.pt + (int64_t)args.lane[b] * kv.max_pages;
  KVT* K = static_cast<KVT*>(kv.k);
  KVT* V = static_cast<KVT*>(kv.v);

  __shared__ float qs[kG * HD];
  __shared__ float sp[kG][kT];
  __shared__ int64_t voff[kT];
  __shared__ float red[kT / 32][kG];
  __shared__ float s_alpha[kG], s_l[kG];
  __shared__ int s_last;

  // rotated queries of this KV head's G query heads
  const float* row = qkv + (int64_t)b * (H + 2 * Hkv) * HD;
  const float* c = rc + (int64_t)pos * kHalf;
  const float* sn = rs + (int64_t)pos * kHalf;
  for (int idx = tid; idx < G * kHalf; idx += kT) {
    const int h = idx / kHalf, i = idx - h * kHalf;
    const float a = row[(g * G + h) * HD + i], e = row[(g * G + h) * HD + i + kHalf];
    rope_pair(a, e, c[i], sn[i], qs[h * HD + i], qs[h * HD + i + kHalf]);
  }
  if (s == ns - 1 && !kv_written) {  // this split holds position pos: append k and v
    const int64_t off = kv_base(kv, ptrow, layer, g, pos);
    const float* kr = row + H * HD + g * HD;
    const float* vr = row + (H + Hkv) * HD + g * HD;
    for (int i = tid; i < kHalf; i += kT) {
      const float a = kr[i], e = kr[i + kHalf];
      float k0, k1;
      rope_pair(a, e, c[i], sn[i], k0, k1);
      KVIO<KVT>::st(K + off + i, k0);
      KVIO<KVT>::st(K + off + i + kHalf, k1);
    }
    for (int i = tid; i < HD; i += kT) KVIO<KVT>::st(V + off + i, vr[i]);
  }
  __syncthreads();

  const float scale = 1.0f / sqrtf((float)HD);
  float m[kG], l[kG], acc[kOut];
#pragma unroll
  for (int h = 0; h < kG; ++h) {
    m[h] = -CUDART_INF_F;
    l[h] = 0.0f;
  }
#pragma unroll
  for (int j = 0; j < kOut; ++j) acc[j] = 0.0f;
  const int warp = tid >> 5, lane = tid & 31;

  for (int c0 = start; c0 < end; c0 += kT) {
    const int t = c0 + tid;
    const bool valid = t < end;
    float sc[kG];
#pragma unroll
    for (int h = 0; h < kG; ++h) sc[h] = 0.0f;
    if (valid) {
      const int64_t ko = kv_base(kv, ptrow, layer, g, t);
      voff[tid] = ko;
#pragma unroll
      for (int e0 = 0; e0 < HD; e0 += kVec) {
        float kk[kVec];
        KVIO<KVT>::load(K + ko + e0, kk);
#pragma unroll
        for (int h = 0; h < kG; ++h)
          if (h < G) {
#pragma unroll
            for (int e = 0; e < kVec; ++e) sc[h] = fmaf(qs[h * HD + e0 + e], kk[e], sc[h]);
          }
      }
    }
    // block max per head (one pass for all heads)
    float mx[kG];
#pragma unroll
    for (int h = 0; h < kG; ++h) {
      float v = (valid && h < G) ? sc[h] * scale : -CUDART_INF_F;
      sc[h] = v;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
      mx[h] = v;
    }
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < kG; ++h) red[warp][h] = mx[h];
    }
    __syncthreads();
    float mnew[kG], alpha[kG];  // block-uniform
#pragma unroll
    for (int h = 0; h < kG; ++h) {
      float v = red[0][h];
#pragma unroll
      for (int w = 1; w < kT / 32; ++w) v = fmaxf(v, red[w][h]);
      mnew[h] = fmaxf(m[h], v);
    }
    __syncthreads();
    // probabilities and block sums
    float ps[kG];
#pragma unroll
    for (int h = 0; h < kG; ++h) {
      const float p = (valid && h < G) ? expf(sc[h] - mnew[h]) : 0.0f;
      sp[h][tid] = p;
      float v = p;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      ps[h] = v;
    }
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < kG; ++h) red[warp][h] = ps[h];
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < kG; ++h) {
      float v = red[0][h];
#pragma unroll
      for (int w = 1; w < kT / 32; ++w) v += red[w][h];
      alpha[h] = (m[h] == -CUDART_INF_F) ? 0.0f : expf(m[h] - mnew[h]);
      l[h] = l[h] * alpha[h] + v;
      m[h] = mnew[h];
      if (tid == 0) {  // block-uniform values, shared for runtime head indices
        s_alpha[h] = alpha[h];
        s_l[h] = l[h];
      }
    }
    __syncthreads();
    // P.V: thread owns outputs o = tid + j*kT, (head o / HD, dim o % HD)
    const int cnt = min(kT, end - c0);
#pragma unroll
    for (int j = 0; j < kOut; ++j) {
      const int o = tid + j * kT;
      if (o < G * HD) {
        const int h = o / HD, i = o - h * HD;
        float a = acc[j] * s_alpha[h];
        for (int u = 0; u < cnt; ++u) a = fmaf(sp[h][u], KVIO<KVT>::ld(V + voff[u] + i), a);
        acc[j] = a;
      }
    }
    __syncthreads();
  }

  OT* orow = o_panel + (int64_t)b * ld_o + g * G * HD;
  if (ns == 1) {
#pragma unroll
    for (int j = 0; j < kOut; ++j) {
      const int o = tid + j * kT;
      if (o < G * HD) st_out(orow + o, acc[j] / s_l[o / HD]);
    }
    return;
  }
  // several splits: publish this split, the last block of (b, g) merges
  const int64_t base = ((int64_t)b * max_splits + s) * H + g * G;
#pragma unroll
  for (int h = 0; h < kG; ++h)
    if (tid == 0 && h < G) {
      part_ml[2 * (base + h)] = m[h];
      part_ml[2 * (base + h) + 1] = l[h];
    }
#pragma unroll
  for (int j = 0; j < kOut; ++j) {
    const int o = tid + j * kT;
    if (o < G * HD) part_acc[base * HD + o] = acc[j];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    int* ctr = counters + (int64_t)b * Hkv + g;
    s_last = atomicAdd(ctr, 1) == ns - 1;
    if (s_last) *ctr = 0;  // every split has arrived: ready for the next step
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
#pragma unroll
  for (int j = 0; j < kOut; ++j) {
    const int o = tid + j * kT;
    if (o < G * HD) {
      const int h = o / HD;
      float mx = -CUDART_INF_F;
      for (int q = 0; q < ns; ++q)
        mx = fmaxf(mx, __ldcg(part_ml + 2 * (((int64_t)b * max_splits + q) * H + g * G + h)));
      float L = 0.0f, A = 0.0f;
      for (int q = 0; q < ns; ++q) {
        const int64_t bq = ((int64_t)b * max_splits + q) * H + g * G + h;
        const float w = expf(__ldcg(part_ml + 2 * bq) - mx);
        L = fmaf(__ldcg(part_ml + 2 * bq + 1), w, L);
        A = fmaf(__ldcg(part_acc + bq * HD + (o - h * HD)), w, A);
      }
      st_out(orow + o, A / L);
    }
  }
}

template <typename KVT, typename OT>
int dispatch_hd(int hd, dim3 grid, cudaStream_t s, const float* qkv, int H, const float* rc,
                const float* rs, const StepArgs& args, const KV& kv, int layer, int split_len,
                int max_splits, float* part_ml, float* part_acc, int* counters, OT* o,
                int ld_o, int kv_written) {
#define FS_ATTN_CASE(D)                                                                  \
  case D:                                                                                \
    launch_k(k_attn_fused<KVT, OT, D>, grid, kT, 0, s, qkv, H, rc, rs, args, kv, layer,        \
                                                 split_len, max_splits, part_ml,         \
                                                 part_acc, counters, o, ld_o, kv_written); \
    return 1;
  switch (hd) {
    FS_ATTN_CASE(16)
    FS_ATTN_CASE(32)
    FS_ATTN_CASE(64)
    FS_ATTN_CASE(128)
    FS_ATTN_CASE(256)
    default:
      return -1;
  }
#undef FS_ATTN_CASE
}

}  // namespace

bool attn_fused_supports(int hd, int G) {
  return (hd == 16 || hd == 32 || hd == 64 || hd == 128 || hd == 256) && G >= 1 && G <= kG;
}

int launch_attention_fused(const float* qkv, int B, int H, const float* rope_cos,
                           const float* rope_sin, const StepArgs& args, const KV& kv,
                           int layer, int max_splits, int split_len, float* part_ml,
                           float* part_acc, int* counters, void* o_panel, int x_type,
                           int ld_o, int kv_written, cudaStream_t s) {
  if (B <= 0) return 0;
  dim3 grid(max_splits, kv.Hkv, B);
  if (kv.kv_f32) {
    if (x_type == X_BF16)
      return dispatch_hd<float, __nv_bfloat16>(kv.hd, grid, s, qkv, H, rope_cos, rope_sin,
                                               args, kv, layer, split_len, max_splits,
                                               part_ml, part_acc, counters,
                                               static_cast<__nv_bfloat16*>(o_panel), ld_o,
                                               kv_written);
    return dispatch_hd<float, float>(kv.hd, grid, s, qkv, H, rope_cos, rope_sin, args, kv,
                                     layer, split_len, max_splits, part_ml, part_acc,
                                     counters, static_cast<float*>(o_panel), ld_o, kv_written);
  }
  if (x_type == X_BF16)
    return dispatch_hd<__nv_bfloat16, __nv_bfloat16>(
        kv.hd, grid, s, qkv, H, rope_cos, rope_sin, args, kv, layer, split_len, max_splits,
        part_ml, part_acc, counters, static_cast<__nv_bfloat16*>(o_panel), ld_o, kv_written);
  return dispatch_hd<__nv_bfloat16, float>(kv.hd, grid, s, qkv, H, rope_cos, rope_sin, args,
                                           kv, layer, split_len, max_splits, part_ml,
                                           part_acc, counters, static_cast<float*>(o_panel),
                                           ld_o, kv_written);
}

}  // namespace fsk
