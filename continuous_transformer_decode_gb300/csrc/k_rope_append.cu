// RoPE + paged KV append of every row of a chunked step.
//
// A chunked step (several rows of one lane at consecutive positions) first
// rotates and appends every row's k and v, so that the attention kernels,
// run afterwards in read-only mode, let a row see its lane's earlier rows of
// the same step. The KV lives in fixed-size pages of a shared arena (mlx-bun
// "Parallel slots", "KV memory", rung 3); lane b's page j holds its tokens
// [j*P, (j+1)*P). The position is read once per row and used for both Q and
// K ("S1b decode: design traps", trap 2).

#include "fs_internal.h"

namespace fsk {
FS_TRACE_TU(attn)
namespace {

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

}  // namespace fsk
