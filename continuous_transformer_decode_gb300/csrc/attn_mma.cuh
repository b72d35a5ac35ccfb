// Warp-level tensor-core helpers shared by the decode-attention kernels
// (k_attn_mma.cu, k_attn_tma.cu): ldmatrix loads, the m16n8k16 bf16 MMA,
// and the split of f32 values into a bf16 pair (hi + lo) that keeps their
// products with exact bf16 keys and values near f32 accuracy.
#pragma once

#include "fs_internal.h"

namespace fsk {
namespace attn {

// 16-byte asynchronous copy global -> shared (L2 only), its group commit and
// the wait for all but N groups.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t r[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t r[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// D += A(16x16) * B(16x8): rows 0..7 of A hold the hi parts of the heads,
// rows 8..15 the lo parts; D rows follow (d0, d1: hi; d2, d3: lo).
__device__ __forceinline__ void mma16816(float d[4], const uint32_t a[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// (lo, hi) f32 pair -> bf16 pair "hi" and the bf16 pair of the remainders.
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = pack_bf16(x0 - hf.x, x1 - hf.y);
}
// An output element; a bf16 panel with a remainder part (lo > 0) also gets
// bf16(v - hi) lo elements further on.
__device__ __forceinline__ void st_out(float* p, float v, int64_t) { *p = v; }
__device__ __forceinline__ void st_out(__nv_bfloat16* p, float v, int64_t lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  *p = h;
  if (lo > 0) p[lo] = __float2bfloat16_rn(v - __bfloat162float(h));
}

}  // namespace attn
}  // namespace fsk
