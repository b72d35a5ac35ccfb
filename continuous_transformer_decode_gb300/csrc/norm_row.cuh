// One row of "residual add, then RMSNorm" computed by 128 threads:
//   if y: x += y (written back, the residual stream);
//   out = x * (1 / sqrt(mean(x^2) + eps)) * g  (bf16 or f32 panel row).
// Thread t owns the float4 chunks t, t + 128, ... of the row; the sum of
// squares is taken per thread in that order, then over the warp with a fixed
// xor butterfly, then over the 4 warps in warp order. Every kernel that
// normalises a row uses this routine, so a row's bits do not depend on which
// kernel did it or on the batch. d must be a multiple of 4, at most 8192.
#pragma once

#include "fs_internal.h"

namespace fsk {

constexpr int kNormRowThreads = 128;
// MaxVec bounds the float4 chunks per thread (d <= 512 * MaxVec). Chunks past
// d contribute exact zeros, so every MaxVec >= d / 512 gives the same bits.

// The routine in two halves, so that what does not depend on the preceding
// kernel (the row of x when it was written two or more kernels earlier, and
// the gains) is loaded before waiting for it: load() reads x and g (or
// load_g() the gains and, after the wait, load_x() a row of x that the
// preceding kernel wrote), finish() adds y (the preceding kernel's output),
// normalises and stores. The arithmetic is that of the one-piece routine
// below.
template <int MaxVec>
struct NormRow {
  float4 v[MaxVec], gg[MaxVec];
  __device__ __forceinline__ void load(const float* __restrict__ x, const float* __restrict__ g,
                                       int d, int t) {
    const int nvec = d >> 2;
#pragma unroll
    for (int j = 0; j < MaxVec; ++j) {
      const int c = t + kNormRowThreads * j;
      v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      gg[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c < nvec) {
        v[j] = *reinterpret_cast<const float4*>(x + 4 * c);
        gg[j] = *reinterpret_cast<const float4*>(g + 4 * c);
      }
    }
  }
  __device__ __forceinline__ void load_g(const float* __restrict__ g, int d, int t) {
    const int nvec = d >> 2;
#pragma unroll
    for (int j = 0; j < MaxVec; ++j) {
      const int c = t + kNormRowThreads * j;
      gg[j] = c < nvec ? *reinterpret_cast<const float4*>(g + 4 * c)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  // through L2: the row may have been written by the preceding kernel
  __device__ __forceinline__ void load_x(const float* x, int d, int t) {
    const int nvec = d >> 2;
#pragma unroll
    for (int j = 0; j < MaxVec; ++j) {
      const int c = t + kNormRowThreads * j;
      v[j] = c < nvec ? __ldcg(reinterpret_cast<const float4*>(x + 4 * c))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  // `bar` is a named barrier id used by exactly the 128 participating
  // threads; `red` is 4 floats of shared memory.
  // lo_off > 0 (bf16 out only): the remainders bf16(v - hi) go to
  // out + lo_off.
  template <typename OT>
  __device__ __forceinline__ void finish(float* __restrict__ x, const float* y, int d, float eps,
                                         OT* __restrict__ out, int t, int bar, float* red,
                                         int64_t lo_off = 0) {
    const int nvec = d >> 2;
    if (y) {
#pragma unroll
      for (int j = 0; j < MaxVec; ++j) {
        const int c = t + kNormRowThreads * j;
        if (c < nvec) {
          const float4 r = __ldcg(reinterpret_cast<const float4*>(y + 4 * c));
          v[j].x += r.x;
          v[j].y += r.y;
          v[j].z += r.z;
          v[j].w += r.w;
        }
      }
    }
    float ss = 0.0f;
#pragma unroll
    for (int j = 0; j < MaxVec; ++j) {
      ss = fmaf(v[j].x, v[j].x, ss);
      ss = fmaf(v[j].y, v[j].y, ss);
      ss = fmaf(v[j].z, v[j].z, ss);
      ss = fmaf(v[j].w, v[j].w, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    asm volatile("bar.sync %0, 128;" ::"r"(bar) : "memory");
    if ((t & 31) == 0) red[t >> 5] = ss;
    asm volatile("bar.sync %0, 128;" ::"r"(bar) : "memory");
    ss = ((red[0] + red[1]) + red[2]) + red[3];
    asm volatile("bar.sync %0, 128;" ::"r"(bar) : "memory");  // red is reusable
    const float rs = 1.0f / sqrtf(ss / (float)d + eps);
#pragma unroll
    for (int j = 0; j < MaxVec; ++j) {
      const int c = t + kNormRowThreads * j;
      if (c < nvec) {
        if (y) *reinterpret_cast<float4*>(x + 4 * c) = v[j];
        const float o0 = v[j].x * rs * gg[j].x, o1 = v[j].y * rs * gg[j].y;
        const float o2 = v[j].z * rs * gg[j].z, o3 = v[j].w * rs * gg[j].w;
        if constexpr (sizeof(OT) == 2) {
          const __nv_bfloat162 lo = __floats2bfloat162_rn(o0, o1);
          const __nv_bfloat162 hi = __floats2bfloat162_rn(o2, o3);
          uint2 pk;
          pk.x = *reinterpret_cast<const uint32_t*>(&lo);
          pk.y = *reinterpret_cast<const uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(out + 4 * c) = pk;
          if (lo_off > 0) {
            const float2 fl = __bfloat1622float2(lo), fh = __bfloat1622float2(hi);
            const __nv_bfloat162 rl = __floats2bfloat162_rn(o0 - fl.x, o1 - fl.y);
            const __nv_bfloat162 rh = __floats2bfloat162_rn(o2 - fh.x, o3 - fh.y);
            pk.x = *reinterpret_cast<const uint32_t*>(&rl);
            pk.y = *reinterpret_cast<const uint32_t*>(&rh);
            *reinterpret_cast<uint2*>(out + lo_off + 4 * c) = pk;
          }
        } else {
          *reinterpret_cast<float4*>(out + 4 * c) = make_float4(o0, o1, o2, o3);
        }
      }
    }
  }
};

// One-piece form: load() then finish().
template <typename OT, int MaxVec>
__device__ __forceinline__ void norm_row_128(float* __restrict__ x, const float* y,
                                             const float* __restrict__ g, int d, float eps,
                                             OT* __restrict__ out, int t, int bar, float* red,
                                             int64_t lo_off = 0) {
  NormRow<MaxVec> n;
  n.load(x, g, d, t);
  n.template finish<OT>(x, y, d, eps, out, t, bar, red, lo_off);
}

}  // namespace fsk
