// Weight-streaming skinny GEMM, warp-per-row form ("GEMV tiles").
//
// Y[b, n] = sum_k X[b, k] * W[n, k] for the B rows of the step panel
// ("MODEL-BATCHING-RESULTS", "The lever": each weight row is read once per
// step and reused for every lane of the [B, *] panel).
//
// One warp owns one output row n (two rows, gate and up, for SwiGLU). The
// row is streamed with 128-bit loads in chunks of 256 elements (8 per
// thread); each weight vector is reused for LG lanes held in registers.
// Every (n, b) element is reduced in the same order whatever B is or which
// lane group b falls in: per thread ascending k inside its 8-element slots,
// chunks ascending, then a fixed xor-butterfly over the warp. That makes a
// lane's result independent of the batch composition (batch invariance).

#include "fs_internal.h"

namespace fsk {
FS_TRACE_TU(gemv)
namespace {

constexpr int kWarps = 8;
constexpr int kLG = 4;  // lanes per register group

__device__ __forceinline__ void load8_w(const Mat& W, int row, int k0,
                                        float w[8]) {
  if (W.wtype == W_BF16) {
    const uint4 u = *reinterpret_cast<const uint4*>(
        static_cast<const __nv_bfloat16*>(W.w) + (int64_t)row * W.Kp + k0);
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float2 f = __bfloat1622float2(p[e]);
      w[2 * e] = f.x;
      w[2 * e + 1] = f.y;
    }
  } else if (W.wtype == W_F32) {
    const float* base = static_cast<const float*>(W.w) + (int64_t)row * W.Kp + k0;
    float4 a = *reinterpret_cast<const float4*>(base);
    float4 b = *reinterpret_cast<const float4*>(base + 4);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  } else {
    const uint2 u = *reinterpret_cast<const uint2*>(
        static_cast<const int8_t*>(W.w) + (int64_t)row * W.Kp + k0);
    const float d = __half2float(W.scales[(int64_t)row * (W.Kp / 32) + k0 / 32]);
    const int8_t* q = reinterpret_cast<const int8_t*>(&u);
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e] = (float)q[e] * d;  // exact in f32
  }
}

__device__ __forceinline__ void load8_x(const void* X, int x_type, int ldx,
                                        int b, int k0, float x[8]) {
  if (x_type == X_BF16) {
    const uint4 u = *reinterpret_cast<const uint4*>(
        static_cast<const __nv_bfloat16*>(X) + (int64_t)b * ldx + k0);
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float2 f = __bfloat1622float2(p[e]);
      x[2 * e] = f.x;
      x[2 * e + 1] = f.y;
    }
  } else {
    const float* base = static_cast<const float*>(X) + (int64_t)b * ldx + k0;
    float4 a = *reinterpret_cast<const float4*>(base);
    float4 c = *reinterpret_cast<const float4*>(base + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = c.x; x[5] = c.y; x[6] = c.z; x[7] = c.w;
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

template <bool kSwiglu>
__global__ void __launch_bounds__(kWarps * 32) k_gemv(GemmArgs a) {
  TraceScope tr(g_trace, kSwiglu ? TR_GEMV_SWIGLU : TR_GEMV);
  pdl_wait();
  tr.ready();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, t = threadIdx.x & 31;
  const int row = blockIdx.x * kWarps + warp;
  if (row >= a.n_out) return;
  const Mat& W = a.W;
  const int Kp = W.Kp;
  const int up_row = kSwiglu ? row + a.n_out : row;
  for (int b0 = 0; b0 < a.B; b0 += kLG) {
    float acc[kLG], acc2[kLG];
#pragma unroll
    for (int l = 0; l < kLG; ++l) acc[l] = acc2[l] = 0.0f;
    for (int k0 = t * 8; k0 < Kp; k0 += 256) {
      float w[8], w2[8], x[8];
      load8_w(W, row, k0, w);
      if (kSwiglu) load8_w(W, up_row, k0, w2);
#pragma unroll
      for (int l = 0; l < kLG; ++l) {
        if (b0 + l < a.B) {
          load8_x(a.X, a.x_type, Kp, b0 + l, k0, x);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            acc[l] = fmaf(w[e], x[e], acc[l]);
            if (kSwiglu) acc2[l] = fmaf(w2[e], x[e], acc2[l]);
          }
        }
      }
    }
#pragma unroll
    for (int l = 0; l < kLG; ++l) {
      const int b = b0 + l;
      float y = warp_sum(acc[l]);
      float y2 = kSwiglu ? warp_sum(acc2[l]) : 0.0f;
      if (t == 0 && b < a.B) {
        if (kSwiglu) {
          const float v = silu(y) * y2;
          if (a.x_type == X_BF16)
            static_cast<__nv_bfloat16*>(a.out_x)[(int64_t)b * a.ldo + row] =
                __float2bfloat16_rn(v);
          else
            static_cast<float*>(a.out_x)[(int64_t)b * a.ldo + row] = v;
        } else if (a.epi == EPI_RESID) {
          a.out_f32[(int64_t)b * a.ldo + row] += y;
        } else {
          a.out_f32[(int64_t)b * a.ldo + row] = y;
        }
      }
    }
  }
}

}  // namespace

int launch_gemv(const GemmArgs& a, cudaStream_t s) {
  if (a.B <= 0) return 0;
  dim3 grid((a.n_out + kWarps - 1) / kWarps);
  if (a.epi == EPI_SWIGLU)
    launch_k(k_gemv<true>, grid, kWarps * 32, 0, s, a);
  else
    launch_k(k_gemv<false>, grid, kWarps * 32, 0, s, a);
  return 1;
}

}  // namespace fsk
