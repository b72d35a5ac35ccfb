// Per-lane GQA decode attention over paged KV, streamed through shared memory.
//
// The attention of f32-KV handles and head dims below 64 (RoPE of q and k at
// the lane's own position, append of k and v at that position, online-softmax attention of
// the lane's query heads over its own keys 0..pos, split-K with an ordered
// merge; "MODEL-BATCHING-RESULTS", "The lever"; mlx-bun "Parallel slots",
// "KV memory" rung 3; "S1b decode: design traps" trap 2), organised for
// bandwidth on long contexts:
//   * a block = (split s, KV head g, panel row b) walks its split in tiles of
//     64 positions; every 16-position page of a tile is one contiguous block
//     per KV head, fetched with one cp.async.bulk (K and V), double-buffered
//     on two mbarriers (every wait bounded, errors reported by flag);
//   * scores: thread -> (head, position) pairs, a 128-bit dot over the
//     position's K row read from shared memory in a rotated chunk order
//     (fixed per position, so the bits do not depend on the batch);
//   * one warp-level max / sum pass per tile serves all heads; P.V reads V
//     from shared memory.
// The appended token's k and v are patched into the tile in shared memory
// from registers, so the block never reads back its own global write.

#include <math_constants.h>

#include "fs_internal.h"

namespace fsk {
FS_TRACE_TU(attn_tiled)
namespace {

constexpr int kT = 128;   // threads
constexpr int kG = 8;     // max query heads per KV head
constexpr int kTT = 64;   // positions per tile
constexpr uint64_t kWaitNs = 1000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  while (!mbar_test(bar, parity))
    if (gtimer() - t0 > kWaitNs) return false;
  return true;
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"((uint64_t)src), "r"(bytes), "r"(bar)
      : "memory");
}

template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kVec = 4;
  __device__ static void load(const float* p, float* o) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
  __device__ static float ld(const float* p) { return *p; }
  __device__ static float round(float v) { return v; }
  __device__ static void st(float* p, float v) { *p = v; }
};
template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kVec = 8;
  __device__ static void load(const __nv_bfloat16* p, float* o) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      o[2 * e] = f.x;
      o[2 * e + 1] = f.y;
    }
  }
  __device__ static float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  __device__ static void st(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};

// An output element; a bf16 panel with a remainder part (lo > 0) also gets
// bf16(v - hi) lo elements further on.
__device__ __forceinline__ void st_out(float* p, float v, int64_t) { *p = v; }
__device__ __forceinline__ void st_out(__nv_bfloat16* p, float v, int64_t lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  *p = h;
  if (lo > 0) p[lo] = __float2bfloat16_rn(v - __bfloat162float(h));
}

template <typename KVT, typename OT, int HD>
__global__ void __launch_bounds__(kT) k_attn_tiled(AttnParams a) {
  TraceScope tr(g_trace, TR_ATTN_TILED);
  pdl_wait();
  tr.ready();
  pdl_trigger();
  constexpr int kHalf = HD / 2;
  constexpr int kVec = Elem<KVT>::kVec;
  constexpr int kChunks = HD / kVec;               // 16-byte chunks per row
  constexpr int kOut = (kG * HD + kT - 1) / kT;
  const KV& kv = a.kv;
  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int pos = a.args.pos[b];
  const int len = pos + 1;
  const int start = s * a.split_len;
  if (start >= len) return;
  const int end = min(len, start + a.split_len);
  const int ns = (len + a.split_len - 1) / a.split_len;
  const int H = a.H, Hkv = kv.Hkv, G = H / Hkv, ps = kv.page_size;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t* ptrow = kv.pt + (int64_t)a.args.lane[b] * kv.max_pages;
  KVT* Kg = static_cast<KVT*>(kv.k);
  KVT* Vg = static_cast<KVT*>(kv.v);
  const bool owns_pos = (s == ns - 1);

  extern __shared__ __align__(128) uint8_t smem[];
  KVT* Kt = reinterpret_cast<KVT*>(smem);                  // [2][kTT][HD]
  KVT* Vt = Kt + 2 * kTT * HD;                              // [2][kTT][HD]
  float* qs = reinterpret_cast<float*>(Vt + 2 * kTT * HD);  // [kG][HD]
  float* P = qs + kG * HD;                                  // [kG][kTT]
  float* knew = P + kG * kTT;                               // [HD]
  float* vnew = knew + HD;                                  // [HD]
  float* s_m = vnew + HD;                                   // [kG]
  float* s_l = s_m + kG;
  float* s_alpha = s_l + kG;
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_alpha + kG);  // 16-byte aligned offset
  __shared__ int s_last, s_abort;

  // ---- rotated queries; the owner of pos also rotates k and appends k, v
  const float* row = a.qkv + (int64_t)b * (H + 2 * Hkv) * HD;
  const float* c = a.rc + (int64_t)pos * kHalf;
  const float* sn = a.rs + (int64_t)pos * kHalf;
  for (int idx = tid; idx < G * kHalf; idx += kT) {
    const int h = idx / kHalf, i = idx - h * kHalf;
    const float x0 = row[(g * G + h) * HD + i], x1 = row[(g * G + h) * HD + i + kHalf];
    rope_pair(x0, x1, c[i], sn[i], qs[h * HD + i], qs[h * HD + i + kHalf]);
  }
  const bool append = owns_pos && !a.kv_written;
  if (append) {
    const float* kr = row + H * HD + g * HD;
    const float* vr = row + (H + Hkv) * HD + g * HD;
    const int pi = pos / ps, slot = pos - pi * ps;
    const int64_t off = (int64_t)a.layer * kv.layer_stride +
                        (((int64_t)ptrow[pi] * Hkv + g) * ps + slot) * HD;
    for (int i = tid; i < kHalf; i += kT) {
      const float x0 = kr[i], x1 = kr[i + kHalf];
      float k0, k1;
      rope_pair(x0, x1, c[i], sn[i], k0, k1);
      Elem<KVT>::st(Kg + off + i, k0);
      Elem<KVT>::st(Kg + off + i + kHalf, k1);
      knew[i] = k0;
      knew[i + kHalf] = k1;
    }
    for (int i = tid; i < HD; i += kT) {
      Elem<KVT>::st(Vg + off + i, vr[i]);
      vnew[i] = vr[i];
    }
  }
  if (tid < kG) {
    s_m[tid] = -CUDART_INF_F;
    s_l[tid] = 0.0f;
  }
  const uint32_t bar0 = smem_u32(bars), bar1 = smem_u32(bars + 1);
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar0));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar1));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_abort = 0;
  }
  __syncthreads();

  const int n_tiles = (end - start + kTT - 1) / kTT;
  const uint32_t page_bytes = (uint32_t)(ps * HD * sizeof(KVT));
  // thread 0: fetch tile i (its pages, K and V) into buffer i % 2
  auto issue = [&](int i) {
    const int t0 = start + i * kTT;
    const int t1 = min(end, t0 + kTT);
    const int p0 = t0 / ps, p1 = (t1 - 1) / ps;
    const uint32_t bar = (i & 1) ? bar1 : bar0;
    const uint32_t bytes = 2u * page_bytes * (uint32_t)(p1 - p0 + 1);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
    KVT* kd = Kt + (i & 1) * kTT * HD;
    KVT* vd = Vt + (i & 1) * kTT * HD;
    for (int p = p0; p <= p1; ++p) {
      const int64_t off = (int64_t)a.layer * kv.layer_stride + ((int64_t)ptrow[p] * Hkv + g) * ps * HD;
      const int r = (p - p0) * ps;
      bulk_load(smem_u32(kd + r * HD), Kg + off, page_bytes, bar);
      bulk_load(smem_u32(vd + r * HD), Vg + off, page_bytes, bar);
    }
  };
  int issued = 0;  // meaningful in thread 0 only
  if (tid == 0) {
    issue(0);
    issued = 1;
    if (n_tiles > 1) {
      issue(1);
      issued = 2;
    }
  }

  const float scale = 1.0f / sqrtf((float)HD);
  float acc[kOut];
#pragma unroll
  for (int j = 0; j < kOut; ++j) acc[j] = 0.0f;

  for (int i = 0; i < n_tiles; ++i) {
    const int t0 = start + i * kTT;
    const int cnt = min(kTT, end - t0);
    const uint32_t bar = (i & 1) ? bar1 : bar0;
    if (!mbar_wait(bar, (uint32_t)(i >> 1) & 1u)) {
      atomicExch(a.err, 11);
      s_abort = 1;
    }
    KVT* Kb = Kt + (i & 1) * kTT * HD;
    KVT* Vb = Vt + (i & 1) * kTT * HD;
    if (append && pos >= t0 && pos < t0 + kTT) {  // the appended token, from registers
      const int r = pos - t0;
      for (int e = tid; e < HD; e += kT) {
        Elem<KVT>::st(Kb + r * HD + e, knew[e]);
        Elem<KVT>::st(Vb + r * HD + e, vnew[e]);
      }
    }
    __syncthreads();
    if (s_abort) {  // block-uniform after the barrier: drain our copies, then stop
      if (tid == 0)
        for (int j = i; j < issued; ++j)
          if (!mbar_wait((j & 1) ? bar1 : bar0, (uint32_t)(j >> 1) & 1u)) atomicExch(a.err, 12);
      break;
    }
    // scores of (head, position) pairs
    for (int pidx = tid; pidx < G * kTT; pidx += kT) {
      const int h = pidx / kTT, tt = pidx - h * kTT;
      float sc = -CUDART_INF_F;
      if (tt < cnt) {
        const KVT* kr = Kb + tt * HD;
        const float* q = qs + h * HD;
        float acc_s = 0.0f;
#pragma unroll
        for (int cc = 0; cc < kChunks; ++cc) {
          const int ch = (cc + tt) % kChunks;  // rotated: distinct banks per row
          float kk[kVec];
          Elem<KVT>::load(kr + ch * kVec, kk);
#pragma unroll
          for (int e = 0; e < kVec; ++e) acc_s = fmaf(q[ch * kVec + e], kk[e], acc_s);
        }
        sc = acc_s * scale;
      }
      P[h * kTT + tt] = sc;
    }
    __syncthreads();
    // online softmax per head: warp w owns heads w, w + 4
    for (int h = warp; h < G; h += kT / 32) {
      float v0 = P[h * kTT + lane], v1 = P[h * kTT + lane + 32];
      float mx = fmaxf(v0, v1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float mold = s_m[h];
      const float mnew = fmaxf(mold, mx);
      const float p0 = (lane < cnt) ? expf(v0 - mnew) : 0.0f;
      const float p1 = (lane + 32 < cnt) ? expf(v1 - mnew) : 0.0f;
      P[h * kTT + lane] = p0;
      P[h * kTT + lane + 32] = p1;
      float sum = p0 + p1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (lane == 0) {
        const float alpha = (mold == -CUDART_INF_F) ? 0.0f : expf(mold - mnew);
        s_alpha[h] = alpha;
        s_l[h] = s_l[h] * alpha + sum;
        s_m[h] = mnew;
      }
    }
    __syncthreads();
    // P.V
#pragma unroll
    for (int j = 0; j < kOut; ++j) {
      const int o = tid + j * kT;
      if (o < G * HD) {
        const int h = o / HD, d = o - h * HD;
        const float* ph = P + h * kTT;
        float accv = acc[j] * s_alpha[h];
        for (int tt = 0; tt < cnt; ++tt) accv = fmaf(ph[tt], Elem<KVT>::ld(Vb + tt * HD + d), accv);
        acc[j] = accv;
      }
    }
    __syncthreads();  // buffer i % 2 is free
    if (tid == 0 && i + 2 < n_tiles) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(i + 2);
      issued = i + 3;
    }
  }
  if (s_abort) return;

  OT* orow = static_cast<OT*>(a.o) + (int64_t)b * a.ld_o + g * G * HD;
  if (ns == 1) {
#pragma unroll
    for (int j = 0; j < kOut; ++j) {
      const int o = tid + j * kT;
      if (o < G * HD) st_out(orow + o, acc[j] / s_l[o / HD], a.o_lo);
    }
    return;
  }
  // several splits: publish (m, l, acc); the last block of (b, g) merges
  const int64_t base = ((int64_t)b * a.max_splits + s) * H + g * G;
  if (tid < G) {
    a.part_ml[2 * (base + tid)] = s_m[tid];
    a.part_ml[2 * (base + tid) + 1] = s_l[tid];
  }
#pragma unroll
  for (int j = 0; j < kOut; ++j) {
    const int o = tid + j * kT;
    if (o < G * HD) a.part_acc[base * HD + o] = acc[j];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    int* ctr = a.counters + (int64_t)b * Hkv + g;
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
        mx = fmaxf(mx, __ldcg(a.part_ml + 2 * (((int64_t)b * a.max_splits + q) * H + g * G + h)));
      float L = 0.0f, A = 0.0f;
      for (int q = 0; q < ns; ++q) {
        const int64_t bq = ((int64_t)b * a.max_splits + q) * H + g * G + h;
        const float w = expf(__ldcg(a.part_ml + 2 * bq) - mx);
        L = fmaf(__ldcg(a.part_ml + 2 * bq + 1), w, L);
        A = fmaf(__ldcg(a.part_acc + bq * HD + (o - h * HD)), w, A);
      }
      st_out(orow + o, A / L, a.o_lo);
    }
  }
}

template <typename KVT, typename OT, int HD>
int launch_hd(const AttnParams& a, int B, cudaStream_t s) {
  const size_t smem = 4 * (size_t)kTT * HD * sizeof(KVT) +
                      sizeof(float) * ((size_t)kG * HD + kG * kTT + 2 * HD + 3 * kG) +
                      2 * sizeof(uint64_t) + 64;
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(k_attn_tiled<KVT, OT, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    attr = true;
  }
  dim3 grid(a.max_splits, a.kv.Hkv, B);
  launch_k(k_attn_tiled<KVT, OT, HD>, grid, kT, smem, s, a);
  return 1;
}

template <typename KVT, typename OT>
int dispatch(const AttnParams& a, int B, cudaStream_t s) {
  switch (a.kv.hd) {
    case 16: return launch_hd<KVT, OT, 16>(a, B, s);
    case 32: return launch_hd<KVT, OT, 32>(a, B, s);
    case 64: return launch_hd<KVT, OT, 64>(a, B, s);
    case 128: return launch_hd<KVT, OT, 128>(a, B, s);
    case 256: return launch_hd<KVT, OT, 256>(a, B, s);
    default: return 0;
  }
}

}  // namespace

bool attn_tiled_supports(int hd, int G, int page_size, int split_len) {
  return (hd == 16 || hd == 32 || hd == 64 || hd == 128 || hd == 256) && G >= 1 && G <= kG &&
         (page_size == 16 || page_size == 32 || page_size == 64) && split_len % kTT == 0;
}

int launch_attention_tiled(const AttnParams& a, int B, int x_type, cudaStream_t s) {
  if (B <= 0) return 0;
  if (a.kv.kv_f32)
    return x_type == X_BF16 ? dispatch<float, __nv_bfloat16>(a, B, s)
                            : dispatch<float, float>(a, B, s);
  return x_type == X_BF16 ? dispatch<__nv_bfloat16, __nv_bfloat16>(a, B, s)
                          : dispatch<__nv_bfloat16, float>(a, B, s);
}

}  // namespace fsk
