// Embedding gather, RMSNorm, the per-lane sampler, the Q8_0 quantiser and
// the weight / KV layout helpers.

#include <math_constants.h>

#include <cstdlib>

#include "fs_internal.h"
#include "norm_row.cuh"

namespace fsk {
FS_TRACE_TU(misc)
namespace {

__device__ __forceinline__ float load_w(const Mat& E, int64_t row, int i) {
  if (E.wtype == W_BF16)
    return __bfloat162float(
        static_cast<const __nv_bfloat16*>(E.w)[row * E.Kp + i]);
  if (E.wtype == W_F32) return static_cast<const float*>(E.w)[row * E.Kp + i];
  const float d = __half2float(E.scales[row * (E.Kp / 32) + i / 32]);
  return (float)static_cast<const int8_t*>(E.w)[row * E.Kp + i] * d;
}

// x[b] = E[tok[b]] and, when g is given, h[b] = RMSNorm(x[b]) * g (the first
// layer's input norm); block b also applies page-table update b of the step.
template <typename OT, int MV>
__global__ void __launch_bounds__(kNormRowThreads)
    k_embed(Mat E, StepArgs args, KV kv, float* __restrict__ x, int d, const float* g,
            float eps, OT* __restrict__ h, int ld_h, int64_t lo_off) {
  TraceMark tr;
  tr.begin(g_trace);
  pdl_wait();
  tr.ready();
  pdl_trigger();
  __shared__ float red[4];
  const int b = blockIdx.x, t = threadIdx.x;
  if (t == 0 && b < *args.n_upd) {
    kv.pt[(int64_t)args.upd_lane[b] * kv.max_pages + args.upd_slot[b]] =
        args.upd_page[b];
  }
  const int64_t tok = args.tok[b];
  float* xr = x + (int64_t)b * d;
  // the same float4 chunks the norm routine gives this thread
  for (int c = t; c < d / 4; c += kNormRowThreads) {
    float4 v;
    v.x = load_w(E, tok, 4 * c);
    v.y = load_w(E, tok, 4 * c + 1);
    v.z = load_w(E, tok, 4 * c + 2);
    v.w = load_w(E, tok, 4 * c + 3);
    *reinterpret_cast<float4*>(xr + 4 * c) = v;
  }
  if (g) norm_row_128<OT, MV>(xr, nullptr, g, d, eps, h + (int64_t)b * ld_h, t, 1, red, lo_off);
  tr.end(TR_EMBED);
}


// Residual add then RMSNorm, one block of 128 threads per panel row (see
// norm_row.cuh for the arithmetic and its fixed reduction order).
template <typename OT, int MV>
__global__ void __launch_bounds__(kNormRowThreads)
    k_rmsnorm(float* __restrict__ x, const float* __restrict__ r,
              const float* __restrict__ g, int d, float eps, OT* __restrict__ out, int ld_out,
              int64_t lo_off) {
  TraceMark tr;
  tr.begin(g_trace);
  __shared__ float red[4];
  const int b = blockIdx.x;
  // The gains are never written: read before the wait. With r given, x was
  // last written two or more kernels back (complete once this kernel runs:
  // every kernel waits for its predecessor before letting its successor
  // start) and is read before the wait too, r is the predecessor's output;
  // without r, x itself is the predecessor's output (a projection that
  // added into the residual stream) and is read after the wait.
  NormRow<MV> n;
  n.load_g(g, d, threadIdx.x);
  if (r) n.load_x(x + (int64_t)b * d, d, threadIdx.x);
  pdl_wait();
  tr.ready();
  pdl_trigger();
  if (!r) n.load_x(x + (int64_t)b * d, d, threadIdx.x);
  n.template finish<OT>(x + (int64_t)b * d, r ? r + (int64_t)b * d : nullptr, d, eps,
               out + (int64_t)b * ld_out, threadIdx.x, 1, red, lo_off);
  tr.end(TR_RMSNORM);
}

// ---------------------------------------------------------------- sampler
// Philox4x32-10 (Salmon et al., SC 2011), written from its definition.
__device__ __forceinline__ void philox(uint32_t c[4], uint32_t k0,
                                       uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * c[0], hi0 = __umulhi(0xD2511F53u, c[0]);
    const uint32_t lo1 = 0xCD9E8D57u * c[2], hi1 = __umulhi(0xCD9E8D57u, c[2]);
    const uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
}

constexpr int kSampThreads = 1024;

// One block per row. Greedy: argmax with the lowest index on ties.
// Temperature: contiguous per-thread segments, an ordered exclusive scan of
// the segment sums, then the owning thread walks its segment.
__global__ void __launch_bounds__(kSampThreads)
    k_sample(const float* __restrict__ logits, int V,
             const float* __restrict__ temps, const uint64_t* __restrict__ seeds,
             const uint64_t* __restrict__ counters, int32_t* __restrict__ out) {
  TraceMark tr;
  tr.begin(g_trace);
  pdl_wait();
  tr.ready();
  pdl_trigger();
  __shared__ double sd[kSampThreads];
  __shared__ int si[kSampThreads];
  const int b = blockIdx.x, t = threadIdx.x;
  const float* lg = logits + (int64_t)b * V;
  const float temp = temps[b];
  const int seg = (V + kSampThreads - 1) / kSampThreads;
  const int lo = min(V, t * seg), hi = min(V, lo + seg);
  if (temp == 0.0f) {
    float best = -CUDART_INF_F;
    int bi = V;  // sentinel: no candidate
    for (int i = lo; i < hi; ++i)
      if (bi == V || lg[i] > best) {
        best = lg[i];
        bi = i;
      }
    sd[t] = best;
    si[t] = bi;
    __syncthreads();
    for (int w = kSampThreads / 2; w > 0; w >>= 1) {
      if (t < w) {
        const double ov = sd[t + w];
        const int oi = si[t + w];
        if (oi != V && (si[t] == V || ov > sd[t] || (ov == sd[t] && oi < si[t]))) {
          sd[t] = ov;
          si[t] = oi;
        }
      }
      __syncthreads();
    }
    if (t == 0) out[b] = si[0] == V ? 0 : si[0];
    tr.end(TR_SAMPLE);
    return;
  }
  // max of z = logit / T
  double mz = -CUDART_INF;
  for (int i = lo; i < hi; ++i) mz = fmax(mz, (double)lg[i] / (double)temp);
  sd[t] = mz;
  __syncthreads();
  for (int w = kSampThreads / 2; w > 0; w >>= 1) {
    if (t < w) sd[t] = fmax(sd[t], sd[t + w]);
    __syncthreads();
  }
  const double m = sd[0];
  __syncthreads();
  double part = 0.0;
  int last_pos = -1;
  for (int i = lo; i < hi; ++i) {
    const double e = exp((double)lg[i] / (double)temp - m);
    part += e;
    if (e > 0.0) last_pos = i;
  }
  sd[t] = part;
  si[t] = last_pos;
  __syncthreads();
  // inclusive scan (Hillis-Steele) of segment sums in thread order
  for (int w = 1; w < kSampThreads; w <<= 1) {
    const double v = t >= w ? sd[t - w] : 0.0;
    __syncthreads();
    sd[t] += v;
    __syncthreads();
  }
  const double total = sd[kSampThreads - 1];
  const double before = t > 0 ? sd[t - 1] : 0.0;
  uint32_t c[4] = {(uint32_t)counters[b], (uint32_t)(counters[b] >> 32), 0u, 0u};
  philox(c, (uint32_t)seeds[b], (uint32_t)(seeds[b] >> 32));
  const uint64_t bits = ((uint64_t)c[0] << 32) | c[1];
  const double u = (double)(bits >> 11) * (1.0 / 9007199254740992.0);
  const double target = u * total;
  __shared__ int found;
  if (t == 0) found = V;
  __syncthreads();
  if (before < target || (t == 0 && target <= 0.0)) {
    double cum = before;
    for (int i = lo; i < hi; ++i) {
      const double e = exp((double)lg[i] / (double)temp - m);
      cum += e;
      if (cum >= target && e > 0.0) {
        atomicMin(&found, i);
        break;
      }
    }
  }
  __syncthreads();
  if (t == 0) {
    int r = found;
    if (r == V) {  // rounding left the target above the total: last positive
      r = 0;
      for (int j = kSampThreads - 1; j >= 0; --j)
        if (si[j] >= 0) {
          r = si[j];
          break;
        }
    }
    out[b] = r;
  }
  tr.end(TR_SAMPLE);
}

// ------------------------------------------------------------- Q8_0 codec
__global__ void k_quantize_q8_0(const float* __restrict__ x, int64_t nblk,
                                uint8_t* __restrict__ blocks) {
  const int64_t blk = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int j = threadIdx.x & 31;
  if (blk >= nblk) return;
  const float v = x[blk * 32 + j];
  float amax = fabsf(v);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float d = amax / 127.0f;
  const float id = d != 0.0f ? 1.0f / d : 0.0f;
  const float q = fminf(127.0f, fmaxf(-127.0f, roundf(v * id)));
  const uint32_t code = (uint32_t)(uint8_t)(int8_t)q;
  const uint32_t dbits = (uint32_t)__half_as_ushort(__float2half_rn(d));
  // byte t of the 34-byte block: 0-1 scale (little endian), 2+i code i.
  // Thread j writes byte j, threads 0 and 1 also bytes 32 and 33.
  const uint32_t code_m2 = __shfl_sync(0xffffffffu, code, (j + 30) & 31);
  const uint32_t code_30 = __shfl_sync(0xffffffffu, code, 30 + (j & 1));
  uint8_t* ob = blocks + blk * 34;
  uint32_t byte_j;
  if (j == 0)
    byte_j = dbits & 0xffu;
  else if (j == 1)
    byte_j = (dbits >> 8) & 0xffu;
  else
    byte_j = code_m2;
  ob[j] = (uint8_t)byte_j;
  if (j < 2) ob[32 + j] = (uint8_t)code_30;
}

// 34-byte blocks of rows [N][K] -> codes [row_offset + n][Kp], scales.
__global__ void k_repack_q8(const uint8_t* __restrict__ blocks, int N, int K,
                            int Kp, int8_t* __restrict__ qs,
                            __half* __restrict__ scales, int row_offset) {
  const int64_t nb_row = K / 32;
  const int64_t blk = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int j = threadIdx.x & 31;
  if (blk >= (int64_t)N * nb_row) return;
  const int64_t n = blk / nb_row, kb = blk - n * nb_row;
  const uint8_t* ib = blocks + blk * 34;
  const int64_t r = row_offset + n;
  qs[r * Kp + kb * 32 + j] = (int8_t)ib[2 + j];
  if (j == 0)
    scales[r * (Kp / 32) + kb] =
        __ushort_as_half((uint16_t)(ib[0] | ((uint16_t)ib[1] << 8)));
}

// ------------------------------------------------------------- KV helpers
__device__ __forceinline__ uint64_t mix64(uint64_t z) {  // splitmix64 finaliser
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Fills whole pages (every layer, K and V) with values uniform in
// [-sqrt(3), sqrt(3)) (unit variance) derived from (seed, element index).
template <typename KVT>
__global__ void k_fill_random_kv(KV kv, int L, const int32_t* __restrict__ pages,
                                 int n_pages, uint64_t seed) {
  const int64_t per_page = (int64_t)kv.Hkv * kv.page_size * kv.hd;
  const int64_t total = (int64_t)L * n_pages * per_page;
  KVT* K = static_cast<KVT*>(kv.k);
  KVT* V = static_cast<KVT*>(kv.v);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t l = i / ((int64_t)n_pages * per_page);
    const int64_t rem = i - l * n_pages * per_page;
    const int64_t p = rem / per_page, e = rem - p * per_page;
    const int64_t off = l * kv.layer_stride + (int64_t)pages[p] * per_page + e;
    const uint64_t h1 = mix64(seed ^ (uint64_t)(2 * off));
    const uint64_t h2 = mix64(seed ^ (uint64_t)(2 * off + 1));
    const float u1 = (float)(h1 >> 40) * (1.0f / 16777216.0f);
    const float u2 = (float)(h2 >> 40) * (1.0f / 16777216.0f);
    const float k = (2.0f * u1 - 1.0f) * 1.7320508f;
    const float v = (2.0f * u2 - 1.0f) * 1.7320508f;
    if constexpr (sizeof(KVT) == 2) {
      K[off] = __float2bfloat16_rn(k);
      V[off] = __float2bfloat16_rn(v);
    } else {
      K[off] = k;
      V[off] = v;
    }
  }
}

// Copies n tokens of one layer between a lane's pages and dense f32
// [n][Hkv][hd] arrays (to_pages: dense -> pages).
template <typename KVT, bool kToPages>
__global__ void k_copy_kv(KV kv, int layer, const int32_t* __restrict__ pages,
                          int n, float* k, float* v) {
  const int64_t row = (int64_t)kv.Hkv * kv.hd;
  const int64_t total = (int64_t)n * row;
  KVT* K = static_cast<KVT*>(kv.k);
  KVT* V = static_cast<KVT*>(kv.v);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / row);
    const int64_t r = i - (int64_t)t * row;
    const int g = (int)(r / kv.hd), e = (int)(r - (int64_t)g * kv.hd);
    const int page = pages[t / kv.page_size], slot = t % kv.page_size;
    const int64_t off = (int64_t)layer * kv.layer_stride +
                        (((int64_t)page * kv.Hkv + g) * kv.page_size + slot) * kv.hd + e;
    if (kToPages) {
      if constexpr (sizeof(KVT) == 2) {
        K[off] = __float2bfloat16_rn(k[i]);
        V[off] = __float2bfloat16_rn(v[i]);
      } else {
        K[off] = k[i];
        V[off] = v[i];
      }
    } else {
      if constexpr (sizeof(KVT) == 2) {
        k[i] = __bfloat162float(K[off]);
        v[i] = __bfloat162float(V[off]);
      } else {
        k[i] = K[off];
        v[i] = V[off];
      }
    }
  }
}

}  // namespace

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = getenv("FS_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

// float4 chunks a thread of a row holds: the smallest of 2, 4, 8, 16 that
// covers d (chunks past d add exact zeros, so the bits do not depend on it)
int norm_chunks(int d) {
  const int per = (d / 4 + kNormRowThreads - 1) / kNormRowThreads;
  return per <= 2 ? 2 : per <= 4 ? 4 : per <= 8 ? 8 : 16;
}

template <typename OT, int MV>
void embed_mv(const Mat& E, const StepArgs& args, int B, const KV& kv, float* x, int d,
              const float* g, float eps, void* h, int ld_h, int64_t lo, cudaStream_t s) {
  launch_k(k_embed<OT, MV>, B, kNormRowThreads, 0, s, E, args, kv, x, d, g, eps,
           static_cast<OT*>(h), ld_h, lo);
}

template <typename OT>
void embed_ot(const Mat& E, const StepArgs& args, int B, const KV& kv, float* x, int d,
              const float* g, float eps, void* h, int ld_h, int64_t lo, cudaStream_t s) {
  switch (norm_chunks(d)) {
    case 2: embed_mv<OT, 2>(E, args, B, kv, x, d, g, eps, h, ld_h, lo, s); break;
    case 4: embed_mv<OT, 4>(E, args, B, kv, x, d, g, eps, h, ld_h, lo, s); break;
    case 8: embed_mv<OT, 8>(E, args, B, kv, x, d, g, eps, h, ld_h, lo, s); break;
    default: embed_mv<OT, 16>(E, args, B, kv, x, d, g, eps, h, ld_h, lo, s); break;
  }
}

int launch_embed(const Mat& E, const StepArgs& args, int B, const KV& kv, float* x, int d,
                 const float* g, float eps, void* h, int x_type, int ld_h, int64_t lo_off,
                 cudaStream_t s) {
  if (B <= 0) return 0;
  if (x_type == X_BF16)
    embed_ot<__nv_bfloat16>(E, args, B, kv, x, d, g, eps, h, ld_h, lo_off, s);
  else
    embed_ot<float>(E, args, B, kv, x, d, g, eps, h, ld_h, 0, s);
  return 1;
}

template <typename OT, int MV>
void rmsnorm_mv(float* x, const float* resid, const float* g, int B, int d, float eps, void* out,
                int ld_out, int64_t lo, cudaStream_t s) {
  launch_k(k_rmsnorm<OT, MV>, B, kNormRowThreads, 0, s, x, resid, g, d, eps,
           static_cast<OT*>(out), ld_out, lo);
}

template <typename OT>
void rmsnorm_ot(float* x, const float* resid, const float* g, int B, int d, float eps, void* out,
                int ld_out, int64_t lo, cudaStream_t s) {
  switch (norm_chunks(d)) {
    case 2: rmsnorm_mv<OT, 2>(x, resid, g, B, d, eps, out, ld_out, lo, s); break;
    case 4: rmsnorm_mv<OT, 4>(x, resid, g, B, d, eps, out, ld_out, lo, s); break;
    case 8: rmsnorm_mv<OT, 8>(x, resid, g, B, d, eps, out, ld_out, lo, s); break;
    default: rmsnorm_mv<OT, 16>(x, resid, g, B, d, eps, out, ld_out, lo, s); break;
  }
}

int launch_rmsnorm(float* x, const float* resid, const float* g, int B, int d, float eps,
                   void* out, int x_type, int ld_out, int64_t lo_off, cudaStream_t s) {
  if (B <= 0) return 0;
  if (x_type == X_BF16)
    rmsnorm_ot<__nv_bfloat16>(x, resid, g, B, d, eps, out, ld_out, lo_off, s);
  else
    rmsnorm_ot<float>(x, resid, g, B, d, eps, out, ld_out, 0, s);
  return 1;
}

int launch_sample(const float* logits, int B, int V, const float* temps,
                  const uint64_t* seeds, const uint64_t* counters, int32_t* out,
                  cudaStream_t s) {
  if (B <= 0) return 0;
  launch_k(k_sample, B, kSampThreads, 0, s, logits, V, temps, seeds, counters, out);
  return 1;
}

int launch_quantize_q8_0(const float* src, int64_t n, uint8_t* blocks,
                         cudaStream_t s) {
  const int64_t nblk = n / 32;
  if (nblk <= 0) return 0;
  const int per = 8;  // blocks per CTA (one warp each)
  k_quantize_q8_0<<<(unsigned)((nblk + per - 1) / per), per * 32, 0, s>>>(
      src, nblk, blocks);
  return 1;
}

int launch_repack_q8(const uint8_t* blocks, int N, int K, int Kp, int8_t* qs,
                     __half* scales, int row_offset, cudaStream_t s) {
  const int64_t nblk = (int64_t)N * (K / 32);
  if (nblk <= 0) return 0;
  const int per = 8;
  k_repack_q8<<<(unsigned)((nblk + per - 1) / per), per * 32, 0, s>>>(
      blocks, N, K, Kp, qs, scales, row_offset);
  return 1;
}

// Rewrites rows [q_begin, q_end) of one lane's history, in every layer, into
// the pages of dst_pt: row q comes from row q (q < a) or from row q + delta
// (q >= a) of the pages of src_pt, and a key that moves down by delta
// positions is turned back by delta positions, R(-delta) R(p) k = R(p - delta) k
// (the rotate-half pairs of the RoPE, with the tables' cos/sin at position
// delta). One block per (layer, kv head, K|V) walks its rows in ascending
// batches; a batch is read whole before any of it is written, and a
// destination row q lies below every source row not yet read (q < q + delta),
// so compaction within a shared page table is safe without a second buffer.
constexpr int kRelocThreads = 256;
constexpr int kRelocPairs = 4;  // rotate-half pairs per thread per batch

template <typename KVT>
__global__ void __launch_bounds__(kRelocThreads)
k_kv_relocate(KV kv, const int32_t* __restrict__ src_pt, const int32_t* __restrict__ dst_pt,
              int q_begin, int q_end, int a, int delta, const float* __restrict__ rc,
              const float* __restrict__ rs) {
  const int half = kv.hd / 2;
  const int which = blockIdx.x & 1;  // 0: K, 1: V
  const int g = (blockIdx.x >> 1) % kv.Hkv;
  const int layer = (blockIdx.x >> 1) / kv.Hkv;
  KVT* base = static_cast<KVT*>(which ? kv.v : kv.k) + (int64_t)layer * kv.layer_stride;
  auto at = [&](int page, int slot) {
    return base + (((int64_t)page * kv.Hkv + g) * kv.page_size + slot) * kv.hd;
  };
  const int rows_per_batch = kRelocThreads * kRelocPairs / half;  // half <= 128
  for (int r0 = q_begin; r0 < q_end; r0 += rows_per_batch) {
    float y0[kRelocPairs], y1[kRelocPairs];
#pragma unroll
    for (int u = 0; u < kRelocPairs; ++u) {
      const int unit = threadIdx.x + u * kRelocThreads;
      const int q = r0 + unit / half, i = unit % half;
      if (unit >= rows_per_batch * half || q >= q_end) continue;
      const int p = q < a ? q : q + delta;
      const KVT* row = at(src_pt[p / kv.page_size], p % kv.page_size);
      float x0, x1;
      if constexpr (sizeof(KVT) == 2) {
        x0 = __bfloat162float(row[i]);
        x1 = __bfloat162float(row[i + half]);
      } else {
        x0 = row[i];
        x1 = row[i + half];
      }
      if (which == 0 && q >= a && delta > 0) {
        const float c = rc[(int64_t)delta * half + i], sn = rs[(int64_t)delta * half + i];
        rope_pair(x0, x1, c, -sn, y0[u], y1[u]);
      } else {
        y0[u] = x0;
        y1[u] = x1;
      }
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kRelocPairs; ++u) {
      const int unit = threadIdx.x + u * kRelocThreads;
      const int q = r0 + unit / half, i = unit % half;
      if (unit >= rows_per_batch * half || q >= q_end) continue;
      KVT* row = at(dst_pt[q / kv.page_size], q % kv.page_size);
      if constexpr (sizeof(KVT) == 2) {
        row[i] = __float2bfloat16_rn(y0[u]);
        row[i + half] = __float2bfloat16_rn(y1[u]);
      } else {
        row[i] = y0[u];
        row[i + half] = y1[u];
      }
    }
    __syncthreads();
  }
}

int launch_kv_relocate(const KV& kv, int L, const int32_t* src_pt, const int32_t* dst_pt,
                       int q_begin, int q_end, int a, int delta, const float* rc,
                       const float* rs, cudaStream_t s) {
  if (q_end <= q_begin || kv.hd > 2 * kRelocThreads * kRelocPairs) return 0;
  const unsigned grid = (unsigned)L * kv.Hkv * 2;
  if (kv.kv_f32)
    k_kv_relocate<float><<<grid, kRelocThreads, 0, s>>>(kv, src_pt, dst_pt, q_begin, q_end, a,
                                                        delta, rc, rs);
  else
    k_kv_relocate<__nv_bfloat16><<<grid, kRelocThreads, 0, s>>>(kv, src_pt, dst_pt, q_begin,
                                                                q_end, a, delta, rc, rs);
  return 1;
}

// Failure-detection check: one thread waits on a barrier that nothing
// arrives on, in the same bounded way as the step kernels' waits (try_wait
// polled against %globaltimer), and on giving up sets the error flag and
// returns, leaving the context usable.
__global__ void k_wait_selftest(uint64_t timeout_ns, int* err) {
  __shared__ uint64_t bar;
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(&bar);
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(a));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  const unsigned long long t0 = gtime();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(a)
        : "memory");
    if (ok) return;  // an arrival (none is made): no error
    if (gtime() - t0 > timeout_ns) {
      atomicExch(err, kErrSelftest);
      return;
    }
  }
}

int launch_wait_selftest(uint64_t timeout_ns, int* err, cudaStream_t s) {
  k_wait_selftest<<<1, 32, 0, s>>>(timeout_ns, err);
  return 1;
}

int launch_fill_random_kv(const KV& kv, int L, const int32_t* pages,
                          int n_pages, uint64_t seed, cudaStream_t s) {
  if (n_pages <= 0) return 0;
  if (kv.kv_f32)
    k_fill_random_kv<float><<<1216, 256, 0, s>>>(kv, L, pages, n_pages, seed);
  else
    k_fill_random_kv<__nv_bfloat16><<<1216, 256, 0, s>>>(kv, L, pages, n_pages,
                                                          seed);
  return 1;
}

int launch_import_kv(const KV& kv, int layer, const int32_t* pages, int n,
                     const float* k, const float* v, cudaStream_t s) {
  if (n <= 0) return 0;
  if (kv.kv_f32)
    k_copy_kv<float, true><<<304, 256, 0, s>>>(kv, layer, pages, n,
                                               const_cast<float*>(k),
                                               const_cast<float*>(v));
  else
    k_copy_kv<__nv_bfloat16, true><<<304, 256, 0, s>>>(
        kv, layer, pages, n, const_cast<float*>(k), const_cast<float*>(v));
  return 1;
}

int launch_export_kv(const KV& kv, int layer, const int32_t* pages, int n,
                     float* k, float* v, cudaStream_t s) {
  if (n <= 0) return 0;
  if (kv.kv_f32)
    k_copy_kv<float, false><<<304, 256, 0, s>>>(kv, layer, pages, n, k, v);
  else
    k_copy_kv<__nv_bfloat16, false><<<304, 256, 0, s>>>(kv, layer, pages, n,
                                                        k, v);
  return 1;
}

}  // namespace fsk
