// Per-lane GQA decode attention over paged bf16 KV with warp-level MMA.
//
// Computes what k_attn_tiled computes (RoPE of q and k at the lane's own
// position, append of k and v there, online-softmax attention of the lane's
// G query heads of one KV head over the lane's own keys 0..pos, split-K with
// an ordered merge; "MODEL-BATCHING-RESULTS", "The lever"; mlx-bun "Parallel
// slots", "KV memory" rung 3; "S1b decode: design traps" trap 2), with the
// two inner products on tensor cores so the kernel is limited by the KV
// stream rather than by instruction issue:
//   * a block = (split s, KV head g, panel row b), 4 warps; the split is
//     walked in tiles of 64 positions, K and V copied by cp.async into
//     XOR-swizzled shared memory (double-buffered), rows past the lane's
//     length zero-filled;
//   * warp w owns positions 16w .. 16w+15 of every tile: S = Q Kᵀ with
//     mma.m16n8k16 (bf16 in, f32 accumulate; the G heads are rows 0..G-1 of
//     the 16-row A operand), a per-warp online softmax, then O += P V with
//     the probabilities re-packed from the S accumulators into A fragments;
//     q and P are f32 values split as hi + lo bf16 parts placed in rows g and
//     g + 8 of the A operand, so one MMA yields both partial products (summed
//     afterwards) and the products with the exact bf16 K and V keep
//     near-f32 accuracy;
//   * the 4 warps' (m, l, O) are merged in warp order, then the splits in
//     split order, so a lane's result does not depend on the batch.

#include <math_constants.h>

#include "attn_mma.cuh"

namespace fsk {
FS_TRACE_TU(attn_mma)
namespace {

using namespace attn;

constexpr int kWarps = 4;
constexpr int kT = 32 * kWarps;
constexpr int kTT = 64;      // positions per tile
constexpr int kG = 8;        // max query heads per KV head

// byte offset of (row, 16-byte chunk) in a swizzled [kTT][HD] bf16 tile
template <int HD>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * (HD * 2) + ((chunk ^ (row & 7)) << 4));
}

// The kernel's body; thread 0's trace marks stay in shared memory (s_tr) so
// that tracing costs the body no registers.
template <typename OT, int HD>
__device__ __forceinline__ void attn_mma_body(const AttnParams& a, unsigned long long* s_tr) {
  constexpr int kHalf = HD / 2;
  constexpr int kCh = HD / 8;            // 16-byte chunks per row
  constexpr int kTileBytes = kTT * HD * 2;
  constexpr int kKs = HD / 16;           // k-steps of Q Kᵀ
  constexpr int kNt = HD / 8;            // n-tiles of P V
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
  const int gq = lane >> 2, cq = lane & 3;  // fragment row (head) and column pair
  const int32_t* ptrow = kv.pt + (int64_t)a.args.lane[b] * kv.max_pages;
  __nv_bfloat16* Kg = static_cast<__nv_bfloat16*>(kv.k);
  __nv_bfloat16* Vg = static_cast<__nv_bfloat16*>(kv.v);
  const bool owns_pos = (s == ns - 1);

  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* Kt = smem;                                       // [2] swizzled tiles
  uint8_t* Vt = smem + 2 * kTileBytes;
  float* qs = reinterpret_cast<float*>(smem + 4 * kTileBytes);  // [kG][HD]
  float* knew = qs + kG * HD;                               // [HD]
  float* vnew = knew + HD;
  float* wm = vnew + HD;                                    // [kWarps][kG]
  float* wl = wm + kWarps * kG;
  float* wo = reinterpret_cast<float*>(smem);  // [kWarps][kG][HD], reuses the idle tiles
  __shared__ int s_last;

  const int n_tiles = (end - start + kTT - 1) / kTT;
  // all threads: copy tile i (valid rows by cp.async, the rest zero) to buffer i % 2
  auto issue = [&](int i) {
    const int t0 = start + i * kTT;
    const int cnt = min(kTT, end - t0);
    uint8_t* kd = Kt + (i & 1) * kTileBytes;
    uint8_t* vd = Vt + (i & 1) * kTileBytes;
    for (int idx = tid; idx < kTT * kCh; idx += kT) {
      const int r = idx / kCh, ch = idx - r * kCh;
      const uint32_t o = swz<HD>(r, ch);
      if (r < cnt) {
        const int t = t0 + r, pi = t / ps, slot = t - pi * ps;
        const int64_t off = (int64_t)a.layer * kv.layer_stride +
                            (((int64_t)ptrow[pi] * Hkv + g) * ps + slot) * HD + ch * 8;
        cp_async16(smem_u32(kd + o), Kg + off);
        cp_async16(smem_u32(vd + o), Vg + off);
      } else {
        *reinterpret_cast<uint4*>(kd + o) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(vd + o) = make_uint4(0, 0, 0, 0);
      }
    }
    cp_commit();
  };
  // Programmatic dependent launch: the KV of earlier positions, the page
  // table and the step arguments were written by kernels that finished before
  // the predecessor started, so the first tiles are fetched before waiting
  // for the predecessor (the QKV projection read below).
  const bool prefetch = !a.kv_written;  // else this step's rows come from the predecessor
  if (prefetch) {
    issue(0);
    if (n_tiles > 1) issue(1);
  }
  // the rotation of position pos (constant tables): thread t rotates pairs
  // i = t mod hd/2 of every head (kT is a multiple of hd/2)
  static_assert(kT % kHalf == 0, "a thread's pairs share one rotation");
  const int ri = tid % kHalf;
  const float rc_i = a.rc[(int64_t)pos * kHalf + ri], rs_i = a.rs[(int64_t)pos * kHalf + ri];
  pdl_wait();
  TraceSmem::ready(s_tr);
  pdl_trigger();
  if (!prefetch) {
    issue(0);
    if (n_tiles > 1) issue(1);
  }

  // ---- rotated queries; the owner of pos also rotates k and appends k, v.
  // Every load of the projection's row is issued before any use.
  const float* row = a.qkv + (int64_t)b * (H + 2 * Hkv) * HD;
  constexpr int kQIt = (kG * kHalf + kT - 1) / kT;
  constexpr int kVIt = (HD + kT - 1) / kT;
  const bool append = owns_pos && !a.kv_written;
  const float* kr = row + H * HD + g * HD;
  const float* vr = row + (H + Hkv) * HD + g * HD;
  float qx0[kQIt], qx1[kQIt], vx[kVIt];
  float kx0 = 0.0f, kx1 = 0.0f;
#pragma unroll
  for (int it = 0; it < kQIt; ++it) {
    const int idx = tid + it * kT, h = idx / kHalf;
    qx0[it] = qx1[it] = 0.0f;
    if (idx < kG * kHalf && h < G) {
      qx0[it] = row[(g * G + h) * HD + ri];
      qx1[it] = row[(g * G + h) * HD + ri + kHalf];
    }
  }
  if (append && tid < kHalf) {
    kx0 = kr[tid];
    kx1 = kr[tid + kHalf];
  }
#pragma unroll
  for (int it = 0; it < kVIt; ++it) {
    const int i = tid + it * kT;
    vx[it] = (append && i < HD) ? vr[i] : 0.0f;
  }
#pragma unroll
  for (int it = 0; it < kQIt; ++it) {
    const int idx = tid + it * kT, h = idx / kHalf;
    if (idx < kG * kHalf) {
      float q0 = 0.0f, q1 = 0.0f;
      if (h < G) rope_pair(qx0[it], qx1[it], rc_i, rs_i, q0, q1);
      qs[h * HD + ri] = q0;
      qs[h * HD + ri + kHalf] = q1;
    }
  }
  if (append) {
    const int pi = pos / ps, slot = pos - pi * ps;
    const int64_t off = (int64_t)a.layer * kv.layer_stride +
                        (((int64_t)ptrow[pi] * Hkv + g) * ps + slot) * HD;
    if (tid < kHalf) {  // ri == tid
      float k0, k1;
      rope_pair(kx0, kx1, rc_i, rs_i, k0, k1);
      Kg[off + tid] = __float2bfloat16_rn(k0);
      Kg[off + tid + kHalf] = __float2bfloat16_rn(k1);
      knew[tid] = k0;
      knew[tid + kHalf] = k1;
    }
#pragma unroll
    for (int it = 0; it < kVIt; ++it) {
      const int i = tid + it * kT;
      if (i < HD) {
        Vg[off + i] = __float2bfloat16_rn(vx[it]);
        vnew[i] = vx[it];
      }
    }
  }
  __syncthreads();

  // Q as bf16 A fragments: row gq = hi part of head gq, row gq + 8 = its lo
  // part (heads >= G are zero)
  uint32_t qa[kKs][4];
#pragma unroll
  for (int ks = 0; ks < kKs; ++ks) {
    const int c0 = ks * 16 + 2 * cq;
    const float* q = qs + gq * HD;
    split_bf16(q[c0], q[c0 + 1], qa[ks][0], qa[ks][1]);
    split_bf16(q[c0 + 8], q[c0 + 9], qa[ks][2], qa[ks][3]);
  }


  const float scale = 1.0f / sqrtf((float)HD);
  float m_run = -CUDART_INF_F, l_run = 0.0f;  // head gq, this warp's positions
  float o_acc[kNt][4];
#pragma unroll
  for (int j = 0; j < kNt; ++j) o_acc[j][0] = o_acc[j][1] = o_acc[j][2] = o_acc[j][3] = 0.0f;

  for (int i = 0; i < n_tiles; ++i) {
    const int t0 = start + i * kTT;
    const int cnt = min(kTT, end - t0);
    if (i + 1 < n_tiles)
      cp_wait<1>();
    else
      cp_wait<0>();
    uint8_t* kb = Kt + (i & 1) * kTileBytes;
    uint8_t* vb = Vt + (i & 1) * kTileBytes;
    __syncthreads();
    if (append && pos >= t0 && pos < t0 + kTT) {  // the appended token, from registers
      const int r = pos - t0;
      for (int ch = tid; ch < kCh; ch += kT) {
        uint4 kk, vv;
        uint32_t* kw = reinterpret_cast<uint32_t*>(&kk);
        uint32_t* vw = reinterpret_cast<uint32_t*>(&vv);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          kw[e] = pack_bf16(knew[ch * 8 + 2 * e], knew[ch * 8 + 2 * e + 1]);
          vw[e] = pack_bf16(vnew[ch * 8 + 2 * e], vnew[ch * 8 + 2 * e + 1]);
        }
        *reinterpret_cast<uint4*>(kb + swz<HD>(r, ch)) = kk;
        *reinterpret_cast<uint4*>(vb + swz<HD>(r, ch)) = vv;
      }
      __syncthreads();
    }
    const int p0 = warp * 16;  // this warp's first position in the tile
    if (p0 < cnt) {
      // S = Q Kᵀ for positions p0 .. p0+15 (two n-tiles of 8)
      float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
      for (int ks = 0; ks < kKs; ++ks) {
        uint32_t bk[4];
        const int rr = p0 + (mi >> 1) * 8 + ri, ch = 2 * ks + (mi & 1);
        ldsm_x4(smem_u32(kb + swz<HD>(rr, ch)), bk);
        mma16816(sacc[0], qa[ks], bk[0], bk[1]);
        mma16816(sacc[1], qa[ks], bk[2], bk[3]);
      }
      // online softmax over this warp's positions, per head (row gq)
      float sv[4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int pp = p0 + nt * 8 + 2 * cq + e;
          sv[nt * 2 + e] = pp < cnt ? (sacc[nt][e] + sacc[nt][2 + e]) * scale : -CUDART_INF_F;
        }
      float mx = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float mnew = fmaxf(m_run, mx);
      const float alpha = (m_run == -CUDART_INF_F) ? 0.0f : expf(m_run - mnew);
      float pv[4], psum = 0.0f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        pv[e] = (sv[e] == -CUDART_INF_F) ? 0.0f : expf(sv[e] - mnew);
        psum += pv[e];
      }
      psum += __shfl_xor_sync(0xffffffffu, psum, 1);
      psum += __shfl_xor_sync(0xffffffffu, psum, 2);
      l_run = l_run * alpha + psum;
      m_run = mnew;
#pragma unroll
      for (int j = 0; j < kNt; ++j) {  // both the hi and the lo accumulators
        o_acc[j][0] *= alpha;
        o_acc[j][1] *= alpha;
        o_acc[j][2] *= alpha;
        o_acc[j][3] *= alpha;
      }
      // O += P V; P's A fragment: positions 2cq..2cq+1 (n-tile 0) and +8,
      // hi parts in row gq, lo parts in row gq + 8
      uint32_t pa[4];
      split_bf16(pv[0], pv[1], pa[0], pa[1]);
      split_bf16(pv[2], pv[3], pa[2], pa[3]);
#pragma unroll
      for (int j = 0; j < kNt; j += 2) {
        uint32_t bv[4];
        const int rr = p0 + (mi & 1) * 8 + ri, ch = j + (mi >> 1);
        ldsm_x4_t(smem_u32(vb + swz<HD>(rr, ch)), bv);
        mma16816(o_acc[j], pa, bv[0], bv[1]);
        mma16816(o_acc[j + 1], pa, bv[2], bv[3]);
      }
    }
    __syncthreads();  // buffer i % 2 is free
    if (i + 2 < n_tiles) issue(i + 2);
  }

  // ---- merge the warps in warp order
  if (cq == 0 && gq < kG) {
    wm[warp * kG + gq] = m_run;
    wl[warp * kG + gq] = l_run;
  }
  if (gq < G) {
#pragma unroll
    for (int j = 0; j < kNt; ++j) {
      wo[(warp * kG + gq) * HD + 8 * j + 2 * cq] = o_acc[j][0] + o_acc[j][2];
      wo[(warp * kG + gq) * HD + 8 * j + 2 * cq + 1] = o_acc[j][1] + o_acc[j][3];
    }
  }
  __syncthreads();
  OT* orow = static_cast<OT*>(a.o) + (int64_t)b * a.ld_o + g * G * HD;
  const int64_t base = ((int64_t)b * a.max_splits + s) * H + g * G;
  for (int o = tid; o < G * HD; o += kT) {
    const int h = o / HD, d = o - h * HD;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * kG + h]);
    float L = 0.0f, A = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = wm[w * kG + h];
      const float sc = (mw == -CUDART_INF_F) ? 0.0f : expf(mw - M);
      L = fmaf(wl[w * kG + h], sc, L);
      A = fmaf(wo[(w * kG + h) * HD + d], sc, A);
    }
    if (ns == 1) {
      st_out(orow + o, A / L, a.o_lo);
    } else {
      if (d == 0) {
        a.part_ml[2 * (base + h)] = M;
        a.part_ml[2 * (base + h) + 1] = L;
      }
      a.part_acc[base * HD + o] = A;
    }
  }
  if (ns == 1) return;
  // several splits: the last block of (b, g) merges them in split order
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
  // merge: every split's (m, l) into shared memory at once, the weights once
  // per (split, head), then the outputs with independent loads; all sums in
  // ascending split order
  float* sm = reinterpret_cast<float*>(smem);     // [ns][kG] m, then weights
  float* sl = sm + (size_t)ns * kG;               // [ns][kG] l
  float* sL = sl + (size_t)ns * kG;               // [kG] merged l
  for (int idx = tid; idx < ns * G; idx += kT) {
    const int q = idx / G, h = idx - q * G;
    const int64_t bq = ((int64_t)b * a.max_splits + q) * H + g * G + h;
    sm[q * kG + h] = __ldcg(a.part_ml + 2 * bq);
    sl[q * kG + h] = __ldcg(a.part_ml + 2 * bq + 1);
  }
  __syncthreads();
  if (tid < G) {
    const int h = tid;
    float mx = -CUDART_INF_F;
    for (int q = 0; q < ns; ++q) mx = fmaxf(mx, sm[q * kG + h]);
    float L = 0.0f;
    for (int q = 0; q < ns; ++q) {
      const float w = expf(sm[q * kG + h] - mx);
      sm[q * kG + h] = w;
      L = fmaf(sl[q * kG + h], w, L);
    }
    sL[h] = L;
  }
  __syncthreads();
  for (int o = tid; o < G * HD; o += kT) {
    const int h = o / HD, d = o - h * HD;
    const float* src = a.part_acc + (((int64_t)b * a.max_splits) * H + g * G + h) * HD + d;
    const int64_t qstride = (int64_t)H * HD;
    float A = 0.0f;
    int q = 0;
    for (; q + 4 <= ns; q += 4) {  // four independent loads in flight
      const float a0 = __ldcg(src + (q + 0) * qstride), a1 = __ldcg(src + (q + 1) * qstride);
      const float a2 = __ldcg(src + (q + 2) * qstride), a3 = __ldcg(src + (q + 3) * qstride);
      A = fmaf(a0, sm[(q + 0) * kG + h], A);
      A = fmaf(a1, sm[(q + 1) * kG + h], A);
      A = fmaf(a2, sm[(q + 2) * kG + h], A);
      A = fmaf(a3, sm[(q + 3) * kG + h], A);
    }
    for (; q < ns; ++q) A = fmaf(__ldcg(src + q * qstride), sm[q * kG + h], A);
    st_out(orow + o, A / sL[h], a.o_lo);
  }
}

// hd 64 keeps to 80 registers: six blocks of an SM (a 256-lane, 3-head
// step is then a single wave)
template <typename OT, int HD>
__global__ void __launch_bounds__(kT, HD == 64 ? 6 : 1) k_attn_mma(AttnParams a) {
  __shared__ unsigned long long s_tr[4];
  TraceSmem::begin(s_tr, g_trace);
  attn_mma_body<OT, HD>(a, s_tr);
  TraceSmem::end(s_tr, TR_ATTN_MMA);
}

template <typename OT, int HD>
int launch_hd(const AttnParams& a, int B, cudaStream_t s) {
  static_assert(kWarps * kG * HD * sizeof(float) <= 4 * (size_t)kTT * HD * 2,
                "the warp-merge buffer must fit in the tile buffers");
  const size_t smem =
      4 * (size_t)kTT * HD * 2 + sizeof(float) * ((size_t)kG * HD + 2 * HD + 2 * kWarps * kG);
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(k_attn_mma<OT, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    attr = true;
  }
  dim3 grid(a.max_splits, a.kv.Hkv, B);
  launch_k(k_attn_mma<OT, HD>, grid, kT, smem, s, a);
  return 1;
}

template <typename OT>
int dispatch(const AttnParams& a, int B, cudaStream_t s) {
  switch (a.kv.hd) {
    case 64: return launch_hd<OT, 64>(a, B, s);
    case 128: return launch_hd<OT, 128>(a, B, s);
    case 256: return launch_hd<OT, 256>(a, B, s);
    default: return 0;
  }
}

}  // namespace

bool attn_mma_supports(int hd, int G, int kv_f32, int split_len, int max_splits) {
  // the split merge stages 2 * kG floats per split in the tile buffers
  const size_t merge_bytes = (size_t)(2 * kG * max_splits + kG) * sizeof(float);
  return !kv_f32 && (hd == 64 || hd == 128 || hd == 256) && G >= 1 && G <= kG &&
         split_len % kTT == 0 && merge_bytes <= 4 * (size_t)kTT * hd * 2;
}

int launch_attention_mma(const AttnParams& a, int B, int x_type, cudaStream_t s) {
  if (B <= 0) return 0;
  return x_type == X_BF16 ? dispatch<__nv_bfloat16>(a, B, s) : dispatch<float>(a, B, s);
}

}  // namespace fsk
