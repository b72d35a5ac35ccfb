// Decode attention for handles whose lanes hold at most 64 positions: one
// warp per (lane, KV head), two per block.
//
// Computes what k_attn_mma computes for a single 64-position tile and a
// single split (RoPE of q and k at the lane's own position, append of k and
// v there, the G query heads of one KV head over the lane's keys 0..pos;
// "MODEL-BATCHING-RESULTS", "The lever"; mlx-bun "Parallel slots"), with
// the same arithmetic in the same order, so the two kernels give the same
// bits: k_attn_mma's warp w takes positions 16w .. 16w+15 of the tile with
// its own online softmax and the four warps' (m, l, O) are merged in warp
// order; here one warp plays the four in turn (chunk w = positions 16w ..
// 16w+15), parks each chunk's (m, l, O) in shared memory (O in the chunk's
// own key rows, dead once its scores are taken) and merges them the same
// way. A pair then needs no block barrier and a block carries two pairs,
// where k_attn_mma spends a 128-thread block and three block barriers on
// each: at short contexts the work per pair is a few hundred instructions
// and those fixed costs were most of it. Two pairs per block (38 KB of
// shared memory at hd 64) let an SM hold ten pairs.

#include <math_constants.h>

#include "attn_mma.cuh"

namespace fsk {
FS_TRACE_TU(attn_warp)
namespace {

using namespace attn;

constexpr int kPairs = 2;          // warps (pairs) per block: five blocks of an SM
constexpr int kT = 32 * kPairs;
constexpr int kTT = 64;            // positions of the one tile
constexpr int kG = 8;              // max query heads per KV head

// byte offset of (row, 16-byte chunk) in a swizzled [kTT][HD] bf16 tile
template <int HD>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * (HD * 2) + ((chunk ^ (row & 7)) << 4));
}

// Shared memory of one warp: K and V tiles, the rotated queries, the
// appended k and v, and the chunks' (m, l).
template <int HD>
struct WarpSmem {
  static constexpr int kTile = kTT * HD * 2;
  static constexpr int kBytes = 2 * kTile + (kG * HD + 2 * HD + 2 * 4 * kG) * 4;
};

template <typename OT, int HD>
__device__ __forceinline__ void attn_warp_body(const AttnParams& a, unsigned long long* s_tr) {
  constexpr int kHalf = HD / 2;
  constexpr int kCh = HD / 8;   // 16-byte chunks per row
  constexpr int kKs = HD / 16;  // k-steps of Q Kᵀ
  constexpr int kNt = HD / 8;   // n-tiles of P V
  constexpr int kTile = WarpSmem<HD>::kTile;
  const KV& kv = a.kv;
  const int H = a.H, Hkv = kv.Hkv, G = H / Hkv, ps = kv.page_size;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = blockIdx.x * kPairs + warp;
  const int b = pair / Hkv, g = pair - b * Hkv;
  const bool live = b < a.n_rows;
  const int gq = lane >> 2, cq = lane & 3;  // fragment row (head) and column pair

  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* base = smem + (size_t)warp * WarpSmem<HD>::kBytes;
  uint8_t* Kt = base;
  uint8_t* Vt = base + kTile;
  float* qs = reinterpret_cast<float*>(base + 2 * kTile);  // [kG][HD]
  float* knew = qs + kG * HD;                              // [HD]
  float* vnew = knew + HD;
  float* wm = vnew + HD;                                   // [4][kG]
  float* wl = wm + 4 * kG;

  int pos = 0, len = 0;
  const int32_t* ptrow = nullptr;
  if (live) {
    pos = a.args.pos[b];
    len = pos + 1;  // <= kTT: the handle's lanes hold at most 64 positions
    ptrow = kv.pt + (int64_t)a.args.lane[b] * kv.max_pages;
  }
  __nv_bfloat16* Kg = static_cast<__nv_bfloat16*>(kv.k);
  __nv_bfloat16* Vg = static_cast<__nv_bfloat16*>(kv.v);
  // the tile: valid rows by cp.async, the rest zero (lanes of this warp)
  auto issue = [&]() {
    for (int idx = lane; idx < kTT * kCh; idx += 32) {
      const int r = idx / kCh, ch = idx - r * kCh;
      const uint32_t o = swz<HD>(r, ch);
      if (r < len) {
        const int pi = r / ps, slot = r - pi * ps;
        const int64_t off = (int64_t)a.layer * kv.layer_stride +
                            (((int64_t)ptrow[pi] * Hkv + g) * ps + slot) * HD + ch * 8;
        cp_async16(smem_u32(Kt + o), Kg + off);
        cp_async16(smem_u32(Vt + o), Vg + off);
      } else {
        *reinterpret_cast<uint4*>(Kt + o) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(Vt + o) = make_uint4(0, 0, 0, 0);
      }
    }
    cp_commit();
  };
  // Programmatic dependent launch: the KV of earlier positions, the page
  // table, the step arguments and the rotation tables are complete before
  // the predecessor starts; only the QKV projection is its output.
  const bool prefetch = !a.kv_written;
  if (live && prefetch) issue();
  constexpr int kRp = (kHalf + 31) / 32;  // rotation pairs of a lane
  float rc[kRp], rsn[kRp];
#pragma unroll
  for (int m = 0; m < kRp; ++m) {
    const int i = lane + 32 * m;
    rc[m] = (live && i < kHalf) ? a.rc[(int64_t)pos * kHalf + i] : 0.0f;
    rsn[m] = (live && i < kHalf) ? a.rs[(int64_t)pos * kHalf + i] : 0.0f;
  }
  pdl_wait();
  TraceSmem::ready(s_tr);
  pdl_trigger();
  if (!live) return;
  if (!prefetch) issue();

  // ---- rotated queries; the block of the last split (here the only one)
  // rotates k and appends k, v. Every load of the projection's row first.
  const float* row = a.qkv + (int64_t)b * (H + 2 * Hkv) * HD;
  const bool append = !a.kv_written;
  const float* kr = row + H * HD + g * HD;
  const float* vr = row + (H + Hkv) * HD + g * HD;
  float qx0[kG][kRp], qx1[kG][kRp], kx0[kRp], kx1[kRp];
  constexpr int kVIt = (HD + 31) / 32;
  float vx[kVIt];
#pragma unroll
  for (int h = 0; h < kG; ++h)
#pragma unroll
    for (int m = 0; m < kRp; ++m) {
      const int i = lane + 32 * m;
      qx0[h][m] = qx1[h][m] = 0.0f;
      if (h < G && i < kHalf) {
        qx0[h][m] = row[(g * G + h) * HD + i];
        qx1[h][m] = row[(g * G + h) * HD + i + kHalf];
      }
    }
#pragma unroll
  for (int m = 0; m < kRp; ++m) {
    const int i = lane + 32 * m;
    kx0[m] = (append && i < kHalf) ? kr[i] : 0.0f;
    kx1[m] = (append && i < kHalf) ? kr[i + kHalf] : 0.0f;
  }
#pragma unroll
  for (int it = 0; it < kVIt; ++it) {
    const int i = lane + 32 * it;
    vx[it] = (append && i < HD) ? vr[i] : 0.0f;
  }
#pragma unroll
  for (int h = 0; h < kG; ++h)
#pragma unroll
    for (int m = 0; m < kRp; ++m) {
      const int i = lane + 32 * m;
      if (i < kHalf) {
        float q0 = 0.0f, q1 = 0.0f;
        if (h < G) rope_pair(qx0[h][m], qx1[h][m], rc[m], rsn[m], q0, q1);
        qs[h * HD + i] = q0;
        qs[h * HD + i + kHalf] = q1;
      }
    }
  if (append) {
    const int pi = pos / ps, slot = pos - pi * ps;
    const int64_t off = (int64_t)a.layer * kv.layer_stride +
                        (((int64_t)ptrow[pi] * Hkv + g) * ps + slot) * HD;
#pragma unroll
    for (int m = 0; m < kRp; ++m) {
      const int i = lane + 32 * m;
      if (i < kHalf) {
        float k0, k1;
        rope_pair(kx0[m], kx1[m], rc[m], rsn[m], k0, k1);
        Kg[off + i] = __float2bfloat16_rn(k0);
        Kg[off + i + kHalf] = __float2bfloat16_rn(k1);
        knew[i] = k0;
        knew[i + kHalf] = k1;
      }
    }
#pragma unroll
    for (int it = 0; it < kVIt; ++it) {
      const int i = lane + 32 * it;
      if (i < HD) {
        Vg[off + i] = __float2bfloat16_rn(vx[it]);
        vnew[i] = vx[it];
      }
    }
  }
  __syncwarp();

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

  cp_wait<0>();
  __syncwarp();
  if (append) {  // the appended token, from registers (row pos of the tile)
    for (int ch = lane; ch < kCh; ch += 32) {
      uint4 kk, vv;
      uint32_t* kw = reinterpret_cast<uint32_t*>(&kk);
      uint32_t* vw = reinterpret_cast<uint32_t*>(&vv);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        kw[e] = pack_bf16(knew[ch * 8 + 2 * e], knew[ch * 8 + 2 * e + 1]);
        vw[e] = pack_bf16(vnew[ch * 8 + 2 * e], vnew[ch * 8 + 2 * e + 1]);
      }
      *reinterpret_cast<uint4*>(Kt + swz<HD>(pos, ch)) = kk;
      *reinterpret_cast<uint4*>(Vt + swz<HD>(pos, ch)) = vv;
    }
    __syncwarp();
  }

  // ---- the four chunks of 16 positions, each with its own online softmax
  const float scale = 1.0f / sqrtf((float)HD);
  const int mi = lane >> 3, ri = lane & 7;
#pragma unroll 1
  for (int w = 0; w < 4; ++w) {
    const int p0 = w * 16;
    float m_run = -CUDART_INF_F, l_run = 0.0f;
    float o_acc[kNt][4];
#pragma unroll
    for (int j = 0; j < kNt; ++j) o_acc[j][0] = o_acc[j][1] = o_acc[j][2] = o_acc[j][3] = 0.0f;
    if (p0 < len) {
      float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < kKs; ++ks) {
        uint32_t bk[4];
        const int rr = p0 + (mi >> 1) * 8 + ri, ch = 2 * ks + (mi & 1);
        ldsm_x4(smem_u32(Kt + swz<HD>(rr, ch)), bk);
        mma16816(sacc[0], qa[ks], bk[0], bk[1]);
        mma16816(sacc[1], qa[ks], bk[2], bk[3]);
      }
      float sv[4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int pp = p0 + nt * 8 + 2 * cq + e;
          sv[nt * 2 + e] = pp < len ? (sacc[nt][e] + sacc[nt][2 + e]) * scale : -CUDART_INF_F;
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
      for (int j = 0; j < kNt; ++j) {
        o_acc[j][0] *= alpha;
        o_acc[j][1] *= alpha;
        o_acc[j][2] *= alpha;
        o_acc[j][3] *= alpha;
      }
      uint32_t pa[4];
      split_bf16(pv[0], pv[1], pa[0], pa[1]);
      split_bf16(pv[2], pv[3], pa[2], pa[3]);
#pragma unroll
      for (int j = 0; j < kNt; j += 2) {
        uint32_t bv[4];
        const int rr = p0 + (mi & 1) * 8 + ri, ch = j + (mi >> 1);
        ldsm_x4_t(smem_u32(Vt + swz<HD>(rr, ch)), bv);
        mma16816(o_acc[j], pa, bv[0], bv[1]);
        mma16816(o_acc[j + 1], pa, bv[2], bv[3]);
      }
    }
    // park the chunk's (m, l, O); O goes into the chunk's own key rows,
    // whose scores are taken (kG x HD f32 = 16 rows x HD bf16)
    __syncwarp();
    float* wo = reinterpret_cast<float*>(Kt + (size_t)p0 * HD * 2);  // [kG][HD]
    if (cq == 0 && gq < kG) {
      wm[w * kG + gq] = m_run;
      wl[w * kG + gq] = l_run;
    }
    if (gq < G) {
#pragma unroll
      for (int j = 0; j < kNt; ++j) {
        wo[gq * HD + 8 * j + 2 * cq] = o_acc[j][0] + o_acc[j][2];
        wo[gq * HD + 8 * j + 2 * cq + 1] = o_acc[j][1] + o_acc[j][3];
      }
    }
  }
  __syncwarp();

  // ---- merge the chunks in chunk order, as k_attn_mma merges its warps
  OT* orow = static_cast<OT*>(a.o) + (int64_t)b * a.ld_o + g * G * HD;
  for (int o = lane; o < G * HD; o += 32) {
    const int h = o / HD, d = o - h * HD;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, wm[w * kG + h]);
    float L = 0.0f, A = 0.0f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float mw = wm[w * kG + h];
      const float sc = (mw == -CUDART_INF_F) ? 0.0f : expf(mw - M);
      const float* wo = reinterpret_cast<const float*>(Kt + (size_t)(w * 16) * HD * 2);
      L = fmaf(wl[w * kG + h], sc, L);
      A = fmaf(wo[h * HD + d], sc, A);
    }
    st_out(orow + o, A / L, a.o_lo);
  }
}

template <typename OT, int HD>
__global__ void __launch_bounds__(kT) k_attn_warp(AttnParams a) {
  __shared__ unsigned long long s_tr[4];
  TraceSmem::begin(s_tr, g_trace);
  attn_warp_body<OT, HD>(a, s_tr);
  TraceSmem::end(s_tr, TR_ATTN_WARP);
}

template <typename OT, int HD>
int launch_hd(const AttnParams& a, int B, cudaStream_t s) {
  static_assert(kG * HD * 4 <= 16 * HD * 2, "a chunk's O fits in its key rows");
  const size_t smem = (size_t)kPairs * WarpSmem<HD>::kBytes;
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(k_attn_warp<OT, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    attr = true;
  }
  AttnParams p = a;
  p.n_rows = B;
  const int pairs = B * a.kv.Hkv;
  launch_k(k_attn_warp<OT, HD>, (pairs + kPairs - 1) / kPairs, kT, smem, s, p);
  return 1;
}

template <typename OT>
int dispatch(const AttnParams& a, int B, cudaStream_t s) {
  switch (a.kv.hd) {
    case 64: return launch_hd<OT, 64>(a, B, s);
    case 128: return launch_hd<OT, 128>(a, B, s);
    default: return 0;
  }
}

}  // namespace

bool attn_warp_supports(int hd, int G, int kv_f32, int max_pos) {
  return !kv_f32 && (hd == 64 || hd == 128) && G >= 1 && G <= kG && max_pos <= kTT;
}

int launch_attention_warp(const AttnParams& a, int B, int x_type, cudaStream_t s) {
  if (B <= 0) return 0;
  return x_type == X_BF16 ? dispatch<__nv_bfloat16>(a, B, s) : dispatch<float>(a, B, s);
}

}  // namespace fsk
