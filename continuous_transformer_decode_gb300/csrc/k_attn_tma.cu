// Per-lane GQA decode attention over paged bf16 KV, pages fetched by TMA.
//
// Computes what k_attn_mma computes (RoPE of q and k at the lane's own
// position, append of k and v there, online-softmax attention of the lane's
// G query heads of one KV head over the lane's own keys 0..pos, split-K with
// an ordered merge; "MODEL-BATCHING-RESULTS", "The lever"; mlx-bun "Parallel
// slots", "KV memory" rung 3; "S1b decode: design traps" trap 2), with the
// same warp-level MMA arithmetic, but the key and value rows reach shared
// memory through the tensor memory accelerator:
//   * the KV arena [layer][page][Hkv][page_size][hd] is a 2-D tensor of
//     rows (layer, page, head, slot) x hd columns, so the rows of one
//     lane's page for one KV head are one contiguous run, copied as boxes of
//     16 rows x 64 columns with 128-byte swizzle (the split's page indices
//     are read into shared memory once);
//   * each of the 4 warps owns rows 16w..16w+15 of every 64-position tile
//     and runs its own ring of 3 slices on its own mbarriers: its lanes issue
//     the slice's copies together (a thread's copies are served one after
//     another, so independent issuers are what keeps several in flight), it
//     zeroes its value rows past the lane's length (a page's unused rows
//     hold stale data), writes the token appended at pos from registers,
//     and refills the slot when done, with no block-wide barrier in the
//     loop;
//   * per slice: S = Q K^T and O += P V on mma.m16n8k16 with q and P split
//     into hi + lo bf16 parts (rows g and g + 8 of the A operand), a per-warp
//     online softmax; the warps' and then the splits' (m, l, O) are merged in
//     a fixed order, so a lane's result does not depend on the batch.

#include <cudaTypedefs.h>
#include <math_constants.h>

#include <algorithm>

#include "attn_mma.cuh"
#include "tma_mbar.cuh"

namespace fsk {
FS_TRACE_TU(attn_tma)
namespace {

using namespace attn;
using namespace tma;

constexpr int kWarps = 4;
constexpr int kT = 32 * kWarps;
constexpr int kTT = 64;       // positions per tile; warp w owns rows 16w..16w+15
constexpr int kG = 8;         // max query heads per KV head
constexpr int kMaxRuns = 64;  // page runs per split (split_len / min(page_size, 16))

template <int HD>
struct Ring {
  static constexpr int kBlocks = HD / 64;          // 128-byte column blocks
  static constexpr int kSlice = 16 * HD * 2;       // one of K or V for 16 rows
  static constexpr int kStages = 3;                // slices in flight per warp
  static constexpr int kWarpBytes = kStages * 2 * kSlice;
};

// Byte offset of (row r < 16, 16-byte chunk) in a 16-row slice laid out as
// [HD / 64] column blocks of [16 rows][128 bytes], each written by TMA with
// 128-byte swizzle (chunk c of row r at (c ^ (r % 8)) * 16 within the row).
__device__ __forceinline__ uint32_t sws(int r, int chunk) {
  return (uint32_t)((chunk >> 3) * 2048 + r * 128 + (((chunk & 7) ^ (r & 7)) << 4));
}

template <typename OT, int HD>
__device__ __forceinline__ void attn_tma_body(const CUtensorMap& tmK, const CUtensorMap& tmV,
                                              const AttnParams& a, unsigned long long* s_tr) {
  using R = Ring<HD>;
  constexpr int kHalf = HD / 2;
  constexpr int kCh = HD / 8;            // 16-byte chunks per row
  constexpr int kKs = HD / 16;           // k-steps of Q K^T
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
  const int64_t layer_row0 = (int64_t)a.layer * (kv.layer_stride / HD);
  const int box = min(ps, 16);  // rows per copy: one page, or 16 rows of one

  extern __shared__ uint8_t smem_raw[];
  // rings 1 KB aligned: the 128-byte swizzle pattern repeats every 8 rows
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* ring = smem + warp * R::kWarpBytes;      // this warp's [kStages][K | V] slices
  float* qs = reinterpret_cast<float*>(smem + kWarps * R::kWarpBytes);  // [kG][HD]
  float* knew = qs + kG * HD;                       // [HD]
  float* vnew = knew + HD;
  float* wm = vnew + HD;                            // [kWarps][kG]
  float* wl = wm + kWarps * kG;
  uint64_t* full = reinterpret_cast<uint64_t*>(wl + kWarps * kG);  // [kWarps][kStages]
  int* srow = reinterpret_cast<int*>(full + kWarps * R::kStages);  // [kMaxRuns]
  float* wo = reinterpret_cast<float*>(smem);       // [kWarps][kG][HD], reuses the idle rings
  uint64_t* my_full = full + warp * R::kStages;
  __shared__ int s_last;

  const int n_tiles = (end - start + kTT - 1) / kTT;
  const int n_runs = (end - start + box - 1) / box;
  // the arena row of every run (box rows of one page) of this split
  for (int r = tid; r < n_runs; r += kT) {
    const int t = start + r * box, pi = t / ps, slot = t - pi * ps;
    srow[r] = (int)(layer_row0 + ((int64_t)ptrow[pi] * Hkv + g) * ps + slot);
  }
  if (tid == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    for (int i = 0; i < kWarps * R::kStages; ++i) mbar_init(smem_u32(full + i), 1);
    mbar_init_fence();
  }
  __syncthreads();
  const int p0 = warp * 16;  // this warp's rows in every tile
  // this warp's slice of tile i: `cnt` valid rows (0 when past the end)
  auto slice_rows = [&](int i) { return max(0, min(16, end - (start + i * kTT + p0))); };
  // lanes 0..: copy the runs of this warp's slice of tile i into stage i % kStages
  auto issue = [&](int i) {
    const int st = i % R::kStages;
    const int cnt = slice_rows(i);
    if (cnt == 0) return;
    const int runs = (cnt + box - 1) / box;
    const uint32_t bar = smem_u32(my_full + st);
    if (lane == 0) mbar_expect_tx(bar, (uint32_t)(2 * runs * box * HD * 2));
    __syncwarp();
    const int n_copies = 2 * runs * R::kBlocks;   // <= 16
    if (lane < n_copies) {
      const int kvsel = lane & 1, rest = lane >> 1;
      const int cb = rest % R::kBlocks, r = rest / R::kBlocks;
      const uint32_t dst = smem_u32(ring + st * 2 * R::kSlice + kvsel * R::kSlice) +
                           (uint32_t)(cb * 2048 + r * box * 128);
      const int run = (i * kTT + p0) / box + r;
      tma_load_2d(dst, kvsel ? &tmV : &tmK, cb * 64, srow[run], bar);
    }
  };
  // Programmatic dependent launch: the KV of earlier positions and the page
  // table were written by kernels that finished before the predecessor
  // started, so each warp's first copies start before waiting for it.
  const bool prefetch = !a.kv_written;  // else this step's rows come from the predecessor
  if (prefetch)
    for (int i = 0; i < min(R::kStages, n_tiles); ++i) issue(i);
  // the rotation of position pos (constant tables): thread t rotates pairs
  // i = t mod hd/2 of every head (kT is a multiple of hd/2)
  static_assert(kT % kHalf == 0, "a thread's pairs share one rotation");
  const int rp = tid % kHalf;
  const float rc_i = a.rc[(int64_t)pos * kHalf + rp], rs_i = a.rs[(int64_t)pos * kHalf + rp];
  pdl_wait();  // the QKV projection's output is read below
  TraceSmem::ready(s_tr);
  pdl_trigger();
  if (!prefetch)
    for (int i = 0; i < min(R::kStages, n_tiles); ++i) issue(i);

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
      qx0[it] = row[(g * G + h) * HD + rp];
      qx1[it] = row[(g * G + h) * HD + rp + kHalf];
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
      qs[h * HD + rp] = q0;
      qs[h * HD + rp + kHalf] = q1;
    }
  }
  if (append) {
    const int pi = pos / ps, slot = pos - pi * ps;
    const int64_t off = (int64_t)a.layer * kv.layer_stride +
                        (((int64_t)ptrow[pi] * Hkv + g) * ps + slot) * HD;
    if (tid < kHalf) {  // rp == tid
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

  const int mi = lane >> 3, ri = lane & 7;
  bool failed = false;
  for (int i = 0; i < n_tiles; ++i) {
    const int cnt = slice_rows(i);
    if (cnt == 0) break;  // past the end: so are all later slices of this warp
    const int st = i % R::kStages;
    uint8_t* kb = ring + st * 2 * R::kSlice;
    uint8_t* vb = kb + R::kSlice;
    const bool ok = mbar_wait(smem_u32(my_full + st), (uint32_t)(i / R::kStages) & 1u);
    if (!__all_sync(0xffffffffu, ok)) {  // uniform over the warp
      if (lane == 0) atomicExch(a.err, 7);
      failed = true;
      break;
    }
    // value rows past the lane's length: zeros (stale page rows)
    for (int idx = lane; idx < (16 - cnt) * kCh; idx += 32) {
      const int r = cnt + idx / kCh, ch = idx % kCh;
      *reinterpret_cast<uint4*>(vb + sws(r, ch)) = make_uint4(0, 0, 0, 0);
    }
    const int t0 = start + i * kTT + p0;
    if (append && pos >= t0 && pos < t0 + 16) {  // the appended token, from registers
      const int r = pos - t0;
      for (int ch = lane; ch < kCh; ch += 32) {
        uint4 kk, vv;
        uint32_t* kw = reinterpret_cast<uint32_t*>(&kk);
        uint32_t* vw = reinterpret_cast<uint32_t*>(&vv);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          kw[e] = pack_bf16(knew[ch * 8 + 2 * e], knew[ch * 8 + 2 * e + 1]);
          vw[e] = pack_bf16(vnew[ch * 8 + 2 * e], vnew[ch * 8 + 2 * e + 1]);
        }
        *reinterpret_cast<uint4*>(kb + sws(r, ch)) = kk;
        *reinterpret_cast<uint4*>(vb + sws(r, ch)) = vv;
      }
    }
    __syncwarp();
    // S = Q K^T for the slice's 16 positions (two n-tiles of 8)
    float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < kKs; ++ks) {
      uint32_t bk[4];
      ldsm_x4(smem_u32(kb + sws((mi >> 1) * 8 + ri, 2 * ks + (mi & 1))), bk);
      mma16816(sacc[0], qa[ks], bk[0], bk[1]);
      mma16816(sacc[1], qa[ks], bk[2], bk[3]);
    }
    // online softmax over this warp's positions, per head (row gq)
    float sv[4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int pp = nt * 8 + 2 * cq + e;
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
      ldsm_x4_t(smem_u32(vb + sws((mi & 1) * 8 + ri, j + (mi >> 1))), bv);
      mma16816(o_acc[j], pa, bv[0], bv[1]);
      mma16816(o_acc[j + 1], pa, bv[2], bv[3]);
    }
    // refill this stage with slice i + kStages: the stores and shared-memory
    // reads above come before the copy's writes
    fence_proxy_async_smem();
    __syncwarp();
    if (i + R::kStages < n_tiles) issue(i + R::kStages);
  }
  if (__syncthreads_or(failed)) {
    // a warp gave up: let every copy in flight land (bounded), then exit
    if (lane == 0)
      for (int i = 0; i < n_tiles; ++i)
        if (slice_rows(i) > 0)
          mbar_wait(smem_u32(my_full + i % R::kStages), (uint32_t)(i / R::kStages) & 1u);
    __syncthreads();
    return;
  }

  // ---- merge the warps in warp order
  if (warp < kWarps && cq == 0 && gq < kG) {
    wm[warp * kG + gq] = m_run;
    wl[warp * kG + gq] = l_run;
  }
  if (warp < kWarps && gq < G) {
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
  // merge: every split's (m, l) into shared memory with plain loads and the
  // splits' outputs by asynchronous copies into the idle rings, all in flight
  // together (`chunk` splits at a time, every split when they fit); the
  // weights once per (split, head); then the outputs from shared memory. All
  // sums in ascending split order.
  constexpr int kOut = (kG * HD + kT - 1) / kT;   // outputs per thread (at most)
  float* sm = reinterpret_cast<float*>(smem);     // [ns][kG] m, then weights
  float* sl = sm + (size_t)ns * kG;               // [ns][kG] l
  float* sL = sl + (size_t)ns * kG;               // [kG] merged l
  const int ml_bytes = ((2 * ns * kG + kG) * (int)sizeof(float) + 15) & ~15;
  float* sp = reinterpret_cast<float*>(smem + ml_bytes);  // [chunk][G * HD]
  const int gh = G * HD;                                  // floats of one split
  const int chunk = (kWarps * R::kWarpBytes - ml_bytes) / (gh * (int)sizeof(float));
  const float* src = a.part_acc + (((int64_t)b * a.max_splits) * H + g * G) * HD;
  const int64_t qstride = (int64_t)H * HD;
  auto stage = [&](int q0) {  // splits q0 .. q0 + chunk - 1 into sp
    const int per = gh / 4;   // 16-byte pieces of one split
    const int n16 = min(chunk, ns - q0) * per;
    for (int c = tid; c < n16; c += kT) {
      const int q = c / per, r = c - q * per;
      cp_async16(smem_u32(sp + q * gh + 4 * r), src + (q0 + q) * qstride + 4 * r);
    }
    cp_commit();
  };
  stage(0);
  for (int idx = tid; idx < ns * G; idx += kT) {
    const int q = idx / G, h = idx - q * G;
    const int64_t bq = ((int64_t)b * a.max_splits + q) * H + g * G + h;
    sm[q * kG + h] = __ldcg(a.part_ml + 2 * bq);
    sl[q * kG + h] = __ldcg(a.part_ml + 2 * bq + 1);
  }
  cp_wait<0>();
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
  float acc[kOut];
#pragma unroll
  for (int j = 0; j < kOut; ++j) acc[j] = 0.0f;
  for (int q0 = 0; q0 < ns; q0 += chunk) {
    if (q0 > 0) {  // every thread is done with the previous chunk
      __syncthreads();
      stage(q0);
      cp_wait<0>();
      __syncthreads();
    }
    const int nq = min(chunk, ns - q0);
    for (int qq = 0; qq < nq; ++qq) {
      const float* pq = sp + qq * gh;
      const float* wq = sm + (q0 + qq) * kG;
#pragma unroll
      for (int j = 0; j < kOut; ++j) {
        const int o = tid + j * kT;
        if (o < gh) acc[j] = fmaf(pq[o], wq[o / HD], acc[j]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kOut; ++j) {
    const int o = tid + j * kT;
    if (o < gh) st_out(orow + o, acc[j] / sL[o / HD], a.o_lo);
  }
}

// Thread 0's trace marks stay in shared memory (s_tr): tracing costs the
// body no registers.
template <typename OT, int HD>
__global__ void __launch_bounds__(kT, HD == 256 ? 1 : 2)
    k_attn_tma(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               AttnParams a) {
  __shared__ unsigned long long s_tr[4];
  TraceSmem::begin(s_tr, g_trace);
  attn_tma_body<OT, HD>(tmK, tmV, a, s_tr);
  TraceSmem::end(s_tr, TR_ATTN_TMA);
}

template <int HD>
constexpr size_t smem_bytes() {
  return 1024 + (size_t)kWarps * Ring<HD>::kWarpBytes +
         sizeof(float) * ((size_t)kG * HD + 2 * HD + 2 * kWarps * kG) +
         8 * (size_t)kWarps * Ring<HD>::kStages + sizeof(int) * kMaxRuns;
}

template <typename OT, int HD>
int launch_hd(const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnParams& a, int B,
              cudaStream_t s) {
  static_assert(kWarps * kG * HD * sizeof(float) <= (size_t)kWarps * Ring<HD>::kWarpBytes,
                "the warp-merge buffer must fit in the rings");
  constexpr size_t smem = smem_bytes<HD>();
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(k_attn_tma<OT, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    attr = true;
  }
  dim3 grid(a.max_splits, a.kv.Hkv, B);
  launch_k(k_attn_tma<OT, HD>, grid, kT, smem, s, tmK, tmV, a);
  return 1;
}

template <typename OT>
int dispatch(const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnParams& a, int B,
             cudaStream_t s) {
  switch (a.kv.hd) {
    case 64: return launch_hd<OT, 64>(tmK, tmV, a, B, s);
    case 128: return launch_hd<OT, 128>(tmK, tmV, a, B, s);
    case 256: return launch_hd<OT, 256>(tmK, tmV, a, B, s);
    default: return 0;
  }
}

}  // namespace

bool attn_tma_supports(int hd, int G, int kv_f32, int page_size, int split_len,
                       int max_splits) {
  if (kv_f32 || !(hd == 64 || hd == 128 || hd == 256) || G < 1 || G > kG) return false;
  // a copy is one page (page_size | 16) or 16 rows of one (16 | page_size),
  // a whole number of 8-row swizzle atoms
  const bool runs = (page_size % 8 == 0) && (16 % page_size == 0 || page_size % 16 == 0);
  const size_t ring_bytes = hd == 64 ? (size_t)kWarps * Ring<64>::kWarpBytes
                            : hd == 128 ? (size_t)kWarps * Ring<128>::kWarpBytes
                                        : (size_t)kWarps * Ring<256>::kWarpBytes;
  // the merge's (m, l) arrays and at least one split's outputs in the rings
  const size_t merge_bytes = (((size_t)(2 * kG * max_splits + kG) * sizeof(float) + 15) & ~15) +
                             (size_t)G * hd * sizeof(float);
  return runs && split_len % kTT == 0 && split_len / std::min(page_size, 16) <= kMaxRuns &&
         merge_bytes <= ring_bytes;
}

// 2-D map over a KV arena [rows][hd] bf16 (rows = layers * pages * Hkv *
// page_size), box [min(page_size, 16) rows][64 columns], 128-byte swizzle.
int attn_tma_make_map(const void* arena, int64_t rows, int hd, int page_size, CUtensorMap* out) {
  if (!tc_available() || rows >= ((int64_t)1 << 31)) return -1;
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return -1;
    enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  cuuint64_t dims[2] = {(cuuint64_t)hd, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)hd * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)std::min(page_size, 16)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(arena), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -2;
}

int launch_attention_tma(const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnParams& a,
                         int B, int x_type, cudaStream_t s) {
  if (B <= 0) return 0;
  return x_type == X_BF16 ? dispatch<__nv_bfloat16>(tmK, tmV, a, B, s)
                          : dispatch<float>(tmK, tmV, a, B, s);
}

}  // namespace fsk
