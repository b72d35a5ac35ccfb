// Weight-streaming GEMM on the 5th-generation tensor cores (tcgen05).
//
// Y[b, n] = sum_k X[b, k] * W[n, k] over the B lanes of the step panel: the
// seven projections and the LM head of every lane run as one GEMM per weight
// matrix, so each weight byte is read once per step ("MODEL-BATCHING-
// RESULTS", "The lever").
//
// Swap-AB: the weight tile is the M = 128 operand (rows of W), the lanes are
// the N operand, so one 128-row weight tile serves every lane and small B
// costs no weight re-reads. Operands are staged by TMA into 128-byte-swizzled
// shared memory; the f32 accumulator lives in tensor memory (TMEM). A stage
// holds several consecutive 64-wide k-blocks of one row tile, filled by one
// 3-D weight copy and one 3-D panel copy: an SM's TMA copies complete one
// after another, so their number, more than their bytes, sets a block's
// time at the small sizes of a decode step.
//
// Block = 6 warps: warp 4 issues TMA loads, warp 5 owns TMEM and issues the
// MMAs, warps 0-3 run the epilogue (warp w reads TMEM lanes 32w..32w+31,
// i.e. weight rows; each thread then holds one output row for every lane).
// Work split (stream-K): the matrix's k-blocks, row tile after row tile, are
// cut into P equal contiguous ranges, and block c of each lane group streams
// range c through one ring of stages, so every block moves the same number
// of weight bytes and no launch ends in a partial wave. The part of a range
// inside one row tile is a piece, accumulated in TMEM; a piece covering the
// whole tile goes straight to the epilogue, a partial one to a workspace,
// and the last piece of a tile to arrive sums the tile's pieces in block
// order, so results never depend on timing. P depends only on the matrix
// shape, the handle's lane capacity and the SM count, never on the number of
// lanes in a call; lane groups split the N dimension only. A lane's output
// is therefore independent of the batch it is computed in.
//
// Every wait on an mbarrier is bounded (1 s of %globaltimer); on timeout the
// block records an error code, stops issuing work, drains the TMA loads it
// issued (again bounded), frees its TMEM and exits.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include <algorithm>
#include <climits>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>

#include "fs_internal.h"
#include "tma_mbar.cuh"

namespace fsk {
FS_TRACE_TU(gemm)
namespace {

using namespace tma;

constexpr int kBM = 128;
constexpr int kBK = 64;                 // bf16 elements per 128-byte row
constexpr int kThreads = 192;
constexpr int kWTileBytes = kBM * kBK * 2;  // 16 KB
// Q8_0 stage: bf16 A tile | int8 codes (8 KB) | fp16 scales (512 B) | X tile
constexpr int kQ8Codes = kBM * kBK;        // 8 KB
constexpr int kQ8Scales = kBM * 2 * 2;     // 512 B
constexpr int kQ8XOff = 25 * 1024;         // 16 + 8 + 0.5 KB, 1 KB aligned
constexpr int kQ8Tile = kQ8Codes + kQ8Scales;  // a tile in global memory: codes, then scales
constexpr int kXbufBytes = 64 * 17 * 4 + 256;  // SwiGLU gate/up exchange, 8-byte aligned end

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
// K-major operand, 128-byte swizzle: rows of 128 bytes, 8-row atoms 1024 B
// apart (stride byte offset), descriptor version 1, layout SWIZZLE_128B (2).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// kind::f16 instruction descriptor: D f32, A and B bf16, both K-major.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
// 1-D bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"((uint64_t)src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          bar)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void epi_bar() {  // the 128 epilogue threads
  asm volatile("bar.sync 1, 128;" ::: "memory");
}
// 16 consecutive f32 columns of this thread's TMEM lane; the caller waits
// (tmem_wait) before reading the registers, so several loads can be in
// flight together.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t r[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32"
      " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Thread-block cluster barrier (every thread of every block of the cluster
// arrives; release / acquire order shared-memory accesses across blocks).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// Address of the same shared-memory location in block `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_dsmem4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ int ld_dsmem_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// z * sigmoid(z) with the fast exponential and division intrinsics (the
// result is rounded to bf16, far coarser than their error); exp(-z)
// overflowing to infinity gives -0.
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// Stream-K bookkeeping. The T = m_tiles * kb_total k-blocks of the matrix,
// taken tile by tile, are cut into P contiguous ranges; block c of a lane
// group owns k-blocks [c T / P, (c + 1) T / P). The part of a range that
// falls in one row tile is a piece: a whole tile goes straight to the
// epilogue, a partial one to the workspace, and the last piece of a tile to
// arrive sums that tile's pieces in block order.
// (32-bit: the host keeps (P + 1) * T below 2^31.)
__device__ __forceinline__ int sk_lo(int c, int T, int P) { return c * T / P; }
// The block whose range holds k-block g.
__device__ __forceinline__ int sk_owner(int g, int T, int P) {
  return ((g + 1) * P - 1) / T;
}
// Workspace piece of block c (slot 0: the first tile of its range, slot 1:
// the last) for one lane of the call: 128 f32, one per row of the tile.
__device__ __forceinline__ float* piece_ptr(const TcParams& p, int slot, int c, int lane) {
  return p.ws + (((int64_t)slot * p.P + c) * p.lanes_total + lane) * kBM;
}
struct TilePieces {
  int cA, cB;  // first and last block contributing to the tile
  int slotA;   // slot of block cA's piece (1 when its range starts in an earlier tile)
};
__device__ __forceinline__ TilePieces tile_pieces(const TcParams& p, int t) {
  const int T = p.m_tiles * p.kb_total;
  const int tb = t * p.kb_total;
  TilePieces r;
  r.cA = sk_owner(tb, T, p.P);
  r.cB = sk_owner(tb + p.kb_total - 1, T, p.P);
  r.slotA = sk_lo(r.cA, T, p.P) < tb ? 1 : 0;
  return r;
}

// Writes one 16-lane chunk of final values of this thread's row.
// SwiGLU: the tile's rows 0-63 are gate rows and 64-127 the matching up
// rows; the gate thread of a pair finishes lanes 0-7 and the up thread
// lanes 8-15, each handing the other half of its values to its partner
// through shared memory (xbuf: two 64 x 9 float arrays).
// Argmax: per lane, (max, lowest row) over the tile's 128 rows. The chunk
// goes through shared memory as order-preserving integer keys (abuf, two
// alternating [16][136] arrays in the idle ring); 8 threads per lane then
// scan 16 rows each in ascending order and combine with 3 shuffles.
template <bool kSplit>
__device__ __forceinline__ void emit_chunk(const TcParams& p, int m_tile, int row_local,
                                           int lane0, int lanes, int c0, const float v[16],
                                           float* xbuf, uint32_t* abuf) {
  if (p.epi == EPI_SWIGLU) {
    const bool up = row_local >= 64;
    const int r = row_local & 63;
    float* mine = xbuf + (up ? 64 * 9 : 0) + r * 9;
    const float* theirs = xbuf + (up ? 0 : 64 * 9) + r * 9;
#pragma unroll
    for (int j = 0; j < 8; ++j) mine[j] = v[up ? j : 8 + j];
    epi_bar();
    const int f = m_tile * 64 + r;
    if (f < p.n_out) {
      __nv_bfloat16* o0 = static_cast<__nv_bfloat16*>(p.out_x) + (int64_t)(lane0 + c0) * p.ldo + f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int jj = up ? 8 + j : j;  // lane of the chunk
        if (c0 + jj < lanes) {
          const float g = up ? theirs[j] : v[j];
          const float u = up ? v[8 + j] : theirs[j];
          const float a = silu(g) * u;
          __nv_bfloat16* o = o0 + (int64_t)jj * p.ldo;
          const __nv_bfloat16 ah = __float2bfloat16_rn(a);
          *o = ah;
          if (kSplit && p.lo_off > 0) o[p.lo_off] = __float2bfloat16_rn(a - __bfloat162float(ah));
        }
      }
    }
    epi_bar();  // xbuf is rewritten by the next chunk
    return;
  }
  if (p.epi == EPI_ARGMAX) {
    constexpr int kLd = 136;  // conflict-free for the writes and the scans
    uint32_t* kb = abuf + ((c0 >> 4) & 1) * 16 * kLd;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint32_t u = __float_as_uint(v[j] + 0.0f);  // -0 as +0
      kb[j * kLd + row_local] = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    }
    epi_bar();
    const int jl = row_local >> 3, q = row_local & 7;
    const int row0 = m_tile * kBM;
    uint32_t bk = 0, br = 0xffffffffu;  // best key and its row (none yet)
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int r = i * 8 + q;  // ascending: the first of equal keys is the lowest row
      const uint32_t k = kb[jl * kLd + r];
      if (row0 + r < p.n_out && (br == 0xffffffffu || k > bk)) {
        bk = k;
        br = (uint32_t)(row0 + r);
      }
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      const uint32_t ok = __shfl_xor_sync(0xffffffffu, bk, o);
      const uint32_t orow = __shfl_xor_sync(0xffffffffu, br, o);
      if (orow != 0xffffffffu &&
          (br == 0xffffffffu || ok > bk || (ok == bk && orow < br))) {
        bk = ok;
        br = orow;
      }
    }
    if (q == 0 && c0 + jl < lanes) {
      const uint32_t u = (bk & 0x80000000u) ? (bk & 0x7fffffffu) : ~bk;
      const int64_t at = (int64_t)(lane0 + c0 + jl) * p.m_tiles + m_tile;
      p.am_val[at] = __uint_as_float(u);
      p.am_idx[at] = (int)br;
    }
    return;  // the next chunk writes the other array; the one after, past
             // that chunk's barrier
  }
  const int row = m_tile * kBM + row_local;
  if (row >= p.n_out) return;
  float* o = p.out_f32 + (int64_t)(lane0 + c0) * p.ldo + row;
  if (p.epi == EPI_RESID) {
    float prev[16];  // every load of the chunk before any store
#pragma unroll
    for (int j = 0; j < 16; ++j) prev[j] = (c0 + j < lanes) ? __ldcg(o + (int64_t)j * p.ldo) : 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (c0 + j < lanes) o[(int64_t)j * p.ldo] = prev[j] + v[j];
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (c0 + j < lanes) o[(int64_t)j * p.ldo] = v[j];
  }
}

__device__ __forceinline__ float4 ld4(const float* q) {
  return __ldcg(reinterpret_cast<const float4*>(q));
}
__device__ __forceinline__ void add4(float4& a, const float4& b) {
  a.x += b.x;
  a.y += b.y;
  a.z += b.z;
  a.w += b.w;
}
// Sum, in block order, of a tile's pieces at rows r0 .. r0+3 of one lane.
__device__ __forceinline__ float4 sum_pieces4(const TcParams& p, const TilePieces& tp,
                                              int lane, int r0) {
  float4 acc = ld4(piece_ptr(p, tp.slotA, tp.cA, lane) + r0);
  int c = tp.cA + 1;
  for (; c + 3 <= tp.cB; c += 4) {  // four independent loads, added in block order
    const float4 v0 = ld4(piece_ptr(p, 0, c, lane) + r0);
    const float4 v1 = ld4(piece_ptr(p, 0, c + 1, lane) + r0);
    const float4 v2 = ld4(piece_ptr(p, 0, c + 2, lane) + r0);
    const float4 v3 = ld4(piece_ptr(p, 0, c + 3, lane) + r0);
    add4(acc, v0);
    add4(acc, v1);
    add4(acc, v2);
    add4(acc, v3);
  }
  for (; c <= tp.cB; ++c) add4(acc, ld4(piece_ptr(p, 0, c, lane) + r0));
  return acc;
}

// Last piece of a row tile to arrive: sum the tile's pieces and apply the
// epilogue with 16-byte accesses (threads map to 4-row groups x lanes).
template <bool kSplit>
__device__ void reduce_tile(const TcParams& p, int m_tile, const TilePieces& tp, int lane0,
                            int lanes) {
  const int t = threadIdx.x;  // 0..127
  if (p.epi == EPI_SWIGLU) {
    const int rq = (t & 15) * 4, lsub = t >> 4;  // 16 threads per lane row
    const int f0 = m_tile * 64 + rq;
    if (f0 >= p.n_out) return;
    for (int b0 = lsub; b0 < lanes; b0 += 16) {
      float4 g[2], u[2];
#pragma unroll
      for (int k = 0; k < 2; ++k)
        if (b0 + 8 * k < lanes) {
          g[k] = sum_pieces4(p, tp, lane0 + b0 + 8 * k, rq);
          u[k] = sum_pieces4(p, tp, lane0 + b0 + 8 * k, 64 + rq);
        }
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int b = b0 + 8 * k;
        if (b >= lanes) break;
        const float a0 = silu(g[k].x) * u[k].x, a1 = silu(g[k].y) * u[k].y;
        const float a2 = silu(g[k].z) * u[k].z, a3 = silu(g[k].w) * u[k].w;
        __nv_bfloat162 lo = __floats2bfloat162_rn(a0, a1);
        __nv_bfloat162 hi = __floats2bfloat162_rn(a2, a3);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t*>(&lo);
        pk.y = *reinterpret_cast<uint32_t*>(&hi);
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out_x) + (int64_t)(lane0 + b) * p.ldo + f0;
        *reinterpret_cast<uint2*>(o) = pk;
        if (kSplit && p.lo_off > 0) {
          const float2 fl = __bfloat1622float2(lo), fh = __bfloat1622float2(hi);
          __nv_bfloat162 rl = __floats2bfloat162_rn(a0 - fl.x, a1 - fl.y);
          __nv_bfloat162 rh = __floats2bfloat162_rn(a2 - fh.x, a3 - fh.y);
          pk.x = *reinterpret_cast<uint32_t*>(&rl);
          pk.y = *reinterpret_cast<uint32_t*>(&rh);
          *reinterpret_cast<uint2*>(o + p.lo_off) = pk;
        }
      }
    }
    return;
  }
  const int rq = (t & 31) * 4, lsub = t >> 5;  // 32 threads per lane row
  const int row0 = m_tile * kBM + rq;
  if (row0 >= p.n_out) return;
  const bool vec = (p.ldo & 3) == 0 && row0 + 4 <= p.n_out;
  constexpr int U = 4;  // lanes in flight per thread: all loads, then stores
  for (int b0 = lsub; b0 < lanes; b0 += 4 * U) {
    float4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (b0 + 4 * u < lanes) v[u] = sum_pieces4(p, tp, lane0 + b0 + 4 * u, rq);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int b = b0 + 4 * u;
      if (b >= lanes) break;
      float* o = p.out_f32 + (int64_t)(lane0 + b) * p.ldo + row0;
      if (vec) {
        if (p.epi == EPI_RESID) add4(v[u], __ldcg(reinterpret_cast<const float4*>(o)));
        *reinterpret_cast<float4*>(o) = v[u];
      } else {
        const float vv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        for (int e = 0; e < 4 && row0 + e < p.n_out; ++e)
          o[e] = p.epi == EPI_RESID ? __ldcg(o + e) + vv[e] : vv[e];
      }
    }
  }
}

// Dequantises one stage's Q8_0 tile (thread r = weight row r) into the
// 128-byte-swizzled bf16 A tile: 16-byte chunk c of row r lands at
// r * 128 + ((c ^ (r % 8)) * 16), the layout a SWIZZLE_128B copy produces.
__device__ __forceinline__ void dequant_q8_tile(uint8_t* stage, int r) {
  const uint8_t* raw = stage + kWTileBytes + r * kBK;
  const __half* sc = reinterpret_cast<const __half*>(stage + kWTileBytes + kQ8Codes) + r * 2;
  const float d0 = __half2float(sc[0]), d1 = __half2float(sc[1]);
  uint8_t* arow = stage + r * 128;
#pragma unroll
  for (int c16 = 0; c16 < 4; ++c16) {
    const uint4 u = *reinterpret_cast<const uint4*>(raw + c16 * 16);
    const int8_t* q = reinterpret_cast<const int8_t*>(&u);
    const float d = c16 < 2 ? d0 : d1;  // inputs 0-31 / 32-63 of the block
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint4 o;
      uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 v = __floats2bfloat162_rn((float)q[half * 8 + 2 * e] * d,
                                                       (float)q[half * 8 + 2 * e + 1] * d);
        ow[e] = *reinterpret_cast<const uint32_t*>(&v);
      }
      const int c = c16 * 2 + half;
      *reinterpret_cast<uint4*>(arow + ((c ^ (r & 7)) * 16)) = o;
    }
  }
}

// kSplit: the panel has a remainder part (TcParams::split), two MMAs per
// k-step; a compile-time switch so that the plain kernel carries none of it.
// How a launch reduces K: plain (whole tiles, or stream-K ranges summed
// through the workspace) or cluster (the K splits of a tile are the blocks
// of a thread-block cluster). A compile-time switch, so that each kernel
// carries only its own reduction.
enum GemmMode { GM_PLAIN = 0, GM_CLUSTER = 1 };

template <bool kQ8, bool kSplit, int kMode>
__device__ __forceinline__ void gemm_tc_body(const CUtensorMap& tmW, const CUtensorMap& tmX,
                                             const CUtensorMap& tmXlo, const TcParams& p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_last;
  __shared__ int s_stop[2];
  __shared__ unsigned long long s_tr[4];
  TraceSmem::begin(s_tr, g_trace);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // cluster reduction: the cs K splits of one (row tile, lane group) are
  // consecutive blocks, one cluster; otherwise the lane groups of one
  // stream-K range are consecutive (they share its weight tiles in L2)
  constexpr bool kCluster = kMode == GM_CLUSTER;
  const int cs = kCluster ? p.cs : 0;
  const int cs_rank = kCluster ? (int)(blockIdx.x % cs) : 0;
  const int cs_unit = kCluster ? (int)(blockIdx.x / cs) : 0;  // tile * groups + group
  const int group = kCluster ? cs_unit % p.groups : (int)(blockIdx.x % p.groups);
  const int cblk = kCluster ? (cs_unit / p.groups) * cs + cs_rank  // stream-K block
                        : (int)(blockIdx.x / p.groups);
  const int lane0 = group * p.lg;
  const int lanes = min(p.lg, p.lanes_total - lane0);
  const int n_tot = (lanes + 15) & ~15;
  const int kbt = p.kb_total;
  const int T = p.m_tiles * kbt;
  const int g0 = sk_lo(cblk, T, p.P), g1 = sk_lo(cblk + 1, T, p.P);  // g1 > g0: P <= T
  const int t_first = g0 / kbt;
  const int n_pieces = (g1 - 1) / kbt - t_first + 1;
  // Stages: the range's k-blocks, piece by piece, in chunks of at most kq
  // consecutive k-blocks of one row tile. A stage is one weight copy (a 3-D
  // box of kq 128 x 64 tiles) and one panel copy per panel part (a box of
  // kq tiles of xh lanes x 64), each tile in the 128-byte-swizzled K-major
  // layout the MMA reads; copies past the range or the matrix are unused or
  // zero-filled.
  const int kq = p.kq, xh = p.xh;
  int n_st = 0;
  for (int q = 0; q < n_pieces; ++q) {
    const int tb = (t_first + q) * kbt;
    n_st += (min(g1, tb + kbt) - max(g0, tb) + kq - 1) / kq;
  }
  // first k-block and k-block count of stage i (0 <= i < n_st)
  auto stage_at = [&](int i, int& g, int& cnt) {
    if (kq == 1) {  // the stages are the range's k-blocks in order
      g = g0 + i;
      cnt = 1;
      return;
    }
    if (n_pieces == 1) {
      g = g0 + i * kq;
      cnt = min(kq, g1 - g);
      return;
    }
    int t = t_first, pb = g0;
    for (;;) {
      const int pe = min(g1, (t + 1) * kbt);
      const int nch = (pe - pb + kq - 1) / kq;
      if (i < nch) {
        g = pb + i * kq;
        cnt = min(kq, pe - g);
        return;
      }
      i -= nch;
      ++t;
      pb = t * kbt;
    }
  };
  const int S = p.stages;
  float* xbuf = reinterpret_cast<float*>(smem + (size_t)S * p.stage_bytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)S * p.stage_bytes + kXbufBytes);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S),
                 conv0 = smem_u32(bars + 2 * S), tfull = smem_u32(bars + 3 * S),
                 tempty = smem_u32(bars + 3 * S + 1), tready = smem_u32(bars + 3 * S + 2);
  const uint32_t ncols = p.tmem_cols;

  if (threadIdx.x == 0) {
    if (!kQ8) prefetch_tensormap(&tmW);
    prefetch_tensormap(&tmX);
    if (kSplit) prefetch_tensormap(&tmXlo);
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
      if (kQ8) mbar_init(conv0 + 8 * s, 128);  // the 128 converters
    }
    mbar_init(tfull, 1);     // the MMA issuer's commit at the end of a piece
    mbar_init(tempty, 128);  // every epilogue thread, after reading TMEM
    mbar_init(tready, 1);    // the MMA warp, once it holds its TMEM columns
    mbar_init_fence();
    s_abort = 0;
    s_last = 0;
  }
  __syncthreads();  // barriers initialised
  uint32_t tmem = 0;  // TMEM base, known to the MMA warp and (after tready) the epilogue
  // TMA producers. Before the wait for the predecessor, one lane per stage
  // issues that stage's weight copy; after it, one lane per panel copy (lanes
  // that issued no weight copy first); in the steady state lane 0 issues the
  // weight copy and lanes 1-2 the panel copies. A block holding a single
  // piece (whole tile, or one K split of one) also lets its 4 epilogue
  // warps, idle until the accumulator is ready, take the stages congruent to
  // their index; otherwise warp 4 issues every stage (the epilogue warps then
  // drain pieces while it keeps the ring full).
  const int npw = p.prod_warps;  // divides S
  const bool warp_prod = !kQ8 && n_pieces == 1 && npw > 1;
  constexpr int nparts = kSplit ? 2 : 1;  // panel copies per stage
  const uint32_t wpart = kQ8 ? (uint32_t)kQ8XOff : (uint32_t)(kq * kWTileBytes);
  const uint32_t xpart = (uint32_t)(kq * xh * 128);  // one panel copy
  const uint32_t x_bytes = xpart * nparts;
  // warp-collective: stages first, first + step, ...
  auto produce = [&](int first, int step) {
    int issued = -1;  // last stage issued
    // g: the stage's first k-block (= m_tile * kb_total + kb)
    auto load_w = [&](int i, int g) {  // weight part of stage i (and its expect_tx)
      const int s = i % S;
      const uint32_t st = smem_u32(smem + (size_t)s * p.stage_bytes);
      if (kQ8) {  // kq = 1
        // one copy: the tile's codes and, right after them, its scales
        mbar_expect_tx(full0 + 8 * s, (uint32_t)kQ8Tile + x_bytes);
        bulk_load(st + kWTileBytes, p.q8_tiles + (int64_t)g * kQ8Tile, kQ8Tile, full0 + 8 * s);
      } else {
        const int tile = g / kbt;
        mbar_expect_tx(full0 + 8 * s, wpart + x_bytes);
        tma_load_3d(st, &tmW, 0, tile * kBM, g - tile * kbt, full0 + 8 * s);
      }
    };
    auto load_x = [&](int i, int g, int part) {  // panel part (1: remainders) of stage i
      const uint32_t st = smem_u32(smem + (size_t)(i % S) * p.stage_bytes) + wpart + part * xpart;
      tma_load_3d(st, part ? &tmXlo : &tmX, 0, lane0, g % kbt, full0 + 8 * (i % S));
    };
    // Programmatic dependent launch: the weight tiles do not depend on the
    // predecessor kernel, so they are issued before waiting for it; the
    // panel is the predecessor's output.
    const int pre = min(S, n_st);  // stages are empty at start: no wait needed
    const int n_pre = pre > first ? (pre - first + step - 1) / step : 0;  // this warp's
    for (int j = lane; j < n_pre; j += 32) {
      int g, cnt;
      stage_at(first + j * step, g, cnt);
      load_w(first + j * step, g);
    }
    __syncwarp();
    pdl_wait();
    TraceSmem::ready(s_tr);
    pdl_trigger();
    for (int c = (lane + 32 - n_pre % 32) % 32; c < n_pre * nparts; c += 32) {
      const int i = first + (c / nparts) * step;
      int g, cnt;
      stage_at(i, g, cnt);
      load_x(i, g, c % nparts);
    }
    if (n_pre > 0) issued = first + (n_pre - 1) * step;
    for (int i = first + n_pre * step; i < n_st; i += step) {
      const int s = i % S;
      const uint32_t ph = (uint32_t)(i / S) & 1u;
      const bool ok = mbar_wait(empty0 + 8 * s, ph ^ 1u);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) {
          atomicExch(p.err, 1);
          s_abort = 1;
        }
        break;
      }
      if (__shfl_sync(0xffffffffu, *(volatile int*)&s_abort, 0)) break;
      int g, cnt;
      stage_at(i, g, cnt);
      if (lane == 0) load_w(i, g);  // the expect_tx comes before any panel copy
      __syncwarp();
      if (lane >= 1 && lane <= nparts) load_x(i, g, lane - 1);
      issued = i;
    }
    // drain: every copy issued here must have landed before the block exits
    for (int i = issued; i >= 0 && i > issued - S; i -= step) {
      const int s = i % S;
      if (!mbar_wait(full0 + 8 * s, (uint32_t)(i / S) & 1u) && lane == 0) atomicExch(p.err, 2);
    }
  };
  const bool early = warp_prod ? warp < npw : warp == 4;  // producers wait inside produce
  if (!early) {
    pdl_wait();
    TraceSmem::ready(s_tr);
    pdl_trigger();
  }

  if (warp == 4) {
    if (!warp_prod) produce(0, 1);
  } else if (warp == 5) {
    // TMEM is taken only now, after the preceding kernel has finished (the
    // wait above): a block brought in early by programmatic dependent launch
    // holds no columns while it waits, so it never stalls the allocation of
    // the running kernel's blocks, nor does its weight prefetch wait for one.
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&s_tmem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(tready);
    tc_fence_after();
    tmem = *(volatile uint32_t*)&s_tmem;
    if (lane == 0) {  // ---- MMA issuer: one TMEM accumulation per piece
      bool ok = true;
      int i = 0;  // stage
      const uint32_t idesc = idesc_bf16(kBM, n_tot);
      for (int q = 0; q < n_pieces && ok; ++q) {
        const int tb = (t_first + q) * kbt;
        const int pb = max(g0, tb), pe = min(g1, tb + kbt);
        if (q > 0) {  // the epilogue has read the previous piece out of TMEM
          if (!mbar_wait(tempty, (uint32_t)(q - 1) & 1u) || *(volatile int*)&s_abort) {
            atomicExch(p.err, 6);
            s_abort = 1;
            ok = false;
          }
          tc_fence_after();
        }
        bool acc = false;
        for (int g = pb; ok && g < pe; g += kq, ++i) {
          const int cnt = min(kq, pe - g);
          const int s = i % S;
          const uint32_t ph = (uint32_t)(i / S) & 1u;
          if (!mbar_wait(full0 + 8 * s, ph) || (kQ8 && !mbar_wait(conv0 + 8 * s, ph)) ||
              *(volatile int*)&s_abort) {
            atomicExch(p.err, 3);
            s_abort = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + (size_t)s * p.stage_bytes);
          const uint32_t b0 = a0 + wpart;
          for (int j = 0; j < cnt; ++j) {
            const uint32_t aj = a0 + (uint32_t)(j * kWTileBytes);
            const uint32_t bj = b0 + (uint32_t)(j * xh * 128);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
              mma_bf16(tmem, sw128_desc(aj + kk * 32), sw128_desc(bj + kk * 32), idesc,
                       (acc || kk > 0) ? 1u : 0u);
              if (kSplit)
                mma_bf16(tmem, sw128_desc(aj + kk * 32), sw128_desc(bj + xpart + kk * 32), idesc,
                         1u);
            }
            acc = true;
          }
          mma_commit(empty0 + 8 * s);  // frees the stage once these MMAs finish
        }
        mma_commit(tfull);  // arrives when every MMA issued above has finished
      }
    }
  } else {  // ---- warps 0-3: Q8_0 dequantisation of each piece, then its epilogue
    if (warp_prod && warp < npw) produce(warp, npw);
    const int row_local = warp * 32 + lane;
    if (!mbar_wait(tready, 0)) {  // the MMA warp's columns
      atomicExch(p.err, 7);
      s_abort = 1;
    }
    tc_fence_after();
    tmem = *(volatile uint32_t*)&s_tmem;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    int i = 0;
    for (int q = 0; q < n_pieces; ++q) {
      const int t = t_first + q;
      const int tb = t * kbt;
      const int pb = max(g0, tb), pe = min(g1, tb + kbt);
      if (kQ8) {
        for (; g0 + i < pe; ++i) {
          const int s = i % S;
          if (!mbar_wait(full0 + 8 * s, (uint32_t)(i / S) & 1u)) {
            atomicExch(p.err, 5);
            s_abort = 1;
            break;
          }
          dequant_q8_tile(smem + (size_t)s * p.stage_bytes, row_local);
          fence_proxy_async_smem();  // visible to the MMA
          mbar_arrive(conv0 + 8 * s);
        }
      }
      if (!mbar_wait(tfull, (uint32_t)q & 1u)) {
        atomicExch(p.err, 4);
        s_abort = 1;
      }
      tc_fence_after();
      // one thread samples the abort flag so that all 128 take the same
      // branch (the slot alternates: a slot is rewritten only two pieces
      // later, after a barrier every thread has passed)
      if (threadIdx.x == 0) s_stop[q & 1] = *(volatile int*)&s_abort;
      epi_bar();
      if (s_stop[q & 1]) break;
      const bool whole = pb == tb && pe == tb + kbt;
      const int slot = q == 0 ? 0 : 1;
      for (int c0 = 0; c0 < n_tot; c0 += 32) {  // two 16-lane loads in flight
        uint32_t r[2][16];
        tmem_ld16(trow + (uint32_t)c0, r[0]);
        if (c0 + 16 < n_tot) tmem_ld16(trow + (uint32_t)(c0 + 16), r[1]);
        tmem_wait();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int cc = c0 + 16 * h;
          if (cc >= n_tot) break;
          float v[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[h][j]);
          if (whole) {
            emit_chunk<kSplit>(p, t, row_local, lane0, lanes, cc, v, xbuf,
                               reinterpret_cast<uint32_t*>(smem));
          } else if (kCluster) {  // the partial tile stays in this block's ring
            float4* dst = reinterpret_cast<float4*>(
                reinterpret_cast<float*>(smem) + row_local * (n_tot + 4) + cc);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          } else {
            float* dst = piece_ptr(p, slot, cblk, lane0 + cc) + row_local;
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (cc + j < lanes) dst[j * kBM] = v[j];
          }
        }
      }
      tc_fence_before();
      mbar_arrive(tempty);  // the accumulator may be overwritten by the next piece
      if (!whole && !kCluster) {
        __threadfence();
        epi_bar();
        const TilePieces tp = tile_pieces(p, t);
        int* ctr = p.counters + t * p.groups + group;
        if (threadIdx.x == 0) s_last = atomicAdd(ctr, 1) == tp.cB - tp.cA;
        epi_bar();
        if (s_last) {
          __threadfence();
          reduce_tile<kSplit>(p, t, tp, lane0, lanes);
          if (threadIdx.x == 0) *ctr = 0;  // ready for the next launch
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (kCluster) {
    // Every thread of every block of the cluster passes both barriers,
    // whatever happened before (an aborted block still arrives), so no
    // block waits on another forever. After the first, every block's
    // partial tile is in its shared memory; block r then sums lane chunks
    // r, r + cs, ... of the tile over the cs blocks in split order and
    // applies the epilogue. The second keeps every block's shared memory
    // alive until the others have read it.
    cluster_sync();
    if (warp < 4) {
      int bad = 0;
      for (int r = 0; r < cs; ++r) bad |= ld_dsmem_s32(dsmem_addr(smem_u32(&s_abort), r));
      if (!bad) {
        const int row_local = warp * 32 + lane;
        const uint32_t mine = smem_u32(smem) + (uint32_t)(row_local * (n_tot + 4)) * 4u;
        for (int c0 = cs_rank * 16; c0 < n_tot; c0 += cs * 16) {
          float v[16];
          for (int r = 0; r < cs; ++r) {
            const uint32_t src = dsmem_addr(mine + (uint32_t)c0 * 4u, r);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float4 q = ld_dsmem4(src + 16u * j);
              if (r == 0) {
                v[4 * j] = q.x;
                v[4 * j + 1] = q.y;
                v[4 * j + 2] = q.z;
                v[4 * j + 3] = q.w;
              } else {
                v[4 * j] += q.x;
                v[4 * j + 1] += q.y;
                v[4 * j + 2] += q.z;
                v[4 * j + 3] += q.w;
              }
            }
          }
          emit_chunk<kSplit>(p, t_first, row_local, lane0, lanes, c0, v, xbuf, nullptr);
        }
      }
    }
    cluster_sync();
  }
  if (warp == 5) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(ncols)
                 : "memory");
  }
  TraceSmem::end(s_tr, TR_GEMM + p.epi);
}

// The kernels: the plain one takes the map of the panel only, the split one
// that of its remainder too (Q8_0 kernels get the panel map in place of the
// unused weight map).
template <bool kQ8, int kMode>
__global__ void __launch_bounds__(kThreads, 2)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
              const TcParams p) {
  gemm_tc_body<kQ8, false, kMode>(tmW, tmX, tmX, p);
}
template <bool kQ8, int kMode>
__global__ void __launch_bounds__(kThreads, 2)
    k_gemm_tc_split(const __grid_constant__ CUtensorMap tmW,
                    const __grid_constant__ CUtensorMap tmX,
                    const __grid_constant__ CUtensorMap tmXlo, const TcParams p) {
  gemm_tc_body<kQ8, true, kMode>(tmW, tmX, tmXlo, p);
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

}  // namespace

bool tc_cluster_reduce() {
  static const bool v = [] {
    const char* e = getenv("FS_TC_CLUSTER");
    return !(e && e[0] == '0');
  }();
  return v;
}

bool tc_available() {
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                       cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

// bf16 map over [rows][Kp] (row stride Kp elements) seen as 3-D (64
// elements, rows, Kp / 64 k-blocks), box (64, box_rows, kq): one copy
// brings kq consecutive k-blocks of box_rows rows, each a [box_rows][64]
// tile in the 128-byte-swizzled K-major layout. Reads beyond the rows or the
// k-blocks return zeros. Encoded maps are kept (keyed by all arguments), so
// a launch finds its maps without encoding them again.
int tc_make_map(const void* base, int64_t rows, int Kp, int box_rows, int kq, CUtensorMap* out) {
  if (!tc_available()) return -1;
  if (box_rows < 1 || box_rows > 256 || kq < 1 || kq > 256 || Kp % kBK) return -2;
  struct Key {
    const void* base;
    int64_t rows;
    int Kp, box_rows, kq;
    bool operator<(const Key& o) const {
      return std::tie(base, rows, Kp, box_rows, kq) <
             std::tie(o.base, o.rows, o.Kp, o.box_rows, o.kq);
    }
  };
  static std::mutex mu;
  static std::map<Key, CUtensorMap> cache;
  const Key key{base, rows, Kp, box_rows, kq};
  std::lock_guard<std::mutex> lock(mu);
  const auto it = cache.find(key);
  if (it != cache.end()) {
    *out = it->second;
    return 0;
  }
  cuuint64_t dims[3] = {(cuuint64_t)kBK, (cuuint64_t)rows, (cuuint64_t)(Kp / kBK)};
  cuuint64_t strides[2] = {(cuuint64_t)Kp * 2, (cuuint64_t)kBK * 2};
  cuuint32_t box[3] = {(cuuint32_t)kBK, (cuuint32_t)box_rows, (cuuint32_t)kq};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
                        dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return -2;
  if (cache.size() >= 4096) cache.clear();  // stale entries of freed buffers
  cache.emplace(key, *out);
  return 0;
}

namespace {

// Dynamic shared memory: 1 KB alignment slack, the stages, the SwiGLU
// exchange buffer, the barriers. The budget lets two blocks share an SM
// (and leaves room for the next kernel's blocks to start under
// programmatic dependent launch); beyond 3-4 stages a block's stream is
// limited by its SM's outstanding-load capacity rather than by the ring.
// the largest dynamic allocation: 227 KB less room for the kernel's static
// shared memory (about 1.6 KB)
constexpr int kSmemAttr = 227 * 1024 - 4096;
constexpr int kMaxStages = 12;
// FS_TC_MAX_STAGES (2..12) lowers the stage cap, a tuning knob read once.
int max_stages() {
  static const int v = [] {
    const char* e = getenv("FS_TC_MAX_STAGES");
    const int x = e ? atoi(e) : kMaxStages;
    return std::max(2, std::min(kMaxStages, x));
  }();
  return v;
}
// Per-block shared memory budget of the ring. A launch whose blocks fit on
// the SMs one each takes most of an SM (FS_TC_SMEM_ALONE_KB, default 208
// KB): more k-blocks per copy and more of the range in flight. A larger
// launch keeps two blocks per SM (FS_TC_SMEM_KB, default 112 KB). Tuning
// knobs (64..208), read once.
int smem_budget(bool alone) {
  static const int shared = [] {
    const char* e = getenv("FS_TC_SMEM_KB");
    const int x = e ? atoi(e) : 112;
    return std::max(64, std::min(208, x)) * 1024;
  }();
  static const int single = [] {
    const char* e = getenv("FS_TC_SMEM_ALONE_KB");
    const int x = e ? atoi(e) : 208;
    return std::max(64, std::min(208, x)) * 1024;
  }();
  return alone ? single : shared;
}
// k-blocks per stage (FS_TC_KQ=1..8 caps it, a tuning knob read once).
int kq_max() {
  static const int v = [] {
    const char* e = getenv("FS_TC_KQ");
    const int x = e ? atoi(e) : 8;
    return std::max(1, std::min(8, x));
  }();
  return v;
}
// Stage layout for panel boxes of xh rows and kq k-blocks per stage: the
// stage size, the stage count within the budget (at least 2) and the
// dynamic shared memory of a block.
int tc_stages_for(int xh, int kq, bool q8, int split, int budget_bytes, int* stage_bytes,
                  int* smem_bytes) {
  const int sb = (q8 ? kQ8XOff : kq * kWTileBytes) + kq * xh * 128 * (split ? 2 : 1);
  const int fixed = 1024 + kXbufBytes + 8 * (3 * kMaxStages + 3);
  const int budget = budget_bytes - fixed;
  const int st = std::max(2, std::min(max_stages(), budget / sb));
  *stage_bytes = sb;
  *smem_bytes = 1024 + st * sb + kXbufBytes + 8 * (3 * st + 3);
  return st;
}
// k-blocks per stage. A small matrix (under 32 MB of weight tiles) is
// covered by one or two stages per block, where the number of copies sets
// the time: as many k-blocks per stage as keep two stages within the budget
// (at most kq_max()). A larger one streams from DRAM through several
// refills of the ring, where the depth of the ring sets the time: at least
// four stages, as few k-blocks per stage as that takes. Then the count is
// evened out over the longest piece of a range so that its stages carry
// equal counts (9 k-blocks: 5 + 4, not 8 + 1).
int tc_choose_kq(const TcParams& p, int xh, bool q8, int split, int budget_bytes) {
  if (q8) return 1;  // Q8_0 stages are dequantised one tile at a time
  const int64_t T = (int64_t)p.m_tiles * p.kb_total;
  const int longest = (int)std::min<int64_t>(p.kb_total, (T + p.P - 1) / p.P);
  const int per_kb = kWTileBytes + xh * 128 * (split ? 2 : 1);
  const int fixed = 1024 + kXbufBytes + 8 * (3 * kMaxStages + 3);
  const int min_stages = T * kWTileBytes >= ((int64_t)32 << 20) ? 4 : 2;
  int kq = std::min(kq_max(), std::min(longest, (budget_bytes - fixed) / (min_stages * per_kb)));
  kq = std::max(1, kq);
  const int chunks = (longest + kq - 1) / kq;
  return (longest + chunks - 1) / chunks;
}

template <bool kQ8, bool kSplit, int kMode>
cudaError_t launch_mode(const CUtensorMap& tmW, const CUtensorMap& tmX, const CUtensorMap& tmXlo,
                        const TcParams& p, int grid, int smem, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e =
        kSplit ? cudaFuncSetAttribute(k_gemm_tc_split<kQ8, kMode>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAttr)
               : cudaFuncSetAttribute(k_gemm_tc<kQ8, kMode>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAttr);
    if (e != cudaSuccess) return e;  // the caller's error check reports it
    attr_set = true;
  }
  if (kSplit) {
    if (kMode == GM_CLUSTER)
      return launch_k_cluster(k_gemm_tc_split<kQ8, kMode>, grid, kThreads, smem, s, p.cs, tmW,
                              tmX, tmXlo, p);
    return launch_k(k_gemm_tc_split<kQ8, kMode>, grid, kThreads, smem, s, tmW, tmX, tmXlo, p);
  }
  if (kMode == GM_CLUSTER)
    return launch_k_cluster(k_gemm_tc<kQ8, kMode>, grid, kThreads, smem, s, p.cs, tmW, tmX, p);
  return launch_k(k_gemm_tc<kQ8, kMode>, grid, kThreads, smem, s, tmW, tmX, p);
}

template <bool kQ8, bool kSplit>
int launch_impl(const TcOperands& o, const TcParams& p0, cudaStream_t s) {
  TcParams p = p0;
  int smem = 0;
  const int grid = p.P * p.groups;
  p.xh = (p.lg + 15) & ~15;
  const int budget = smem_budget(grid <= p.sms);
  p.kq = tc_choose_kq(p, p.xh, kQ8, kSplit, budget);
  p.stages = tc_stages_for(p.xh, p.kq, kQ8, kSplit, budget, &p.stage_bytes, &smem);
  // producer warps of single-piece blocks: up to 4, dividing the stage count
  p.prod_warps = 1;
  if (!kQ8) {
    p.prod_warps = p.stages >= 4 ? 4 : p.stages;
    if (p.stages % p.prod_warps) {
      p.stages -= p.stages % p.prod_warps;
      smem = 1024 + p.stages * p.stage_bytes + kXbufBytes + 8 * (3 * p.stages + 3);
    }
  }
  CUtensorMap tw, tx, txlo;
  if (tc_make_map(o.x, o.x_rows, o.Kp, p.xh, p.kq, &tx) ||
      (kSplit && tc_make_map(static_cast<const __nv_bfloat16*>(o.x) + o.x_lo, o.x_rows, o.Kp,
                             p.xh, p.kq, &txlo)) ||
      (!kQ8 && tc_make_map(o.w, o.w_rows, o.Kp, kBM, p.kq, &tw)))
    return -1;
  if (!kSplit) txlo = tx;
  if (kQ8) tw = tx;  // unused
  // cluster reduction when every stream-K range is one of cs <= 8 equal K
  // splits of a row tile and the partial tile (128 rows x (lanes + 4) f32)
  // fits in the ring; the argmax epilogue needs whole tiles anyway
  p.cs = 0;
  {
    const int n_tot = (p.lg + 15) & ~15;
    const int cs = p.P / p.m_tiles;
    if (tc_cluster_reduce() && !p.cs_off && p.epi != EPI_ARGMAX && p.P % p.m_tiles == 0 &&
        cs >= 2 && cs <= 8 && (size_t)kBM * (n_tot + 4) * 4 <= (size_t)p.stages * p.stage_bytes)
      p.cs = cs;
  }
  if (p.cs)
    launch_mode<kQ8, kSplit, GM_CLUSTER>(tw, tx, txlo, p, grid, smem, s);
  else
    launch_mode<kQ8, kSplit, GM_PLAIN>(tw, tx, txlo, p, grid, smem, s);
  return 1;
}

__global__ void k_tile_q8(const int8_t* __restrict__ codes, const __half* __restrict__ scales,
                          int N, int Kp, int8_t* __restrict__ tiles) {
  const int kb_total = Kp / kBK;
  const int64_t tile = blockIdx.x;  // (m_tile, kb)
  const int m_tile = (int)(tile / kb_total), kb = (int)(tile % kb_total);
  const int r = threadIdx.x;        // row in the tile (128 threads)
  const int row = m_tile * kBM + r;
  int8_t* dst = tiles + tile * kQ8Tile + r * kBK;
  __half* sdst = reinterpret_cast<__half*>(tiles + tile * kQ8Tile + kQ8Codes) + r * 2;
  if (row < N) {
    const int8_t* src = codes + (int64_t)row * Kp + kb * kBK;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      reinterpret_cast<uint4*>(dst)[c] = reinterpret_cast<const uint4*>(src)[c];
    sdst[0] = scales[(int64_t)row * (Kp / 32) + kb * 2];
    sdst[1] = scales[(int64_t)row * (Kp / 32) + kb * 2 + 1];
  } else {
#pragma unroll
    for (int c = 0; c < 4; ++c) reinterpret_cast<uint4*>(dst)[c] = make_uint4(0, 0, 0, 0);
    sdst[0] = __float2half_rn(0.0f);
    sdst[1] = __float2half_rn(0.0f);
  }
}

// bf16 copy of a Q8_0 matrix: out[row][k] = bf16(q * d), the value and the
// rounding dequant_q8_tile gives the same weight inside the GEMM, so either
// operand source feeds the MMAs the same bits. One thread per 8 inputs.
__global__ void k_dequant_q8_bf16(const int8_t* __restrict__ codes,
                                  const __half* __restrict__ scales, int64_t n8, int Kp,
                                  __nv_bfloat16* __restrict__ out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const int64_t e = i * 8;  // first of the thread's 8 inputs (row-major [N][Kp])
  const int64_t row = e / Kp;
  const int k = (int)(e % Kp);
  const float d = __half2float(scales[row * (Kp / 32) + k / 32]);
  const uint2 u = *reinterpret_cast<const uint2*>(codes + e);
  const int8_t* q = reinterpret_cast<const int8_t*>(&u);
  uint4 o;
  uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __nv_bfloat162 v = __floats2bfloat162_rn((float)q[2 * j] * d, (float)q[2 * j + 1] * d);
    ow[j] = *reinterpret_cast<const uint32_t*>(&v);
  }
  *reinterpret_cast<uint4*>(out + e) = o;
}

}  // namespace

int launch_dequant_q8_bf16(const int8_t* codes, const __half* scales, int N, int Kp,
                           __nv_bfloat16* out, cudaStream_t s) {
  const int64_t n8 = (int64_t)N * Kp / 8;
  if (n8 == 0) return 0;
  k_dequant_q8_bf16<<<(unsigned)((n8 + 255) / 256), 256, 0, s>>>(codes, scales, n8, Kp, out);
  return 1;
}

int launch_gemm_tc(const TcOperands& o, const TcParams& p, cudaStream_t s) {
  return p.split ? launch_impl<false, true>(o, p, s) : launch_impl<false, false>(o, p, s);
}

int launch_gemm_tc_q8(const TcOperands& o, const TcParams& p, cudaStream_t s) {
  return p.split ? launch_impl<true, true>(o, p, s) : launch_impl<true, false>(o, p, s);
}

namespace {
// One warp per lane: the argmax over the lane's tile maxima, lowest index on
// ties (each lane of the warp scans tiles t = lane, lane + 32, ... upward).
__global__ void k_argmax_tiles(const float* __restrict__ am_val, const int* __restrict__ am_idx,
                               int B, int m_tiles, int32_t* __restrict__ tokens_out) {
  TraceMark tr;
  tr.begin(g_trace);
  pdl_wait();
  tr.ready();
  pdl_trigger();
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int ln = threadIdx.x & 31;
  if (b >= B) return;  // never thread 0: the grid has ceil(B / warps) blocks
  float bv = -CUDART_INF_F;
  int bi = INT_MAX;
  for (int t = ln; t < m_tiles; t += 32) {
    const float v = am_val[(int64_t)b * m_tiles + t];
    const int i = am_idx[(int64_t)b * m_tiles + t];
    if (v > bv || (v == bv && i < bi)) {
      bv = v;
      bi = i;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > bv || (ov == bv && oi < bi)) {
      bv = ov;
      bi = oi;
    }
  }
  if (ln == 0) tokens_out[b] = bi;
  tr.end(TR_ARGMAX);
}
}  // namespace

int launch_argmax_tiles(const float* am_val, const int* am_idx, int B, int m_tiles,
                        int32_t* tokens_out, cudaStream_t s) {
  if (B <= 0) return 0;
  launch_k(k_argmax_tiles, (B + 3) / 4, 128, 0, s, am_val, am_idx, B, m_tiles, tokens_out);
  return 1;
}

int launch_tile_q8(const int8_t* codes, const __half* scales, int N, int Kp, int8_t* tiles,
                   cudaStream_t s) {
  const int m_tiles = (N + kBM - 1) / kBM;
  k_tile_q8<<<m_tiles * (Kp / kBK), kBM, 0, s>>>(codes, scales, N, Kp, tiles);
  return 1;
}

}  // namespace fsk
