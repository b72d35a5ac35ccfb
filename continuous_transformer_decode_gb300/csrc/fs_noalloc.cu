// fs_gemm_bf16_noalloc: the tcgen05 weight-streaming GEMM without any device
// allocation.
//
// Some callers cannot call cudaMalloc or cudaFree. One example is a process
// whose device memory belongs to another framework's caching allocator, where
// raw allocations would compete with that pool. Another is a latency-critical
// loop, where cudaFree synchronises the whole device and allocation time is
// unbounded. A third is an embedder with a fixed, pre-planned device-memory
// budget. For them, this entry point runs the same GEMM kernel as
// fs_gemm_bf16. The K-split workspace of that kernel (partial tiles, arrival
// counters and the error flag) lives in the file-scope array below instead of
// memory allocated per call. Every GPU that loads this library keeps the array
// until the process exits.
//
// Set-up: every call looks up the array's device address on the current
// device with cudaGetSymbolAddress (the lookup allocates nothing), so no
// address outlives a device reset or a re-created context. The call then synchronises its stream and copies the kernel's
// error flag to the host before it returns.
//
// Sharing: every call on a device uses the same array, which keeps the last
// call's contents. Each call clears the counters and the error flag before
// its launch. Calls that overlap on the GPU (on different streams, or from
// different threads) race on the array and must be serialised by the caller.

#include "../../include/fs.h"
#include "fs_internal.h"

namespace {

constexpr size_t kScratchBytes = (size_t)8 << 20;  // 8 MiB in all
constexpr size_t kCtrBytes = (size_t)64 << 10;     // counters + error flag
constexpr size_t kPartialBytes = kScratchBytes - kCtrBytes;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the scratch array on the current device.
unsigned char* scratch_on_current_device(int* rc) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
    *rc = FS_ERR_CUDA;
    return nullptr;
  }
  *rc = FS_OK;
  return static_cast<unsigned char*>(p);
}

}  // namespace

extern "C" int fs_gemm_bf16_noalloc(const uint16_t* W, int32_t N, int32_t K,
                                    const uint16_t* X, int32_t B, float* Y,
                                    int32_t splits, void* stream) {
  using namespace fsk;
  if (!W || !X || !Y || N < 1 || K < 64 || K % 64 || B < 1 || splits < 1 ||
      splits > K / 64 || splits > 8)
    return FS_ERR_ARG;
  const int64_t m_tiles = (N + 127) / 128;
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FS_ERR_CUDA;
  // stream-K width m_tiles * splits: each block's range is the K split of one
  // tile, so only the first workspace slot of each block is ever written
  const int P = (int)(m_tiles * splits);
  if (!tc_width_ok((int)m_tiles, K / 64, P)) return FS_ERR_ARG;
  int lg = 0, groups = 0;
  tc_lane_groups(B, P, sms, &lg, &groups);
  const size_t ctr_bytes = (size_t)(m_tiles * groups + 1) * sizeof(int);
  const size_t part_bytes =
      splits > 1 ? (size_t)splits * B * m_tiles * 128 * sizeof(float) : 0;
  if (ctr_bytes > kCtrBytes || part_bytes > kPartialBytes) return FS_ERR_SCRATCH;

  int rc = FS_OK;
  unsigned char* base = scratch_on_current_device(&rc);
  if (rc != FS_OK) return rc;
  int* counters = reinterpret_cast<int*>(base);
  int* err = counters + m_tiles * groups;
  float* ws = reinterpret_cast<float*>(base + kCtrBytes);

  cudaStream_t s = (cudaStream_t)stream;
  // what must start at zero: the arrival counters and the error flag
  if (cudaMemsetAsync(counters, 0, ctr_bytes, s) != cudaSuccess) return FS_ERR_CUDA;
  TcParams p{};
  p.m_tiles = (int)m_tiles;
  p.P = P;
  p.kb_total = K / 64;
  p.lanes_total = B;
  p.sms = sms;
  p.lg = lg;
  p.groups = groups;
  p.tmem_cols = tc_tmem_cols(lg);
  p.epi = EPI_STORE;
  p.out_f32 = Y;
  p.ldo = N;
  p.n_out = N;
  p.ws = ws;
  p.counters = counters;
  p.err = err;
  p.cs_off = 1;  // K splits sum through the static workspace
  const TcOperands o{W, N, X, B, K, 0};
  if (launch_gemm_tc(o, p, s) < 0) return FS_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
    return FS_ERR_CUDA;
  int herr = 0;
  if (cudaMemcpy(&herr, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FS_ERR_CUDA;
  return herr ? FS_ERR_DEVICE : FS_OK;
}
