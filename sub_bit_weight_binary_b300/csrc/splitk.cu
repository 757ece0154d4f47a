// splitk.cu -- decode product y[n] = x . (s (.) W)^T with K split across
// CTAs, for matrices with few rows (where one CTA per 16-row tile leaves most
// SMs idle). Each CTA sums a range of 128-code groups for 16 rows and writes
// FP32 partials; the last CTA of a row tile adds the partials in split order
// (deterministic) and writes FP16 y.
//
// The partials and the per-tile arrival counters live in one file-scope
// device array of fixed size, so this entry point allocates nothing. It is
// meant for callers that cannot allocate at call time: a serving loop that
// must not stall on cudaMalloc/cudaFree (both synchronise the device), or a
// process whose device memory is budgeted up front and handed out by its own
// pool. The price is shared state: two calls that overlap in time (different
// streams, or different host threads on one device) use the same scratch and
// corrupt each other's partials; calls must be ordered (same stream, or
// synchronised between).
#include <mutex>

#include "common.cuh"

namespace bonsai {
namespace splitk {

constexpr int kRowsPerCta = 16;                 // one warp per row
constexpr int kThreads = kRowsPerCta * 32;
constexpr int kMaxRows = 8192;
constexpr int kMaxSplits = 32;
constexpr int kMaxTiles = kMaxRows / kRowsPerCta;
constexpr size_t kPartialBytes = size_t(kMaxSplits) * kMaxRows * sizeof(float);  // 1 MiB
constexpr size_t kScratchBytes = kPartialBytes + kMaxTiles * sizeof(unsigned int);

// [split][row] FP32 partials, then one arrival counter per row tile. The
// counters must be zero when a call starts; the last CTA of a tile resets its
// counter, and the first call on a device clears them all.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

struct Params {
  const uint8_t* packed;
  const __half* scales;
  const __half* x;
  __half* y;
  long long row_bytes;
  int n, k, G, ternary;
  int splits, groups_per_split;
  float* partials;
  unsigned int* counters;
};

// code of weight (row, k): +-1 (binary bit 1 = +1) or -1/0/+1 (base-3 digit
// minus one, least significant digit first)
__device__ __forceinline__ float code_at(const Params& p, const uint8_t* row, int k) {
  if (p.ternary) {
    unsigned int b = row[k / 5];
    const int d = k % 5;
    for (int i = 0; i < d; ++i) b /= 3u;
    return float(int(b % 3u) - 1);
  }
  const uint32_t word = reinterpret_cast<const uint32_t*>(row)[k >> 5];
  return ((word >> (k & 31)) & 1u) ? 1.f : -1.f;
}

__global__ void __launch_bounds__(kThreads) splitk_kernel(const Params p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.y * kRowsPerCta + warp;
  const int split = blockIdx.x;
  const int g0 = split * p.groups_per_split;
  const int g1 = min(p.G, g0 + p.groups_per_split);
  float acc = 0.f;
  if (row < p.n) {
    const uint8_t* wrow = p.packed + (long long)row * p.row_bytes;
    for (int g = g0; g < g1; ++g) {
      float part = 0.f;
      for (int i = lane; i < 128; i += 32) {
        const int k = g * 128 + i;
        part = fmaf(code_at(p, wrow, k), __half2float(p.x[k]), part);
      }
      acc = fmaf(__half2float(p.scales[(size_t)row * p.G + g]), part, acc);
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  if (lane == 0 && row < p.n) p.partials[(size_t)split * p.n + row] = acc;
  __threadfence();
  __syncthreads();
  __shared__ unsigned int last;
  if (threadIdx.x == 0) last = atomicAdd(&p.counters[blockIdx.y], 1u) == unsigned(p.splits - 1);
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (lane == 0 && row < p.n) {
    float sum = 0.f;
    for (int sp = 0; sp < p.splits; ++sp) sum += __ldcg(&p.partials[(size_t)sp * p.n + row]);
    p.y[row] = __float2half_rn(sum);
  }
  if (threadIdx.x == 0) p.counters[blockIdx.y] = 0u;  // zero again for the next call
}

}  // namespace splitk

// Host side. The scratch address is looked up once per device; the first
// call on a device also clears the counters (on the caller's stream, before
// its kernel).
bonsai_status splitk_launch(const bonsai_weights* w, const uint16_t* x, uint16_t* y,
                            cudaStream_t stream) {
  using namespace splitk;
  if (w->n > kMaxRows) return BONSAI_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BONSAI_ERR_CUDA;
  static void* scratch[64] = {};
  static bool cleared[64] = {};
  static std::mutex mu;
  void* base = nullptr;
  bool first = false;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!scratch[dev]) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || !ptr) return BONSAI_ERR_CUDA;
      scratch[dev] = ptr;
    }
    base = scratch[dev];
    first = !cleared[dev];
    cleared[dev] = true;
  }
  unsigned int* counters = reinterpret_cast<unsigned int*>(static_cast<unsigned char*>(base) +
                                                           kPartialBytes);
  if (first &&
      cudaMemsetAsync(counters, 0, kMaxTiles * sizeof(unsigned int), stream) != cudaSuccess) {
    std::lock_guard<std::mutex> lock(mu);
    cleared[dev] = false;  // not cleared after all: the next call tries again
    return BONSAI_ERR_CUDA;
  }

  Params p{};
  p.packed = static_cast<const uint8_t*>(w->packed);
  p.scales = reinterpret_cast<const __half*>(w->scales);
  p.x = reinterpret_cast<const __half*>(x);
  p.y = reinterpret_cast<__half*>(y);
  p.row_bytes = w->row_bytes;
  p.n = (int)w->n;
  p.k = (int)w->k;
  p.G = p.k / 128;
  p.ternary = w->format == BONSAI_FMT_TERNARY ? 1 : 0;
  const int tiles = (p.n + kRowsPerCta - 1) / kRowsPerCta;
  int splits = (2 * device_sm_count() + tiles - 1) / tiles;
  splits = splits < 1 ? 1 : (splits > kMaxSplits ? kMaxSplits : splits);
  if (splits > p.G) splits = p.G;
  p.groups_per_split = (p.G + splits - 1) / splits;
  p.splits = (p.G + p.groups_per_split - 1) / p.groups_per_split;  // no empty split
  p.partials = static_cast<float*>(base);
  p.counters = counters;
  splitk_kernel<<<dim3(p.splits, tiles), kThreads, 0, stream>>>(p);
  return cuda_status(cudaGetLastError());
}

}  // namespace bonsai
