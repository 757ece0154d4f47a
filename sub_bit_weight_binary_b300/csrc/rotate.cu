// rotate.cu -- block-diagonal signed Hadamard rotation of FP16 activation
// rows, applied online before a product whose weights were rotated offline.
//
// The OpenBonsai page ("工作原理") names a signed Hadamard rotation among its
// compression steps; this library applies it to x along K in power-of-two
// blocks b:
//   out[r][b0 + i] = b^(-1/2) * sum_j H[i][j] * s[b0 + j] * x[r][b0 + j],
//   H[i][j] = (-1)^popcount(i & j)   (Sylvester),  s = +-1 per feature.
// The fast transform needs log2(b) butterfly stages (a, b) -> (a + b, a - b):
// a thread holds 8 consecutive elements (one 16-byte load) and does strides
// 1, 2, 4 in registers; strides 8..128 pair lanes of a warp (shuffles);
// strides 256 and 512 go through shared memory. A CTA of 128 threads covers
// a tile of 1024 elements of one row, which always holds whole blocks. Each
// element is read and written by the same thread, so the rotation may run in
// place. Arithmetic is FP32; the output is rounded once to FP16.
#include <cmath>

#include "common.cuh"

namespace bonsai {
namespace rotate {

constexpr int kThreads = 128;
constexpr int kTile = kThreads * 8;  // elements of a row per CTA pass

__device__ __forceinline__ void unpack8(const uint4& q, float (&v)[8]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <int LOGB>
__global__ void __launch_bounds__(kThreads) hadamard_kernel(
    const uint4* x, uint4* out, const uint32_t* __restrict__ signs, long long m, int k,
    int tiles_per_row, float scale) {
  static_assert(LOGB >= 3 && LOGB <= 10, "blocks of 8 .. 1024 elements");
  constexpr int kLaneStages = (LOGB < 8 ? LOGB : 8) - 3;  // lane strides 8 .. 128
  __shared__ float sm[LOGB > 8 ? kTile : 1];
  pdl_wait();  // x may be written by earlier work on the stream
  pdl_launch_dependents();
  const int t = threadIdx.x, lane = t & 31;
  const long long tiles = m * tiles_per_row;
  for (long long tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const long long row = tile / tiles_per_row;
    const int e0 = (int)(tile - row * tiles_per_row) * kTile + 8 * t;
    // k is a multiple of the block and of 8: a block is all live or all dead
    const bool live = e0 < k;
    float v[8];
    if (live) {
      unpack8(x[(row * k + e0) >> 3], v);
      if (signs) {
        const uint32_t byte = (signs[e0 >> 5] >> (e0 & 31)) & 0xFFu;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (!((byte >> i) & 1u)) v[i] = -v[i];
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
    }
    // strides 1, 2, 4 inside the thread
#pragma unroll
    for (int h = 1; h < 8 && h < (1 << LOGB); h <<= 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (!(i & h)) {
          const float a = v[i], b = v[i | h];
          v[i] = a + b;
          v[i | h] = a - b;
        }
      }
    }
    // strides 8 .. 128: partner lane t ^ mask holds the other element
#pragma unroll
    for (int s = 0; s < kLaneStages; ++s) {
      const int mask = 1 << s;
      const float sgn = (lane & mask) ? -1.f : 1.f;  // upper lane: p - v, lower: v + p
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float p = __shfl_xor_sync(0xFFFFFFFFu, v[i], mask);
        v[i] = fmaf(sgn, v[i], p);  // one rounding, as the plain sum or difference
      }
    }
    if constexpr (LOGB > 8) {
      // strides 256 (and 512): groups of 2^(LOGB-8) elements 256 apart
      constexpr int kPts = 1 << (LOGB - 8);
      constexpr int kGroups = kTile / kPts;
#pragma unroll
      for (int i = 0; i < 8; ++i) sm[8 * t + i] = v[i];
      __syncthreads();
      for (int g = t; g < kGroups; g += kThreads) {
        const int base = (g & 255) + (g >> 8) * (256 * kPts);
        float u[kPts];
#pragma unroll
        for (int j = 0; j < kPts; ++j) u[j] = sm[base + 256 * j];
#pragma unroll
        for (int h = 1; h < kPts; h <<= 1) {
#pragma unroll
          for (int j = 0; j < kPts; ++j) {
            if (!(j & h)) {
              const float a = u[j], b = u[j | h];
              u[j] = a + b;
              u[j | h] = a - b;
            }
          }
        }
#pragma unroll
        for (int j = 0; j < kPts; ++j) sm[base + 256 * j] = u[j];
      }
      __syncthreads();
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = sm[8 * t + i];
      __syncthreads();  // the next tile overwrites sm
    }
    if (live)
      out[(row * k + e0) >> 3] = make_uint4(pack2(v[0] * scale, v[1] * scale),
                                            pack2(v[2] * scale, v[3] * scale),
                                            pack2(v[4] * scale, v[5] * scale),
                                            pack2(v[6] * scale, v[7] * scale));
  }
}

}  // namespace rotate

bonsai_status hadamard_launch(const uint16_t* x, int64_t m, int64_t k, int32_t block,
                              const uint32_t* signs, uint16_t* out, cudaStream_t stream) {
  using namespace rotate;
  int logb = 0;
  while ((1 << logb) < block) ++logb;
  const int tiles_per_row = (int)((k + kTile - 1) / kTile);
  const long long tiles = (long long)m * tiles_per_row;
  const long long cap = 16LL * device_sm_count();  // 16 CTAs of 128 threads fill an SM
  const float scale = (float)(1.0 / std::sqrt((double)block));
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(tiles < cap ? tiles : cap));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const uint4* xi = reinterpret_cast<const uint4*>(x);
  uint4* oi = reinterpret_cast<uint4*>(out);
  cudaError_t e;
  switch (logb) {
    case 3: e = cudaLaunchKernelEx(&cfg, hadamard_kernel<3>, xi, oi, signs, (long long)m, (int)k, tiles_per_row, scale); break;
    case 4: e = cudaLaunchKernelEx(&cfg, hadamard_kernel<4>, xi, oi, signs, (long long)m, (int)k, tiles_per_row, scale); break;
    case 5: e = cudaLaunchKernelEx(&cfg, hadamard_kernel<5>, xi, oi, signs, (long long)m, (int)k, tiles_per_row, scale); break;
    case 6: e = cudaLaunchKernelEx(&cfg, hadamard_kernel<6>, xi, oi, signs, (long long)m, (int)k, tiles_per_row, scale); break;
    case 7: e = cudaLaunchKernelEx(&cfg, hadamard_kernel<7>, xi, oi, signs, (long long)m, (int)k, tiles_per_row, scale); break;
    case 8: e = cudaLaunchKernelEx(&cfg, hadamard_kernel<8>, xi, oi, signs, (long long)m, (int)k, tiles_per_row, scale); break;
    case 9: e = cudaLaunchKernelEx(&cfg, hadamard_kernel<9>, xi, oi, signs, (long long)m, (int)k, tiles_per_row, scale); break;
    case 10: e = cudaLaunchKernelEx(&cfg, hadamard_kernel<10>, xi, oi, signs, (long long)m, (int)k, tiles_per_row, scale); break;
    default: return BONSAI_ERR_UNSUPPORTED;
  }
  return cuda_status(e);
}

}  // namespace bonsai
