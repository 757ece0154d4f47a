// xnor.cu -- XNOR-popcount product of +-1 activations and +-1 weights.
//
// "1-bit 嘅數學" (1-bit diffusion page): a binary GEMM can be done with
// XOR + popcount. With bit 1 = +1 and bit 0 = -1, the product of two codes is
// +1 when the bits agree, so over a 128-code group
//     d_g = sum a*w = 128 - 2 * popc(a XOR w)      (4 words)
//     D   = sum_g d_g = K - 2 * popc(a XOR w)       (exact int32)
//     Y   = a_s[m] * sum_g s[n][g] * d_g            (FP32, FP16 out)
// The kernel is bound by the popcount pipe: one XOR and one POPC per 32
// codes of each (m, n) pair; everything else is amortised over a 64x64 tile.
// A carry-save step lets 3 popcounts cover the 4 words of a group.
#include "common.cuh"

namespace bonsai {
BONSAI_DEFINE_STATUS(g_status_xnor)

unsigned int read_clear_status_xnor() {
  unsigned int v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_status_xnor, sizeof(v));
  cudaMemcpyToSymbol(g_status_xnor, &z, sizeof(z));
  return v;
}

namespace xnor {

constexpr int kBM = 64, kBN = 64;      // output tile
constexpr int kThreads = 256;          // 16 x 16 threads, 4 x 4 outputs each
constexpr int kCW = 32;                // words of K per smem chunk (8 groups)
constexpr int kPitch = kCW + 4;        // padded row pitch (words)
constexpr int kSPitch = kCW / 4 + 1;   // group scales per W row, padded: 16 rows -> 16 banks

// popc(a XOR w) over one 128-code group (4 words) with 3 popcounts: a full
// adder over words 0..2 and a half adder with word 3 give per-bit
// sum s (weight 1) and carries c1, c2 (weight 2):
//   popc = popc(s) + 2 * (popc(c1) + popc(c2)).
__device__ __forceinline__ int group_popc(uint4 a, uint4 w) {
  const uint32_t x0 = a.x ^ w.x, x1 = a.y ^ w.y, x2 = a.z ^ w.z, x3 = a.w ^ w.w;
  const uint32_t s1 = x0 ^ x1 ^ x2;
  const uint32_t c1 = (x0 & x1) | (x2 & (x0 ^ x1));
  const uint32_t s = s1 ^ x3;
  const uint32_t c2 = s1 & x3;
  return __popc(s) + 2 * (__popc(c1) + __popc(c2));
}

__global__ void __launch_bounds__(kThreads) xnor_kernel(
    const uint32_t* __restrict__ a_bits, const __half* __restrict__ a_scale,
    const uint32_t* __restrict__ w_bits, long long w_row_words, const __half* __restrict__ scales,
    int m, int n, int k, int32_t* __restrict__ d_out, __half* __restrict__ y_out) {
  __shared__ __align__(16) uint32_t As[kBM * kPitch];
  __shared__ __align__(16) uint32_t Ws[kBN * kPitch];
  __shared__ float Ss[kBN * kSPitch];

  pdl_wait();
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;
  const int kw = k / 32, G = k / 128;

  int dacc[4][4];
  float yacc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) { dacc[i][j] = 0; yacc[i][j] = 0.f; }

  for (int c0 = 0; c0 < kw; c0 += kCW) {
    const int cw = min(kCW, kw - c0);  // multiple of 4
    __syncthreads();
    // stage A and W chunks (rows past m / n are clamped; never stored)
    for (int t = threadIdx.x; t < kBM * (kCW / 4); t += kThreads) {
      const int r = t / (kCW / 4), v = t - r * (kCW / 4);
      if (4 * v < cw) {
        const int ra = min(m0 + r, m - 1), rw = min(n0 + r, n - 1);
        *reinterpret_cast<uint4*>(&As[r * kPitch + 4 * v]) =
            *reinterpret_cast<const uint4*>(a_bits + (long long)ra * kw + c0 + 4 * v);
        *reinterpret_cast<uint4*>(&Ws[r * kPitch + 4 * v]) =
            *reinterpret_cast<const uint4*>(w_bits + (long long)rw * w_row_words + c0 + 4 * v);
      }
    }
    for (int t = threadIdx.x; t < kBN * (kCW / 4); t += kThreads) {
      const int r = t / (kCW / 4), gg = t - r * (kCW / 4);
      const int rw = min(n0 + r, n - 1);
      const int gi = min(c0 / 4 + gg, G - 1);
      Ss[r * kSPitch + gg] = __half2float(scales[(long long)rw * G + gi]);
    }
    __syncthreads();
    for (int gg = 0; gg < cw / 4; ++gg) {
      uint4 av[4], wv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        av[i] = *reinterpret_cast<const uint4*>(&As[(ty + 16 * i) * kPitch + 4 * gg]);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        wv[j] = *reinterpret_cast<const uint4*>(&Ws[(tx + 16 * j) * kPitch + 4 * gg]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float sg = Ss[(tx + 16 * j) * kSPitch + gg];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int pc = group_popc(av[i], wv[j]);
          const int dg = 128 - 2 * pc;
          dacc[i][j] += dg;
          // exact int -> float for |dg| <= 128 without the conversion pipe
          const float fd = __int_as_float(0x4B400000 + dg) - 12582912.0f;
          yacc[i][j] = fmaf(sg, fd, yacc[i][j]);
        }
      }
    }
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = m0 + ty + 16 * i;
    if (row >= m) continue;
    const float as = __half2float(a_scale[row]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = n0 + tx + 16 * j;
      if (col >= n) continue;
      if (d_out) d_out[(long long)row * n + col] = dacc[i][j];
      if (y_out) y_out[(long long)row * n + col] = __float2half_rn(as * yacc[i][j]);
    }
  }
}

// ---- activation binarisation (the A operand from FP16 rows) ----
// The pages give XOR + popcount for +-1 operands but no rule for turning an
// FP16 activation row into one. This library's reading: code +1 where
// x >= 0 (both zeros included; a NaN compares false and gives -1), and the
// row scale a_s = mean |x|, the least-squares scale for those codes
// (d/dalpha sum (x - alpha*a)^2 = 0 gives alpha = sum |x| / K).
// One pass over x: each thread reads 8 halves (16 B), forms one byte of the
// code row, and 4 neighbouring lanes make one LE word; |x| is summed in FP32.
// Few rows: a CTA owns a row and reduces over its 8 warps. Many rows (at
// least 16 per SM): a warp owns a row, keeps 8 loads per lane in flight and
// needs no CTA barrier (measured about 1.8x faster at 4096 x 4096, slower at
// 512 rows where it leaves SMs idle).
constexpr int kBinThreads = 256;
constexpr int kBinUnroll = 4;
constexpr int kBinWarpUnroll = 8;

// bit = (x >= 0) on the FP16 pattern h: +0..+inf are 0x0000..0x7C00, -0 is
// 0x8000; positive NaNs (0x7C01..0x7FFF) and every negative fall outside.
__device__ __forceinline__ uint32_t nonneg2(uint32_t w) {
  const uint32_t le = __vcmpleu2(w, 0x7C007C00u);  // 0xFFFF per half where h <= 0x7C00
  const uint32_t z = __vcmpeq2(w, 0x80008000u);    // 0xFFFF per half where h == -0
  const uint32_t m = le | z;
  return (m & 1u) | ((m >> 15) & 2u);
}

__device__ __forceinline__ float abs_sum2(uint32_t w) {
  const uint32_t a = w & 0x7FFF7FFFu;  // clear both sign bits
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&a));
  return f.x + f.y;
}

__device__ __forceinline__ uint32_t code_byte(const uint4& v) {
  return nonneg2(v.x) | (nonneg2(v.y) << 2) | (nonneg2(v.z) << 4) | (nonneg2(v.w) << 6);
}
__device__ __forceinline__ float abs_sum8(const uint4& v) {
  return (abs_sum2(v.x) + abs_sum2(v.y)) + (abs_sum2(v.z) + abs_sum2(v.w));
}

__global__ void __launch_bounds__(kBinThreads) binarize_rows_warp(
    const uint4* __restrict__ x, long long m, int k, uint32_t* __restrict__ a_bits,
    __half* __restrict__ a_scale) {
  pdl_wait();  // x may be written by earlier work on the stream
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (kBinThreads / 32);
  const int chunks = k / 8;  // a multiple of 16: 4-lane word groups are all in or all out
  for (long long row = (long long)blockIdx.x * (kBinThreads / 32) + (threadIdx.x >> 5); row < m;
       row += warps) {
    const uint4* xr = x + row * chunks;
    uint32_t* br = a_bits + row * (k / 32);
    float sum = 0.f;
    for (int base = 0; base < chunks; base += 32 * kBinWarpUnroll) {
      uint4 v[kBinWarpUnroll];
#pragma unroll
      for (int u = 0; u < kBinWarpUnroll; ++u) {
        const int c = base + 32 * u + lane;
        v[u] = c < chunks ? __ldcs(xr + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kBinWarpUnroll; ++u) {
        const int c = base + 32 * u + lane;
        uint32_t byte = code_byte(v[u]);
        sum += abs_sum8(v[u]);
        byte |= __shfl_down_sync(0xFFFFFFFFu, byte, 1) << 8;
        byte |= __shfl_down_sync(0xFFFFFFFFu, byte, 2) << 16;
        if ((lane & 3) == 0 && c < chunks) br[c >> 2] = byte;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    if (lane == 0) a_scale[row] = __float2half_rn(sum / float(k));
  }
}

__global__ void __launch_bounds__(kBinThreads) binarize_kernel(
    const uint4* __restrict__ x, long long m, int k, uint32_t* __restrict__ a_bits,
    __half* __restrict__ a_scale) {
  __shared__ float red[kBinThreads / 32];
  pdl_wait();  // x may be written by earlier work on the stream
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int chunks = k / 8;  // 16-byte chunks per row; a multiple of 16
  for (long long row = blockIdx.x; row < m; row += gridDim.x) {
    const uint4* xr = x + row * chunks;
    uint32_t* br = a_bits + row * (k / 32);
    float sum = 0.f;
    for (int base = warp * 32; base < chunks; base += kBinThreads * kBinUnroll) {
      uint4 v[kBinUnroll];
#pragma unroll
      for (int u = 0; u < kBinUnroll; ++u) {
        const int c = base + u * kBinThreads + lane;
        v[u] = c < chunks ? __ldcs(xr + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kBinUnroll; ++u) {
        const int c = base + u * kBinThreads + lane;
        uint32_t byte = code_byte(v[u]);
        sum += abs_sum8(v[u]);
        // lanes 4j..4j+3 hold consecutive chunks (bytes) of one word
        byte |= __shfl_down_sync(0xFFFFFFFFu, byte, 1) << 8;
        byte |= __shfl_down_sync(0xFFFFFFFFu, byte, 2) << 16;
        if ((lane & 3) == 0 && c < chunks) br[c >> 2] = byte;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    if (lane == 0) red[warp] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.f;
#pragma unroll
      for (int i = 0; i < kBinThreads / 32; ++i) t += red[i];
      a_scale[row] = __float2half_rn(t / float(k));
    }
    __syncthreads();
  }
}

}  // namespace xnor

bonsai_status xnor_launch(const uint32_t* a_bits, const uint16_t* a_scale, int64_t m,
                          const bonsai_weights* w, int32_t* d_out, uint16_t* y_out,
                          cudaStream_t stream) {
  using namespace xnor;
  dim3 grid((unsigned)((w->n + kBN - 1) / kBN), (unsigned)((m + kBM - 1) / kBM));
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(
      &cfg, xnor_kernel, a_bits, reinterpret_cast<const __half*>(a_scale),
      static_cast<const uint32_t*>(w->packed), (long long)(w->row_bytes / 4),
      reinterpret_cast<const __half*>(w->scales), (int)m, (int)w->n, (int)w->k, d_out,
      reinterpret_cast<__half*>(y_out));
  return cuda_status(e);
}

bonsai_status binarize_launch(const uint16_t* x, int64_t m, int64_t k, uint32_t* a_bits,
                              uint16_t* a_scale, cudaStream_t stream) {
  using namespace xnor;
  const long long cap = 8LL * device_sm_count();  // 8 CTAs of 256 threads fill an SM
  const long long rows_per_cta = kBinThreads / 32;
  const bool per_warp = m >= 2 * cap;  // 16 rows per SM
  const long long want = per_warp ? (m + rows_per_cta - 1) / rows_per_cta : m;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(want < cap ? want : cap));
  cfg.blockDim = dim3(kBinThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, per_warp ? binarize_rows_warp : binarize_kernel,
                                     reinterpret_cast<const uint4*>(x), (long long)m, (int)k,
                                     a_bits, reinterpret_cast<__half*>(a_scale));
  return cuda_status(e);
}

}  // namespace bonsai
