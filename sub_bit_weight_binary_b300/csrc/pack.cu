// pack.cu -- int8 codes -> packed BINARY / TERNARY layouts (offline step).
//
// Binary: bit (k % 32) of word k/32 is 1 for code +1 and 0 for code -1
// ("1-bit 嘅數學": every weight is +1 or -1). Ternary: byte b holds codes
// 5b..5b+4 as the base-3 number sum (code+1)*3^i, least significant digit
// first ("三值权重到底做了什么": values -1, 0, +1); codes past k and the row
// padding are zero codes (byte 121). A code outside the format's set records
// BONSAI_ERR_BAD_CODE in the status word; the output word is then unspecified.
#include "common.cuh"

namespace bonsai {
BONSAI_DEFINE_STATUS(g_status_pack)

unsigned int read_clear_status_pack() {
  unsigned int v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_status_pack, sizeof(v));
  cudaMemcpyToSymbol(g_status_pack, &z, sizeof(z));
  return v;
}

namespace {

// One thread per output word. 32 codes are read as two 16-byte vectors.
__global__ void pack_binary_kernel(const int8_t* __restrict__ codes, long long rows, int k,
                                   uint32_t* __restrict__ out, int words_per_row) {
  const long long total = rows * (long long)words_per_row;
  const int data_words = k / 32;
  bool bad = false;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const long long r = t / words_per_row;
    const int j = (int)(t - r * words_per_row);
    uint32_t word = 0;
    if (j < data_words) {
      const int4* src = reinterpret_cast<const int4*>(codes + r * k + 32LL * j);
      const int4 v0 = src[0], v1 = src[1];
      const uint32_t u[8] = {(uint32_t)v0.x, (uint32_t)v0.y, (uint32_t)v0.z, (uint32_t)v0.w,
                             (uint32_t)v1.x, (uint32_t)v1.y, (uint32_t)v1.z, (uint32_t)v1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        // +1 is 0x01 and -1 is 0xFF: the code bit is the inverted sign bit of
        // each byte; one multiply gathers the four sign bits into bits 28..31
        const uint32_t sgn = ~u[i] & 0x80808080u;
        word |= ((sgn * 0x00204081u) >> 28) << (4 * i);
        const uint32_t expect = ((u[i] >> 7) & 0x01010101u) * 0xFEu + 0x01010101u;
        bad |= u[i] != expect;
      }
    }
    out[t] = word;
  }
  if (bad) set_status(BONSAI_ERR_BAD_CODE);
}

// Digit bytes (code + 1) of four int8 codes, with a carry-free byte add;
// a code outside {-1,0,+1} gives a digit above 2.
__device__ __forceinline__ uint32_t digits4(uint32_t w) {
  return ((w & 0x7F7F7F7Fu) + 0x01010101u) ^ (w & 0x80808080u);
}

// One thread per 16 output bytes (80 codes, five 16-byte loads). Output byte
// b = d0 + 3 d1 + 9 d2 + 27 d3 + 81 d4 of its five digit bytes: a byte
// permute gathers d0..d3 and one 4-way byte dot product weighs them.
__global__ void pack_ternary_kernel(const int8_t* __restrict__ codes, long long rows, int k,
                                    uint8_t* __restrict__ out, int row_bytes) {
  const int chunks = row_bytes / 16;
  const long long total = rows * (long long)chunks;
  bool bad = false;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const long long r = t / chunks;
    const int j = (int)(t - r * chunks);
    const int k0 = 80 * j;
    uint32_t d[21];
    if (k0 + 80 <= k) {
      const int4* src = reinterpret_cast<const int4*>(codes + r * k + k0);
#pragma unroll
      for (int i = 0; i < 5; ++i) {
        const int4 v = src[i];
        d[4 * i] = digits4((uint32_t)v.x);
        d[4 * i + 1] = digits4((uint32_t)v.y);
        d[4 * i + 2] = digits4((uint32_t)v.z);
        d[4 * i + 3] = digits4((uint32_t)v.w);
      }
#pragma unroll
      for (int i = 0; i < 20; ++i)  // a digit byte above 2: bits above 1 set, or both low bits
        bad |= ((d[i] & 0xFCFCFCFCu) | (d[i] & (d[i] >> 1) & 0x01010101u)) != 0u;
    } else {  // row tail and padding: codes past k are zero codes (digit 1)
#pragma unroll
      for (int i = 0; i < 20; ++i) {
        uint32_t v = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kk = k0 + 4 * i + e;
          int c = 0;
          if (kk < k) {
            c = codes[r * k + kk];
            if (c < -1 || c > 1) { bad = true; c = 0; }
          }
          v |= uint32_t(c + 1) << (8 * e);
        }
        d[i] = v;
      }
    }
    d[20] = 0;
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t word = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int b = 4 * q + e;      // output byte within the chunk
        const int p = 5 * b;          // its first digit byte
        const int w0 = p >> 2, o0 = p & 3;
        const uint32_t lo4 = __byte_perm(d[w0], d[w0 + 1],
                                         o0 | ((o0 + 1) << 4) | ((o0 + 2) << 8) | ((o0 + 3) << 12));
        const uint32_t d4 = (d[(p + 4) >> 2] >> (8 * ((p + 4) & 3))) & 0xFFu;
        const uint32_t value = (uint32_t)__dp4a(lo4, 0x1B090301u, 81u * d4);
        word |= (value & 0xFFu) << (8 * e);
      }
      o[q] = word;
    }
    *reinterpret_cast<uint4*>(out + r * row_bytes + 16LL * j) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (bad) set_status(BONSAI_ERR_BAD_CODE);
}

int grid_for(long long items, int threads) {
  long long g = (items + threads - 1) / threads;
  const long long cap = 16LL * device_sm_count();
  if (g > cap) g = cap;
  return g < 1 ? 1 : (int)g;
}

}  // namespace

bonsai_status pack_binary_launch(const int8_t* codes, int64_t rows, int64_t k, void* out,
                                 int64_t row_bytes, cudaStream_t stream) {
  const int wpr = (int)(row_bytes / 4);
  const long long items = rows * (long long)wpr;
  if (items == 0) return BONSAI_OK;
  pack_binary_kernel<<<grid_for(items, 256), 256, 0, stream>>>(
      codes, rows, (int)k, static_cast<uint32_t*>(out), wpr);
  return cuda_status(cudaGetLastError());
}

bonsai_status pack_ternary_launch(const int8_t* codes, int64_t rows, int64_t k, void* out,
                                  int64_t row_bytes, cudaStream_t stream) {
  const long long items = rows * (long long)(row_bytes / 16);
  if (items == 0) return BONSAI_OK;
  pack_ternary_kernel<<<grid_for(items, 256), 256, 0, stream>>>(
      codes, rows, (int)k, static_cast<uint8_t*>(out), (int)row_bytes);
  return cuda_status(cudaGetLastError());
}

}  // namespace bonsai
