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
      for (int i = 0; i < 32; ++i) {
        const uint32_t c = (u[i >> 2] >> (8 * (i & 3))) & 0xFFu;
        if (c == 0x01u) word |= 1u << i;
        else if (c != 0xFFu) bad = true;
      }
    }
    out[t] = word;
  }
  if (bad) set_status(BONSAI_ERR_BAD_CODE);
}

// One thread per output byte.
__global__ void pack_ternary_kernel(const int8_t* __restrict__ codes, long long rows, int k,
                                    uint8_t* __restrict__ out, int row_bytes) {
  const long long total = rows * (long long)row_bytes;
  bool bad = false;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const long long r = t / row_bytes;
    const int b = (int)(t - r * row_bytes);
    int value = 0;
#pragma unroll
    for (int i = 4; i >= 0; --i) {
      const int kk = 5 * b + i;
      int c = 0;
      if (kk < k) {
        c = codes[r * k + kk];
        if (c < -1 || c > 1) { bad = true; c = 0; }
      }
      value = 3 * value + (c + 1);
    }
    out[t] = (uint8_t)value;
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
  const long long items = rows * (long long)row_bytes;
  if (items == 0) return BONSAI_OK;
  pack_ternary_kernel<<<grid_for(items, 256), 256, 0, stream>>>(
      codes, rows, (int)k, static_cast<uint8_t*>(out), (int)row_bytes);
  return cuda_status(cudaGetLastError());
}

}  // namespace bonsai
