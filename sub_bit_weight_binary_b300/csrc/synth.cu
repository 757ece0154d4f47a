// synth.cu -- device twin of synth.py: seeded synthetic inputs generated on
// the GPU (the multi-gigabyte decode-sweep weights). Input generation only.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/bonsai_synth.h"

namespace {

__device__ __forceinline__ uint64_t splitmix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t host_splitmix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t key_of(uint64_t seed, uint64_t tid) { return host_splitmix64(seed ^ (tid << 40)); }

enum Kind { kBits32, kTernary, kBinary, kUniform };

template <int KIND, typename T>
__global__ void synth_kernel(uint64_t key, int64_t start, int64_t count, double lo, double hi,
                             T* out) {
  for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < count;
       j += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t r = splitmix64(key + (uint64_t)(start + j));
    if (KIND == kBits32) {
      out[j] = (T)(uint32_t)(r >> 32);
    } else if (KIND == kTernary) {
      const uint32_t t = (uint32_t)(r >> 40);
      out[j] = (T)(t < 5033165u ? -1 : (t < 11744051u ? 0 : 1));
    } else if (KIND == kBinary) {
      out[j] = (T)((r >> 63) ? 1 : -1);
    } else {
      const double u = (double)(r >> 11) * 0x1.0p-53;
      const double v = __dadd_rn(lo, __dmul_rn(u, __dsub_rn(hi, lo)));
      out[j] = (T)__half_as_ushort(__double2half(v));
    }
  }
}

template <int KIND, typename T>
int launch(uint64_t seed, uint64_t tid, int64_t start, int64_t count, double lo, double hi,
           T* out, cudaStream_t stream) {
  if (!out || start < 0 || count < 0) return 1;
  if (count == 0) return 0;
  int64_t blocks = (count + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  synth_kernel<KIND, T><<<(unsigned)blocks, 256, 0, stream>>>(key_of(seed, tid), start, count,
                                                               lo, hi, out);
  return cudaGetLastError() == cudaSuccess ? 0 : 5;
}

}  // namespace

extern "C" {
int bonsai_synth_bits32(uint64_t seed, uint64_t tid, int64_t start, int64_t count, uint32_t* out,
                        bonsai_synth_stream stream) {
  return launch<kBits32>(seed, tid, start, count, 0.0, 0.0, out, stream);
}
int bonsai_synth_ternary_codes(uint64_t seed, uint64_t tid, int64_t start, int64_t count,
                               int8_t* out, bonsai_synth_stream stream) {
  return launch<kTernary>(seed, tid, start, count, 0.0, 0.0, out, stream);
}
int bonsai_synth_binary_codes(uint64_t seed, uint64_t tid, int64_t start, int64_t count,
                              int8_t* out, bonsai_synth_stream stream) {
  return launch<kBinary>(seed, tid, start, count, 0.0, 0.0, out, stream);
}
int bonsai_synth_uniform_f16(uint64_t seed, uint64_t tid, int64_t start, int64_t count, double lo,
                             double hi, uint16_t* out, bonsai_synth_stream stream) {
  return launch<kUniform>(seed, tid, start, count, lo, hi, out, stream);
}
}
