/*
 * bonsai_synth.h -- device twin of the seeded synthetic-input generator
 * (sub_bit_weight_binary_b300/synth.py). Input generation only: it holds
 * none of the products' arithmetic and is not part of libbonsai.
 *
 * Element i of tensor `tid` under `seed`:
 *   key = splitmix64(seed XOR (tid << 40)),  r(i) = splitmix64(key + i)
 * (splitmix64 as published by S. Vigna). All outputs are device buffers owned
 * by the caller; each call launches one kernel on `stream` and returns
 * 0 on success, 1 on bad arguments, 5 on a CUDA error.
 */
#ifndef BONSAI_SYNTH_H
#define BONSAI_SYNTH_H
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif
typedef struct CUstream_st* bonsai_synth_stream;

/* out[j] = high 32 bits of r(start + j), j < count. */
int bonsai_synth_bits32(uint64_t seed, uint64_t tid, int64_t start, int64_t count,
                        uint32_t* out, bonsai_synth_stream stream);
/* out[j] = -1 / 0 / +1 with P = 0.3 / 0.4 / 0.3 from the top 24 bits of r. */
int bonsai_synth_ternary_codes(uint64_t seed, uint64_t tid, int64_t start, int64_t count,
                               int8_t* out, bonsai_synth_stream stream);
/* out[j] = +1 if the top bit of r is 1, else -1. */
int bonsai_synth_binary_codes(uint64_t seed, uint64_t tid, int64_t start, int64_t count,
                              int8_t* out, bonsai_synth_stream stream);
/* out[j] = FP16 bits of lo + u*(hi-lo), u = (r >> 11) * 2^-53, two float64
 * roundings (multiply, add), then round-to-nearest-even to FP16. */
int bonsai_synth_uniform_f16(uint64_t seed, uint64_t tid, int64_t start, int64_t count,
                             double lo, double hi, uint16_t* out, bonsai_synth_stream stream);
#ifdef __cplusplus
}
#endif
#endif
