// gemv.cu -- streaming decode product y = x . (s (.) W)^T for binary and
// ternary weights and up to 8 token columns (batch-1 decode, speculative
// verification). Memory-bandwidth bound ("第一の壁": every weight is
// re-streamed per token): each packed byte is read from HBM once.
//
// Shared structure (sm_103a):
//  * A persistent grid, one CTA per SM. A producer warp streams tiles of
//    16 rows of packed weights into a 3-stage shared-memory ring with 1-D
//    bulk copies (TMA engine), one copy per row and chunk of <= 1024 bytes,
//    completion counted on an mbarrier. With BONSAI_WEIGHTS_PREFETCH the
//    producer starts before the previous kernel on the stream has finished
//    (programmatic dependent launch), so consecutive products keep HBM busy.
//  * Eight consumer warps split each chunk along K, expand codes to MMA
//    operands in registers and accumulate on the tensor core with warp-level
//    mma.sync; the FP16 group scale (one per 128 codes, OpenBonsai page,
//    "工作原理") multiplies each group's FP32 partial. A shared-memory
//    reduction across the warps finishes each tile.
//
// Binary (gemv_binary_kernel): operands are exact e4m3 +1/-1, four codes per
// LOP3 (the sign bit of each byte is the code bit). x is split per token and
// 128-group into four e5m2 pieces after a power-of-two scale,
//   x * 2^e = p0 + p1 + p2 + p3  (exact for every x within 2^20 of the group
//   maximum), and the pieces ride in the MMA's N columns, so one
//   m16n8k32 e4m3 x e5m2 instruction applies 16 rows x 32 codes to all four
//   pieces: y_g = s_g * 2^-e * sum over pieces.
//
// Ternary (gemv_ternary_kernel): a 256-entry table (byte -> five 2-bit
// digits, one copy per lane) decodes the base-3 bytes. Each digit c in
// {0,1,2} is placed into mantissa bits j..j+1 of an FP16 whose exponent is
// 15-j, giving 2^-j + c*2^-10 with one LOP3 per two codes ("multiplication
// degenerates to addition and sign flip", 三值权重 page). The constant part
// is removed exactly by the tile's 16th row, which holds the all-zero code
// byte 121: its MMA sum is the correction, computed by the same instruction
// as every real row, so an all-zero group contributes exactly 0:
//   sum_k (c_k - 1) x_k = 2^10 * (acc_row - acc_neutral).
#include "common.cuh"

namespace bonsai {
BONSAI_DEFINE_STATUS(g_status_gemv)

unsigned int read_clear_status_gemv() {
  unsigned int v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_status_gemv, sizeof(v));
  cudaMemcpyToSymbol(g_status_gemv, &z, sizeof(z));
  return v;
}

namespace gemv {

constexpr int kWarps = 8;                  // consumer warps
constexpr int kThreads = (kWarps + 1) * 32;
constexpr int kMaxStages = 8;
constexpr int kStageBudget = 96 * 1024;   // bytes in flight per CTA (HBM read saturates near this)
constexpr int kChunk = 1024;               // packed bytes per row per stage
constexpr int kLutBytes = 256 * 256;       // ternary: 256 entries x (32 lanes x 4 B + pad)
constexpr int kTerEntry = 48;              // ternary x-table bytes per (variant, lane)
constexpr int kTerVariants = 12;           // (round, group) pairs per 640-code super-group
constexpr uint32_t kZeroTrits = 121;       // byte of five zero codes

struct Params {
  const uint8_t* w;
  const __half* scales;
  const __half* x;
  __half* y;
  long long row_bytes;
  int n, k, m, G;
  int rows;        // real rows per tile: 16 binary, 15 ternary (row 15 = neutral)
  int data_bytes;  // packed bytes per row that are streamed
  int chunks;      // stages per tile
  int pitch;       // smem row pitch, bytes (pitch/4 = 4 mod 32: conflict-free words)
  int tiles;
  int n_sg;        // ternary: super-groups per row
  int ncolp;       // binary: B columns per pass (4 for one token, 8 for two)
  int xt_stride;   // ternary: bytes per token column of the x table
  int prefetch;    // may read weights before the previous grid completes
  int sc_tma;      // group scales travel with the weights (k % 1024 == 0)
  int sc_chunk;    // groups per chunk (64 binary, 40 ternary)
  int sc_pitch;    // smem bytes per row of staged scales
  int stage_bytes; // weights (16 rows x pitch) + scales (16 rows x sc_pitch)
  int stages;      // ring depth
  int off_bar, off_red, off_p2e, off_lut, off_xt, off_stage;
};

// ---------------------------------------------------------------------------
// producer warp: tiles of `rows` rows x chunks of <= kChunk bytes into the
// ring with 16-byte asynchronous copies from all 32 lanes (weights, then the
// chunk's group scales); each lane's completion is one arrival on the
// stage's full barrier (count 32).
__device__ __forceinline__ void produce(const Params& p, uint32_t sbase, uint32_t bar_full,
                                        uint32_t bar_empty, int lane) {
  if (!p.prefetch) pdl_wait();
  const uint64_t pol = policy_evict_first();
  int s = 0;
  uint32_t ph = 0;
  for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x) {
    const int row0 = tile * p.rows;
    const int rows = min(p.rows, p.n - row0);
    for (int c = 0; c < p.chunks; ++c) {
      const int off = c * kChunk;
      const int len = min(kChunk, p.data_bytes - off);
      const int g0 = c * p.sc_chunk;
      const int scb = p.sc_tma ? 2 * (min(g0 + p.sc_chunk, p.G) - g0) : 0;
      int ok = 1;
      if (lane == 0) {
        ok = mbar_wait(bar_empty + 8 * s, ph ^ 1);
        if (!ok) set_status(BONSAI_ERR_TIMEOUT);
      }
      if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) return;
      const uint32_t dst = sbase + p.off_stage + s * p.stage_bytes;
      const uint8_t* src = p.w + (long long)row0 * p.row_bytes + off;
      for (int r = 0; r < rows; ++r)
        for (int b = lane * 16; b < len; b += 32 * 16)
          cp_async16(dst + r * p.pitch + b, src + (long long)r * p.row_bytes + b, pol);
      if (scb) {
        const uint8_t* ssrc = reinterpret_cast<const uint8_t*>(p.scales + (size_t)row0 * p.G + g0);
        const int pieces = scb / 16;
        for (int i = lane; i < rows * pieces; i += 32) {
          const int r = i / pieces, b = (i - r * pieces) * 16;
          cp_async16(dst + 16 * p.pitch + r * p.sc_pitch + b, ssrc + (size_t)r * p.G * 2 + b, pol);
        }
      }
      cp_async_arrive(bar_full + 8 * s);
      if (++s == p.stages) { s = 0; ph ^= 1; }
    }
  }
}

__device__ __forceinline__ void init_barriers(uint32_t bar_full, uint32_t bar_empty, int stages) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(bar_full + 8 * s, 32);  // one arrival per producer lane
      mbar_init(bar_empty + 8 * s, kWarps);
    }
    fence_barrier_init();
  }
}

// ===========================================================================
// binary: e4m3 x e5m2 MMA
// ===========================================================================

// Codes c, c+8, c+16, c+24 of a word as e4m3 +1 (0x38) / -1 (0xB8): the
// code bit is moved to the byte's sign bit.
template <int C>
__device__ __forceinline__ uint32_t bin_cls(uint32_t w) {
  const uint32_t s = C == 7 ? w : (w << (7 - C));
  return (s & 0x80808080u) ^ 0xB8B8B8B8u;
}

__device__ __forceinline__ void mma_e4m3_e5m2(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e5m2.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// FP32 -> e5m2 (round to nearest even, low byte) and back.
__device__ __forceinline__ uint32_t f32_to_e5m2(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(v));
  return r & 0xFFu;
}
__device__ __forceinline__ float e5m2_to_f32(uint32_t b) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"(uint16_t(b)));
  return __half2float(__ushort_as_half(uint16_t(h2 & 0xFFFFu)));
}

// x table: for pass P, group gi, half h (MMAs 2h, 2h+1), column col and
// lane-quad index q, 16 bytes = 4 B-registers {b0,b1 of MMA 2h; b0,b1 of
// MMA 2h+1}. Byte j of the register of class c holds the piece of code
// k = 32q + c + 8j of the group. p2e[token][gi] = 2^-e.
__device__ void build_binary_tables(const Params& p, uint8_t* smem, int npass) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* xt = smem + p.off_xt;
  float* p2e = reinterpret_cast<float*>(smem + p.off_p2e);
  const int xt_bytes = npass * p.G * 2 * p.ncolp * 64;
  for (int i = tid; i < xt_bytes / 16; i += kWarps * 32)
    reinterpret_cast<uint4*>(xt)[i] = make_uint4(0, 0, 0, 0);
  named_bar_sync(1, kWarps * 32);
  // one warp per (token, group); lane l holds codes 4l..4l+3 of the group.
  // The x loads of up to 8 items are issued together, then processed.
  const int items = p.m * p.G;
  for (int base = warp; base < items; base += 8 * kWarps) {
    uint2 raw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int item = base + i * kWarps;
      raw[i] = make_uint2(0, 0);
      if (item < items) {
        const int tok = item / p.G, gi = item - tok * p.G;
        raw[i] = *reinterpret_cast<const uint2*>(p.x + (size_t)tok * p.k + 128 * gi + 4 * lane);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int item = base + i * kWarps;
      if (item >= items) break;
      const int tok = item / p.G, gi = item - tok * p.G;
      const __half2 h01 = *reinterpret_cast<const __half2*>(&raw[i].x);
      const __half2 h23 = *reinterpret_cast<const __half2*>(&raw[i].y);
      const float v[4] = {__low2float(h01), __high2float(h01), __low2float(h23),
                          __high2float(h23)};
      const float am = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
      const unsigned amax = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(am));
      // power-of-two scale putting the group maximum in [2^14, 2^15) (e5m2 max 57344)
      const int E = amax ? int((amax >> 23) & 0xFF) - 127 : 0;
      const int e = 14 - E;
      const float up = __uint_as_float(uint32_t(127 + e) << 23);
      if (lane == 0) p2e[tok * p.G + gi] = __uint_as_float(uint32_t(127 - e) << 23);
      const int pass = tok >> 1, colbase = 4 * (tok & 1);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int kg = 4 * lane + t;  // code within the group
        const int q = kg >> 5, c = kg & 7, j = (kg >> 3) & 3;
        float r = v[t] * up;          // exact: a power-of-two scale
        uint8_t* dst = xt + (((size_t)pass * p.G + gi) * 2 + (c >> 2)) * (p.ncolp * 64) +
                       q * 16 + (c & 3) * 4 + j;
#pragma unroll
        for (int pc = 0; pc < 4; ++pc) {  // four e5m2 pieces
          const uint32_t b = f32_to_e5m2(r);
          r -= e5m2_to_f32(b);            // exact residual
          dst[(colbase + pc) * 64] = uint8_t(b);
        }
      }
    }
  }
}

template <int NPASS>
__global__ void __launch_bounds__(kThreads, 1) gemv_binary_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + p.off_bar, bar_empty = bar_full + 8 * kMaxStages;
  init_barriers(bar_full, bar_empty, p.stages);
  __syncthreads();
  pdl_launch_dependents();
  if (warp == kWarps) {
    produce(p, sbase, bar_full, bar_empty, lane);
    return;
  }
  pdl_wait();  // x is written by earlier work on the stream; y may be read by it
  build_binary_tables(p, smem, NPASS);
  named_bar_sync(1, kWarps * 32);

  const int g = lane >> 2, q = lane & 3;
  const bool bcol = g < p.ncolp;
  const int pw = p.pitch >> 2;
  const uint8_t* xt = smem + p.off_xt + (bcol ? g : 0) * 64 + q * 16;
  const float* p2e = reinterpret_cast<const float*>(smem + p.off_p2e);
  const int pass_stride = p.G * 2 * p.ncolp * 64;
  int s = 0;
  uint32_t ph = 0;
  bool alive = true;
  int tcount = 0;
  for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x, ++tcount) {
    const int row0 = tile * 16;
    const int rg = min(row0 + g, p.n - 1), rg8 = min(row0 + g + 8, p.n - 1);
    const __half* sc0p = p.scales + (size_t)rg * p.G;
    const __half* sc1p = p.scales + (size_t)rg8 * p.G;
    float yacc[NPASS][2];
#pragma unroll
    for (int ps = 0; ps < NPASS; ++ps) yacc[ps][0] = yacc[ps][1] = 0.f;
    for (int c = 0; c < p.chunks; ++c) {
      const int len = min(kChunk, p.data_bytes - c * kChunk);
      const int cg = len >> 4;  // 128-code groups in this chunk
      const int gb = (warp * cg) >> 3, ge = ((warp + 1) * cg) >> 3;
      const int gbase = c * (kChunk / 16);
      float s0[8], s1[8];
      if (!p.sc_tma) {  // scales not staged: global loads issued before the wait
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int gi = min(gbase + gb + j, p.G - 1);
          s0[j] = __half2float(sc0p[gi]);
          s1[j] = __half2float(sc1p[gi]);
        }
      }
      const uint8_t* stage = smem + p.off_stage + s * p.stage_bytes;
      const uint32_t* stg = reinterpret_cast<const uint32_t*>(stage);
      const __half* scs = reinterpret_cast<const __half*>(stage + 16 * p.pitch);
      const int scp = p.sc_pitch >> 1;
      if (alive && !mbar_wait(bar_full + 8 * s, ph)) { set_status(BONSAI_ERR_TIMEOUT); alive = false; }
      if (alive) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (gb + j < ge) {
            const int gl = gb + j, gi = gbase + gl;
            if (p.sc_tma) {
              s0[j] = __half2float(scs[g * scp + gl]);
              s1[j] = __half2float(scs[(g + 8) * scp + gl]);
            }
            const uint32_t w0 = stg[g * pw + gl * 4 + q];
            const uint32_t w1 = stg[(g + 8) * pw + gl * 4 + q];
            const uint32_t a00 = bin_cls<0>(w0), a01 = bin_cls<1>(w0), a02 = bin_cls<2>(w0),
                           a03 = bin_cls<3>(w0), a04 = bin_cls<4>(w0), a05 = bin_cls<5>(w0),
                           a06 = bin_cls<6>(w0), a07 = bin_cls<7>(w0);
            const uint32_t a10 = bin_cls<0>(w1), a11 = bin_cls<1>(w1), a12 = bin_cls<2>(w1),
                           a13 = bin_cls<3>(w1), a14 = bin_cls<4>(w1), a15 = bin_cls<5>(w1),
                           a16 = bin_cls<6>(w1), a17 = bin_cls<7>(w1);
#pragma unroll
            for (int ps = 0; ps < NPASS; ++ps) {
              const uint8_t* xg = xt + ps * pass_stride + gi * 2 * (p.ncolp * 64);
              const uint4 b0 = bcol ? *reinterpret_cast<const uint4*>(xg) : make_uint4(0, 0, 0, 0);
              const uint4 b1 = bcol ? *reinterpret_cast<const uint4*>(xg + p.ncolp * 64)
                                    : make_uint4(0, 0, 0, 0);
              float acc[4] = {0.f, 0.f, 0.f, 0.f};
              mma_e4m3_e5m2(acc, a00, a10, a01, a11, b0.x, b0.y);
              mma_e4m3_e5m2(acc, a02, a12, a03, a13, b0.z, b0.w);
              mma_e4m3_e5m2(acc, a04, a14, a05, a15, b1.x, b1.y);
              mma_e4m3_e5m2(acc, a06, a16, a07, a17, b1.z, b1.w);
              // columns 2q, 2q+1 are two pieces of token 2*ps + q/2
              const int tok = min(2 * ps + (q >> 1), p.m - 1);
              const float f = p2e[tok * p.G + gi];
              yacc[ps][0] = fmaf(s0[j] * f, acc[0] + acc[1], yacc[ps][0]);
              yacc[ps][1] = fmaf(s1[j] * f, acc[2] + acc[3], yacc[ps][1]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
      if (++s == p.stages) { s = 0; ph ^= 1; }
    }
    // reduction over warps and over the two lanes holding a token's pieces
    float* red = reinterpret_cast<float*>(smem + p.off_red) + (tcount & 1) * (kWarps * 16 * 16);
#pragma unroll
    for (int ps = 0; ps < NPASS; ++ps) {
      red[(warp * 16 + g) * 16 + ps * 4 + q] = yacc[ps][0];
      red[(warp * 16 + g + 8) * 16 + ps * 4 + q] = yacc[ps][1];
    }
    named_bar_sync(1, kWarps * 32);
    if (threadIdx.x < 16 * p.m) {
      const int row = threadIdx.x & 15, tok = threadIdx.x >> 4;
      if (row0 + row < p.n) {
        const int slot = (tok >> 1) * 4 + (tok & 1) * 2;
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
          sum += red[(w * 16 + row) * 16 + slot] + red[(w * 16 + row) * 16 + slot + 1];
        p.y[(size_t)tok * p.n + row0 + row] = __float2half_rn(sum);
      }
    }
  }
}

// ===========================================================================
// ternary: FP16 MMA with the neutral 16th row
// ===========================================================================
__host__ __device__ constexpr uint32_t mant_mask2(int j) { return (3u << j) | (3u << (j + 16)); }
__host__ __device__ constexpr uint32_t exp_base(int j) {
  return (uint32_t(15 - j) << 10) | (uint32_t(15 - j) << 26);
}
// The table gives digit i at bits 2i..2i+1; digits 0,1 are used from F<<4
// (mantissa bits j = 4, 6), digits 2,3,4 in place (j = 4, 6, 8): j >= 4
// keeps the constant 2^-j within 2^6 of the step 2^-10.
__host__ __device__ constexpr int ter_j(int md) { return md <= 1 ? 2 * md + 4 : 2 * md; }

template <int MD>
__device__ __forceinline__ uint32_t ter_operand(uint32_t f, uint32_t fl) {
  constexpr int j = ter_j(MD);
  return ((MD <= 1 ? fl : f) & mant_mask2(j)) | exp_base(j);
}

// variant v of a super-group: round (4 words = 80 codes) and the group
// (0..4) whose codes it keeps
__constant__ int c_var_round[kTerVariants] = {0, 1, 1, 2, 3, 3, 4, 4, 5, 6, 6, 7};
__constant__ int c_var_group[kTerVariants] = {0, 0, 1, 1, 1, 2, 2, 3, 3, 3, 4, 4};

__device__ void build_ternary_tables(const Params& p, uint8_t* smem) {
  const int tid = threadIdx.x, nthr = kWarps * 32;
  // 1. x -> shared memory (the byte table's region, free until step 3)
  __half* xs_all = reinterpret_cast<__half*>(smem + p.off_lut);
  {
    const int n16 = p.m * p.k / 8;  // 16-byte pieces
    const uint4* src = reinterpret_cast<const uint4*>(p.x);
    uint4* dst = reinterpret_cast<uint4*>(xs_all);
    for (int base = tid; base < n16; base += 8 * nthr) {
      uint4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (base + i * nthr < n16) v[i] = src[base + i * nthr];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (base + i * nthr < n16) dst[base + i * nthr] = v[i];
    }
  }
  named_bar_sync(1, nthr);
  // 2. x table: (token, super-group, variant, lane q) -> 10 words (b0,b1 per digit)
  const int items = p.m * p.n_sg * kTerVariants * 4;
  for (int t = tid; t < items; t += nthr) {
    int r = t;
    const int q = r & 3;
    r >>= 2;
    const int v = r % kTerVariants;
    r /= kTerVariants;
    const int sg = r % p.n_sg;
    const int col = r / p.n_sg;
    const int rnd = c_var_round[v], grp = c_var_group[v];
    const __half* xs = xs_all + (size_t)col * p.k;
    uint32_t e[12];
#pragma unroll
    for (int md = 0; md < 5; ++md) {
      __half h[4];
#pragma unroll
      for (int bj = 0; bj < 4; ++bj) {
        const int kr = 5 * (4 * (4 * rnd + q) + bj) + md;  // code index in the super-group
        const int kg = 640 * sg + kr;
        h[bj] = (kg < p.k && (kr >> 7) == grp) ? xs[kg] : __ushort_as_half(0);
      }
      e[2 * md] = pack_half2(h[0], h[1]);
      e[2 * md + 1] = pack_half2(h[2], h[3]);
    }
    e[10] = e[11] = 0;
    uint4* dst = reinterpret_cast<uint4*>(smem + p.off_xt + col * p.xt_stride +
                                          ((sg * kTerVariants + v) * 4 + q) * kTerEntry);
    dst[0] = make_uint4(e[0], e[1], e[2], e[3]);
    dst[1] = make_uint4(e[4], e[5], e[6], e[7]);
    dst[2] = make_uint4(e[8], e[9], e[10], e[11]);
  }
  named_bar_sync(1, nthr);
  {  // 3. byte -> digits, one copy per lane (entry e at e*256 + lane*4)
    const int e = tid;  // 256 consumer threads, one entry each
    uint32_t v = 0;
    if (e < 243) {
      int r = e;
#pragma unroll
      for (int i = 0; i < 5; ++i) { v |= uint32_t(r % 3) << (2 * i); r /= 3; }
    }
    uint4* dst = reinterpret_cast<uint4*>(smem + p.off_lut + e * 256);
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = make_uint4(v, v, v, v);
  }
}

template <int MD>
__device__ __forceinline__ void ter_fill(uint32_t (&A)[5][4], uint32_t fa01, uint32_t fb01,
                                         uint32_t fa23, uint32_t fb23) {
  A[MD][0] = ter_operand<MD>(fa01, fa01 << 4);
  A[MD][1] = ter_operand<MD>(fb01, fb01 << 4);
  A[MD][2] = ter_operand<MD>(fa23, fa23 << 4);
  A[MD][3] = ter_operand<MD>(fb23, fb23 << 4);
}

__global__ void __launch_bounds__(kThreads, 1) gemv_ternary_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + p.off_bar, bar_empty = bar_full + 8 * kMaxStages;
  init_barriers(bar_full, bar_empty, p.stages);
  // row 15 of every stage holds all-zero codes and is never overwritten
  for (int i = threadIdx.x; i < p.stages * (p.pitch / 4); i += kThreads) {
    const int s = i / (p.pitch / 4), wd = i - s * (p.pitch / 4);
    reinterpret_cast<uint32_t*>(smem + p.off_stage + s * p.stage_bytes + 15 * p.pitch)[wd] =
        kZeroTrits * 0x01010101u;
  }
  for (int i = threadIdx.x; i < p.stages * (p.sc_pitch / 4); i += kThreads) {
    const int s = i / (p.sc_pitch / 4), wd = i - s * (p.sc_pitch / 4);
    reinterpret_cast<uint32_t*>(smem + p.off_stage + s * p.stage_bytes + 16 * p.pitch +
                                15 * p.sc_pitch)[wd] = 0u;
  }
  __syncthreads();
  pdl_launch_dependents();
  if (warp == kWarps) {
    produce(p, sbase, bar_full, bar_empty, lane);
    return;
  }
  pdl_wait();
  build_ternary_tables(p, smem);
  named_bar_sync(1, kWarps * 32);

  const int g = lane >> 2, q = lane & 3;
  const bool bcol = g < p.m;
  const uint8_t* xt_col = smem + p.off_xt + (bcol ? g : 0) * p.xt_stride;
  const uint32_t lut_lane = uint32_t(lane * 4);
  const uint8_t* lut = smem + p.off_lut;
  const int pw = p.pitch >> 2;
  int s = 0;
  uint32_t ph = 0;
  bool alive = true;
  int tcount = 0;
  for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x, ++tcount) {
    const int row0 = tile * 15;
    const int rg = min(row0 + g, p.n - 1), rg8 = min(row0 + g + 8, p.n - 1);
    const __half* sc0p = p.scales + (size_t)rg * p.G;
    const __half* sc1p = p.scales + (size_t)rg8 * p.G;
    float yacc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int c = 0; c < p.chunks; ++c) {
      const int len = min(kChunk, p.data_bytes - c * kChunk);
      const int nsg = (len + 127) >> 7;
      const int sg = c * (kChunk / 128) + warp;
      float s0[5], s1[5];
      if (!p.sc_tma) {  // scales not staged: global loads issued before the wait
#pragma unroll
        for (int j = 0; j < 5; ++j) {
          const int gi = min(5 * sg + j, p.G - 1);
          s0[j] = __half2float(sc0p[gi]);
          s1[j] = __half2float(sc1p[gi]);
        }
      }
      const uint8_t* stage = smem + p.off_stage + s * p.stage_bytes;
      const uint32_t* stg = reinterpret_cast<const uint32_t*>(stage);
      if (alive && !mbar_wait(bar_full + 8 * s, ph)) { set_status(BONSAI_ERR_TIMEOUT); alive = false; }
      if (p.sc_tma && alive && warp < nsg) {
        const __half* scs = reinterpret_cast<const __half*>(stage + 16 * p.pitch);
        const int scp = p.sc_pitch >> 1;
#pragma unroll
        for (int j = 0; j < 5; ++j) {
          const int gl = min(5 * warp + j, p.G - 1 - c * p.sc_chunk);  // staged group
          s0[j] = __half2float(scs[g * scp + gl]);
          s1[j] = __half2float(scs[(g + 8) * scp + gl]);
        }
      }
      if (alive && warp < nsg) {
        const uint32_t* r0 = stg + g * pw + warp * 32 + q;
        const uint32_t* r1 = stg + (g + 8) * pw + warp * 32 + q;
        const uint8_t* xt = xt_col + (sg * kTerVariants * 4 + q) * kTerEntry;
        float accA[4] = {0.f, 0.f, 0.f, 0.f}, accB[4] = {0.f, 0.f, 0.f, 0.f};
        // finished group: subtract the neutral row's sum (lanes 28..31 hold row 15)
        auto epi = [&](int grp, const float (&acc)[4]) {
          const float t0 = __shfl_sync(0xFFFFFFFFu, acc[2], 28 + q);
          const float t1 = __shfl_sync(0xFFFFFFFFu, acc[3], 28 + q);
          yacc[0] = fmaf(s0[grp], (acc[0] - t0) * 1024.f, yacc[0]);
          yacc[1] = fmaf(s0[grp], (acc[1] - t1) * 1024.f, yacc[1]);
          yacc[2] = fmaf(s1[grp], (acc[2] - t0) * 1024.f, yacc[2]);
          yacc[3] = fmaf(s1[grp], (acc[3] - t1) * 1024.f, yacc[3]);
        };
#pragma unroll
        for (int rnd = 0; rnd < 8; ++rnd) {
          uint32_t A[5][4];
          {
            const uint32_t wa = r0[4 * rnd], wb = r1[4 * rnd];
            auto lookup = [&](uint32_t wd, int i) -> uint32_t {
              const uint32_t off = __byte_perm(wd, lut_lane, 0x5504 | (i << 4));
              return *reinterpret_cast<const uint32_t*>(lut + off);
            };
            const uint32_t fa01 = lookup(wa, 0) + (lookup(wa, 1) << 16);
            const uint32_t fa23 = lookup(wa, 2) + (lookup(wa, 3) << 16);
            const uint32_t fb01 = lookup(wb, 0) + (lookup(wb, 1) << 16);
            const uint32_t fb23 = lookup(wb, 2) + (lookup(wb, 3) << 16);
            ter_fill<0>(A, fa01, fb01, fa23, fb23);
            ter_fill<1>(A, fa01, fb01, fa23, fb23);
            ter_fill<2>(A, fa01, fb01, fa23, fb23);
            ter_fill<3>(A, fa01, fb01, fa23, fb23);
            ter_fill<4>(A, fa01, fb01, fa23, fb23);
          }
          // first variant of the round; a second if it straddles a group edge
          const int v0 = (rnd == 0) ? 0 : (rnd == 1) ? 1 : (rnd == 2) ? 3 : (rnd == 3) ? 4
                       : (rnd == 4) ? 6 : (rnd == 5) ? 8 : (rnd == 6) ? 9 : 11;
          const bool split = (rnd == 1 || rnd == 3 || rnd == 4 || rnd == 6);
          const int grp0 = (rnd <= 1) ? 0 : (rnd <= 3) ? 1 : (rnd == 4) ? 2 : (rnd <= 6) ? 3 : 4;
          auto run = [&](float (&acc)[4], int v) {
            const uint4* bp = reinterpret_cast<const uint4*>(xt + v * 4 * kTerEntry);
            const uint4 b0 = bcol ? bp[0] : make_uint4(0, 0, 0, 0);
            const uint4 b1 = bcol ? bp[1] : make_uint4(0, 0, 0, 0);
            const uint4 b2 = bcol ? bp[2] : make_uint4(0, 0, 0, 0);
            mma_16816(acc, A[0][0], A[0][1], A[0][2], A[0][3], b0.x, b0.y);
            mma_16816(acc, A[1][0], A[1][1], A[1][2], A[1][3], b0.z, b0.w);
            mma_16816(acc, A[2][0], A[2][1], A[2][2], A[2][3], b1.x, b1.y);
            mma_16816(acc, A[3][0], A[3][1], A[3][2], A[3][3], b1.z, b1.w);
            mma_16816(acc, A[4][0], A[4][1], A[4][2], A[4][3], b2.x, b2.y);
          };
          // groups 0,2,4 accumulate in accA, groups 1,3 in accB
          if ((grp0 & 1) == 0) run(accA, v0); else run(accB, v0);
          if (split) {
            if ((grp0 & 1) == 0) {
              run(accB, v0 + 1);
              epi(grp0, accA);
              accA[0] = accA[1] = accA[2] = accA[3] = 0.f;
            } else {
              run(accA, v0 + 1);
              epi(grp0, accB);
              accB[0] = accB[1] = accB[2] = accB[3] = 0.f;
            }
          }
        }
        epi(4, accA);  // group 4 ends with round 7
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
      if (++s == p.stages) { s = 0; ph ^= 1; }
    }
    float* red = reinterpret_cast<float*>(smem + p.off_red) + (tcount & 1) * (kWarps * 16 * 8);
    red[(warp * 16 + g) * 8 + 2 * q] = yacc[0];
    red[(warp * 16 + g) * 8 + 2 * q + 1] = yacc[1];
    red[(warp * 16 + g + 8) * 8 + 2 * q] = yacc[2];
    red[(warp * 16 + g + 8) * 8 + 2 * q + 1] = yacc[3];
    named_bar_sync(1, kWarps * 32);
    if (threadIdx.x < 128) {
      const int row = threadIdx.x & 15, col = threadIdx.x >> 4;
      if (row < 15 && col < p.m && row0 + row < p.n) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) sum += red[(w * 16 + row) * 8 + col];
        p.y[(size_t)col * p.n + row0 + row] = __float2half_rn(sum);
      }
    }
  }
}

}  // namespace gemv

// Host launcher. Returns UNSUPPORTED when the per-CTA tables do not fit.
bonsai_status gemv_launch(const bonsai_weights* w, const uint16_t* x, int64_t m,
                          uint16_t* y, cudaStream_t stream) {
  using namespace gemv;
  const bool ter = w->format == BONSAI_FMT_TERNARY;
  const int k = (int)w->k;
  const int n = (int)w->n;
  if (m < 1 || m > 8) return BONSAI_ERR_UNSUPPORTED;
  Params p{};
  p.w = static_cast<const uint8_t*>(w->packed);
  p.scales = reinterpret_cast<const __half*>(w->scales);
  p.x = reinterpret_cast<const __half*>(x);
  p.y = reinterpret_cast<__half*>(y);
  p.row_bytes = w->row_bytes;
  p.n = n;
  p.k = k;
  p.m = (int)m;
  p.G = k / 128;
  p.prefetch = (w->flags & BONSAI_WEIGHTS_PREFETCH) ? 1 : 0;
  const int npass = (p.m + 1) / 2;
  if (!ter) {
    p.rows = 16;
    p.data_bytes = k / 8;
    p.ncolp = p.m == 1 ? 4 : 8;
  } else {
    p.rows = 15;
    p.data_bytes = (int)bonsai_packed_row_bytes(BONSAI_FMT_TERNARY, k);
    p.n_sg = (p.data_bytes + 127) / 128;
    p.xt_stride = p.n_sg * kTerVariants * 4 * kTerEntry + 64;
  }
  if (ter && p.m * k * 2 > kLutBytes) return BONSAI_ERR_UNSUPPORTED;  // x staged in the table region
  p.chunks = (p.data_bytes + kChunk - 1) / kChunk;
  p.sc_chunk = ter ? kChunk * 5 / 128 : kChunk / 16;  // groups per chunk: 40 / 64
  p.sc_tma = (p.G % 8 == 0) ? 1 : 0;
  {
    int scp = (2 * p.sc_chunk + 15) / 16 * 16;
    if ((scp / 4) % 8 == 0) scp += 16;  // words = 4 mod 8: 8 rows hit 8 distinct banks
    p.sc_pitch = scp;
  }
  const int chunk_max = p.data_bytes < kChunk ? p.data_bytes : kChunk;
  const int cw = chunk_max / 4;
  const int pw = ((cw - 4 + 31) / 32) * 32 + 4;
  p.pitch = pw * 4;
  p.tiles = (n + p.rows - 1) / p.rows;
  p.stage_bytes = 16 * p.pitch + 16 * p.sc_pitch;

  auto up = [](int v, int a) { return (v + a - 1) / a * a; };
  int off = 0;
  p.off_bar = off;   off = up(off + 16 * kMaxStages, 128);
  p.off_red = off;   off = up(off + 2 * kWarps * 16 * 16 * 4, 128);
  p.off_p2e = off;   if (!ter) off = up(off + p.m * p.G * 4, 128);
  p.off_lut = off;   if (ter) off = up(off + kLutBytes, 128);
  p.off_xt = off;
  off = ter ? up(off + p.m * p.xt_stride, 1024) : up(off + npass * p.G * 2 * p.ncolp * 64, 1024);
  p.off_stage = off;
  {
    const int room = (device_max_smem_optin() - off) / p.stage_bytes;
    int st = kStageBudget / p.stage_bytes;
    st = st < 3 ? 3 : (st > kMaxStages ? kMaxStages : st);
    p.stages = st < room ? st : room;
  }
  if (p.stages < 2) return BONSAI_ERR_UNSUPPORTED;
  off = up(off + p.stages * p.stage_bytes, 128);
  const int smem = off;

  const void* fn;
  if (ter) fn = (const void*)gemv_ternary_kernel;
  else if (npass == 1) fn = (const void*)gemv_binary_kernel<1>;
  else if (npass == 2) fn = (const void*)gemv_binary_kernel<2>;
  else if (npass == 3) fn = (const void*)gemv_binary_kernel<3>;
  else fn = (const void*)gemv_binary_kernel<4>;
  if (ensure_dynamic_smem(fn, smem) != cudaSuccess) return BONSAI_ERR_CUDA;

  const int sms = device_sm_count();
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p.tiles < sms ? p.tiles : sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&p};
  return cuda_status(cudaLaunchKernelExC(&cfg, fn, args));
}

}  // namespace bonsai
