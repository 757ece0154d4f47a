// gemm.cu -- multi-token product Y = X . (s (.) W)^T on the 5th-generation
// tensor cores (tcgen05), for prompt processing (pp512) and
// diffusion-transformer image tokens. This case is a dense contraction:
// every dequantised weight tile is reused by 256 (or 512) tokens.
//
// One persistent CTA per SM, 16 warps with fixed roles:
//   warp 0      TMA producer: X tiles [256 tokens x 64 k] FP16, 128-byte
//               swizzle, straight into the MMA's canonical K-major layout
//               (two per stage for 512-token tiles); it also prefetches the
//               packed weight rows of its tiles into L2.
//   warp 1      MMA issuer (one thread): tcgen05.mma kind::f16, M=128
//               features x N=256 tokens x K=16, FP32 accumulators in TMEM.
//   warp 2      TMEM allocator (512 columns: two 256-column accumulators, so
//               the epilogue of tile i overlaps the main loop of tile i+1,
//               or one 512-column accumulator for 512-token tiles).
//   warps 4-7   epilogue: tcgen05.ld -> FP16 (round to nearest even) -> Y.
//   warps 8-15  dequantisers: packed codes -> FP16 s*w written into the
//               swizzled A stage. The value is exact: s*(+-1) only flips the
//               sign bit and s*0 is 0, so FP16 x FP16 products are exact in
//               FP32 and only the FP32 sums round.
// Scales follow the one-FP16-per-128-weights rule of the OpenBonsai page
// ("工作原理"); the weights are +-1 ("1-bit 嘅數學") or -1/0/+1 (ternary).
// Every mbarrier wait is bounded; a wait that runs out records
// BONSAI_ERR_TIMEOUT and the kernel drains and leaves.
#include "tcgen05.cuh"

namespace bonsai {
BONSAI_DEFINE_STATUS(g_status_gemm)

unsigned int read_clear_status_gemm() {
  unsigned int v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_status_gemm, sizeof(v));
  cudaMemcpyToSymbol(g_status_gemm, &z, sizeof(z));
  return v;
}

namespace gemm {

constexpr int BM = 128;                 // features per tile  (MMA M)
constexpr int BN = 256;                 // tokens per MMA     (MMA N)
constexpr int BK = 64;                  // K per stage: one 128-byte swizzle row of FP16
// Three tile shapes. Narrow: 128 features x 256 tokens, two TMEM
// accumulators of 256 columns, so the epilogue of one tile overlaps the main
// loop of the next. Wide (ternary): 128 x 512, one accumulator of 512
// columns; every dequantised weight stage feeds two N=256 MMAs, which halves
// the dequantisation per FLOP (the ternary dequantisers limit). Tall
// (binary): 256 x 256, one accumulator of 512 columns; every activation
// stage feeds two M=128 MMAs, which halves the X traffic per FLOP (binary's
// MMA thread waits on the X ring). Both larger tiles give up the overlapped
// epilogue.
// Separate rings: dequantised weight tiles (A) are produced on chip, X tiles
// (B) arrive by TMA from L2. Narrow ternary dequantisation has the longer
// latency per stage, so it gets the deeper A ring; wide X stages are 64 KB,
// tall A stages 32 KB.
constexpr int NARROW = 0, WIDE = 1, TALL = 2;
template <int FMT, int MODE> struct Cfg {
  static constexpr int TT = MODE == WIDE ? 512 : 256;      // tokens per tile
  static constexpr int FM = MODE == TALL ? 256 : BM;       // features per tile
  static constexpr int HALVES = TT / BN;                   // token halves (N=256 MMAs)
  static constexpr int FHALVES = FM / BM;                  // feature halves (M=128 MMAs)
  static constexpr int NACC = MODE == NARROW ? 2 : 1;      // TMEM accumulators of 256 columns x halves
  static constexpr int A = MODE == WIDE ? 4 : MODE == TALL ? 3 : (FMT == BONSAI_FMT_TERNARY ? 6 : 4);
  static constexpr int B = MODE == WIDE ? 2 : (FMT == BONSAI_FMT_TERNARY ? 3 : 4);
  static constexpr int A_BYTES = FM * BK * 2;              // 16 or 32 KB
  static constexpr int B_BYTES = TT * BK * 2;              // 32 or 64 KB
};
constexpr int A_HALF = BM * BK * 2;     // 16 KB: one M=128 operand tile
constexpr int B_HALF = BN * BK * 2;     // 32 KB: one TMA box of X
constexpr int TMEM_COLS = 512;
constexpr int THREADS = 512;
constexpr int W_TMA = 0, W_MMA = 1, W_TMEM = 2, W_EPI = 4, W_DQ = 8;
constexpr int LUT_BYTES = 256 * 128;    // byte -> five 2-bit digits, one copy per lane
constexpr int BAR_BYTES = 256;

struct Params {
  const uint8_t* w;
  const __half* scales;
  __half* y;
  long long row_bytes;
  int m, n, k, G, nk;
  int tiles, tok_tiles;
  int prefetch;
  int swiglu;    // rows 16t..16t+7 gate, 16t+8..16t+15 up: write silu(g)*u
  int y_stride;  // elements per token row of y: n, or n/2 with swiglu
  // Stream-K (128 x 256 tiles, caller workspace): tiles [0, dp) run whole,
  // one per CTA and wave; the k-steps of tiles [dp, tiles) are cut into
  // sk_ctas equal ranges. sk_ctas = 0: every tile whole.
  int dp, sk_ctas;
  int sk_iters;                // (tiles - dp) * nk; sk_iters * sk_ctas < 2^31
  float* ws;                   // one BM x BN FP32 partial tile per stream-K CTA
  unsigned int* ws_count;      // partials delivered, one counter per stream-K tile
};

// A tile is split over at most kMaxPartners + 1 stream-K ranges.
constexpr int kMaxPartners = 12;

// ---- the work of a CTA -----------------------------------------------------
// Segments: its whole tiles blockIdx.x + i * gridDim.x below dp, then at most
// two stream-K pieces [a, b) of the cut k-steps (b - a <= nk, so a piece
// ends the first tile it starts in, or begins the next). The piece that
// holds k-step 0 of a tile finishes it: it adds the partial tiles of the
// CTAs that hold the rest (their first pieces) and writes Y.
__device__ __forceinline__ int sk_start(const Params& p, int c) {
  return c * p.sk_iters / p.sk_ctas;
}
// SK = false (the larger tiles, never cut): whole tiles only.
template <bool SK>
struct Segs {
  int whole, count;
  int a, b;
  __device__ __forceinline__ explicit Segs(const Params& p) {
    const int c = blockIdx.x, gd = gridDim.x;
    whole = p.dp > c ? (p.dp - c + gd - 1) / gd : 0;
    count = whole;
    a = b = 0;
    if (SK && c < p.sk_ctas) {
      a = sk_start(p, c);
      b = sk_start(p, c + 1);
      if (b > a) count += b > (a / p.nk + 1) * p.nk ? 2 : 1;
    }
  }
  // tile and k-step range [j0, j1) (in the tile's K order) of segment i
  __device__ __forceinline__ void at(const Params& p, int i, int& tile, int& j0, int& j1) const {
    if (!SK || i < whole) {
      tile = blockIdx.x + i * (int)gridDim.x;
      j0 = 0;
      j1 = p.nk;
      return;
    }
    const int t0 = a / p.nk;
    if (i == whole) {
      tile = p.dp + t0;
      j0 = a - t0 * p.nk;
      j1 = b - t0 * p.nk < p.nk ? b - t0 * p.nk : p.nk;
    } else {
      tile = p.dp + t0 + 1;
      j0 = 0;
      j1 = b - (t0 + 1) * p.nk;
    }
  }
};

// Number of CTAs after this one whose first stream-K range lies in `tile`
// (the partners whose partial tiles this CTA's finishing range adds).
__device__ __forceinline__ int sk_partners(const Params& p, int tile) {
  const int t_end = (tile - p.dp + 1) * p.nk;
  int np = 0;
  while ((int)blockIdx.x + 1 + np < p.sk_ctas && sk_start(p, (int)blockIdx.x + 1 + np) < t_end) ++np;
  return np;
}

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* a) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}
// Waits until *c >= target; false if kWaitNs of wall-clock time ran out.
__device__ bool wait_at_least(const unsigned int* c, unsigned int target) {
  if (ld_acquire_u32(c) >= target) return true;
  const uint64_t t0 = global_ns();
  while (ld_acquire_u32(c) < target) {
    __nanosleep(100);
    if (global_ns() - t0 > kWaitNs) return false;
  }
  return true;
}

// Instruction descriptor, kind::f16: D=F32 (bits 4-5 = 1), A=B=F16 (0),
// both K-major, N>>3 at bits 17-22, M>>4 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24);

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// ---- dequantisation of one row x 64 k into the swizzled A stage ------------
// Row r of the stage lives at r*128 bytes; its 16-byte chunk c (codes
// 8c..8c+7) is stored at chunk position c ^ (r & 7).
__device__ __forceinline__ void dq_binary(uint2 wv, uint32_t s2, uint32_t dst_row, int sw) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t x = ~(c < 4 ? wv.x : wv.y) >> (8 * (c & 3));
    uint32_t h[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t t2 = (x >> (2 * i)) & 3u;  // bit0: code k is -1, bit1: code k+1 is -1
      h[i] = ((t2 * 0x40008000u) & 0x80008000u) ^ s2;
    }
    sts128(dst_row + ((c ^ sw) << 4), h[0], h[1], h[2], h[3]);
  }
}

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Ternary digit pairs without a table: a digit c (0..2) placed in mantissa
// bits p, p+1 of a half whose exponent field is 25 - p is the value
// 2^(10-p) + c; minus the same half with c = 1 it is c - 1 in {-1, 0, +1},
// exactly (both operands lie within a factor of two). The product with the
// FP16 scale is then exact as well. Five pair shapes occur: digits (d, d+1)
// of one byte for d = 0..3 (p = 2d low, 2d+2 high, from the byte's digit
// word in both halves) and digit 4 of a byte with digit 0 of the next.
__host__ __device__ constexpr uint32_t ter_exp(int p) { return uint32_t(25 - p) << 10; }
__host__ __device__ constexpr int ter_plo(int d) { return d < 4 ? 2 * d : 8; }
__host__ __device__ constexpr int ter_phi(int d) { return d < 4 ? 2 * d + 2 : 0; }
__host__ __device__ constexpr uint32_t ter_mask(int d) {
  return (3u << ter_plo(d)) | (3u << (ter_phi(d) + 16));
}
__host__ __device__ constexpr uint32_t ter_e(int d) {
  return ter_exp(ter_plo(d)) | (ter_exp(ter_phi(d)) << 16);
}
__host__ __device__ constexpr uint32_t ter_one(int d) {
  return ter_e(d) | (1u << ter_plo(d)) | (1u << (ter_phi(d) + 16));
}

// Exponent fields and c = 1 operands of the five pair shapes, in registers
// (LOP3 takes one immediate; HSUB2 subtracts a register).
struct TerConsts {
  uint32_t e[5], one[5];
  __device__ __forceinline__ TerConsts() {
#pragma unroll
    for (int d = 0; d < 5; ++d) {
      uint32_t a = ter_e(d), b = ter_one(d);
      asm volatile("" : "+r"(a), "+r"(b));  // keep them in registers
      e[d] = a;
      one[d] = b;
    }
  }
};

template <int D>
__device__ __forceinline__ uint32_t ter_pair(uint32_t w, uint32_t s2, const TerConsts& K) {
  uint32_t u;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(u) : "r"(w), "n"(ter_mask(D)), "r"(K.e[D]));
  return hmul2_u32(hsub2_u32(u, K.one[D]), s2);
}

// Ternary k-step kk = 5u + V covers codes 64V..64V+63 of the 64-byte block u
// (320 codes): they start in byte 64V/5 at digit 64V%5, known at compile time.
// The byte table gives a byte's five digits (digit i at bits 2i, 2i+1).
template <int V>
__device__ __forceinline__ void dq_ternary(const uint32_t (&wd)[16], uint32_t s2, uint32_t lut,
                                           const TerConsts& K, uint32_t dst_row, int sw) {
  constexpr int T0 = 64 * V;
  constexpr int B0 = T0 / 5;
  constexpr int B1 = (T0 + 63) / 5;
  uint32_t F[B1 - B0 + 1];
#pragma unroll
  for (int b = B0; b <= B1; ++b) {
    const uint32_t byte = (wd[b >> 2] >> (8 * (b & 3))) & 0xFFu;
    F[b - B0] = lds32(lut + byte * 128u);
  }
  uint32_t pv[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int T = T0 + 2 * j;
    const int b = T / 5 - B0, d = T % 5;
    // the pair's digit word: the byte's digits in both halves, or (d = 4)
    // this byte's digits low and the next byte's high
    const uint32_t w = d < 4 ? __byte_perm(F[b], 0u, 0x1010) : __byte_perm(F[b], F[b + 1], 0x5410);
    switch (d) {
      case 0: pv[j] = ter_pair<0>(w, s2, K); break;
      case 1: pv[j] = ter_pair<1>(w, s2, K); break;
      case 2: pv[j] = ter_pair<2>(w, s2, K); break;
      case 3: pv[j] = ter_pair<3>(w, s2, K); break;
      default: pv[j] = ter_pair<4>(w, s2, K); break;
    }
  }
#pragma unroll
  for (int c = 0; c < 8; ++c)
    sts128(dst_row + ((c ^ sw) << 4), pv[4 * c], pv[4 * c + 1], pv[4 * c + 2], pv[4 * c + 3]);
}

// K order of a tile. All CTAs stream the same activation tiles; in the same
// K order they would all ask L2 for the same X tile at the same moment (the
// MMA thread measured 140-325 cycles per k-step waiting on the X ring). Each
// tile therefore starts at its own block of 5 k-steps and wraps around:
// k = (j + 5 * rot) mod nk, rot = tile mod (number of blocks). Blocks stay
// whole (the ternary dequantisers read 64-byte blocks of 5 k-steps).
__device__ __forceinline__ int k_blocks(const Params& p) { return (p.nk + 4) / 5; }
__device__ __forceinline__ int k_rot(const Params& p, int tile) { return tile % k_blocks(p); }
__device__ __forceinline__ int k_at(const Params& p, int tile, int j) {
  const int k = j + 5 * k_rot(p, tile);
  return k < p.nk ? k : k - p.nk;
}

// Finishing a cut tile. Its range holds k-step 0 and is its CTA's last
// segment, so all the CTA's MMAs have completed, the A and B rings are idle
// and so are the dequantiser warps. Three groups of four warps (the epilogue
// warps, then the two dequantiser groups), each covering the 128
// tensor-memory lanes, share the tile's 16-token steps round robin. The np
// partners' partial tiles come into the rings by bulk copies, a group of
// steps of every partner into one of two 96 KB buffers, so the next group is
// copied while one is added (measured: ~4 us of copies and ~6 us of adds and
// FP16 stores at 512 tokens when the 4 epilogue warps did it alone). The sum
// is this CTA's accumulator, then the partners in CTA order. `issuer` (one
// thread) issues the copies; fin_bar has 12 arrivals per group.
constexpr int kFinishBufSteps = 12;  // 16-token steps of one partner per 96 KB buffer
__device__ void finish_cut_tile(const Params& p, int tile, int np, uint32_t acc, uint32_t ring,
                                uint32_t stg_bar, uint32_t fin_bar, int grp, bool issuer) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;          // tensor-memory lanes 32 quarter ..
  const int row = 32 * quarter + lane;   // feature row of the tile
  const int n0 = (tile / p.tok_tiles) * BM, m0 = (tile % p.tok_tiles) * BN;
  const int steps = (p.m - m0 + 15) / 16 < BN / 16 ? (p.m - m0 + 15) / 16 : BN / 16;
  const uint32_t tl = acc + ((uint32_t)(32 * quarter) << 16);
  constexpr int STEP_BYTES = BM * 16 * 4;  // one partner, one step: 8 KB
  const int gsz = np > 0 ? (kFinishBufSteps / np < steps ? kFinishBufSteps / np : steps) : steps;
  const int groups = (steps + gsz - 1) / gsz;
  auto copy_group = [&](int j) {
    const int s0 = j * gsz, gn = steps - s0 < gsz ? steps - s0 : gsz;
    const uint32_t buf = ring + (j & 1) * kFinishBufSteps * STEP_BYTES, bar = stg_bar + 8 * (j & 1);
    mbar_arrive_expect_tx(bar, (uint32_t)(np * gn * STEP_BYTES));
    for (int q = 0; q < np; ++q)
      for (int st = 0; st < gn; ++st)
        bulk_g2s(buf + (q * gsz + st) * STEP_BYTES,
                 p.ws + (size_t)(blockIdx.x + 1 + q) * (BM * BN) + (size_t)(s0 + st) * (BM * 16),
                 STEP_BYTES, bar, policy_evict_first());
  };
  if (np > 0 && issuer) {
    copy_group(0);
    if (groups > 1) copy_group(1);
  }
  const int feat = n0 + row;
  const bool fok = feat < p.n;
  for (int j = 0; j < groups; ++j) {
    const int s0 = j * gsz, gn = steps - s0 < gsz ? steps - s0 : gsz;
    const uint32_t buf = ring + (j & 1) * kFinishBufSteps * STEP_BYTES;
    if (np > 0 && !mbar_wait(stg_bar + 8 * (j & 1), (j >> 1) & 1)) set_status(BONSAI_ERR_TIMEOUT);
    for (int st = s0 + ((grp - s0 % 3) + 3) % 3; st < s0 + gn; st += 3) {  // steps = grp mod 3
      uint32_t v[16];
      TMEM_LD_16(tl + 16 * st, v);
      tmem_ld_wait();
      for (int q = 0; q < np; ++q) {
        const uint32_t src = buf + (q * gsz + st - s0) * STEP_BYTES + row * 16;
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4) {
          float4 f;
          asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                       : "=f"(f.x), "=f"(f.y), "=f"(f.z), "=f"(f.w)
                       : "r"(src + i4 * BM * 16));
          v[4 * i4] = __float_as_uint(__uint_as_float(v[4 * i4]) + f.x);
          v[4 * i4 + 1] = __float_as_uint(__uint_as_float(v[4 * i4 + 1]) + f.y);
          v[4 * i4 + 2] = __float_as_uint(__uint_as_float(v[4 * i4 + 2]) + f.z);
          v[4 * i4 + 3] = __float_as_uint(__uint_as_float(v[4 * i4 + 3]) + f.w);
        }
      }
      if (p.swiglu) {
        const int hcol = (feat >> 4) * 8 + (feat & 7);
#pragma unroll
        for (int j2 = 0; j2 < 16; ++j2) {
          const float g = __uint_as_float(v[j2]);
          const float u = __shfl_down_sync(0xFFFFFFFFu, g, 8);
          const int tok = m0 + 16 * st + j2;
          if (fok && !(lane & 8) && tok < p.m)
            p.y[(size_t)tok * p.y_stride + hcol] = __float2half_rn(silu(g) * u);
        }
      } else if (fok) {
#pragma unroll
        for (int j2 = 0; j2 < 16; ++j2) {
          const int tok = m0 + 16 * st + j2;
          if (tok < p.m) p.y[(size_t)tok * p.y_stride + feat] = __float2half_rn(__uint_as_float(v[j2]));
        }
      }
    }
    if (np > 0) {  // every warp done with this buffer before its next copy
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(fin_bar);
      if (!mbar_wait(fin_bar, j & 1)) set_status(BONSAI_ERR_TIMEOUT);
      if (issuer && j + 2 < groups) copy_group(j + 2);
    }
  }
}

// Outputs of a whole tile from its TMEM accumulator (column a*256, feature
// half f at +256 f): the 32-token chunks grp, grp + ngrp, ... of the tile,
// read by this warp's lane quarter. On a CTA's last tile the epilogue warps
// (grp 0) share the chunks with the two dequantiser groups, which have no
// k-steps left (a tile's epilogue is otherwise exposed when no next tile
// follows: the larger tiles' one accumulator, or the last wave). acc_empty
// (not 0): arrived on after this warp's last TMEM load. Wide (ternary
// 512-token) tiles do not take the help: with it the kernel rose from 110 to
// 117 registers and the M=4096 product lost 2% (A/B on one GPU), more than
// the M=512 product gained; out of line it cost 28%.
template <int FM, int TT, int FHALVES>
__device__ void store_tile(const Params& p, int tile, uint32_t tmem_base, uint32_t a, int grp,
                           int ngrp, uint32_t acc_empty) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, quarter = warp & 3;
  const int n0 = (tile / p.tok_tiles) * FM, m0 = (tile % p.tok_tiles) * TT;
  // column chunks that hold tokens (the MMAs wrote only the used halves)
  const int chunks = (p.m - m0 + 31) / 32 < TT / 32 ? (p.m - m0 + 31) / 32 : TT / 32;
  const int total = chunks * FHALVES;
  const int last = grp < total ? grp + (total - 1 - grp) / ngrp * ngrp : -1;
#pragma unroll 1
  for (int cf = grp; cf < total; cf += ngrp) {
    const int f = cf / chunks, c = cf - f * chunks;  // feature half, token chunk
    const int feat = n0 + BM * f + 32 * quarter + lane;
    const bool fok = feat < p.n;
    uint32_t v[32];
    TMEM_LD_32(tmem_base + ((uint32_t)(32 * quarter) << 16) + (a + f) * 256 + 32 * c, v);
    tmem_ld_wait();
    if (cf == last && acc_empty) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
    }
    if (p.swiglu) {
      // lanes 0-7 / 16-23 hold gate features, lanes 8-15 / 24-31 the up
      // features of the same outputs (n % 16 == 0, so fok is uniform
      // over each 16-lane block)
      const int hcol = (feat >> 4) * 8 + (feat & 7);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float g = __uint_as_float(v[j]);
        const float u = __shfl_down_sync(0xFFFFFFFFu, g, 8);
        const int tok = m0 + 32 * c + j;
        if (fok && !(lane & 8) && tok < p.m)
          p.y[(size_t)tok * p.y_stride + hcol] = __float2half_rn(silu(g) * u);
      }
    } else if (fok) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int tok = m0 + 32 * c + j;
        if (tok < p.m)
          p.y[(size_t)tok * p.y_stride + feat] = __float2half_rn(__uint_as_float(v[j]));
      }
    }
  }
  if (last < 0 && acc_empty) {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(acc_empty);
  }
}

template <int FMT, int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  using C = Cfg<FMT, MODE>;
  static_assert(MODE != TALL || FMT == BONSAI_FMT_BINARY, "256-feature tiles are for binary");
  constexpr int A_STAGES = C::A, B_STAGES = C::B, B_BYTES = C::B_BYTES, TT = C::TT, FM = C::FM;
  constexpr int A_BYTES = C::A_BYTES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sA = smem_u32(smem);
  const uint32_t sB = sA + A_STAGES * A_BYTES;
  const uint32_t sLut = sB + B_STAGES * B_BYTES;
  const uint32_t sBar = FMT == BONSAI_FMT_TERNARY ? sLut + LUT_BYTES : sLut;
  // full_a[s]: the 4 dequantiser warps of the k-step's parity group;
  // full_b[s][h]: the X copy of half h of stage s (transaction bytes; one
  // half per 256 tokens, so the MMAs of the first half of a 512-token stage
  // start, and its refill begins, without waiting for the second);
  // empty_a / empty_b: the MMAs
  // that read the stage have completed.
  const uint32_t full_a = sBar, empty_a = full_a + 8 * A_STAGES;
  constexpr int NB = B_STAGES * C::HALVES;  // X barriers: one per (stage, half)
  const uint32_t full_b = empty_a + 8 * A_STAGES, empty_b = full_b + 8 * NB;
  const uint32_t acc_full = empty_b + 8 * NB, acc_empty = acc_full + 16;
  const uint32_t drain = acc_empty + 16;
  const uint32_t tmem_slot = drain + 8;
  const uint32_t epi_bar = sBar + 192;  // the epilogue warps' own barrier (stream-K)
  const uint32_t stg_bar = sBar + 200;  // two: partial tiles copied into the idle rings
  const uint32_t fin_bar = sBar + 216;  // the 12 warps that finish a cut tile
  // The epilogue warps arrive here once the CTA's last accumulator is
  // complete; the dequantisers wait on it (once) before they help store it.
  // They must not wait on acc_full themselves: they can finish their k-steps
  // two accumulator phases ahead of the MMAs (short K), and a parity wait
  // cannot tell those phases apart.
  const uint32_t help_bar = sBar + 224;
  static_assert(8 * (2 * A_STAGES + 2 * NB + 5) + 4 <= 192, "barriers overlap epi_bar");

  if ((sA & 1023u) != 0) {  // the swizzle atoms need 1024-byte alignment
    if (threadIdx.x == 0) set_status(BONSAI_ERR_UNSUPPORTED);
    return;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < A_STAGES; ++s) {
      mbar_init(full_a + 8 * s, 4);
      mbar_init(empty_a + 8 * s, 1);
    }
    for (int s = 0; s < NB; ++s) {
      mbar_init(full_b + 8 * s, 1);
      mbar_init(empty_b + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(acc_full + 8 * a, 1);
      mbar_init(acc_empty + 8 * a, 4);
    }
    mbar_init(drain, 1);
    mbar_init(epi_bar, 4);
    mbar_init(stg_bar, 1);
    mbar_init(stg_bar + 8, 1);
    mbar_init(fin_bar, 12);
    mbar_init(help_bar, 4);
    fence_barrier_init();
  }
  if (FMT == BONSAI_FMT_TERNARY && warp >= W_DQ) {
    const int t = threadIdx.x - W_DQ * 32;  // 0..255
    for (int i = t; i < 256 * 32; i += 256) {
      const int e = i >> 5, ln = i & 31;
      uint32_t v = 0;
      if (e < 243) {
        int r = e;
        for (int d = 0; d < 5; ++d) { v |= uint32_t(r % 3) << (2 * d); r /= 3; }
      }
      asm volatile("st.shared.b32 [%0], %1;" ::"r"(sLut + e * 128 + ln * 4), "r"(v) : "memory");
    }
  }
  if (warp == W_TMEM) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  uint32_t tmem_base;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(tmem_base) : "r"(tmem_slot) : "memory");

  if (warp == W_TMA) {
    // ------------------------------ X producer ------------------------------
    if (lane == 0) {
      pdl_wait();
      // The dequantisers read packed weight rows straight from global memory
      // one 64-byte block ahead; with the rows of this tile and of the next
      // one already on their way to L2, those reads do not wait on DRAM. A
      // tile's rows are contiguous (row_bytes apart).
      auto prefetch_tile = [&](int tile) {
        if (tile >= p.tiles) return;
        const int n0 = (tile / p.tok_tiles) * FM;
        const int rows = p.n - n0 < FM ? p.n - n0 : FM;
        prefetch_l2(p.w + (long long)n0 * p.row_bytes, (long long)rows * p.row_bytes);
      };
      const Segs<MODE == NARROW> sg(p);
      int tile = p.tiles, j0 = 0, j1 = 0;
      if (sg.count > 0) {
        sg.at(p, 0, tile, j0, j1);
        prefetch_tile(tile);
      }
      uint32_t g = 0;
      bool ok = true;
      for (int i = 0; i < sg.count && ok; ++i) {
        sg.at(p, i, tile, j0, j1);
        const int m0 = (tile % p.tok_tiles) * TT;
        // token halves of a wide tile that hold tokens (rows past m read as 0)
        const int halves = (p.m - m0 + BN - 1) / BN < C::HALVES ? (p.m - m0 + BN - 1) / BN : C::HALVES;
        if (i + 1 < sg.count) {
          int t2, a2, b2;
          sg.at(p, i + 1, t2, a2, b2);
          if (t2 != tile) prefetch_tile(t2);
        }
        for (int kk = j0; kk < j1; ++kk, ++g) {
          const int s = g % B_STAGES;
          const uint32_t ph = (g / B_STAGES) & 1;
          for (int h = 0; h < C::HALVES && ok; ++h) {
            const uint32_t bf = full_b + 8 * (s * C::HALVES + h);
            if (!mbar_wait(empty_b + 8 * (s * C::HALVES + h), ph ^ 1)) {
              set_status(BONSAI_ERR_TIMEOUT);
              ok = false;
              break;
            }
            if (h < halves) {
              mbar_arrive_expect_tx(bf, (uint32_t)B_HALF);
              tma_load_2d(sB + s * B_BYTES + h * B_HALF, &tmx, k_at(p, tile, kk) * BK,
                          m0 + h * BN, bf);
            } else {
              mbar_arrive(bf);  // a half without tokens: complete its phase, load nothing
            }
          }
          if (!ok) break;
        }
      }
    }
  } else if (warp == W_MMA) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      uint32_t g = 0, it = 0;
      bool ok = true;
      const Segs<MODE == NARROW> sg(p);
      for (int i = 0; i < sg.count && ok; ++i, ++it) {
        int tile, j0, j1;
        sg.at(p, i, tile, j0, j1);
        const uint32_t a = it % C::NACC, use = it / C::NACC;
        if (!mbar_wait(acc_empty + 8 * a, (use & 1) ^ 1)) { set_status(BONSAI_ERR_TIMEOUT); break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + a * 256;
        const int m0 = (tile % p.tok_tiles) * TT;
        const int halves = (p.m - m0 + BN - 1) / BN < C::HALVES ? (p.m - m0 + BN - 1) / BN : C::HALVES;
        for (int kk = j0; kk < j1; ++kk, ++g) {
          const int sa = g % A_STAGES, sb = g % B_STAGES;
          const uint32_t pb = (g / B_STAGES) & 1;
          if (!mbar_wait(full_a + 8 * sa, (g / A_STAGES) & 1)) {
            set_status(BONSAI_ERR_TIMEOUT);
            ok = false;
            break;
          }
          for (int h = 0; h < C::HALVES; ++h) {  // token half h: tokens m0 + 256h ..
            const int ib = sb * C::HALVES + h;
            if (!mbar_wait(full_b + 8 * ib, pb)) {
              set_status(BONSAI_ERR_TIMEOUT);
              ok = false;
              break;
            }
            if (h < halves) {
              tc_fence_after();
              const uint64_t bd = smem_desc_sw128(sB + sb * B_BYTES + h * B_HALF);
#pragma unroll
              for (int f = 0; f < C::FHALVES; ++f) {  // feature half f: rows 128f .. of the stage
                const uint64_t ad = smem_desc_sw128(sA + sa * A_BYTES + f * A_HALF);
                // accumulator of (f, h): TMEM columns 256 (f + h) (one of them is 0)
#pragma unroll
                for (int k4 = 0; k4 < BK / 16; ++k4)  // +32 bytes per K=16 step inside the atom
                  mma_f16_ss(d_tmem + (f + h) * 256, ad + 2 * k4, bd + 2 * k4, kIdesc,
                             ((kk - j0) | k4) != 0);
              }
              mma_commit(empty_b + 8 * ib);
            } else {
              mbar_arrive(empty_b + 8 * ib);  // nothing read this half
            }
          }
          if (!ok) break;
          mma_commit(empty_a + 8 * sa);
        }
        if (ok) mma_commit(acc_full + 8 * a);
      }
      mma_commit(drain);
      if (!mbar_wait(drain, 0)) set_status(BONSAI_ERR_TIMEOUT);
    }
  } else if (warp >= W_EPI && warp < W_EPI + 4) {
    // ------------------------------- epilogue -------------------------------
    pdl_wait();
    const int e = warp - W_EPI;  // TMEM lanes 32e .. 32e+31
    const int et = threadIdx.x - W_EPI * 32;  // 0..127
    uint32_t it = 0;
    // all four epilogue warps at one point (bounded: a warp that gave up on
    // a wait still arrives, and a wait that runs out is recorded)
    uint32_t ephase = 0;
    auto epi_sync = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(epi_bar);
      if (!mbar_wait(epi_bar, ephase & 1)) set_status(BONSAI_ERR_TIMEOUT);
      ++ephase;
    };
    const Segs<MODE == NARROW> sg(p);
    for (int i = 0; i < sg.count; ++i, ++it) {
      int tile, j0, j1;
      sg.at(p, i, tile, j0, j1);
      // stream-K: a piece that does not hold k-step 0 leaves its sums in its
      // partial tile; the piece that does adds those of the next CTAs
      // (their first pieces lie in this tile), in CTA order
      const bool sk = MODE == NARROW && i >= sg.whole;
      const bool partial = sk && j0 > 0;
      int np = 0;
      if (sk && !partial) {
        np = sk_partners(p, tile);
        if (np > kMaxPartners) {  // the host keeps ranges long enough for this never to happen
          if (et == 0) set_status(BONSAI_ERR_UNSUPPORTED);
          np = kMaxPartners;
        }
        if (np > 0) {
          if (et == 0 && !wait_at_least(p.ws_count + (tile - p.dp), (unsigned)np))
            set_status(BONSAI_ERR_TIMEOUT);
          epi_sync();
        }
      }
      const uint32_t a = it % C::NACC, use = it / C::NACC;
      if (!mbar_wait(acc_full + 8 * a, use & 1)) { set_status(BONSAI_ERR_TIMEOUT); break; }
      tc_fence_after();
      if (i == sg.count - 1) {  // the last accumulator is complete: the dequantisers may help
        __syncwarp();
        if (lane == 0) mbar_arrive(help_bar);
      }
      const int n0 = (tile / p.tok_tiles) * FM, m0 = (tile % p.tok_tiles) * TT;
      if constexpr (MODE == NARROW) {
        if (sk) {
          // Stream-K pieces, 16 tokens (a step) at a time. Partial tile
          // layout [step][i4][feature row][4 tokens] FP32: a warp's float4
          // stores and loads cover 512 contiguous bytes. The finishing piece
          // is its CTA's last segment, so its MMAs have completed and the A
          // and B rings (192 KB) are idle: the partners' partial tiles are
          // brought there by bulk copies, a group of steps of all partners
          // at a time, and added from shared memory.
          const int steps = (p.m - m0 + 15) / 16 < BN / 16 ? (p.m - m0 + 15) / 16 : BN / 16;
          const uint32_t tl = tmem_base + ((uint32_t)(32 * e) << 16) + a * 256;
          constexpr int STEP_BYTES = BM * 16 * 4;  // 8 KB
          auto part_at = [&](int cta, int st) {
            return p.ws + (size_t)cta * (BM * BN) + (size_t)st * (BM * 16);
          };
          if (partial) {
            for (int st = 0; st < steps; ++st) {
              uint32_t v[16];
              TMEM_LD_16(tl + 16 * st, v);
              tmem_ld_wait();
              float4* dst = reinterpret_cast<float4*>(part_at(blockIdx.x, st)) + et;
#pragma unroll
              for (int i4 = 0; i4 < 4; ++i4)
                dst[i4 * BM] = make_float4(__uint_as_float(v[4 * i4]), __uint_as_float(v[4 * i4 + 1]),
                                           __uint_as_float(v[4 * i4 + 2]), __uint_as_float(v[4 * i4 + 3]));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty + 8 * a);
          } else {
            static_assert(A_STAGES * A_BYTES + B_STAGES * B_BYTES >= 2 * kFinishBufSteps * STEP_BYTES,
                          "two finishing buffers fit the rings");
            finish_cut_tile(p, tile, np, tmem_base + a * 256, sA, stg_bar, fin_bar, 0, et == 0);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty + 8 * a);
          }
        }
      }
      if (!(MODE == NARROW && sk)) {
        // the last tile: with the dequantisers (not for wide tiles)
        const int ngrp = MODE != WIDE && i == sg.count - 1 ? 3 : 1;
        store_tile<FM, TT, C::FHALVES>(p, tile, tmem_base, a, 0, ngrp, acc_empty + 8 * a);
      }
      if (partial) {  // every row stored, then one count for the tile
        __threadfence();
        epi_sync();
        if (et == 0)
          asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.ws_count + (tile - p.dp))
                       : "memory");
      } else if (np > 0) {  // every partial read: the counter is zero again for the next call
        epi_sync();
        if (et == 0) p.ws_count[tile - p.dp] = 0;
      }
    }
  } else if (warp >= W_DQ) {
    // ------------------------------ dequantisers -----------------------------
    if (!p.prefetch) pdl_wait();
    const int dq = warp - W_DQ;         // 0..7
    const uint32_t h = dq >> 2;         // parity group: even / odd k-steps
    const int r = (dq & 3) * 32 + lane; // feature row within the tile
    const int sw = r & 7;
    const uint32_t lut = sLut + lane * 4;
    const TerConsts K;
    // Ternary: the packed row is read in 64-byte blocks (320 codes = 5
    // k-steps) one block ahead, so the load latency hides behind the
    // dequantisation of the current block; the block's group scales travel
    // with it.
    constexpr int KPB = 5;
    const int nblk = (p.nk + KPB - 1) / KPB;
    uint32_t cur[16], nxt[16];
    uint16_t csc[3], nsc[3];
    int cur_key = -1, nxt_key = -1;
    auto load_block = [&](int tile, int u, uint32_t (&dst)[16], uint16_t (&sc)[3]) {
      const int n = (tile / p.tok_tiles) * FM + r;
      const bool nok = n < p.n;
      const unsigned short* srow = reinterpret_cast<const unsigned short*>(p.scales) +
                                   (size_t)(nok ? n : 0) * p.G;
      const int g0 = (KPB * u) >> 1;
#pragma unroll
      for (int i = 0; i < 3; ++i) sc[i] = (nok && g0 + i < p.G) ? srow[g0 + i] : (uint16_t)0;
      const uint4* src =
          reinterpret_cast<const uint4*>(p.w + (long long)(nok ? n : 0) * p.row_bytes + 64 * u);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 q4 = src[i];  // ternary rows hold whole 64-byte blocks
        dst[4 * i] = q4.x; dst[4 * i + 1] = q4.y; dst[4 * i + 2] = q4.z; dst[4 * i + 3] = q4.w;
      }
    };
    uint32_t g = 0;
    bool ok = true;
    const Segs<MODE == NARROW> sg(p);
    for (int i = 0; i < sg.count && ok; ++i) {
      int tile, j0, j1;
      sg.at(p, i, tile, j0, j1);
      const int n = (tile / p.tok_tiles) * FM + r;
      const bool nok = n < p.n;
      const uint8_t* wrow = p.w + (long long)(nok ? n : 0) * p.row_bytes;
      const __half* srow = p.scales + (size_t)(nok ? n : 0) * p.G;
      // 256-feature tiles: this thread also expands row r + 128 into the
      // stage's second M=128 operand tile
      const bool nok2 = FM > BM && n + BM < p.n;
      const uint8_t* wrow2 = p.w + (long long)(nok2 ? n + BM : 0) * p.row_bytes;
      const __half* srow2 = p.scales + (size_t)(nok2 ? n + BM : 0) * p.G;
      for (int j = j0; j < j1; ++j, ++g) {
        if ((g & 1) != h) continue;
        const int kk = k_at(p, tile, j);  // the k-step this stage holds
        const int s = g % A_STAGES;
        const uint32_t ph = (g / A_STAGES) & 1;
        const uint32_t dst = sA + s * A_BYTES + r * 128;
        if constexpr (FMT == BONSAI_FMT_BINARY) {
          // 8 bytes and one scale per k-step, loaded directly (measured
          // faster than loading one own k-step or one 64-byte block ahead)
          const uint2 wv = *reinterpret_cast<const uint2*>(wrow + 8 * kk);
          const __half sc = srow[kk >> 1];
          const uint32_t s2 = nok ? (uint32_t(__half_as_ushort(sc)) * 0x10001u) : 0u;
          uint2 wv2 = make_uint2(0u, 0u);
          uint32_t s22 = 0u;
          if constexpr (FM > BM) {
            wv2 = *reinterpret_cast<const uint2*>(wrow2 + 8 * kk);
            const __half sc2 = srow2[kk >> 1];
            s22 = nok2 ? (uint32_t(__half_as_ushort(sc2)) * 0x10001u) : 0u;
          }
          if (!mbar_wait(empty_a + 8 * s, ph ^ 1)) { set_status(BONSAI_ERR_TIMEOUT); ok = false; break; }
          dq_binary(wv, s2, dst, sw);
          if constexpr (FM > BM) dq_binary(wv2, s22, dst + A_HALF, sw);
        } else {
          const int u = kk / KPB;
          const int key = tile * nblk + u;
          if (key != cur_key) {
            if (key == nxt_key) {
#pragma unroll
              for (int i = 0; i < 16; ++i) cur[i] = nxt[i];
#pragma unroll
              for (int i = 0; i < 3; ++i) csc[i] = nsc[i];
            } else {
              load_block(tile, u, cur, csc);
            }
            cur_key = key;
            // prefetch the block that follows in this thread's order: the
            // one of the segment's next k-step outside this block, or the
            // next segment's first
            const int jn = j + (KPB - kk % KPB < p.nk - kk ? KPB - kk % KPB : p.nk - kk);
            int nt = -1, nj = 0;
            if (jn < j1) {
              nt = tile;
              nj = jn;
            } else if (i + 1 < sg.count) {
              int b2;
              sg.at(p, i + 1, nt, nj, b2);
            }
            if (nt >= 0) {
              const int nu = k_at(p, nt, nj) / KPB;
              load_block(nt, nu, nxt, nsc);
              nxt_key = nt * nblk + nu;
            }
          }
          const int si = (kk >> 1) - ((KPB * u) >> 1);  // 0..2
          const uint32_t sc = si == 0 ? csc[0] : si == 1 ? csc[1] : csc[2];
          const uint32_t s2 = sc * 0x10001u;  // rows past n carry scale 0
          if (!mbar_wait(empty_a + 8 * s, ph ^ 1)) { set_status(BONSAI_ERR_TIMEOUT); ok = false; break; }
          switch (kk % 5) {
            case 0: dq_ternary<0>(cur, s2, lut, K, dst, sw); break;
            case 1: dq_ternary<1>(cur, s2, lut, K, dst, sw); break;
            case 2: dq_ternary<2>(cur, s2, lut, K, dst, sw); break;
            case 3: dq_ternary<3>(cur, s2, lut, K, dst, sw); break;
            default: dq_ternary<4>(cur, s2, lut, K, dst, sw); break;
          }
        }
        fence_proxy_async_smem();  // generic-proxy stores -> tensor-core reads
        __syncwarp();
        if (lane == 0) mbar_arrive(full_a + 8 * s);
      }
    }
    // no k-steps left: help with this CTA's last tile (its stores, or finishing a cut tile)
    if (ok && sg.count > 0) {
      const int i = sg.count - 1;
      int tile, j0, j1;
      sg.at(p, i, tile, j0, j1);
      const uint32_t a = (uint32_t)i % C::NACC;
      if (MODE != WIDE && !(MODE == NARROW && i >= sg.whole)) {
        if (!mbar_wait(help_bar, 0)) {
          set_status(BONSAI_ERR_TIMEOUT);
        } else {
          tc_fence_after();
          store_tile<FM, TT, C::FHALVES>(p, tile, tmem_base, a, 1 + (dq >> 2), 3, 0);
        }
      }
    }
    if constexpr (MODE == NARROW) {
      if (ok && sg.count > sg.whole) {
        const int i = sg.count - 1;
        int tile, j0, j1;
        sg.at(p, i, tile, j0, j1);
        if (j0 == 0) {
          int np = sk_partners(p, tile);
          np = np > kMaxPartners ? kMaxPartners : np;
          const uint32_t a = (uint32_t)i % C::NACC;
          if (!mbar_wait(help_bar, 0)) {
            set_status(BONSAI_ERR_TIMEOUT);
          } else {
            tc_fence_after();
            finish_cut_tile(p, tile, np, tmem_base + a * 256, sA, stg_bar, fin_bar, 1 + (dq >> 2),
                            false);
          }
        }
      }
    }
  }

  pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == W_TMEM) tmem_dealloc(tmem_base, TMEM_COLS);
}

// Stream-K schedule of `tiles` 128 x 256 tiles of nk k-steps on `sms` CTAs:
// the whole waves stay data-parallel; when the plain schedule would leave
// more than a sixteenth of the SM time idle, the last wave is cut into equal
// k-step ranges of at least kMinSkSteps, each CTA's range within two
// consecutive tiles. (A finishing range adds the others' partial tiles at
// the end of the kernel, ~10 us measured at 512 tokens, so an almost full
// last wave is not worth cutting.)
constexpr int kMinSkSteps = 8;
struct SkPlan {
  int dp = 0, sk_ctas = 0;
  long long iters = 0;
  long long bytes = 0;  // workspace: counters, then the partial tiles
  long long count_bytes = 0;
};
static SkPlan sk_plan(long long tiles, int nk, int sms) {
  SkPlan s;
  const long long rest = tiles % sms;
  const long long waves = (tiles + sms - 1) / sms;
  if (rest == 0 || tiles * 16 >= 15 * waves * sms) return s;
  const long long iters = rest * nk;
  if (iters * sms >= (1LL << 31)) return s;  // the device splits ranges in 32-bit
  long long ctas = iters / kMinSkSteps;
  if (ctas > sms) ctas = sms;
  // ranges of at least nk / (kMaxPartners - 1) k-steps: a tile meets at most
  // kMaxPartners + 1 of them
  if (ctas > (kMaxPartners - 1) * rest) ctas = (kMaxPartners - 1) * rest;
  if (ctas <= rest) return s;  // ranges of a whole tile: nothing to gain
  s.dp = (int)(tiles - rest);
  s.sk_ctas = (int)ctas;
  s.iters = iters;
  s.count_bytes = (rest * 4 + 255) / 256 * 256;
  s.bytes = s.count_bytes + ctas * (long long)BM * BN * 4;
  return s;
}

// The tile shape (NARROW / WIDE / TALL) and, for NARROW tiles with a
// workspace, the stream-K schedule.
struct Shape {
  int mode, tt, fm;
  long long tiles;
  SkPlan sk;
};
static Shape gemm_shape(const bonsai_weights* w, int64_t m, bool stream_k) {
  const bool ter = w->format == BONSAI_FMT_TERNARY;
  auto smem_of = [](int a, int a_bytes, int b, int b_bytes, bool lut) {
    return a * a_bytes + b * b_bytes + (lut ? LUT_BYTES : 0) + BAR_BYTES;
  };
  using CTW = Cfg<BONSAI_FMT_TERNARY, WIDE>;
  using CBT = Cfg<BONSAI_FMT_BINARY, TALL>;
  const int smem_big = ter ? smem_of(CTW::A, CTW::A_BYTES, CTW::B, CTW::B_BYTES, true)
                           : smem_of(CBT::A, CBT::A_BYTES, CBT::B, CBT::B_BYTES, false);
  // Besides the 128-feature x 256-token tiles (two TMEM accumulators, the
  // epilogue overlapping the next tile), each format has a larger tile with
  // one 512-column accumulator: ternary 512 tokens (halves the dequantisation
  // per FLOP, the ternary limiter: +7% at M=512, N=17408), binary 256
  // features (halves the activation-tile traffic per FLOP, where binary's MMA
  // thread waits; 512-token tiles measured -9% for binary). The larger tile
  // is taken when the SMs stay about as busy (busy = tiles / (waves * SMs);
  // 0.9 for stream-K narrow tiles): a layer's N=5120 products would
  // otherwise drop from 80 to 40 tiles.
  const long long sms_l = device_sm_count();
  auto busy = [&](long long tiles) {
    return (double)tiles / (double)(((tiles + sms_l - 1) / sms_l) * sms_l);
  };
  const long long ft = (w->n + BM - 1) / BM, ft2 = (w->n + 2 * BM - 1) / (2 * BM);
  const long long tok = (m + 255) / 256, tok2 = (m + 511) / 512;
  const int nk = (int)(w->k / BK);
  const SkPlan skn = stream_k ? sk_plan(ft * tok, nk, (int)sms_l) : SkPlan{};
  // a cut last wave fills the SMs, less its partial-tile traffic
  const double busy_narrow = skn.sk_ctas ? 0.9 : busy(ft * tok);
  const double busy_big = ter ? busy(ft * tok2) : busy(ft2 * tok);
  // Binary takes 256-feature tiles only while every SM gets at most one: the
  // gain is the halved X traffic, and with several tiles per SM the
  // epilogue no longer overlapped cancels it (interleaved A/B on one GPU:
  // M=512, N=17408 +13%, M=4096 even, a layer whose q/k/v and gate/up took
  // them -4.5%).
  const bool big = (ter ? m > BN : ft2 * tok <= sms_l) && busy_big >= 0.85 * busy_narrow &&
                   smem_big <= device_max_smem_optin();
  Shape sh;
  sh.mode = !big ? NARROW : (ter ? WIDE : TALL);
  sh.tt = sh.mode == WIDE ? 512 : 256;
  sh.fm = sh.mode == TALL ? 256 : BM;
  sh.tiles = ((w->n + sh.fm - 1) / sh.fm) * ((m + sh.tt - 1) / sh.tt);
  if (sh.mode == NARROW) sh.sk = skn;
  return sh;
}
}  // namespace gemm

int64_t gemm_workspace_bytes(const bonsai_weights* w, int64_t m) {
  return gemm::gemm_shape(w, m, true).sk.bytes;
}

bonsai_status gemm_launch(const bonsai_weights* w, const uint16_t* x, int64_t m, uint16_t* y,
                          bool swiglu, cudaStream_t stream, void* ws, int64_t ws_bytes) {
  using namespace gemm;
  if (m > 0x7FFFFFFF / 2) return BONSAI_ERR_UNSUPPORTED;
  CUtensorMap tm;
  if (!encode_tensor_map_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, const_cast<uint16_t*>(x),
                            (uint64_t)w->k, (uint64_t)m, (uint64_t)w->k * 2, BK, BN,
                            CU_TENSOR_MAP_SWIZZLE_128B))
    return BONSAI_ERR_CUDA;
  const bool ter = w->format == BONSAI_FMT_TERNARY;
  auto smem_of = [](int a, int a_bytes, int b, int b_bytes, bool lut) {
    return a * a_bytes + b * b_bytes + (lut ? LUT_BYTES : 0) + BAR_BYTES;
  };
  using CTN = Cfg<BONSAI_FMT_TERNARY, NARROW>;
  using CTW = Cfg<BONSAI_FMT_TERNARY, WIDE>;
  using CBN = Cfg<BONSAI_FMT_BINARY, NARROW>;
  using CBT = Cfg<BONSAI_FMT_BINARY, TALL>;
  const int smem_narrow = ter ? smem_of(CTN::A, CTN::A_BYTES, CTN::B, CTN::B_BYTES, true)
                              : smem_of(CBN::A, CBN::A_BYTES, CBN::B, CBN::B_BYTES, false);
  const int smem_big = ter ? smem_of(CTW::A, CTW::A_BYTES, CTW::B, CTW::B_BYTES, true)
                           : smem_of(CBT::A, CBT::A_BYTES, CBT::B, CBT::B_BYTES, false);
  Shape sh = gemm_shape(w, m, ws != nullptr);
  if (sh.sk.sk_ctas && sh.sk.bytes > ws_bytes) {  // workspace too small: whole tiles
    sh = gemm_shape(w, m, false);
  }
  const bool big = sh.mode != NARROW;
  const int tt = sh.tt, fm = sh.fm;

  Params p{};
  p.w = static_cast<const uint8_t*>(w->packed);
  p.scales = reinterpret_cast<const __half*>(w->scales);
  p.y = reinterpret_cast<__half*>(y);
  p.row_bytes = w->row_bytes;
  p.m = (int)m;
  p.n = (int)w->n;
  p.k = (int)w->k;
  p.G = p.k / 128;
  p.nk = p.k / BK;
  p.tok_tiles = (int)((m + tt - 1) / tt);
  p.tiles = ((p.n + fm - 1) / fm) * p.tok_tiles;
  p.prefetch = (w->flags & BONSAI_WEIGHTS_PREFETCH) ? 1 : 0;
  p.swiglu = swiglu ? 1 : 0;
  p.y_stride = swiglu ? p.n / 2 : p.n;
  if (sh.sk.sk_ctas) {
    p.dp = sh.sk.dp;
    p.sk_ctas = sh.sk.sk_ctas;
    p.sk_iters = (int)sh.sk.iters;
    p.ws_count = static_cast<unsigned int*>(ws);
    p.ws = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + sh.sk.count_bytes);
  } else {
    p.dp = p.tiles;
  }

  const int smem = big ? smem_big : smem_narrow;
  if (smem > device_max_smem_optin()) return BONSAI_ERR_UNSUPPORTED;
  const void* fn = ter ? (big ? (const void*)gemm_kernel<BONSAI_FMT_TERNARY, WIDE>
                              : (const void*)gemm_kernel<BONSAI_FMT_TERNARY, NARROW>)
                       : (big ? (const void*)gemm_kernel<BONSAI_FMT_BINARY, TALL>
                              : (const void*)gemm_kernel<BONSAI_FMT_BINARY, NARROW>);
  if (ensure_dynamic_smem(fn, smem) != cudaSuccess)
    return BONSAI_ERR_CUDA;

  const int sms = device_sm_count();
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p.sk_ctas ? sms : (p.tiles < sms ? p.tiles : sms));
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&tm, &p};
  return cuda_status(cudaLaunchKernelExC(&cfg, fn, args));
}

}  // namespace bonsai
