// gemv.cu -- streaming decode product y = x . (s (.) W)^T for binary and
// ternary weights and up to 8 token columns (batch-1 decode, speculative
// verification). Memory-bandwidth bound: each packed byte is read once.
//
// Design (sm_103a):
//  * One persistent CTA per SM. A producer warp streams 16-row tiles of
//    packed weights into a 4-stage shared-memory ring with 1-D bulk copies
//    (TMA engine), one copy per row and chunk of up to 1024 bytes.
//  * Eight consumer warps split each chunk along K and expand codes to FP16
//    operands in registers, then feed mma.sync m16n8k16 (FP16 x FP16 -> FP32):
//    the tensor core serves as the wide FP32 accumulator of a 16-row x
//    16-code slab per instruction; the 8 columns of the B operand carry up
//    to 8 tokens.
//  * Code -> FP16 without a multiply per weight: a code c in {0,1,2} (ternary
//    digit, or the binary bit) placed into mantissa bits j..j+1 of an FP16
//    whose exponent is 15-j gives the value 2^-j + c * 2^-10, one LOP3 per
//    two codes. With the same 2^-10 step for every j, the per-group MMA sum
//    is acc = sum 2^-j(k) x_k + 2^-10 sum c_k x_k, so
//      binary : sum (2b-1) x = 2^11 acc - T,  T = sum (2^(11-j)+1) x
//      ternary: sum (c-1) x  = 2^10 acc - T,  T = sum (2^(10-j)+1) x
//    where T depends only on x and is built once per CTA. This is the pages'
//    "multiplication degenerates to addition and sign flip" carried out by
//    the tensor core's adders ("三值权重到底做了什么").
//  * The FP16 group scale (one per 128 codes, OpenBonsai "工作原理") multiplies
//    each group's FP32 partial: y += s_g * (2^e acc_g - T_g).
//  * Ternary bytes decode through a 256-entry table (byte -> five 2-bit
//    digits) replicated once per lane so that lookups never conflict.
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
constexpr int kRows = 16;                  // rows per tile (MMA M)
constexpr int kStages = 4;
constexpr int kChunk = 1024;               // packed bytes per row per stage
constexpr int kLutBytes = 256 * 256;       // 256 entries x (32 lanes x 4 B, padded)
constexpr int kTerEntry = 48;              // bytes per (variant, lane) x-table entry
constexpr int kTerVariants = 12;           // (round, group) pairs per super-group

struct Params {
  const uint8_t* w;
  const __half* scales;
  const __half* x;
  __half* y;
  long long row_bytes;
  int n, k, m, G;
  int data_bytes;  // packed bytes per row that are streamed
  int chunks;      // stages per tile
  int pitch;       // smem row pitch, bytes (pitch/4 = 4 mod 32)
  int tiles;
  int n_sg;        // ternary: 640-code super-groups per row
  int t_rows;      // rows of the T table
  int xt_stride;   // bytes per token column of the x table
  int prefetch;    // may read weights before the previous grid completes
  int off_bar, off_red, off_t, off_lut, off_xt, off_stage;
};

// ---- operand expansion constants -----------------------------------------
// FP16 pair with both exponents 15-j and mantissa bits j..j+1 selected.
__host__ __device__ constexpr uint32_t mant_mask1(int j) { return (1u << j) | (1u << (j + 16)); }
__host__ __device__ constexpr uint32_t mant_mask2(int j) { return (3u << j) | (3u << (j + 16)); }
__host__ __device__ constexpr uint32_t exp_base(int j) {
  return (uint32_t(15 - j) << 10) | (uint32_t(15 - j) << 26);
}

// Binary: bit p (0..15) of each 16-bit half is moved to mantissa bit j(p)
// in 4..9 by a shift of the word: p<4 via w<<4, 4<=p<=9 in place, p>=10 via
// w>>6. Keeping j >= 4 bounds the constant term 2^-j against the step 2^-10.
__host__ __device__ constexpr int bin_j(int p) { return p < 4 ? p + 4 : (p <= 9 ? p : p - 6); }

template <int P>
__device__ __forceinline__ uint32_t bin_operand(uint32_t w, uint32_t wl, uint32_t wr) {
  constexpr int j = bin_j(P);
  const uint32_t src = P < 4 ? wl : (P <= 9 ? w : wr);
  return (src & mant_mask1(j)) | exp_base(j);
}

// Ternary: the table gives digit i at bits 2i..2i+1; digits 0,1 are used
// from F<<4 (j = 4, 6), digits 2,3,4 in place (j = 4, 6, 8).
__host__ __device__ constexpr int ter_j(int mdig) { return mdig <= 1 ? 2 * mdig + 4 : 2 * mdig; }

template <int MD>
__device__ __forceinline__ uint32_t ter_operand(uint32_t f, uint32_t fl) {
  constexpr int j = ter_j(MD);
  const uint32_t src = MD <= 1 ? fl : f;
  return (src & mant_mask2(j)) | exp_base(j);
}

// Variant v of a super-group: round (4 words = 80 codes) and the group
// (0..4) whose codes it keeps.
__constant__ int c_var_round[kTerVariants] = {0, 1, 1, 2, 3, 3, 4, 4, 5, 6, 6, 7};
__constant__ int c_var_group[kTerVariants] = {0, 0, 1, 1, 1, 2, 2, 3, 3, 3, 4, 4};

// Fills the operands of digit MD for rows g (fa*) and g+8 (fb*).
template <int MD>
__device__ __forceinline__ void ter_fill(uint32_t (&A)[5][4], uint32_t fa01, uint32_t fb01,
                                         uint32_t fa23, uint32_t fb23) {
  A[MD][0] = ter_operand<MD>(fa01, fa01 << 4);
  A[MD][1] = ter_operand<MD>(fb01, fb01 << 4);
  A[MD][2] = ter_operand<MD>(fa23, fa23 << 4);
  A[MD][3] = ter_operand<MD>(fb23, fb23 << 4);
}

// Operands of a row whose five digits all equal 1 (code 0): the neutral
// pattern whose MMA sum is subtracted from every row's sum.
__device__ __forceinline__ void ter_neutral(uint32_t (&A)[5][4]) {
#pragma unroll
  for (int md = 0; md < 5; ++md) {
    const int j = ter_j(md);
    const uint32_t v = exp_base(j) | (1u << j) | (1u << (j + 16));
    A[md][0] = A[md][1] = A[md][2] = A[md][3] = v;
  }
}

// One 640-code super-group of a 16-row tile: 8 rounds of 80 codes, 5 MMAs
// per round, plus a second pass with the next group's x-table variant when
// a round straddles a 128-code group edge. `operands(rnd, A)` produces the
// expanded codes of a round, `epi(grp, acc)` consumes a finished group.
// The same sequence of MMAs runs for the neutral pattern in the prologue,
// so an all-zero group cancels exactly.
template <typename Ops, typename Epi>
__device__ __forceinline__ void ter_supergroup(const uint8_t* xt, bool bcol, Ops&& operands,
                                               Epi&& epi) {
  float accA[4] = {0.f, 0.f, 0.f, 0.f}, accB[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int rnd = 0; rnd < 8; ++rnd) {
    uint32_t A[5][4];
    operands(rnd, A);
    // first variant of the round; second one if the round straddles a group edge
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

// ---- per-CTA tables from x -------------------------------------------------
template <int FMT>
__device__ void build_tables(const Params& p, uint8_t* smem) {
  const int tid = threadIdx.x;  // 0 .. 255 (consumer threads)
  const int nthr = kWarps * 32;
  float* T = reinterpret_cast<float*>(smem + p.off_t);
  // T[row][8]: zero-fill, then the real entries.
  for (int i = tid; i < p.t_rows * 8; i += nthr) T[i] = 0.f;
  named_bar_sync(1, nthr);
  if (FMT == BONSAI_FMT_BINARY) {
    const int words = p.k / 32;
    for (int t = tid; t < p.m * words; t += nthr) {
      const int col = t / words, wd = t - col * words;
      const __half* xs = p.x + (size_t)col * p.k + 32 * wd;
      uint32_t e[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        e[2 * i] = pack_half2(xs[i], xs[i + 16]);
        e[2 * i + 1] = pack_half2(xs[i + 8], xs[i + 24]);
      }
      uint4* dst = reinterpret_cast<uint4*>(smem + p.off_xt + col * p.xt_stride +
                                            (wd >> 2) * 256 + (wd & 3) * 16);
#pragma unroll
      for (int c = 0; c < 4; ++c)
        dst[c * 4] = make_uint4(e[4 * c], e[4 * c + 1], e[4 * c + 2], e[4 * c + 3]);
    }
    for (int t = tid; t < p.m * p.G; t += nthr) {
      const int col = t / p.G, gi = t - col * p.G;
      const __half* xs = p.x + (size_t)col * p.k + 128 * gi;
      float S[6] = {0, 0, 0, 0, 0, 0}, X = 0.f;
#pragma unroll
      for (int wd = 0; wd < 4; ++wd) {
#pragma unroll
        for (int pp = 0; pp < 16; ++pp) {
          const float v = __half2float(xs[32 * wd + pp]) + __half2float(xs[32 * wd + pp + 16]);
          S[bin_j(pp) - 4] += v;
          X += v;
        }
      }
      float acc = X;
#pragma unroll
      for (int j = 4; j <= 9; ++j) acc += float(1 << (11 - j)) * S[j - 4];
      T[gi * 8 + col] = acc;
    }
  } else {
    // Byte -> digits table, one copy per lane: entry e at e*256 + lane*4.
    uint32_t* lut = reinterpret_cast<uint32_t*>(smem + p.off_lut);
    for (int t = tid; t < 256 * 32; t += nthr) {
      const int e = t >> 5, ln = t & 31;
      uint32_t v = 0;
      if (e < 243) {
        int r = e;
#pragma unroll
        for (int i = 0; i < 5; ++i) {
          v |= uint32_t(r % 3) << (2 * i);
          r /= 3;
        }
      }
      lut[e * 64 + ln] = v;
    }
    // x table: (col, super-group, variant, lane) -> 10 words (b0,b1 per digit).
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
      const __half* xs = p.x + (size_t)col * p.k;
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
    // T = MMA sum of the neutral (all-zero-code) pattern per group and
    // token, computed with the very MMA sequence of the main loop.
    named_bar_sync(1, nthr);  // x table complete
    {
      const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, q = lane & 3;
      const bool bcol = g < p.m;
      const uint8_t* xt_col = smem + p.off_xt + (bcol ? g : 0) * p.xt_stride;
      for (int sg = warp; sg < p.n_sg; sg += kWarps) {
        const uint8_t* xt = xt_col + (sg * kTerVariants * 4 + q) * kTerEntry;
        auto operands = [&](int, uint32_t (&A)[5][4]) { ter_neutral(A); };
        auto epi = [&](int grp, const float (&acc)[4]) {
          if (g == 0) {
            T[(5 * sg + grp) * 8 + 2 * q] = acc[0];
            T[(5 * sg + grp) * 8 + 2 * q + 1] = acc[1];
          }
        };
        ter_supergroup(xt, bcol, operands, epi);
      }
    }
  }
}

// ---- epilogue of one group ---------------------------------------------------
template <int FMT>
__device__ __forceinline__ void group_epilogue(float (&yacc)[4], const float (&acc)[4],
                                               float2 tt, float s0, float s1) {
  constexpr float kStep = FMT == BONSAI_FMT_BINARY ? 2048.f : 1024.f;
  yacc[0] = fmaf(s0, fmaf(acc[0], kStep, -tt.x), yacc[0]);
  yacc[1] = fmaf(s0, fmaf(acc[1], kStep, -tt.y), yacc[1]);
  yacc[2] = fmaf(s1, fmaf(acc[2], kStep, -tt.x), yacc[2]);
  yacc[3] = fmaf(s1, fmaf(acc[3], kStep, -tt.y), yacc[3]);
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + p.off_bar;
  const uint32_t bar_empty = bar_full + 8 * kStages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kWarps) {
    // ------------------------------ producer -------------------------------
    if (lane == 0) {
      if (!p.prefetch) pdl_wait();
      const uint64_t pol = policy_evict_first();
      int s = 0;
      uint32_t ph = 0;
      for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x) {
        const int row0 = tile * kRows;
        const int rows = min(kRows, p.n - row0);
        const uint8_t* src = p.w + (long long)row0 * p.row_bytes;
        for (int c = 0; c < p.chunks; ++c) {
          if (!mbar_wait(bar_empty + 8 * s, ph ^ 1)) {
            set_status(BONSAI_ERR_TIMEOUT);
            return;
          }
          const int off = c * kChunk;
          const int len = min(kChunk, p.data_bytes - off);
          mbar_arrive_expect_tx(bar_full + 8 * s, uint32_t(rows * len));
          const uint32_t dst = sbase + p.off_stage + s * kRows * p.pitch;
          for (int r = 0; r < rows; ++r)
            bulk_g2s(dst + r * p.pitch, src + r * p.row_bytes + off, len, bar_full + 8 * s, pol);
          if (++s == kStages) { s = 0; ph ^= 1; }
        }
      }
    }
    pdl_launch_dependents();
    return;
  }

  // -------------------------------- consumers ---------------------------------
  pdl_wait();  // x is written by earlier work on the stream; y may be read by it
  build_tables<FMT>(p, smem);
  named_bar_sync(1, kWarps * 32);
  pdl_launch_dependents();

  const int g = lane >> 2, q = lane & 3;
  const bool bcol = g < p.m;
  const uint8_t* xt_col = smem + p.off_xt + (bcol ? g : 0) * p.xt_stride;  // never past the table
  const float* T = reinterpret_cast<const float*>(smem + p.off_t);
  const uint32_t lut_lane = uint32_t(lane * 4);
  const uint8_t* lut = smem + p.off_lut;
  const int pw = p.pitch >> 2;  // pitch in words

  int s = 0;
  uint32_t ph = 0;
  bool alive = true;
  int tcount = 0;
  for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x, ++tcount) {
    const int row0 = tile * kRows;
    const int rg = min(row0 + g, p.n - 1), rg8 = min(row0 + g + 8, p.n - 1);
    const __half* sc0p = p.scales + (size_t)rg * p.G;
    const __half* sc1p = p.scales + (size_t)rg8 * p.G;
    float yacc[4] = {0.f, 0.f, 0.f, 0.f};

    for (int c = 0; c < p.chunks; ++c) {
      const int len = min(kChunk, p.data_bytes - c * kChunk);
      const uint32_t* stg =
          reinterpret_cast<const uint32_t*>(smem + p.off_stage + s * kRows * p.pitch);
      if (FMT == BONSAI_FMT_BINARY) {
        const int cg = len >> 4;  // groups in this chunk (16 bytes each)
        const int gb = (warp * cg) >> 3, ge = ((warp + 1) * cg) >> 3;
        const int gbase = c * (kChunk / 16);
        float s0[8], s1[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int gi = min(gbase + gb + j, p.G - 1);
          s0[j] = __half2float(sc0p[gi]);
          s1[j] = __half2float(sc1p[gi]);
        }
        if (alive && !mbar_wait(bar_full + 8 * s, ph)) { set_status(BONSAI_ERR_TIMEOUT); alive = false; }
        if (alive) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (gb + j < ge) {
              const int gl = gb + j;       // group within the chunk
              const int gi = gbase + gl;   // group within the row
              const uint32_t w0 = stg[g * pw + gl * 4 + q];
              const uint32_t w1 = stg[(g + 8) * pw + gl * 4 + q];
              const uint32_t w0l = w0 << 4, w0r = w0 >> 6, w1l = w1 << 4, w1r = w1 >> 6;
              const uint4* xt = reinterpret_cast<const uint4*>(xt_col + gi * 256) + q;
              float acc[4] = {0.f, 0.f, 0.f, 0.f};
#define BIN_MMA(I, BX, BY)                                                        \
  mma_16816(acc, bin_operand<I>(w0, w0l, w0r), bin_operand<I>(w1, w1l, w1r),      \
            bin_operand<I + 8>(w0, w0l, w0r), bin_operand<I + 8>(w1, w1l, w1r), BX, BY)
              {
                uint4 b = bcol ? xt[0] : make_uint4(0, 0, 0, 0);
                BIN_MMA(0, b.x, b.y);
                BIN_MMA(1, b.z, b.w);
                b = bcol ? xt[4] : make_uint4(0, 0, 0, 0);
                BIN_MMA(2, b.x, b.y);
                BIN_MMA(3, b.z, b.w);
                b = bcol ? xt[8] : make_uint4(0, 0, 0, 0);
                BIN_MMA(4, b.x, b.y);
                BIN_MMA(5, b.z, b.w);
                b = bcol ? xt[12] : make_uint4(0, 0, 0, 0);
                BIN_MMA(6, b.x, b.y);
                BIN_MMA(7, b.z, b.w);
              }
#undef BIN_MMA
              const float2 tt = *reinterpret_cast<const float2*>(T + gi * 8 + 2 * q);
              group_epilogue<FMT>(yacc, acc, tt, s0[j], s1[j]);
            }
          }
        }
      } else {
        const int nsg = (len + 127) >> 7;  // super-groups in this chunk
        const int sg = c * (kChunk / 128) + warp;
        float s0[5], s1[5];
#pragma unroll
        for (int j = 0; j < 5; ++j) {
          const int gi = min(5 * sg + j, p.G - 1);
          s0[j] = __half2float(sc0p[gi]);
          s1[j] = __half2float(sc1p[gi]);
        }
        if (alive && !mbar_wait(bar_full + 8 * s, ph)) { set_status(BONSAI_ERR_TIMEOUT); alive = false; }
        if (alive && warp < nsg) {
          const uint32_t* r0 = stg + g * pw + warp * 32 + q;
          const uint32_t* r1 = stg + (g + 8) * pw + warp * 32 + q;
          const uint8_t* xt = xt_col + (sg * kTerVariants * 4 + q) * kTerEntry;
          auto operands = [&](int rnd, uint32_t (&A)[5][4]) {
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
          };
          auto epi = [&](int grp, const float (&acc)[4]) {
            const int gi = 5 * sg + grp;
            const float2 tt = *reinterpret_cast<const float2*>(T + gi * 8 + 2 * q);
            yacc[0] = fmaf(s0[grp], (acc[0] - tt.x) * 1024.f, yacc[0]);
            yacc[1] = fmaf(s0[grp], (acc[1] - tt.y) * 1024.f, yacc[1]);
            yacc[2] = fmaf(s1[grp], (acc[2] - tt.x) * 1024.f, yacc[2]);
            yacc[3] = fmaf(s1[grp], (acc[3] - tt.y) * 1024.f, yacc[3]);
          };
          ter_supergroup(xt, bcol, operands, epi);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
      if (++s == kStages) { s = 0; ph ^= 1; }
    }

    // cross-warp reduction of the tile
    float* red = reinterpret_cast<float*>(smem + p.off_red) + (tcount & 1) * (kWarps * 16 * 8);
    red[(warp * 16 + g) * 8 + 2 * q] = yacc[0];
    red[(warp * 16 + g) * 8 + 2 * q + 1] = yacc[1];
    red[(warp * 16 + g + 8) * 8 + 2 * q] = yacc[2];
    red[(warp * 16 + g + 8) * 8 + 2 * q + 1] = yacc[3];
    named_bar_sync(1, kWarps * 32);
    if (threadIdx.x < 128) {
      const int row = threadIdx.x & 15, col = threadIdx.x >> 4;
      if (col < p.m && row0 + row < p.n) {
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
  const int fmt = w->format;
  const int k = (int)w->k;
  const int n = (int)w->n;
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
  if (fmt == BONSAI_FMT_BINARY) {
    p.data_bytes = k / 8;
    p.n_sg = 0;
    p.t_rows = p.G;
    p.xt_stride = p.G * 256 + 64;
  } else {
    p.data_bytes = (int)bonsai_packed_row_bytes(BONSAI_FMT_TERNARY, k);
    p.n_sg = (p.data_bytes + 127) / 128;
    p.t_rows = p.n_sg * 5;
    p.xt_stride = p.n_sg * kTerVariants * 4 * kTerEntry + 64;
  }
  p.chunks = (p.data_bytes + kChunk - 1) / kChunk;
  const int chunk_max = p.data_bytes < kChunk ? p.data_bytes : kChunk;
  const int cw = chunk_max / 4;
  const int pw = ((cw - 4 + 31) / 32) * 32 + 4;
  p.pitch = pw * 4;
  p.tiles = (n + kRows - 1) / kRows;

  auto up = [](int v, int a) { return (v + a - 1) / a * a; };
  int off = 0;
  p.off_bar = off;   off = up(off + 16 * kStages, 128);
  p.off_red = off;   off = up(off + 2 * kWarps * 16 * 8 * 4, 128);
  p.off_t = off;     off = up(off + p.t_rows * 8 * 4, 128);
  p.off_lut = off;   if (fmt == BONSAI_FMT_TERNARY) off = up(off + kLutBytes, 128);
  p.off_xt = off;    off = up(off + p.m * p.xt_stride, 1024);
  p.off_stage = off; off = up(off + kStages * kRows * p.pitch, 128);
  const int smem = off;
  if (smem > device_max_smem_optin()) return BONSAI_ERR_UNSUPPORTED;

  const void* fn = fmt == BONSAI_FMT_BINARY ? (const void*)gemv_kernel<BONSAI_FMT_BINARY>
                                            : (const void*)gemv_kernel<BONSAI_FMT_TERNARY>;
  cudaError_t e = ensure_dynamic_smem(fn, smem);
  if (e != cudaSuccess) return BONSAI_ERR_CUDA;

  const int sms = device_sm_count();
  int grid = p.tiles < sms ? p.tiles : sms;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (fmt == BONSAI_FMT_BINARY)
    e = cudaLaunchKernelEx(&cfg, gemv_kernel<BONSAI_FMT_BINARY>, p);
  else
    e = cudaLaunchKernelEx(&cfg, gemv_kernel<BONSAI_FMT_TERNARY>, p);
  return e == cudaSuccess ? BONSAI_OK : BONSAI_ERR_CUDA;
}

}  // namespace bonsai
