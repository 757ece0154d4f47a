// gemv.cu -- streaming decode product y = x . (s (.) W)^T for binary and
// ternary weights and up to 8 token columns (batch-1 decode, speculative
// verification). Memory-bandwidth bound ("第一の壁": every weight is
// re-streamed per token): each packed byte is read from HBM once.
//
// Structure (sm_103a):
//  * A persistent grid, one CTA per SM: 16 consumer warps, a producer warp and
//    a reducer warp. The producer streams tiles of 16 rows in chunks of
//    <= 1024 bytes per row into a shared-memory ring
//    with 2-D TMA boxes, one box for the weights and one for the chunk's
//    group scales. A box is as wide as the padded row pitch (pitch/4 = 4
//    mod 32 words), so the consumers' word loads are conflict-free; the
//    extra columns are either the next chunk's first bytes or read as zero.
//    About 96 KB are in flight per SM.
//  * With BONSAI_WEIGHTS_PREFETCH the producer starts before the previous
//    kernel on the stream has finished (programmatic dependent launch).
//  * Consumers split each chunk along K, expand codes to FP16 operands in
//    registers and accumulate 16 rows x 16 codes per mma.sync m16n8k16
//    (FP16 x FP16 -> FP32; the B columns carry the tokens). The FP16 group
//    scale (one per 128 codes, OpenBonsai page, "工作原理") multiplies each
//    group's FP32 partial; a shared-memory reduction finishes a tile.
//
// Codes -> FP16 without a multiply per code: a code value c in {0,1,2}
// (binary bit, or ternary digit = code + 1) placed into mantissa bits j..
// of an FP16 whose exponent field is 15-j is the number 2^-j + c*2^-10, one
// LOP3 per two codes ("multiplication degenerates to addition and sign
// flip", 三值权重 page). The same 2^-10 step for every j gives, per group,
//   acc = sum_k 2^-j(k) x_k + 2^-10 sum_k c_k x_k.
//  * binary:  sum (2b-1) x = 2^11 acc - T,  T = sum (2^(11-j)+1) x, built
//    once per CTA from x. Every binary code is +-1, so the rounding of the
//    offset sums stays small against the output's own sum |x s w|.
//  * ternary: one packed FP16 subtraction of the digit-1 operand (same j)
//    turns each operand into (c-1)*2^-10 exactly (both values share the
//    exponent), so a zero code contributes an exact 0 product, an all-zero
//    group gives exactly 0 and the accumulation only rounds the nonzero
//    terms: sum (c-1) x = 2^10 acc.
#include <type_traits>
#include <vector>

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

// Consumer warps per CTA; warp W issues the TMA copies, warp W+1 sums the
// warps' partials of a tile.
constexpr int kBinWarps = 16;
constexpr int kTerWarps = 16;
__host__ __device__ constexpr int threads_for(int w) { return (w + 2) * 32; }
constexpr int kMaxStages = 8;
// Stages the producer may issue before the consumers have their activations:
// the weight boxes and the activation loads share the SM's return path from
// L2, so a full ring requested ahead of x delays x by its whole size.
constexpr int kEarlyStages = 2;
constexpr int kStageBudget = 96 * 1024;    // bytes in flight per CTA
constexpr int kChunk = 1024;               // packed bytes per row per stage
constexpr int kLutBytes = 256 * 256;       // ternary: 256 entries x (32 lanes x 4 B + pad)
constexpr int kLutBytes8 = 256 * 128;      // the same, packed (5..8 tokens)
constexpr int kTerEntry = 48;              // ternary x-table bytes per (round, side, lane)
constexpr int kTerMaxTokens = 4;           // two B columns (group parities) per token

struct Params {
  const __half* scales;
  const __half* x;
  __half* y;
  int n, k, m, G;
  int rows;         // rows per tile (16)
  int data_bytes;   // packed bytes per row that are streamed
  int chunks;       // stages per tile
  int pitch;        // smem row pitch, bytes = TMA box width
  int tiles;
  int n_sg;         // ternary: 640-code super-groups per row
  int xt_stride;    // bytes per token of the x table
  int prefetch;     // may read weights before the previous grid completes
  int swiglu;       // rows 16t..16t+7 gate, 16t+8..16t+15 up: write silu(g)*u
  int y_stride;     // elements per token row of y: n, or n/2 with swiglu
  int sc_tma;       // group scales streamed with the weights (G % 8 == 0)
  int sc_chunk;     // groups per chunk (64 binary, 40 ternary)
  int sc_pitch;     // smem bytes per row of streamed scales = TMA box width
  int stage_bytes;  // 16 rows x pitch + 16 rows x sc_pitch, rounded to 128
  int stages;       // ring depth
  int red_cols;     // token columns held per row in the partial-sum slots (m)
  int off_bar, off_red, off_t, off_lut, off_xt, off_stage;
};

// ---------------------------------------------------------------------------
// Barriers at off_bar: full[kMaxStages], empty[kMaxStages] of the weight
// ring, then red_full[2], red_empty[2] of the two partial-sum slots, then
// x_ready (the consumers' tables are built).
constexpr int kBarriers = 2 * kMaxStages + 5;
__device__ __forceinline__ uint32_t x_ready_bar(uint32_t bar_full) {
  return bar_full + 8 * (2 * kMaxStages + 4);
}
template <int W>
__device__ __forceinline__ void init_barriers(uint32_t bar_full, uint32_t bar_empty, int stages) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, W);
    }
    const uint32_t red_full = bar_full + 16 * kMaxStages;
    for (int s = 0; s < 2; ++s) {
      mbar_init(red_full + 8 * s, W);
      mbar_init(red_full + 16 + 8 * s, 1);
    }
    mbar_init(x_ready_bar(bar_full), 1);
    fence_barrier_init();
  }
}

// Partial sums of a tile: red[slot][warp][row][token], two slots used in
// turn. A consumer warp waits until its slot is free, stores its partials
// and arrives on red_full; the reducer warp sums the 16 warps' partials,
// writes y and frees the slot. The consumer warps never wait for each other.
template <int W>
__device__ __forceinline__ float* partial_slot(const Params& p, uint8_t* smem, uint32_t red_full,
                                               int tcount, bool& alive) {
  const int slot = tcount & 1;
  const uint32_t ph = (tcount >> 1) & 1;
  if (alive && !__all_sync(0xFFFFFFFFu, mbar_wait(red_full + 16 + 8 * slot, ph ^ 1))) {
    set_status(BONSAI_ERR_TIMEOUT);
    alive = false;
  }
  return reinterpret_cast<float*>(smem + p.off_red) + slot * (W * 16 * p.red_cols);
}

__device__ __forceinline__ void partial_done(uint32_t red_full, int tcount, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(red_full + 8 * (tcount & 1));
}

// One product's tiles; tcount counts the CTA's tiles over all products of a
// launch (it selects the slot and its phase). Returns false after a timeout.
template <int W>
__device__ bool reduce_tiles(const Params& p, uint8_t* smem, uint32_t red_full, int lane,
                             int& tcount) {
  for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x, ++tcount) {
    const int slot = tcount & 1;
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(red_full + 8 * slot, (tcount >> 1) & 1))) {
      set_status(BONSAI_ERR_TIMEOUT);
      return false;
    }
    const float* red =
        reinterpret_cast<const float*>(smem + p.off_red) + slot * (W * 16 * p.red_cols);
    const int rc = p.red_cols;
    const int row0 = tile * p.rows;
    if (p.swiglu) {
      // 8 gate rows then the 8 up rows of the same features (n % 16 == 0)
      for (int o = lane; o < 8 * p.m; o += 32) {
        const int r = o & 7, col = o >> 3;
        float g = 0.f, u = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
          g += red[(w * 16 + r) * rc + col];
          u += red[(w * 16 + r + 8) * rc + col];
        }
        p.y[(size_t)col * p.y_stride + tile * 8 + r] = __float2half_rn(silu(g) * u);
      }
    } else {
      for (int o = lane; o < 16 * p.m; o += 32) {
        const int row = o & 15, col = o >> 4;
        if (row < p.rows && row0 + row < p.n) {
          float sum = 0.f;
#pragma unroll
          for (int w = 0; w < W; ++w) sum += red[(w * 16 + row) * rc + col];
          p.y[(size_t)col * p.y_stride + row0 + row] = __float2half_rn(sum);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(red_full + 16 + 8 * slot);
  }
  return true;
}

template <int W>
__device__ void reducer(const Params& p, uint8_t* smem, uint32_t red_full, int lane) {
  pdl_wait();  // y may be read by earlier work on the stream
  int tcount = 0;
  reduce_tiles<W>(p, smem, red_full, lane, tcount);
}

// Producer (one thread): per chunk one weight box and, if streamed, one
// scale box, both completing on the stage's full barrier. The ring position
// (s, ph) carries over from product to product within a launch. With x_ready
// (not 0) only the first kEarlyStages stages go out before the consumers
// signal it. Returns false after a timeout.
__device__ __forceinline__ bool produce_tiles(const CUtensorMap* tmw, const CUtensorMap* tms,
                                              const Params& p, uint32_t sbase, uint32_t bar_full,
                                              uint32_t bar_empty, int& s, uint32_t& ph,
                                              uint32_t x_ready = 0) {
  const uint32_t tx = uint32_t(p.rows * p.pitch + (p.sc_tma ? p.rows * p.sc_pitch : 0));
  int issued = 0;
  for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x) {
    const int row0 = tile * p.rows;
    for (int c = 0; c < p.chunks; ++c, ++issued) {
      if (x_ready && issued == kEarlyStages && !mbar_wait(x_ready, 0)) {
        set_status(BONSAI_ERR_TIMEOUT);
        return false;
      }
      if (!mbar_wait(bar_empty + 8 * s, ph ^ 1)) {
        set_status(BONSAI_ERR_TIMEOUT);
        return false;
      }
      mbar_arrive_expect_tx(bar_full + 8 * s, tx);
      const uint32_t dst = sbase + p.off_stage + s * p.stage_bytes;
      tma_load_2d(dst, tmw, c * (kChunk / 8), row0, bar_full + 8 * s);
      if (p.sc_tma) tma_load_2d(dst + 16 * p.pitch, tms, c * p.sc_chunk, row0, bar_full + 8 * s);
      if (++s == p.stages) { s = 0; ph ^= 1; }
    }
  }
  return true;
}

__device__ __forceinline__ void produce(const CUtensorMap* tmw, const CUtensorMap* tms,
                                        const Params& p, uint32_t sbase, uint32_t bar_full,
                                        uint32_t bar_empty) {
  if (!p.prefetch) pdl_wait();
  int s = 0;
  uint32_t ph = 0;
  produce_tiles(tmw, tms, p, sbase, bar_full, bar_empty, s, ph, x_ready_bar(bar_full));
}

// Consumer wait on a stage, with the same outcome in every lane of the warp.
__device__ __forceinline__ bool wait_full(uint32_t bar, uint32_t ph, bool& alive) {
  if (alive) {
    const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar, ph));
    if (!ok) {
      set_status(BONSAI_ERR_TIMEOUT);
      alive = false;
    }
  }
  return alive;
}

// Scale of (row, group gi), gl = gi's index within the chunk: the streamed
// copy, else a global load.
template <bool SC>
__device__ __forceinline__ float scale_of(const Params& p, const uint8_t* stage, int row_in_tile,
                                          int row_global, int gl, int gi) {
  if constexpr (SC)
    return __half2float(
        reinterpret_cast<const __half*>(stage + 16 * p.pitch + row_in_tile * p.sc_pitch)[gl]);
  return __half2float(p.scales[(size_t)min(row_global, p.n - 1) * p.G + min(gi, p.G - 1)]);
}

__host__ __device__ constexpr uint32_t exp_base(int j) {
  return (uint32_t(15 - j) << 10) | (uint32_t(15 - j) << 26);
}

// Exponent fields exp_base(0..9) held in registers: (src & mask) | E is then
// one LOP3 with the mask as its immediate.
struct ExpRegs {
  uint32_t e[10];
  uint32_t one[5];  // ternary: digit-1 operand per digit position
  __device__ __forceinline__ ExpRegs() {
#pragma unroll
    for (int j = 0; j < 10; ++j) {
      uint32_t v = exp_base(j);
      asm volatile("" : "+r"(v));  // keep the value in a register
      e[j] = v;
    }
#pragma unroll
    for (int md = 0; md < 5; ++md) {
      uint32_t v = (uint32_t(15 - 2 * md) << 10 | (1u << (2 * md))) * 0x10001u;
      asm volatile("" : "+r"(v));
      one[md] = v;
    }
  }
};

template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t e) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "r"(e));
  return d;
}

// ===========================================================================
// binary
// ===========================================================================
// Bit p (0..15) of each 16-bit half is used as mantissa bit j(p): bits 0..9
// in place, bits 10..15 from w>>6 (j = 4..9).
__host__ __device__ constexpr int bin_j(int p) { return p <= 9 ? p : p - 6; }

template <int P>
__device__ __forceinline__ uint32_t bin_operand(uint32_t w, uint32_t wr, const ExpRegs& E) {
  constexpr int j = bin_j(P);
  return and_or<(1u << j) | (1u << (j + 16))>(P <= 9 ? w : wr, E.e[j]);
}

// x table (binary): token t, group gi, pair c2 (MMAs 2c2, 2c2+1), lane quad
// index q -> 16 bytes {b0,b1 of MMA 2c2; b0,b1 of MMA 2c2+1} at
// t*stride + gi*256 + c2*64 + q*16. MMA i takes the codes of class i
// (bits i, i+16 of word q of the group) and class i+8 (bits i+8, i+24).
// T[gi][t] = sum over the group of (2^(11-j)+1) x. One thread per word of
// x; the four words of a group sit in four neighbouring lanes.
template <int W>
__device__ void build_binary_tables(const Params& p, uint8_t* smem) {
  const int lane = threadIdx.x & 31, nthr = W * 32;
  float* T = reinterpret_cast<float*>(smem + p.off_t);
  const int words = p.k / 32, total = p.m * words;
  for (int base = threadIdx.x - lane; base < total; base += nthr) {
    const int t = base + lane;
    const bool valid = t < total;
    const int col = valid ? t / words : 0, wd = valid ? t - col * words : 0;
    uint4 v[4] = {};
    if (valid) {
      const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)col * p.k + 32 * wd);
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = src[i];
    }
    uint32_t u[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      u[4 * i] = v[i].x;
      u[4 * i + 1] = v[i].y;
      u[4 * i + 2] = v[i].z;
      u[4 * i + 3] = v[i].w;
    }
    // x of code i of the word: half (i & 1) of u[i >> 1]
    auto xh = [&](int i) -> uint32_t { return (u[i >> 1] >> (16 * (i & 1))) & 0xFFFFu; };
    uint32_t e[16];
    float tsum = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      e[2 * i] = xh(i) | (xh(i + 16) << 16);
      e[2 * i + 1] = xh(i + 8) | (xh(i + 24) << 16);
    }
#pragma unroll
    for (int i = 0; i < 32; ++i)
      tsum = fmaf(float((1 << (11 - bin_j(i & 15))) + 1), __half2float(__ushort_as_half(xh(i))),
                  tsum);
    tsum += __shfl_xor_sync(0xFFFFFFFFu, tsum, 1);
    tsum += __shfl_xor_sync(0xFFFFFFFFu, tsum, 2);
    if (valid) {
      uint4* dst = reinterpret_cast<uint4*>(smem + p.off_xt + col * p.xt_stride + (wd >> 2) * 256 +
                                            (wd & 3) * 16);
#pragma unroll
      for (int c = 0; c < 4; ++c)
        dst[c * 4] = make_uint4(e[4 * c], e[4 * c + 1], e[4 * c + 2], e[4 * c + 3]);
      if ((wd & 3) == 0) T[(wd >> 2) * 8 + col] = tsum;
    }
  }
}

template <bool SC>
__global__ void __launch_bounds__(threads_for(kBinWarps), 1)
    gemv_binary_kernel(const __grid_constant__ CUtensorMap tmw,
                       const __grid_constant__ CUtensorMap tms, const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + p.off_bar, bar_empty = bar_full + 8 * kMaxStages;
  const uint32_t red_full = bar_full + 16 * kMaxStages;
  init_barriers<kBinWarps>(bar_full, bar_empty, p.stages);
  __syncthreads();
  pdl_launch_dependents();
  if (warp == kBinWarps) {
    if (lane == 0) produce(&tmw, &tms, p, sbase, bar_full, bar_empty);
    return;
  }
  if (warp == kBinWarps + 1) {
    reducer<kBinWarps>(p, smem, red_full, lane);
    return;
  }
  pdl_wait();  // x is written by earlier work on the stream
  build_binary_tables<kBinWarps>(p, smem);
  named_bar_sync(1, kBinWarps * 32);
  if (threadIdx.x == 0) mbar_arrive(x_ready_bar(bar_full));

  const int g = lane >> 2, q = lane & 3;
  const bool bcol = g < p.m;
  const int pw = p.pitch >> 2;
  const uint8_t* xt_col = smem + p.off_xt + (bcol ? g : 0) * p.xt_stride;
  const float* T = reinterpret_cast<const float*>(smem + p.off_t);
  const ExpRegs E;
  uint4 bx = make_uint4(0, 0, 0, 0);
  int s = 0;
  uint32_t ph = 0;
  bool alive = true;
  int tcount = 0;
  for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x, ++tcount) {
    const int row0 = tile * 16;
    float yacc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int c = 0; c < p.chunks; ++c) {
      const int len = min(kChunk, p.data_bytes - c * kChunk);
      const int cg = len >> 4;  // 128-code groups in this chunk
      const uint8_t* stage = smem + p.off_stage + s * p.stage_bytes;
      const uint32_t* stg = reinterpret_cast<const uint32_t*>(stage);
      if (wait_full(bar_full + 8 * s, ph, alive)) {
        // Groups gl = r, r + kBinWarps, ... of the chunk; r alternates between
        // the two halves of the warp range from tile to tile, so a warp's
        // share evens out over two tiles. x-table loads only in the lanes of
        // real columns (the others keep stale values, and their columns are
        // not stored).
        const int r = (warp + (kBinWarps / 2) * (tcount & 1)) % kBinWarps;
        for (int gl = r; gl < cg; gl += kBinWarps) {
          const int gi = c * (kChunk / 16) + gl;
          const uint32_t w0 = stg[g * pw + gl * 4 + q];
          const uint32_t w1 = stg[(g + 8) * pw + gl * 4 + q];
          const uint32_t w0r = w0 >> 6, w1r = w1 >> 6;
          const uint4* xt = reinterpret_cast<const uint4*>(xt_col + gi * 256) + q;
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
#define BIN_MMA(I, BX, BY)                                                  \
  mma_16816(acc, bin_operand<I>(w0, w0r, E), bin_operand<I>(w1, w1r, E),    \
            bin_operand<I + 8>(w0, w0r, E), bin_operand<I + 8>(w1, w1r, E), BX, BY)
#pragma unroll
          for (int c2 = 0; c2 < 4; ++c2) {
            if (bcol) bx = xt[4 * c2];
            switch (c2) {
              case 0: BIN_MMA(0, bx.x, bx.y); BIN_MMA(1, bx.z, bx.w); break;
              case 1: BIN_MMA(2, bx.x, bx.y); BIN_MMA(3, bx.z, bx.w); break;
              case 2: BIN_MMA(4, bx.x, bx.y); BIN_MMA(5, bx.z, bx.w); break;
              default: BIN_MMA(6, bx.x, bx.y); BIN_MMA(7, bx.z, bx.w); break;
            }
          }
#undef BIN_MMA
          const float2 tt = *reinterpret_cast<const float2*>(T + gi * 8 + 2 * q);
          const float s0 = scale_of<SC>(p, stage, g, row0 + g, gl, gi);
          const float s1 = scale_of<SC>(p, stage, g + 8, row0 + g + 8, gl, gi);
          yacc[0] = fmaf(s0, fmaf(acc[0], 2048.f, -tt.x), yacc[0]);
          yacc[1] = fmaf(s0, fmaf(acc[1], 2048.f, -tt.y), yacc[1]);
          yacc[2] = fmaf(s1, fmaf(acc[2], 2048.f, -tt.x), yacc[2]);
          yacc[3] = fmaf(s1, fmaf(acc[3], 2048.f, -tt.y), yacc[3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
      if (++s == p.stages) { s = 0; ph ^= 1; }
    }
    float* red = partial_slot<kBinWarps>(p, smem, red_full, tcount, alive);
    const int rc = p.red_cols;  // token columns 2q, 2q+1; only real tokens are kept
    if (2 * q < rc) {
      red[(warp * 16 + g) * rc + 2 * q] = yacc[0];
      red[(warp * 16 + g + 8) * rc + 2 * q] = yacc[2];
    }
    if (2 * q + 1 < rc) {
      red[(warp * 16 + g) * rc + 2 * q + 1] = yacc[1];
      red[(warp * 16 + g + 8) * rc + 2 * q + 1] = yacc[3];
    }
    partial_done(red_full, tcount, lane);
  }
}

// ===========================================================================
// ternary
// ===========================================================================
// A 640-code super-group (128 bytes, exactly 5 groups) is processed in 8
// rounds of 80 codes: in a round lane q of a quad takes word 4*round+q of
// its two rows, and digit md (0..4) of the word's 4 bytes feeds MMA md.
// Four rounds straddle a group edge (128 codes = 25.6 bytes); instead of a
// second MMA, B carries two columns per token: column 2t+side holds token
// t's x restricted to the groups of parity `side`, so one MMA accumulates
// both groups of a round apart.
// The byte table gives digit i at bits 2i..2i+1, used in place as mantissa
// bits j = 2i, 2i+1.
__host__ __device__ constexpr uint32_t mant_mask2(int j) { return (3u << j) | (3u << (j + 16)); }

// digit-1 operand of position MD in both halves: 2^-j + 2^-10, j = 2 MD
__host__ __device__ constexpr uint32_t ter_one(int md) {
  return exp_base(2 * md) | (1u << (2 * md)) | (1u << (2 * md + 16));
}

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// (c-1) * 2^-10 for the two codes of digit position MD: the offset operand
// 2^-j + d*2^-10 minus the digit-1 operand, exact (same exponent, Sterbenz)
template <int MD>
__device__ __forceinline__ uint32_t ter_operand(uint32_t f, const ExpRegs& E) {
  return hsub2_u32(and_or<mant_mask2(2 * MD)>(f, E.e[2 * MD]), E.one[MD]);
}

// group (0..4) of the super-group that the first / last code of round r falls in
__host__ __device__ constexpr int round_first_group(int r) { return (80 * r) >> 7; }
__host__ __device__ constexpr int round_last_group(int r) { return (80 * r + 79) >> 7; }

// the super-group's 8 rounds are split over kTerParts warps
constexpr int kTerParts = kTerWarps / 8;
static_assert(kTerParts == 2 || kTerParts == 4, "8 rounds over 2 or 4 warps");

struct TerDigits {
  uint32_t a01, a23, b01, b23;  // rows g (a) and g+8 (b), bytes (0,1) and (2,3)
};

// Rounds [R0, R0+N) of a super-group: all lookups first (their shared-memory
// latencies overlap), then the MMAs; a group is flushed after its last round
// in the range.
template <int R0, int N, typename Fetch, typename Round, typename Epi>
__device__ __forceinline__ void ter_range(Fetch& fetch, Round& round, Epi& epi) {
  TerDigits f[N];
#pragma unroll
  for (int i = 0; i < N; ++i) fetch(R0 + i, f[i]);
#pragma unroll
  for (int i = 0; i < N; ++i) {
    round(R0 + i, f[i]);
    if (round_last_group(R0 + i) != round_first_group(R0 + i)) epi(round_first_group(R0 + i));
  }
  epi(round_last_group(R0 + N - 1));
}

// Byte -> digits table, one copy per lane: digit i at bits 2i..2i+1. Entry e
// of lane l at e*ROW + l*4; ROW = 256 lets one PRMT build the address from
// the byte (64 KB, half of each row unused), ROW = 128 packs it into 32 KB
// (two instructions per address), for the many-token mode whose x tables
// are large. Independent of x, so it is built before the wait for the
// previous grid.
template <int ROW>
__device__ void build_byte_table(uint8_t* smem) {
  // one 16-byte piece (4 lanes' copies) per thread and store: 8 threads fill
  // an entry's 128 bytes, so a warp's stores cover 4 entries bank-free
  for (int t = threadIdx.x; t < 256 * 8; t += kTerWarps * 32) {
    const int e = t >> 3, piece = t & 7;
    uint32_t v = 0;
    if (e < 243) {
      int r = e;
#pragma unroll
      for (int i = 0; i < 5; ++i) { v |= uint32_t(r % 3) << (2 * i); r /= 3; }
    }
    reinterpret_cast<uint4*>(smem + e * ROW)[piece] = make_uint4(v, v, v, v);
  }
}

// x table: item (token, super-group, round, side, lane q) -> 10 words, the B
// pair (b0, b1) of each digit MMA, at token*stride + (item within the
// token)*48. An item covers the 20 consecutive codes 640 sg + 80 rnd + 20 q
// (bytes 4 (4 rnd + q) + 0..3), read from global memory as 5 x 8 bytes.
// CG: read x through L2 only. A plan step whose x another step of the same
// launch wrote needs it (this SM's L1 may hold older lines of that buffer);
// otherwise the ordinary cached loads are faster (neighbouring threads share
// sectors), and x was written before the launch.
template <bool CG>
__device__ void build_ternary_xtable(const Params& p, uint8_t* smem) {
  const int per_token = p.n_sg * 64;
  for (int t = threadIdx.x; t < p.m * per_token; t += kTerWarps * 32) {
    const int col = t / per_token, it = t - col * per_token;
    const int q = it & 3, side = (it >> 2) & 1, rnd = (it >> 3) & 7, sg = it >> 6;
    const int k0 = 640 * sg + 80 * rnd + 20 * q;
    uint32_t u[10];
#pragma unroll
    for (int i = 0; i < 5; ++i) {
      uint2 v = make_uint2(0, 0);
      if (k0 + 4 * i < p.k)  // k % 128 == 0: a 4-code piece is all in or all out
        v = CG ? __ldcg(reinterpret_cast<const uint2*>(p.x + (size_t)col * p.k + k0 + 4 * i))
               : *reinterpret_cast<const uint2*>(p.x + (size_t)col * p.k + k0 + 4 * i);
      u[2 * i] = v.x;
      u[2 * i + 1] = v.y;
    }
    // code c of the item (0..19): half (c & 1) of u[c >> 1]; it is kept if
    // its group within the super-group has parity `side`
    auto xh = [&](int c) -> uint32_t {
      const int kr = 80 * rnd + 20 * q + c;
      return (((kr >> 7) & 1) == side) ? (u[c >> 1] >> (16 * (c & 1))) & 0xFFFFu : 0u;
    };
    uint32_t e[12];
#pragma unroll
    for (int md = 0; md < 5; ++md) {
      e[2 * md] = xh(md) | (xh(5 + md) << 16);
      e[2 * md + 1] = xh(10 + md) | (xh(15 + md) << 16);
    }
    e[10] = e[11] = 0;
    uint4* dst = reinterpret_cast<uint4*>(smem + p.off_xt + col * p.xt_stride + it * kTerEntry);
    dst[0] = make_uint4(e[0], e[1], e[2], e[3]);
    dst[1] = make_uint4(e[4], e[5], e[6], e[7]);
    dst[2] = make_uint4(e[8], e[9], e[10], e[11]);
  }
}

// TOK8 = false: up to 4 tokens, B column 2t + side (the group-parity trick
// above). TOK8 = true: 5..8 tokens, B column t; a round that straddles a
// group edge issues its five MMAs once per side (x of the other side's
// groups is zero in that B) into separate accumulators, the others once.
// Consumer warps: the tiles of one product. The ring position (s, ph), the
// partial-sum slot counter and the timeout state carry over from product to
// product within a launch.
template <bool SC, bool TOK8>
__device__ void ternary_consume(const Params& p, uint8_t* smem, uint32_t bar_full,
                                uint32_t bar_empty, uint32_t red_full, int warp, int lane,
                                int& s, uint32_t& ph, int& tcount, bool& alive) {
  const int g = lane >> 2, q = lane & 3;
  // B column g: token g>>1, side g&1 (up to 4 tokens), or token g (TOK8)
  const bool bcol = (TOK8 ? g : (g >> 1)) < p.m;
  const uint8_t* xt_lane =
      TOK8 ? smem + p.off_xt + (bcol ? g : 0) * p.xt_stride + q * kTerEntry
           : smem + p.off_xt + (bcol ? (g >> 1) : 0) * p.xt_stride + ((g & 1) * 4 + q) * kTerEntry;
  const uint32_t lut_lane = uint32_t(lane * 4);
  const uint8_t* lut = smem;  // the byte table sits at offset 0
  const int pw = p.pitch >> 2;
  const int sgw = warp / kTerParts, part = warp % kTerParts;  // super-group of the chunk, rounds
  const ExpRegs E;
  uint4 b0 = make_uint4(0, 0, 0, 0), b1 = b0, b2 = b0;
  for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x, ++tcount) {
    const int row0 = tile * 16;
    // token q, rows g and g+8; TOK8: rows g, g+8 x tokens 2q, 2q+1
    float yacc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int c = 0; c < p.chunks; ++c) {
      const int len = min(kChunk, p.data_bytes - c * kChunk);
      const int nsg = (len + 127) >> 7;
      const int sg = c * (kChunk / 128) + sgw;
      const uint8_t* stage = smem + p.off_stage + s * p.stage_bytes;
      const uint32_t* stg = reinterpret_cast<const uint32_t*>(stage);
      if (wait_full(bar_full + 8 * s, ph, alive) && sgw < nsg) {
        const uint32_t* r0 = stg + g * pw + sgw * 32 + q;
        const uint32_t* r1 = stg + (g + 8) * pw + sgw * 32 + q;
        const uint8_t* xt = xt_lane + sg * (64 * kTerEntry);
        // acc: (row g, token q, side 0 / 1), (row g+8, token q, side 0 / 1);
        // TOK8: accs[side] = (row g, tokens 2q, 2q+1), (row g+8, same)
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        float accs[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        // the part of group grp held in this warp -> yacc; clears its side
        auto epi = [&](int grp) {
          const int side = grp & 1;
          const int gl = min(5 * sgw + grp, p.G - 1 - c * p.sc_chunk);  // group within the chunk
          const int gi = 5 * sg + grp;
          const float sa = scale_of<SC>(p, stage, g, row0 + g, gl, gi);
          const float sb = scale_of<SC>(p, stage, g + 8, row0 + g + 8, gl, gi);
          if constexpr (TOK8) {
            float(&a)[4] = accs[side];
            yacc[0] = fmaf(sa, a[0] * 1024.f, yacc[0]);
            yacc[1] = fmaf(sa, a[1] * 1024.f, yacc[1]);
            yacc[2] = fmaf(sb, a[2] * 1024.f, yacc[2]);
            yacc[3] = fmaf(sb, a[3] * 1024.f, yacc[3]);
            a[0] = a[1] = a[2] = a[3] = 0.f;
          } else {
            const float va = side ? acc[1] : acc[0];
            const float vb = side ? acc[3] : acc[2];
            yacc[0] = fmaf(sa, va * 1024.f, yacc[0]);
            yacc[1] = fmaf(sb, vb * 1024.f, yacc[1]);
            if (side) {
              acc[1] = 0.f;
              acc[3] = 0.f;
            } else {
              acc[0] = 0.f;
              acc[2] = 0.f;
            }
          }
        };
        // word loads and byte-table lookups of a round (digits of bytes (0,1)
        // and (2,3) side by side in the two halves)
        auto fetch = [&](int rnd, TerDigits& f) {
          const uint32_t wa = r0[4 * rnd], wb = r1[4 * rnd];
          auto lookup = [&](uint32_t wd, int i) -> uint32_t {
            uint32_t off;
            if constexpr (TOK8)  // byte * 128 + lane * 4
              off = ((i == 0 ? (wd << 7) : (wd >> (8 * i - 7))) & 0x7F80u) | lut_lane;
            else  // byte * 256 + lane * 4
              off = __byte_perm(wd, lut_lane, 0x5504 | (i << 4));
            return *reinterpret_cast<const uint32_t*>(lut + off);
          };
          f.a01 = __byte_perm(lookup(wa, 0), lookup(wa, 1), 0x5410);
          f.a23 = __byte_perm(lookup(wa, 2), lookup(wa, 3), 0x5410);
          f.b01 = __byte_perm(lookup(wb, 0), lookup(wb, 1), 0x5410);
          f.b23 = __byte_perm(lookup(wb, 2), lookup(wb, 3), 0x5410);
        };
        // the round's five digit MMAs
#define TER_MMA(D, MD, BX, BY)                                                  \
  mma_16816(D, ter_operand<MD>(f.a01, E), ter_operand<MD>(f.b01, E),            \
            ter_operand<MD>(f.a23, E), ter_operand<MD>(f.b23, E), BX, BY)
        auto round = [&](int rnd, const TerDigits& f) {
          if constexpr (TOK8) {
            // one pass per side that holds codes of this round
            for (int side = 0; side < 2; ++side) {
              const bool used = side == (round_first_group(rnd) & 1) ||
                                side == (round_last_group(rnd) & 1);
              if (!used) continue;
              const uint4* bp =
                  reinterpret_cast<const uint4*>(xt + (rnd * 8 + side * 4) * kTerEntry);
              if (bcol) {
                b0 = bp[0];
                b1 = bp[1];
                b2 = bp[2];
              } else {
                b0 = b1 = b2 = make_uint4(0, 0, 0, 0);
              }
              float(&a)[4] = accs[side];
              TER_MMA(a, 0, b0.x, b0.y);
              TER_MMA(a, 1, b0.z, b0.w);
              TER_MMA(a, 2, b1.x, b1.y);
              TER_MMA(a, 3, b1.z, b1.w);
              TER_MMA(a, 4, b2.x, b2.y);
            }
          } else {
            // only lanes of real tokens load x; the other columns are not stored
            const uint4* bp = reinterpret_cast<const uint4*>(xt + rnd * (8 * kTerEntry));
            if (bcol) {
              b0 = bp[0];
              b1 = bp[1];
              b2 = bp[2];
            }
            TER_MMA(acc, 0, b0.x, b0.y);
            TER_MMA(acc, 1, b0.z, b0.w);
            TER_MMA(acc, 2, b1.x, b1.y);
            TER_MMA(acc, 3, b1.z, b1.w);
            TER_MMA(acc, 4, b2.x, b2.y);
          }
        };
#undef TER_MMA
        // this warp's rounds of the super-group; a group is flushed after its
        // last round in the range
        if constexpr (kTerParts == 2) {
          if (part == 0) ter_range<0, 4>(fetch, round, epi);
          else ter_range<4, 4>(fetch, round, epi);
        } else {
          switch (part) {
            case 0: ter_range<0, 2>(fetch, round, epi); break;
            case 1: ter_range<2, 2>(fetch, round, epi); break;
            case 2: ter_range<4, 2>(fetch, round, epi); break;
            default: ter_range<6, 2>(fetch, round, epi); break;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
      if (++s == p.stages) { s = 0; ph ^= 1; }
    }
    float* red = partial_slot<kTerWarps>(p, smem, red_full, tcount, alive);
    const int rc = p.red_cols;  // only real tokens are kept
    if constexpr (TOK8) {  // token columns 2q, 2q+1
      if (2 * q < rc) {
        red[(warp * 16 + g) * rc + 2 * q] = yacc[0];
        red[(warp * 16 + g + 8) * rc + 2 * q] = yacc[2];
      }
      if (2 * q + 1 < rc) {
        red[(warp * 16 + g) * rc + 2 * q + 1] = yacc[1];
        red[(warp * 16 + g + 8) * rc + 2 * q + 1] = yacc[3];
      }
    } else if (q < rc) {  // token column q
      red[(warp * 16 + g) * rc + q] = yacc[0];
      red[(warp * 16 + g + 8) * rc + q] = yacc[1];
    }
    partial_done(red_full, tcount, lane);
  }
}


template <bool SC, bool TOK8>
__global__ void __launch_bounds__(threads_for(kTerWarps), 1)
    gemv_ternary_kernel(const __grid_constant__ CUtensorMap tmw,
                        const __grid_constant__ CUtensorMap tms, const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + p.off_bar, bar_empty = bar_full + 8 * kMaxStages;
  const uint32_t red_full = bar_full + 16 * kMaxStages;
  init_barriers<kTerWarps>(bar_full, bar_empty, p.stages);
  __syncthreads();
  pdl_launch_dependents();
  if (warp == kTerWarps) {
    if (lane == 0) produce(&tmw, &tms, p, sbase, bar_full, bar_empty);
    return;
  }
  if (warp == kTerWarps + 1) {
    reducer<kTerWarps>(p, smem, red_full, lane);
    return;
  }
  build_byte_table<TOK8 ? 128 : 256>(smem);
  pdl_wait();  // x is written by earlier work on the stream
  build_ternary_xtable<false>(p, smem);
  named_bar_sync(1, kTerWarps * 32);
  if (threadIdx.x == 0) mbar_arrive(x_ready_bar(bar_full));
  int s = 0, tcount = 0;
  uint32_t ph = 0;
  bool alive = true;
  ternary_consume<SC, TOK8>(p, smem, bar_full, bar_empty, red_full, warp, lane, s, ph, tcount,
                            alive);
}

// ===========================================================================
// a decode plan: many one-token ternary products in one persistent launch
// ===========================================================================
// Every weight is re-streamed per token ("第一の壁"), and a token of a deep
// decoder is hundreds of products; as separate launches each pays the
// launch, the dependency wait and the table prologue. Here one launch walks
// the products of a plan in order: the producer streams each product's tiles
// through the same ring without a break (weights are static, so it runs
// ahead into the next product), the consumers rebuild the x table per
// product, and the reducer counts each finished product in the plan's
// completion counters. A product whose x is another product's y waits (one
// thread, bounded) until every CTA has counted that product.
struct alignas(128) PlanStep {
  CUtensorMap tmw;  // packed weights (and scales) of the product
  CUtensorMap tms;
  Params p;         // the product's parameters, with the launch's shared geometry
  int after;        // earlier product whose y is this x, or -1
};

__device__ __forceinline__ unsigned int ld_acquire(const unsigned int* a) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}

// Waits until *c >= target; false if `limit_ns` of wall-clock time ran out.
__device__ bool wait_count(const unsigned int* c, unsigned int target,
                           uint64_t limit_ns = kWaitNs) {
  if (ld_acquire(c) >= target) return true;
  const uint64_t t0 = global_ns();
  while (ld_acquire(c) < target) {
    __nanosleep(200);
    if (global_ns() - t0 > limit_ns) return false;
  }
  return true;
}

__global__ void __launch_bounds__(threads_for(kTerWarps), 1)
    gemv_ternary_plan_kernel(const PlanStep* __restrict__ steps, int count, unsigned int* done,
                             const __grid_constant__ Params g) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + g.off_bar, bar_empty = bar_full + 8 * kMaxStages;
  const uint32_t red_full = bar_full + 16 * kMaxStages;
  init_barriers<kTerWarps>(bar_full, bar_empty, g.stages);
  __syncthreads();
  pdl_launch_dependents();
  if (warp == kTerWarps) {  // producer: all products' tiles through one ring
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      for (int j = 0; j < count; ++j) {
        const Params p = steps[j].p;
        // the descriptors live in global memory (written by the host before
        // the launch): acquire them for the tensor-map proxy
        asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(&steps[j].tmw)
                     : "memory");
        asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(&steps[j].tms)
                     : "memory");
        if (!produce_tiles(&steps[j].tmw, &steps[j].tms, p, sbase, bar_full, bar_empty, s, ph))
          break;
      }
    }
    return;
  }
  if (warp == kTerWarps + 1) {  // reducer: y of each product, then its count
    pdl_wait();
    int tcount = 0;
    bool ok = true;
    for (int j = 0; j < count; ++j) {
      const Params p = steps[j].p;
      if (ok) ok = reduce_tiles<kTerWarps>(p, smem, red_full, lane, tcount);
      __threadfence();  // this lane's stores of y before the count
      __syncwarp();
      if (lane == 0) atomicAdd(done + j, 1u);
    }
    named_bar_sync(2, (kTerWarps + 1) * 32);  // the consumers are past their last wait
    // the last CTA to finish resets the counters for the next run of the plan
    if (lane == 0 && atomicAdd(done + count, 1u) == gridDim.x - 1)
      for (int j = 0; j <= count; ++j) done[j] = 0u;
    return;
  }
  build_byte_table<256>(smem);
  pdl_wait();  // the first products' x may be written by earlier work on the stream
  int s = 0, tcount = 0;
  uint32_t ph = 0;
  bool alive = true, deps = true;  // after a wait runs out, later waits are skipped
  for (int j = 0; j < count; ++j) {
    const Params p = steps[j].p;
    const int after = steps[j].after;
    if (threadIdx.x == 0 && after >= 0 && deps && !wait_count(done + after, gridDim.x)) {
      set_status(BONSAI_ERR_TIMEOUT);
      deps = false;
    }
    named_bar_sync(1, kTerWarps * 32);  // also: every warp is done with the previous x table
    __threadfence();
    if (after >= 0) build_ternary_xtable<true>(p, smem);
    else build_ternary_xtable<false>(p, smem);
    named_bar_sync(1, kTerWarps * 32);
    if (p.sc_tma)
      ternary_consume<true, false>(p, smem, bar_full, bar_empty, red_full, warp, lane, s, ph,
                                   tcount, alive);
    else
      ternary_consume<false, false>(p, smem, bar_full, bar_empty, red_full, warp, lane, s, ph,
                                    tcount, alive);
  }
  named_bar_sync(2, (kTerWarps + 1) * 32);
}

// Self-test of the plan's dependency wait: one thread waits, with a limit of
// limit_ns, on a counter that nothing increments; the wait gives up and
// records BONSAI_ERR_TIMEOUT.
static __device__ unsigned int g_never_counted;  // stays 0

__global__ void plan_wait_selftest_kernel(uint64_t limit_ns) {
  if (!wait_count(&g_never_counted, 1u, limit_ns)) set_status(BONSAI_ERR_TIMEOUT);
}

// ===========================================================================
// binary, one token: subset-sum tables
// ===========================================================================
// For one token the products x . w of four consecutive codes take only 16
// values, sum_{i<4} (2 b_i - 1) x_i over the 16 bit patterns b of a nibble
// ("multiplication degenerates to addition and sign flip", 三值权重 page).
// The CTA tabulates them once per launch from x (FP32), and each nibble of a
// packed word then costs one table load and one add: no MMA and no operand
// construction. Lanes are rows: lane (r, h) of a warp takes row r of the
// 16-row tile and words 2h, 2h+1 of each 128-code group it handles, so at
// every step the 32 lanes read two 16-word tables (one per half-warp) and
// never conflict on a bank.
//
// Table layout, group g, position pos = 16 hp + j of the group (word
// pos >> 3, nibble pos & 7): entry e at byte
//   (g >> 1) * 4096 + j * 256 + (g & 1) * 128 + hp * 64 + 4 e.
// Half hp lands in banks 16 hp .. 16 hp + 15. The part below 256 of that
// offset, 4 e | 64 hp | 128 (g & 1), is the low byte of the address; it is
// built in the nibble extraction (one LOP3 per four nibbles), and one PRMT
// merges it with the 256-aligned group base; j * 256 is the load's
// immediate offset.
constexpr int kLutGroupBytes = 2048;   // table bytes per 128-code group
constexpr int kLutMaxGroups = 64;      // K <= 8192: at most 128 KB of tables

// The tables are written one 16-byte piece (4 entries) per thread and store:
// a table row (a group pair, position j) is 256 contiguous bytes, 16 pieces
// (group parity, half hp, entry block b), so the 32 lanes of a warp store
// two whole rows (512 contiguous bytes) and no two lanes of a wavefront share
// a bank. A thread's x loads (the four activations of its position, 8 bytes)
// are all issued before its first entry is computed, so the build waits on
// memory once.
constexpr int kLutBuildPasses = (kLutMaxGroups / 2 * 16 * 16 + kBinWarps * 32 - 1) / (kBinWarps * 32);

__device__ void build_nibble_tables(const Params& p, uint32_t tab) {
  const int rows = (p.G + 1) / 2 * 16;  // (group pair, position j)
  const int passes = (rows * 16 + kBinWarps * 32 - 1) / (kBinWarps * 32);  // uniform
  uint2 xv[kLutBuildPasses];
#pragma unroll
  for (int it = 0; it < kLutBuildPasses; ++it) {
    if (it >= passes) break;
    const int t = threadIdx.x + it * kBinWarps * 32;
    const int row = t >> 4, piece = t & 15;
    const int g = 2 * (row >> 4) + (piece >> 3), pos = 16 * ((piece >> 2) & 1) + (row & 15);
    xv[it] = (row < rows && g < p.G) ? *reinterpret_cast<const uint2*>(p.x + 128 * g + 4 * pos)
                                     : make_uint2(0, 0);
  }
#pragma unroll
  for (int it = 0; it < kLutBuildPasses; ++it) {
    if (it >= passes) break;
    const int t = threadIdx.x + it * kBinWarps * 32;
    const int row = t >> 4, piece = t & 15, b = piece & 3;
    if (row < rows) {
      const float x0 = __half2float(__ushort_as_half(uint16_t(xv[it].x & 0xFFFFu)));
      const float x1 = __half2float(__ushort_as_half(uint16_t(xv[it].x >> 16)));
      const float x2 = __half2float(__ushort_as_half(uint16_t(xv[it].y & 0xFFFFu)));
      const float x3 = __half2float(__ushort_as_half(uint16_t(xv[it].y >> 16)));
      // entries 4b .. 4b+3: index bit i set = code i is +1; codes 2,3 fixed by b
      const float hi = ((b & 1) ? x2 : -x2) + ((b & 2) ? x3 : -x3);
      // piece offset within the row = (g & 1) * 128 + hp * 64 + b * 16 = piece * 16
      asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(tab + 256 * row + 16 * piece),
                   "f"(-x0 - x1 + hi), "f"(x0 - x1 + hi), "f"(x1 - x0 + hi), "f"(x0 + x1 + hi)
                   : "memory");
    }
  }
}

__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

// The 8 nibbles of word w as table loads: t1 holds nibbles 0,2,4,6 and t2
// nibbles 1,3,5,7, each as 4 e | low address bits `lowbits`; J0 is the
// word's first position j (0 or 8).
template <int J0>
__device__ __forceinline__ void lut_word(uint32_t w, uint32_t lowbits, uint32_t base,
                                         float& a0, float& a1) {
  uint32_t t1, t2;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(t1) : "r"(w << 2), "r"(0x3C3C3C3Cu), "r"(lowbits));
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(t2) : "r"(w >> 2), "r"(0x3C3C3C3Cu), "r"(lowbits));
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const uint32_t ae = __byte_perm(t1, base, 0x7650 | b);   // nibble 2b
    const uint32_t ao = __byte_perm(t2, base, 0x7650 | b);   // nibble 2b + 1
    a0 += lds_f32(ae + (J0 + 2 * b) * 256);
    a1 += lds_f32(ao + (J0 + 2 * b + 1) * 256);
  }
}

template <bool SC>
__global__ void __launch_bounds__(threads_for(kBinWarps), 1)
    gemv_binary_lut_kernel(const __grid_constant__ CUtensorMap tmw,
                           const __grid_constant__ CUtensorMap tms,
                           const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + p.off_bar, bar_empty = bar_full + 8 * kMaxStages;
  const uint32_t red_full = bar_full + 16 * kMaxStages;
  const uint32_t tab = sbase + p.off_lut;
  if (tab & 255u) {  // the PRMT address merge needs 256-byte aligned group bases
    if (threadIdx.x == 0) set_status(BONSAI_ERR_UNSUPPORTED);
    return;
  }
  init_barriers<kBinWarps>(bar_full, bar_empty, p.stages);
  __syncthreads();
  pdl_launch_dependents();
  if (warp == kBinWarps) {
    if (lane == 0) produce(&tmw, &tms, p, sbase, bar_full, bar_empty);
    return;
  }
  if (warp == kBinWarps + 1) {
    reducer<kBinWarps>(p, smem, red_full, lane);
    return;
  }
  pdl_wait();  // x is written by earlier work on the stream
  build_nibble_tables(p, tab);
  named_bar_sync(1, kBinWarps * 32);
  if (threadIdx.x == 0) mbar_arrive(x_ready_bar(bar_full));

  const int r = lane & 15, h = lane >> 4;
  const int pw = p.pitch >> 2;
  const uint32_t hbits = h ? 0x40404040u : 0u;
  int s = 0;
  uint32_t ph = 0;
  bool alive = true;
  int tcount = 0;
  for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x, ++tcount) {
    const int row0 = tile * 16;
    float yacc = 0.f;
    for (int c = 0; c < p.chunks; ++c) {
      const int len = min(kChunk, p.data_bytes - c * kChunk);
      const int cg = len >> 4;  // 128-code groups in this chunk
      const uint8_t* stage = smem + p.off_stage + s * p.stage_bytes;
      const uint32_t* stg = reinterpret_cast<const uint32_t*>(stage);
      if (wait_full(bar_full + 8 * s, ph, alive)) {
        // groups gl = gs, gs + kBinWarps, ...; gs alternates between the two
        // halves of the warp range from tile to tile
        const int gs = (warp + (kBinWarps / 2) * (tcount & 1)) % kBinWarps;
        for (int gl = gs; gl < cg; gl += kBinWarps) {
          const int gi = c * (kChunk / 16) + gl;
          const uint4 wv = *reinterpret_cast<const uint4*>(stg + r * pw + gl * 4);
          const uint32_t w0 = h ? wv.z : wv.x, w1 = h ? wv.w : wv.y;
          const uint32_t lowbits = hbits | ((gi & 1) ? 0x80808080u : 0u);
          const uint32_t base = tab + (gi >> 1) * 4096;
          float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
          lut_word<0>(w0, lowbits, base, a0, a1);
          lut_word<8>(w1, lowbits, base, a2, a3);
          const float sc = scale_of<SC>(p, stage, r, row0 + r, gl, gi);
          yacc = fmaf(sc, (a0 + a1) + (a2 + a3), yacc);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
      if (++s == p.stages) { s = 0; ph ^= 1; }
    }
    yacc += __shfl_xor_sync(0xFFFFFFFFu, yacc, 16);  // words 0,1 + words 2,3
    float* red = partial_slot<kBinWarps>(p, smem, red_full, tcount, alive);
    if (h == 0) red[(warp * 16 + r) * p.red_cols] = yacc;
    partial_done(red_full, tcount, lane);
  }
}

}  // namespace gemv

// One launch for up to 8 binary / 4 ternary tokens. Returns UNSUPPORTED
// when the per-CTA tables do not fit in shared memory.
namespace gemv {
// A product ready to launch: parameters, tensor maps, shared memory, kernel.
struct Prepared {
  Params p;
  CUtensorMap tmw, tms;
  int smem;
  const void* fn;
  int threads;
};
}  // namespace gemv

// Parameters of one launch over w (tensor maps too when `maps`). Returns
// UNSUPPORTED when the per-CTA tables do not fit in shared memory.
static bonsai_status gemv_prepare(const bonsai_weights* w, const uint16_t* x, int m, uint16_t* y,
                                  bool swiglu, bool maps, gemv::Prepared& out) {
  using namespace gemv;
  Params& p = out.p;
  const bool ter = w->format == BONSAI_FMT_TERNARY;
  const int k = (int)w->k;
  const int n = (int)w->n;
  p = Params{};
  p.scales = reinterpret_cast<const __half*>(w->scales);
  p.x = reinterpret_cast<const __half*>(x);
  p.y = reinterpret_cast<__half*>(y);
  p.n = n;
  p.k = k;
  p.m = m;
  p.G = k / 128;
  p.prefetch = (w->flags & BONSAI_WEIGHTS_PREFETCH) ? 1 : 0;
  p.swiglu = swiglu ? 1 : 0;
  p.y_stride = swiglu ? n / 2 : n;
  if (!ter) {
    p.rows = 16;
    p.data_bytes = k / 8;
    p.xt_stride = p.G * 256 + 64;
  } else {
    p.rows = 16;
    p.data_bytes = (int)bonsai_packed_row_bytes(BONSAI_FMT_TERNARY, k);
    p.n_sg = (p.data_bytes + 127) / 128;
    p.xt_stride = p.n_sg * 64 * kTerEntry + 64;
  }
  p.chunks = (p.data_bytes + kChunk - 1) / kChunk;
  p.sc_chunk = ter ? kChunk * 5 / 128 : kChunk / 16;  // groups per chunk: 40 / 64
  p.sc_tma = (p.G % 8 == 0) ? 1 : 0;
  {
    int scp = (2 * p.sc_chunk + 15) / 16 * 16;
    if ((scp / 4) % 8 == 0) scp += 16;  // words = 4 mod 8: 8 rows hit 8 distinct banks
    p.sc_pitch = scp;
    const int chunk_max = p.data_bytes < kChunk ? p.data_bytes : kChunk;
    const int cw = chunk_max / 4;
    const int pw = ((cw - 4 + 31) / 32) * 32 + 4;  // >= cw words, = 4 mod 32
    p.pitch = pw * 4;
  }
  p.tiles = (n + p.rows - 1) / p.rows;
  p.stage_bytes = (16 * p.pitch + 16 * p.sc_pitch + 127) / 128 * 128;
  // one binary token with K <= 8192: the subset-sum kernel
  const bool lut = !ter && m == 1 && p.G <= kLutMaxGroups;

  auto up = [](int v, int a) { return (v + a - 1) / a * a; };
  int off = 0;
  p.off_lut = off;   // at 0: the kernels rely on it (1024-byte aligned)
  if (ter) off = up(off + (m > kTerMaxTokens ? kLutBytes8 : kLutBytes), 128);
  else if (lut) off = up(off + ((p.G + 1) / 2) * 2 * kLutGroupBytes, 128);
  p.off_bar = off;   off = up(off + 8 * kBarriers, 128);
  const int warps = ter ? kTerWarps : kBinWarps;
  p.red_cols = m;
  p.off_red = off;   off = up(off + 2 * warps * 16 * p.red_cols * 4, 128);
  p.off_t = off;     if (!ter && !lut) off = up(off + p.G * 8 * 4, 128);
  p.off_xt = off;    if (!lut) off = up(off + p.m * p.xt_stride, 1024);
  off = up(off, 1024);
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

  CUtensorMap& tmw = out.tmw;
  CUtensorMap& tms = out.tms;
  if (maps && !encode_tensor_map_2d(&tmw, CU_TENSOR_MAP_DATA_TYPE_UINT64, const_cast<void*>(w->packed),
                            (uint64_t)(w->row_bytes / 8), (uint64_t)n, (uint64_t)w->row_bytes,
                            (uint32_t)(p.pitch / 8), (uint32_t)p.rows, CU_TENSOR_MAP_SWIZZLE_NONE))
    return BONSAI_ERR_CUDA;
  tms = tmw;  // unused unless the scales are streamed
  if (maps && p.sc_tma &&
      !encode_tensor_map_2d(&tms, CU_TENSOR_MAP_DATA_TYPE_UINT16, const_cast<uint16_t*>(w->scales),
                            (uint64_t)p.G, (uint64_t)n, (uint64_t)p.G * 2,
                            (uint32_t)(p.sc_pitch / 2), (uint32_t)p.rows,
                            CU_TENSOR_MAP_SWIZZLE_NONE))
    return BONSAI_ERR_CUDA;

  const bool tok8 = ter && m > kTerMaxTokens;
  const void* fn = ter ? (tok8 ? (p.sc_tma ? (const void*)gemv_ternary_kernel<true, true>
                                           : (const void*)gemv_ternary_kernel<false, true>)
                               : (p.sc_tma ? (const void*)gemv_ternary_kernel<true, false>
                                           : (const void*)gemv_ternary_kernel<false, false>))
                 : lut ? (p.sc_tma ? (const void*)gemv_binary_lut_kernel<true>
                                   : (const void*)gemv_binary_lut_kernel<false>)
                       : (p.sc_tma ? (const void*)gemv_binary_kernel<true>
                                   : (const void*)gemv_binary_kernel<false>);
  out.smem = smem;
  out.fn = fn;
  out.threads = threads_for(warps);
  return BONSAI_OK;
}

static bonsai_status gemv_launch_one(const bonsai_weights* w, const uint16_t* x, int m,
                                     uint16_t* y, bool swiglu, cudaStream_t stream) {
  using namespace gemv;
  Prepared pr;
  const bonsai_status st = gemv_prepare(w, x, m, y, swiglu, true, pr);
  if (st != BONSAI_OK) return st;
  if (ensure_dynamic_smem(pr.fn, pr.smem) != cudaSuccess) return BONSAI_ERR_CUDA;
  const int sms = device_sm_count();
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(pr.p.tiles < sms ? pr.p.tiles : sms);
  cfg.blockDim = dim3(pr.threads);
  cfg.dynamicSmemBytes = pr.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&pr.tmw, &pr.tms, &pr.p};
  return cuda_status(cudaLaunchKernelExC(&cfg, pr.fn, args));
}

// Up to 8 tokens in one launch; ternary products of more than 4 tokens whose
// x tables do not fit beside the ring take two launches (4 + the rest).
bonsai_status gemv_launch(const bonsai_weights* w, const uint16_t* x, int64_t m, uint16_t* y,
                          bool swiglu, cudaStream_t stream) {
  if (m < 1 || m > 8) return BONSAI_ERR_UNSUPPORTED;
  if (w->format != BONSAI_FMT_TERNARY || m <= gemv::kTerMaxTokens)
    return gemv_launch_one(w, x, (int)m, y, swiglu, stream);
  {
    const bonsai_status st = gemv_launch_one(w, x, (int)m, y, swiglu, stream);
    if (st != BONSAI_ERR_UNSUPPORTED) return st;
  }
  const bonsai_status st = gemv_launch_one(w, x, gemv::kTerMaxTokens, y, swiglu, stream);
  if (st != BONSAI_OK) return st;
  const int64_t y_stride = swiglu ? w->n / 2 : w->n;
  return gemv_launch_one(w, x + gemv::kTerMaxTokens * w->k, (int)m - gemv::kTerMaxTokens,
                         y + gemv::kTerMaxTokens * y_stride, swiglu, stream);
}

// ------------------------------------------------------------------ plans
// Plan memory: count PlanStep records, then count + 1 counters (one per
// product, one for the CTAs that finished the run).
int64_t gemv_plan_bytes(int64_t count) {
  const int64_t b = count * (int64_t)sizeof(gemv::PlanStep) + 4 * (count + 1);
  return (b + 127) / 128 * 128;
}

// Parameters of every product of a plan (with tensor maps when `host` is
// given) and the launch's shared shared-memory geometry.
static bonsai_status gemv_plan_prepare(const bonsai_decode_step* steps, int64_t count,
                                       gemv::PlanStep* host, gemv::Params& g, int& smem) {
  using namespace gemv;
  auto up = [](int v, int a) { return (v + a - 1) / a * a; };
  int xt_max = 0, stage_max = 0;
  for (int64_t j = 0; j < count; ++j) {
    const bonsai_decode_step& st = steps[j];
    if (st.w.format != BONSAI_FMT_TERNARY) return BONSAI_ERR_FORMAT;
    Prepared pr;
    const bonsai_status e =
        gemv_prepare(&st.w, st.x, 1, st.y, st.swiglu != 0, host != nullptr, pr);
    if (e != BONSAI_OK) return e;
    xt_max = pr.p.xt_stride > xt_max ? pr.p.xt_stride : xt_max;
    stage_max = pr.p.stage_bytes > stage_max ? pr.p.stage_bytes : stage_max;
    if (host) {
      host[j].tmw = pr.tmw;
      host[j].tms = pr.tms;
      host[j].p = pr.p;
      host[j].after = st.after;
    }
    if (j == 0) g = pr.p;
  }
  // one layout for all products: byte table, barriers, one-token partial
  // slots, the largest x table, a ring of the largest stages
  int off = 0;
  g.off_lut = off;   off = up(off + kLutBytes, 128);
  g.off_bar = off;   off = up(off + 8 * kBarriers, 128);
  g.red_cols = 1;
  g.off_red = off;   off = up(off + 2 * kTerWarps * 16 * 4, 128);
  g.off_t = off;
  g.off_xt = off;    off = up(off + xt_max, 1024);
  g.off_stage = off;
  g.stage_bytes = stage_max;
  {
    const int room = (device_max_smem_optin() - off) / stage_max;
    int st = kStageBudget / stage_max;
    st = st < 3 ? 3 : (st > kMaxStages ? kMaxStages : st);
    g.stages = st < room ? st : room;
  }
  if (g.stages < 2) return BONSAI_ERR_UNSUPPORTED;
  smem = up(off + g.stages * g.stage_bytes, 128);
  if (host)
    for (int64_t j = 0; j < count; ++j) {
      Params& p = host[j].p;
      p.off_lut = g.off_lut; p.off_bar = g.off_bar; p.red_cols = g.red_cols;
      p.off_red = g.off_red; p.off_t = g.off_t; p.off_xt = g.off_xt;
      p.off_stage = g.off_stage; p.stage_bytes = g.stage_bytes; p.stages = g.stages;
      p.prefetch = 1;
    }
  return BONSAI_OK;
}

bonsai_status gemv_plan_init(const bonsai_decode_step* steps, int64_t count, void* plan,
                             cudaStream_t stream) {
  std::vector<gemv::PlanStep> host((size_t)count);
  gemv::Params g;
  int smem = 0;
  bonsai_status st = gemv_plan_prepare(steps, count, host.data(), g, smem);
  if (st != BONSAI_OK) return st;
  const size_t rec = (size_t)count * sizeof(gemv::PlanStep);
  // pageable source: the copy is staged before the call returns
  if (cudaMemcpyAsync(plan, host.data(), rec, cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return BONSAI_ERR_CUDA;
  return cuda_status(cudaMemsetAsync(static_cast<uint8_t*>(plan) + rec, 0,
                                     4 * (size_t)(count + 1), stream));
}

bonsai_status gemv_plan_run(const bonsai_decode_step* steps, int64_t count, void* plan,
                            cudaStream_t stream) {
  gemv::Params g;
  int smem = 0;
  bonsai_status st = gemv_plan_prepare(steps, count, nullptr, g, smem);
  if (st != BONSAI_OK) return st;
  const void* fn = (const void*)gemv::gemv_ternary_plan_kernel;
  if (ensure_dynamic_smem(fn, smem) != cudaSuccess) return BONSAI_ERR_CUDA;
  const gemv::PlanStep* recs = static_cast<const gemv::PlanStep*>(plan);
  unsigned int* done = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(plan) +
                                                       (size_t)count * sizeof(gemv::PlanStep));
  int cnt = (int)count;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(device_sm_count());  // every CTA takes part in every product
  cfg.blockDim = dim3(gemv::threads_for(gemv::kTerWarps));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&recs, &cnt, &done, &g};
  return cuda_status(cudaLaunchKernelExC(&cfg, fn, args));
}

bonsai_status plan_wait_selftest_launch(uint64_t limit_ns, cudaStream_t stream) {
  gemv::plan_wait_selftest_kernel<<<1, 1, 0, stream>>>(limit_ns);
  return cuda_status(cudaGetLastError());
}

}  // namespace bonsai
