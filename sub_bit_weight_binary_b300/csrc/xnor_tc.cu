// xnor_tc.cu -- the +-1 x +-1 product of bonsai_xnor_gemm on the tensor
// cores (tcgen05), bit-exact with the XOR + popcount definition
// ("1-bit 嘅數學": d = k - 2 * popcount(a XOR w)).
//
// A +-1 code is exact in FP16, so is a product of two of them, and an FP32
// accumulator holds every sum of up to 2^24 of them exactly: the tensor-core
// sum sum_k a*w IS k - 2 popc(a XOR w). The per-group scales of Y are exact
// too (s * (+-1) = +-s in FP16), so Y's MMA differs from D's only in the
// weight operand:
//   D[m][n] = sum_k a[m][k] w[n][k]                  (A = +-1)
//   Y[m][n] = a_s[m] * sum_k a[m][k] s[n][k/128] w[n][k]   (A = +-s)
//
// One persistent CTA per SM, 16 warps, tile = 128 features x 128 tokens:
//   warp 0      MMA issuer (one thread): per 64-code k-step, 4 MMAs
//               (M=128, N=128, K=16) into D and 4 into Y
//   warp 1      tensor-memory allocator (all 512 columns)
//   warps 4-7   per tile, first the activation expanders (one token row per
//               thread: 64 bits -> 64 FP16 +-1 in the 128-byte swizzled
//               K-major layout of a shared-memory B stage, the layout a TMA
//               load would give; the bits are loaded 4 k-steps ahead), then
//               the epilogue: tcgen05.ld of D and Y; D rounded to int32 (it
//               is an integer), Y times a_s[m] rounded once to FP16
//   warps 8-15  weight expanders: one feature row per thread, its 64 codes
//               as +-1 and +-s FP16 pairs written straight into tensor
//               memory (the A operand of the MMA), two groups for even and
//               odd k-steps, each loading its codes 4 own k-steps ahead
// Tensor memory: D in columns 0..127, Y in 128..255, then the A stages in
// the other 256 columns: 4 of 64 columns when both outputs are wanted (+-1
// codes in the first 32, +-s in the next 32), else 8 of 32; column c holds
// codes 2c, 2c+1 of the row, the lower code in the low half.
// Every mbarrier wait is bounded; a wait that runs out records
// BONSAI_ERR_TIMEOUT and the roles drain and leave.
#include "tcgen05.cuh"

namespace bonsai {
BONSAI_DEFINE_STATUS(g_status_xnor_tc)

unsigned int read_clear_status_xnor_tc() {
  unsigned int v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_status_xnor_tc, sizeof(v));
  cudaMemcpyToSymbol(g_status_xnor_tc, &z, sizeof(z));
  return v;
}

namespace xtc {

constexpr int TM = 128;       // features per tile (MMA M, tensor-memory lanes)
constexpr int TN = 128;       // tokens per tile (MMA N)
constexpr int BK = 64;        // codes per k-step: one 128-byte swizzle row of FP16
constexpr int THREADS = 512;
constexpr int A_STAGES = 8;   // in tensor memory: 8 of 32 columns (one output), 4 of 64 (both)
constexpr int B_STAGES = A_STAGES;  // in shared memory, 16 KB each; one ring index for A and B
constexpr int B_BYTES = TN * BK * 2;
constexpr int TMEM_COLS = 512;
constexpr int COL_D = 0, COL_Y = TN, COL_A = 2 * TN;
static_assert(COL_A + A_STAGES * 32 <= TMEM_COLS, "tensor memory holds D, Y and the A stages");
constexpr int W_MMA = 0, W_TMEM = 1, W_EPI = 4, W_AX = 8;
constexpr int B_AHEAD = 4;  // k-steps of activation bits loaded ahead
constexpr int W_AHEAD = 4;  // own k-steps of weight codes loaded ahead (one L2/DRAM round trip
                            // is longer than one own k-step)
constexpr int SMEM_BYTES = B_STAGES * B_BYTES + 256 + 1024;  // + barriers, + alignment slack

// Instruction descriptor, kind::f16: D=F32 (bits 4-5 = 1), A=B=F16, both
// K-major, N>>3 at bits 17-22, M>>4 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (uint32_t(TN >> 3) << 17) | (uint32_t(TM >> 4) << 24);

struct Params {
  const uint32_t* a_bits;  // [m][k/32]
  const __half* a_scale;   // [m]
  const uint8_t* w;        // [n][row_bytes]
  const __half* scales;    // [n][k/128]
  int32_t* d;              // [m][n] or null
  __half* y;               // [m][n] or null
  long long row_bytes;
  int m, n, k, G, nk;
  int tok_tiles, tiles;
  int prefetch;  // the weights may be read before the previous grid completes
};

// A from tensor memory, B from shared memory.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

#define TMEM_ST_16(taddr, v)                                                              \
  asm volatile(                                                                           \
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,"  \
      "%12,%13,%14,%15,%16};" ::"r"(taddr),                                                \
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),         \
      "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]),     \
      "r"(v[14]), "r"(v[15])                                                               \
      : "memory")

#define TMEM_ST_32(taddr, v)                                                              \
  asm volatile(                                                                           \
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,"  \
      "%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"   \
      "%32};" ::"r"(taddr),                                                               \
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),         \
      "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]),     \
      "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]),  \
      "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),  \
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])                                       \
      : "memory")

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Sign masks of the code pair (2i, 2i+1) of the complemented bits nb (bit
// set = code -1): 0x8000 in a half whose code is -1. XOR with the pair of
// magnitudes (+1 = 0x3C00, or the FP16 scale) gives the signed pair.
__device__ __forceinline__ uint32_t sign_pair(uint32_t nb, int i) {
  return (((nb >> (2 * i)) & 3u) * 0x40008000u) & 0x80008000u;
}

// D and Y of a tile from tensor memory: its 16-token chunks grp, grp + ngrp,
// ... read by this warp's lane quarter. On a CTA's last tile the epilogue
// warps (grp 0) share the chunks with the two weight-expander groups, which
// have no k-steps left (with one tile per CTA the whole epilogue is
// otherwise exposed). acc_empty (not 0): arrived on after this warp's last
// tensor-memory load.
__device__ __forceinline__ void store_dy(const Params& p, int tile, uint32_t tmem_base, int grp,
                                         int ngrp, uint32_t acc_empty) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, quarter = warp & 3;
  const bool do_d = p.d != nullptr, do_y = p.y != nullptr;
  const int n0 = (tile / p.tok_tiles) * TM, m0 = (tile % p.tok_tiles) * TN;
  const int feat = n0 + 32 * quarter + lane;
  const bool fok = feat < p.n;
  const int chunks = (p.m - m0 + 15) / 16 < TN / 16 ? (p.m - m0 + 15) / 16 : TN / 16;
  const int last = grp < chunks ? grp + (chunks - 1 - grp) / ngrp * ngrp : -1;
  const uint32_t tl = tmem_base + ((uint32_t)(32 * quarter) << 16);
#pragma unroll 1
  for (int c = grp; c < chunks; c += ngrp) {
    uint32_t vd[16], vy[16];
    if (do_d) TMEM_LD_16(tl + COL_D + 16 * c, vd);
    if (do_y) TMEM_LD_16(tl + COL_Y + 16 * c, vy);
    tmem_ld_wait();
    if (c == last && acc_empty) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
    }
    if (!fok) continue;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int tok = m0 + 16 * c + j;
      if (tok >= p.m) break;
      if (do_d) p.d[(size_t)tok * p.n + feat] = __float2int_rn(__uint_as_float(vd[j]));
      if (do_y)
        p.y[(size_t)tok * p.n + feat] =
            __float2half_rn(__half2float(p.a_scale[tok]) * __uint_as_float(vy[j]));
    }
  }
  if (last < 0 && acc_empty) {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(acc_empty);
  }
}

__global__ void __launch_bounds__(THREADS, 1) xnor_tc_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  // the swizzled B stages need 1024-byte alignment
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sB = (raw + 1023u) & ~1023u;
  const uint32_t sBar = sB + B_STAGES * B_BYTES;
  // One ring for both operands (stage s of the A stages in tensor memory and
  // of the B stages in shared memory hold the same k-step): full[s] gets the
  // 4 weight-expander warps of the k-step's group and the 4 activation
  // expanders, empty[s] one commit. One wait and one commit per k-step for
  // the MMA thread (each commit costs ~85 cycles of its issue).
  const uint32_t full = sBar, empty = full + 8 * A_STAGES;
  const uint32_t acc_full = empty + 8 * A_STAGES, acc_empty = acc_full + 8;
  const uint32_t drain = acc_empty + 8, tmem_slot = drain + 8;
  // the epilogue warps arrive once the CTA's last accumulator is complete;
  // the weight expanders wait on it (once) before they help store it (not
  // on acc_full: they may finish their k-steps two accumulator phases ahead)
  const uint32_t help_bar = tmem_slot + 8;
  static_assert(8 * (2 * A_STAGES + 5) <= 256, "barrier area");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool do_d = p.d != nullptr, do_y = p.y != nullptr;
  // A stages: 32 columns per wanted output (+-1 codes first, then +-s)
  const int a_cols = (do_d && do_y) ? 64 : 32;
  const int a_stages = (TMEM_COLS - COL_A) / a_cols;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a_stages; ++s) {
      mbar_init(full + 8 * s, 8);  // 4 weight expanders (the k-step's group) + 4 activation expanders
      mbar_init(empty + 8 * s, 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 4);
    mbar_init(drain, 1);
    mbar_init(help_bar, 4);
    fence_barrier_init();
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

  if (warp == W_MMA) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      pdl_wait();
      uint32_t ga = 0, gb = 0, it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x, ++it) {
        if (!mbar_wait(acc_empty, (it & 1) ^ 1)) { set_status(BONSAI_ERR_TIMEOUT); break; }
        tc_fence_after();
        for (int kk = 0; kk < p.nk; ++kk, ++ga, ++gb) {
          const int sa = ga % a_stages, sb = sa;
          if (!mbar_wait(full + 8 * sa, (ga / a_stages) & 1)) {
            set_status(BONSAI_ERR_TIMEOUT);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bd = smem_desc_sw128(sB + sb * B_BYTES);
          const uint32_t a_u = tmem_base + COL_A + a_cols * sa, a_s = a_u + (do_d ? 32 : 0);
#pragma unroll
          for (int k4 = 0; k4 < BK / 16; ++k4) {  // K=16: 8 A columns, 32 B bytes
            if (do_d) mma_f16_ts(tmem_base + COL_D, a_u + 8 * k4, bd + 2 * k4, kIdesc, (kk | k4) != 0);
            if (do_y) mma_f16_ts(tmem_base + COL_Y, a_s + 8 * k4, bd + 2 * k4, kIdesc, (kk | k4) != 0);
          }
          mma_commit(empty + 8 * sa);
        }
        if (ok) mma_commit(acc_full);
      }
      mma_commit(drain);
      if (!mbar_wait(drain, 0)) set_status(BONSAI_ERR_TIMEOUT);
    }
  } else if (warp >= W_AX) {
    // ---------------------------- weight expanders ----------------------------
    const int ax = warp - W_AX;          // 0..7
    const uint32_t h = ax >> 2;          // group: even / odd k-steps
    const int q = warp & 3;              // tensor-memory lane quarter
    const int r = 32 * q + lane;         // feature row of the tile
    if (!p.prefetch) pdl_wait();
    bool ok = true;
    // codes and scale of an own k-step (zeros past the last tile or row)
    auto load = [&](int tile, int kk, uint2& wv, uint32_t& sc) {
      const int n = (tile / p.tok_tiles) * TM + r;
      const bool nok = n < p.n && tile < p.tiles && kk < p.nk;
      wv = nok ? *reinterpret_cast<const uint2*>(p.w + (long long)n * p.row_bytes + 8 * kk)
               : make_uint2(0u, 0u);
      sc = nok ? uint32_t(__half_as_ushort(p.scales[(size_t)n * p.G + (kk >> 1)])) * 0x10001u : 0u;
    };
    // this thread's k-steps in order: every tile's kk = h, h + 2, ... (nk is
    // even, so g % 2 == kk % 2); (t_ld, k_ld) is the next one to load
    int t_ld = blockIdx.x, k_ld = (int)h;
    auto advance = [&]() {
      k_ld += 2;
      if (k_ld >= p.nk) { k_ld -= p.nk; t_ld += gridDim.x; }
    };
    uint2 ring_w[W_AHEAD];
    uint32_t ring_s[W_AHEAD];
#pragma unroll
    for (int i = 0; i < W_AHEAD; ++i) { load(t_ld, k_ld, ring_w[i], ring_s[i]); advance(); }
    for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x) {
      const int n = (tile / p.tok_tiles) * TM + r;
      const bool nok = n < p.n;
      const uint32_t one = nok ? 0x3C003C00u : 0u;  // rows past n give zeros
      for (int kk = (int)h; kk < p.nk; kk += 2) {
        const uint32_t g = (uint32_t)((tile - (int)blockIdx.x) / (int)gridDim.x) * p.nk + kk;
        const int s = g % a_stages;
        uint2 wv = ring_w[0];
        uint32_t sc = ring_s[0];
        // the ring rotates by one: static indices only (no local memory)
#pragma unroll
        for (int i = 0; i < W_AHEAD - 1; ++i) { ring_w[i] = ring_w[i + 1]; ring_s[i] = ring_s[i + 1]; }
        load(t_ld, k_ld, ring_w[W_AHEAD - 1], ring_s[W_AHEAD - 1]);
        advance();
        if (!mbar_wait(empty + 8 * s, ((g / a_stages) & 1) ^ 1)) {
          set_status(BONSAI_ERR_TIMEOUT);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ta = tmem_base + ((uint32_t)(32 * q) << 16) + COL_A + a_cols * s;
        // 16 columns (32 codes) at a time
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint32_t bits = ~(half ? wv.y : wv.x);
          uint32_t v[16];
          if (do_d) {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = sign_pair(bits >> (2 * j), 0) ^ one;
            TMEM_ST_16(ta + 16 * half, v);
          }
          if (do_y) {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = sign_pair(bits >> (2 * j), 0) ^ sc;
            TMEM_ST_16(ta + (do_d ? 32 : 0) + 16 * half, v);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(full + 8 * s);
      }
    }
    // no k-steps left: help store this CTA's last tile
    if (ok && (int)blockIdx.x < p.tiles) {
      const int last = (int)blockIdx.x + (p.tiles - 1 - (int)blockIdx.x) / (int)gridDim.x * (int)gridDim.x;
      if (!mbar_wait(help_bar, 0)) {
        set_status(BONSAI_ERR_TIMEOUT);
      } else {
        tc_fence_after();
        store_dy(p, last, tmem_base, 1 + (int)h, 3, 0);
      }
    }
  } else if (warp >= W_EPI && warp < W_EPI + 4) {
    // ------------------------------- epilogue -------------------------------
    pdl_wait();
    const int e = warp - W_EPI;  // tensor-memory lanes 32e .. 32e+31
    const int r = 32 * e + lane; // token row of the B stages
    const int words = p.k / 32;
    uint32_t it = 0, gb = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x, ++it) {
      // ---- activation expansion for the whole tile
      {
        const int m0 = (tile % p.tok_tiles) * TN;
        const bool real = m0 + r < p.m;
        const uint2* src = reinterpret_cast<const uint2*>(p.a_bits + (size_t)(real ? m0 + r : 0) * words);
        const uint32_t one = real ? 0x3C003C00u : 0u;  // rows past m hold zeros
        uint2 pre[B_AHEAD];
#pragma unroll
        for (int i = 0; i < B_AHEAD; ++i) pre[i] = real && i < p.nk ? src[i] : make_uint2(0u, 0u);
        for (int k0 = 0; k0 < p.nk && ok; k0 += B_AHEAD) {
#pragma unroll
          for (int i = 0; i < B_AHEAD; ++i) {
            const int kk = k0 + i;
            if (kk >= p.nk) break;
            const uint2 bits = pre[i];
            pre[i] = real && kk + B_AHEAD < p.nk ? src[kk + B_AHEAD] : make_uint2(0u, 0u);
            const int s = gb % a_stages;
            if (!mbar_wait(empty + 8 * s, ((gb / a_stages) & 1) ^ 1)) {
              set_status(BONSAI_ERR_TIMEOUT);
              ok = false;
              break;
            }
            const uint32_t dst_row = sB + s * B_BYTES + r * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {  // 16-byte chunk c: codes 8c .. 8c+7
              const uint32_t nb = ~(c < 4 ? bits.x : bits.y) >> (8 * (c & 3));
              sts128(dst_row + ((c ^ (r & 7)) << 4), sign_pair(nb, 0) ^ one, sign_pair(nb, 1) ^ one,
                     sign_pair(nb, 2) ^ one, sign_pair(nb, 3) ^ one);
            }
            fence_proxy_async_smem();  // generic-proxy stores -> tensor-core reads
            __syncwarp();
            if (lane == 0) mbar_arrive(full + 8 * s);
            ++gb;
          }
        }
      }
      if (!ok) break;
      // ---- epilogue of the tile
      if (!mbar_wait(acc_full, it & 1)) { set_status(BONSAI_ERR_TIMEOUT); break; }
      tc_fence_after();
      const bool last_tile = tile + (int)gridDim.x >= p.tiles;
      if (last_tile) {  // the weight expanders may help
        __syncwarp();
        if (lane == 0) mbar_arrive(help_bar);
      }
      store_dy(p, tile, tmem_base, 0, last_tile ? 3 : 1, acc_empty);
    }
  }

  pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == W_TMEM) tmem_dealloc(tmem_base, TMEM_COLS);
}

}  // namespace xtc

bonsai_status xnor_tc_launch(const uint32_t* a_bits, const uint16_t* a_scale, int64_t m,
                             const bonsai_weights* w, int32_t* d_out, uint16_t* y_out,
                             cudaStream_t stream) {
  using namespace xtc;
  if (m > 0x7FFFFFFF / 2 || w->k > (1LL << 24)) return BONSAI_ERR_UNSUPPORTED;
  if (SMEM_BYTES > device_max_smem_optin()) return BONSAI_ERR_UNSUPPORTED;
  Params p{};
  p.a_bits = a_bits;
  p.a_scale = reinterpret_cast<const __half*>(a_scale);
  p.w = static_cast<const uint8_t*>(w->packed);
  p.scales = reinterpret_cast<const __half*>(w->scales);
  p.d = d_out;
  p.y = reinterpret_cast<__half*>(y_out);
  p.row_bytes = w->row_bytes;
  p.m = (int)m;
  p.n = (int)w->n;
  p.k = (int)w->k;
  p.G = p.k / 128;
  p.nk = p.k / BK;
  p.tok_tiles = (int)((m + TN - 1) / TN);
  const long long tiles = ((w->n + TM - 1) / TM) * (long long)p.tok_tiles;
  if (tiles > 0x7FFFFFFF) return BONSAI_ERR_UNSUPPORTED;
  p.tiles = (int)tiles;
  p.prefetch = (w->flags & BONSAI_WEIGHTS_PREFETCH) ? 1 : 0;
  if (ensure_dynamic_smem((const void*)xnor_tc_kernel, SMEM_BYTES) != cudaSuccess)
    return BONSAI_ERR_CUDA;
  const int sms = device_sm_count();
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p.tiles < sms ? p.tiles : sms);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&p};
  return cuda_status(cudaLaunchKernelExC(&cfg, (const void*)xnor_tc_kernel, args));
}

}  // namespace bonsai
