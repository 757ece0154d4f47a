// gemv_lut.cu -- one-token decode product (ternary, and binary at the end of
// the file) through per-position tables of partial sums, with K split
// across thread blocks.
//
// "Multiplication degenerates to addition and sign flip" (三值权重 page): a
// packed byte holds five codes, so x . w over those five codes is one of 243
// numbers fixed by x alone. The kernel tabulates them in FP32 for every byte
// position of a slice of K, and each byte of each row then costs one table
// load and one add; no code is expanded into an operand.
//
// Structure (sm_103a):
//  * K is cut into slices of 640 codes (128 packed bytes, five whole 128-code
//    groups); the rows into C chunks. One CTA per (chunk, slice), at most one
//    per SM, 16 warps.
//  * Tables, one bank per lane: lane p handles bytes 4p..4p+3 of every row
//    (one 32-bit word), and the table of byte 4p+j is stored entry-major with
//    entry e of lane p at e*256 + (j&1)*128 + 4p in table pair j>>1, so the
//    32 lookups of a warp hit 32 banks. One PRMT puts the byte into bits
//    8..15, one add gives the address, one LDS fetches the FP32 sum.
//  * Group scales (one FP16 per 128 codes, OpenBonsai page, "工作原理"): the
//    slice's group edges fall inside bytes 25, 51, 76 and 102. The table of
//    such a byte holds only its codes below the edge; its codes above the
//    edge are looked up in a small table by the byte's upper base-3 digits
//    (index = byte / 3^k, a multiply-high). The lane adds them, with any
//    later bytes of its word (all above the edge), into a hand-over sum that
//    the next lane (whose four bytes are all in the upper group) takes with
//    one shuffle. So every lane multiplies by exactly one scale per row.
//  * Streaming: a row's slice is only 128 bytes, and a 2-D TMA box of such
//    short rows costs the copy engine far more per byte than wide boxes
//    (measured: ~190 ns per 8-row stage from one issuing thread). So every
//    warp streams its own stages (8 rows of weights and their scales) with
//    16-byte cp.async copies into four private ring slots, three stages
//    ahead of the one it reads; warp w takes stages w, w+16, ...
//  * A warp sums its 8 rows' lane values with a transposed butterfly and
//    stores one FP32 partial per (row, slice) in the caller's workspace.
//    The chunk's rows are split into S parts with one arrival counter each;
//    the CTA that completes a part adds its S partials in slice order (the
//    same order every call) and writes FP16 y, or silu(g)*u for a gated
//    feed-forward weight, then re-arms the counter.
#include "common.cuh"

namespace bonsai {
BONSAI_DEFINE_STATUS(g_status_lut)

unsigned int read_clear_status_lut() {
  unsigned int v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_status_lut, sizeof(v));
  cudaMemcpyToSymbol(g_status_lut, &z, sizeof(z));
  return v;
}

namespace lut {

constexpr int kWarps = 16;  // every warp streams its own rows
constexpr int kThreads = kWarps * 32;
constexpr int kRows = 8;           // rows per stage
constexpr int kDepth = 3;          // a warp's stages in flight beyond the one it reads
constexpr int kWarpSlots = kDepth + 1;
constexpr int kSlots = kWarps * kWarpSlots;
constexpr int kSliceBytes = 128;   // packed bytes per row per slice
constexpr int kSliceCodes = 640;
constexpr int kStageW = kRows * kSliceBytes;  // weights of a stage
constexpr int kScaleRow = 32;                 // 16 scales per row and stage
constexpr int kStageBytes = kStageW + kRows * kScaleRow;
constexpr int kEntries = 256;                 // 243 byte values; 256 keeps any byte in bounds
constexpr int kPairBytes = kEntries * 256;    // two byte positions per 256-byte table row
constexpr int kHRows = 86;                    // upper-digit table rows (255 / 3 + 1)
constexpr int kMaxSlices = 160;

constexpr int kOffT = 0;
constexpr int kOffH = kOffT + 2 * kPairBytes;
constexpr int kOffX = kOffH + kHRows * 128;
constexpr int kOffFlags = kOffX + kSliceCodes * 4;
constexpr int kOffRing = kOffFlags + kMaxSlices * 4;
constexpr int kSmem = kOffRing + kSlots * kStageBytes;
static_assert(kOffRing % 128 == 0, "ring stages are 128-byte aligned");
static_assert(kSmem <= 232448, "fits the opt-in shared memory of one SM");

struct Params {
  const uint8_t* packed;
  const __half* scales;
  const __half* x;
  __half* y;
  float* ws;          // partial sums [chunk][slice][rc]
  unsigned int* cnt;  // arrival counters [chunk][part]
  long long row_bytes;
  int n, k, G, S, C, rc, part_rows;
  int prefetch, swiglu;
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
// Shared-memory reads by 32-bit shared address. Not volatile, so the
// compiler may schedule them freely across the unrolled rows; the reads of a
// ring stage take their address from a value produced after the stage's
// copies were waited for (opaque_zero), which keeps them behind that wait.
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
  uint32_t v;
  asm("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float lds_f32(uint32_t a) {
  float v;
  asm("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float lds_h2f(uint32_t a) {
  unsigned short v;
  asm("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return __half2float(__ushort_as_half(v));
}
__device__ __forceinline__ uint32_t opaque_zero() {
  uint32_t z;
  asm volatile("mov.u32 %0, 0;" : "=r"(z)::"memory");
  return z;
}

// 16-byte asynchronous copy global -> shared; with src_bytes 0 the 16 bytes
// are zero-filled and nothing is read.
__device__ __forceinline__ void cp16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// The four bytes whose codes cross a group edge inside one slice, as
// (lane, byte of the lane's word, digits below the edge): bytes 25, 51, 76
// and 102 hold codes 125..129, 255..259, 380..384 and 510..514.
__host__ __device__ constexpr int edge_byte(int lane) {
  return lane == 6 ? 1 : lane == 12 ? 3 : lane == 19 ? 0 : lane == 25 ? 2 : -1;
}
__host__ __device__ constexpr int edge_low_digits(int lane) {
  return lane == 6 ? 3 : lane == 12 ? 1 : lane == 19 ? 4 : lane == 25 ? 2 : 0;
}

// A warp's copies of one stage (8 rows x 128 bytes of weights, and the 8
// rows' 16-group scale window from group sx) into a ring slot: two 16-byte
// pieces of weights per lane (rows r and r+4, piece col of the row's slice),
// one piece of scales for lanes 0..15. The per-lane offsets are fixed for
// the kernel; bytes past the row and groups past k/128 read as zero, and
// rows past n re-read row n-1 (their sums are never used).
struct StageCopy {
  const uint8_t* w;      // weights of row 0 of the chunk, at this lane's piece
  const __half* sc;      // scales of row 0 of the chunk, at this lane's piece
  long long row_bytes;
  int G, n, r_w, r_s;
  uint32_t wbytes, sbytes, dw, ds;

  __device__ __forceinline__ StageCopy(const Params& p, int row0, int s, int sx, int lane) {
    const int col = lane & 7;
    r_w = lane >> 3;
    r_s = lane >> 1;
    const long long off = (long long)s * kSliceBytes + 16 * col;
    wbytes = off < p.row_bytes ? 16u : 0u;
    w = p.packed + (size_t)row0 * p.row_bytes + (wbytes ? off : 0);
    const int g0 = sx + 8 * (lane & 1);
    sbytes = (lane < 16 && g0 < p.G) ? 16u : 0u;
    sc = p.scales + (size_t)row0 * p.G + (g0 < p.G ? g0 : 0);
    row_bytes = p.row_bytes;
    G = p.G;
    n = p.n - row0;  // rows of the chunk that exist (and beyond)
    dw = r_w * kSliceBytes + 16 * col;
    ds = kStageW + (r_s & 7) * kScaleRow + 16 * (lane & 1);
  }
  // stage i: rows 8i .. 8i+7 of the chunk
  __device__ __forceinline__ void issue(uint32_t dst, int i, int lane) const {
    int ra = kRows * i + r_w, rb = ra + 4, rs = kRows * i + (r_s & 7);
    if (kRows * i + kRows > n) {
      ra = min(ra, n - 1);
      rb = min(rb, n - 1);
      rs = min(rs, n - 1);
    }
    cp16(dst + dw, w + (size_t)ra * row_bytes, wbytes);
    cp16(dst + dw + 4 * kSliceBytes, w + (size_t)rb * row_bytes, wbytes);
    if (lane < 16) cp16(dst + ds, sc + (size_t)rs * G, sbytes);
  }
};

// Tables of the CTA's slice from x (FP32, zero past K). T: for the 128 byte
// positions, every byte value's sum over the codes below the position's
// group edge (all five codes but for the four edge bytes); H: for the edge
// bytes, the sum over the codes above the edge by the upper digits (row 0
// of the other lanes is zero: their index is always 0). Both with the same
// unrolled code: a byte value (or upper-digit index) e = a + 27*b, digits
// 0..2 in a and digits 3..4 in b, sums A[a] + B[b].
__device__ __forceinline__ void table_rows(float* dst, int stride, const float (&xv)[5], int q,
                                           int limit) {
  float A[27];
#pragma unroll
  for (int a = 0; a < 27; ++a) {
    const int d0 = a % 3, d1 = (a / 3) % 3, d2 = a / 9;
    float v = d0 == 0 ? -xv[0] : d0 == 2 ? xv[0] : 0.f;
    v += d1 == 0 ? -xv[1] : d1 == 2 ? xv[1] : 0.f;
    v += d2 == 0 ? -xv[2] : d2 == 2 ? xv[2] : 0.f;
    A[a] = v;
  }
  for (int b = q; 27 * b < limit; b += 4) {
    const int d3 = b % 3, d4 = b / 3;
    const float B = (d3 == 0 ? -xv[3] : d3 == 2 ? xv[3] : 0.f) +
                    (d4 == 0 ? -xv[4] : d4 == 2 ? xv[4] : 0.f);
    float* rb = dst + 27 * stride * b;
#pragma unroll
    for (int a = 0; a < 27; ++a)
      if (27 * b + a < limit) rb[a * stride] = A[a] + B;
  }
}

__device__ __forceinline__ void build_tables(const Params& p, uint8_t* smem, int s) {
  float* xs = reinterpret_cast<float*>(smem + kOffX);
  const int t = threadIdx.x;
  for (int i = t; i < kSliceCodes; i += kThreads) {
    const int kk = s * kSliceCodes + i;
    xs[i] = kk < p.k ? __half2float(p.x[kk]) : 0.f;
  }
  if (t < 32 && edge_byte(t) < 0) reinterpret_cast<float*>(smem + kOffH)[t] = 0.f;
  __syncthreads();
  const int pos = t & 127, q = t >> 7;
  const int pj = pos >> 5, pl = pos & 31;
  const int byte = 4 * pl + pj;
  const bool edge = edge_byte(pl) == pj;
  const int nd = edge ? edge_low_digits(pl) : 5;
  float xv[5];
#pragma unroll
  for (int i = 0; i < 5; ++i) xv[i] = i < nd ? xs[5 * byte + i] : 0.f;
  table_rows(reinterpret_cast<float*>(smem + kOffT + (pj >> 1) * kPairBytes + (pj & 1) * 128) + pl,
             64, xv, q, 243);
  if (edge) {  // the codes above the edge, as digits 0.. of the index
#pragma unroll
    for (int i = 0; i < 5; ++i) xv[i] = i + nd < 5 ? xs[5 * byte + nd + i] : 0.f;
    const int lim = nd == 1 ? 81 : nd == 2 ? 27 : nd == 3 ? 9 : 3;
    table_rows(reinterpret_cast<float*>(smem + kOffH) + pl, 32, xv, q, lim);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    gemv_ter_lut_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const int s = blockIdx.x % p.S, c = blockIdx.x / p.S;
  const int row0 = c * p.rc;
  const int rows = min(p.rc, p.n - row0);
  const int nst = (rows + kRows - 1) / kRows;
  const int mine = nst > warp ? (nst - warp + kWarps - 1) / kWarps : 0;  // stages warp, warp+16, ..
  const int sx = 8 * ((5 * s) / 8);  // first group of the 16-byte aligned scale window
  const uint32_t ring = sbase + kOffRing + warp * kWarpSlots * kStageBytes;
  pdl_launch_dependents();

  // weights never depend on earlier work on the stream: with the prefetch
  // flag the first stages stream in while the previous kernel finishes
  const StageCopy cpy(p, row0, s, sx, lane);
  if (!p.prefetch) pdl_wait();
  for (int d = 0; d < kDepth; ++d) {
    if (d < mine) cpy.issue(ring + d * kStageBytes, warp + kWarps * d, lane);
    cp_commit();
  }

  // lane constants
  const int js = edge_byte(lane);
  // upper-digit index byte / 3^k as the high word of byte * ceil(2^16 / 3^k) * 2^16
  const uint32_t magic = (lane == 6 ? 2428u : lane == 12 ? 21846u : lane == 19 ? 810u
                          : lane == 25 ? 7282u : 0u) << 16;
  const float b1 = (js >= 0 && 1 > js) ? 1.f : 0.f;  // byte 1..3 wholly above the edge
  const float b2 = (js >= 0 && 2 > js) ? 1.f : 0.f;
  const float b3 = (js >= 0 && 3 > js) ? 1.f : 0.f;
  const float a1 = 1.f - b1, a2 = 1.f - b2, a3 = 1.f - b3;
  // table address of byte j: the pair's base (the same for every lane) plus
  // PRMT(word, c) = byte << 8 | the lane's offset in its half of the row
  const uint32_t tb0 = sbase + kOffT, tb1 = tb0 + kPairBytes;
  const uint32_t c0 = 4u * lane, c1 = 128u + 4u * lane;
  const uint32_t hq = sbase + kOffH + 4u * lane;
  const uint32_t sel_e = 0x4440u | uint32_t(js < 0 ? 0 : js);
  const int g = (20 * lane) >> 7;  // the lane's (lower) group in the slice
  const uint32_t so = 2u * uint32_t(5 * s - sx + g);

  pdl_wait();  // x, y and the workspace are used by earlier work on the stream
  build_tables(p, smem, s);
  __syncthreads();

  float* part = p.ws + (size_t)(c * p.S + s) * p.rc;
  // One stage's rows in two phases, so that no shuffle sits between one row's
  // loads and the next row's: first every shared-memory load of the 8 rows,
  // then the arithmetic with the 8 hand-over shuffles back to back.
  struct Loads {
    float v0[kRows], v1[kRows], v2[kRows], v3[kRows], h[kRows], sc[kRows];
  };
  auto stage_loads = [&](uint32_t st, Loads& L) {
    uint32_t w[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) w[r] = lds_u32(st + r * kSliceBytes + 4 * lane);
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      L.v0[r] = lds_f32(tb0 + prmt(w[r], c0, 0x5504u));
      L.v1[r] = lds_f32(tb0 + prmt(w[r], c1, 0x5514u));
      L.v2[r] = lds_f32(tb1 + prmt(w[r], c0, 0x5524u));
      L.v3[r] = lds_f32(tb1 + prmt(w[r], c1, 0x5534u));
      L.h[r] = lds_f32(hq + 128u * __umulhi(prmt(w[r], 0u, sel_e), magic));
      L.sc[r] = lds_h2f(st + kStageW + r * kScaleRow + so);
    }
  };
  auto stage_values = [&](const Loads& L, float (&cr)[kRows]) {
    float hs[kRows], own[kRows], hp[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      hs[r] = fmaf(b3, L.v3[r], fmaf(b2, L.v2[r], fmaf(b1, L.v1[r], L.h[r])));
      own[r] = fmaf(a3, L.v3[r], fmaf(a2, L.v2[r], fmaf(a1, L.v1[r], L.v0[r])));
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) hp[r] = __shfl_up_sync(0xFFFFFFFFu, hs[r], 1);  // lane 0: 0
#pragma unroll
    for (int r = 0; r < kRows; ++r) cr[r] = L.sc[r] * (own[r] + hp[r]);
  };
  // transposed butterfly over the 32 lanes (lanes 4R..4R+3 end with row R)
  // and the stage's 8 partial sums to the workspace
  const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4;
  auto reduce_store = [&](const float (&cr)[kRows], int stage) {
    float t4[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float keep = h16 ? cr[q + 4] : cr[q];
      const float send = h16 ? cr[q] : cr[q + 4];
      t4[q] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
    }
    float t2[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const float keep = h8 ? t4[q + 2] : t4[q];
      const float send = h8 ? t4[q] : t4[q + 2];
      t2[q] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 8);
    }
    float v = (h4 ? t2[1] : t2[0]) + __shfl_xor_sync(0xFFFFFFFFu, h4 ? t2[0] : t2[1], 4);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
    if ((lane & 3) == 0) part[stage * kRows + (lane >> 2)] = v;
  };
  // software pipeline: stage j's lookups, then stage j-1's butterfly, so the
  // butterfly's dependent shuffles overlap the next stage's loads
  float prev[kRows];
  for (int j = 0; j < mine; ++j) {
    const int jn = j + kDepth;
    if (jn < mine) cpy.issue(ring + (jn % kWarpSlots) * kStageBytes, warp + kWarps * jn, lane);
    cp_commit();
    cp_wait<kDepth>();  // this lane's copies of stage j have landed
    __syncwarp();       // and every other lane's
    Loads L;
    stage_loads(ring + (j % kWarpSlots) * kStageBytes + opaque_zero(), L);
    if (j > 0) reduce_store(prev, warp + kWarps * (j - 1));  // overlaps the loads
    float cur[kRows];
    stage_values(L, cur);
#pragma unroll
    for (int r = 0; r < kRows; ++r) prev[r] = cur[r];
    __syncwarp();  // the slot is refilled by the next iteration's copies
  }
  if (mine > 0) reduce_store(prev, warp + kWarps * (mine - 1));
  cp_wait<0>();
  __syncthreads();  // every partial of the CTA is written (program order)

  // arrivals: one counter per part of the chunk's rows. Release: the CTA's
  // partials before the arrival; acquire: the other CTAs' partials after it
  // (the barrier below extends both to the whole CTA).
  unsigned int* flags = reinterpret_cast<unsigned int*>(smem + kOffFlags);
  if (threadIdx.x < p.S) {
    unsigned int* ctr = p.cnt + c * p.S + threadIdx.x;
    unsigned int old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;"
                 : "=r"(old)
                 : "l"(ctr)
                 : "memory");
    const bool last = old == unsigned(p.S - 1);
    if (last) *ctr = 0u;  // every CTA of the chunk has arrived: re-arm for the next call
    flags[threadIdx.x] = last ? 1u : 0u;
  }
  __syncthreads();
  // the parts this CTA completed, all rows at once
  const float* base = p.ws + (size_t)c * p.S * p.rc;
  int nf = 0;
  for (int q = 0; q < p.S; ++q) nf += flags[q] ? 1 : 0;
  const int span = p.swiglu ? p.part_rows / 2 : p.part_rows;  // outputs per part
  const int total = nf * span;
  // two outputs per thread and pass, all their partials loaded at once (one
  // L2 round trip), each output's partials added in slice order
  for (int o0 = threadIdx.x; o0 < total; o0 += 2 * kThreads) {
    int rr[2], ff[2];
    bool ok[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int o = o0 + t * kThreads;
      ok[t] = false;
      rr[t] = ff[t] = 0;
      if (o < total) {
        int q = -1;
        for (int u = o / span; u >= 0; --u)  // the (o/span)-th completed part
          do ++q; while (!flags[q]);
        // row of the output (the gate row with swiglu: 8 gate rows, then the
        // 8 up rows of the same features, per 16-row block)
        ff[t] = q * span + (o - (o / span) * span);
        rr[t] = p.swiglu ? (ff[t] >> 3) * 16 + (ff[t] & 7) : ff[t];
        ok[t] = rr[t] < rows;
      }
    }
    float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};  // [output][gate or plain, up]
    for (int j0 = 0; j0 < p.S; j0 += 8) {
      float v[2][2][8];
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const bool in = ok[t] && j0 + u < p.S && (hh == 0 || p.swiglu);
            v[t][hh][u] = in ? __ldcg(base + (size_t)(j0 + u) * p.rc + rr[t] + 8 * hh) : 0.f;
          }
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int u = 0; u < 8; ++u) acc[t][hh] += v[t][hh][u];
    }
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if (!ok[t]) continue;
      if (p.swiglu) p.y[row0 / 2 + ff[t]] = __float2half_rn(silu(acc[t][0]) * acc[t][1]);
      else p.y[row0 + rr[t]] = __float2half_rn(acc[t][0]);
    }
  }
}

// ------------------------------------------------------------------ binary
// The same structure for binary weights: a byte holds eight codes, so a
// position's table has 256 entries (the sum of +-x over the eight codes,
// bit i of the byte giving the sign of code i) and a slice is 1024 codes
// (eight whole groups); a lane's 32 codes are a quarter of one group, so
// there is no group edge inside a lane's word and no hand-over.
constexpr int kBinSliceCodes = 1024;
constexpr int kBinOffFlags = kOffX + kBinSliceCodes * 4;
constexpr int kBinOffRing = kBinOffFlags + kMaxSlices * 4;
constexpr int kBinSmem = kBinOffRing + kSlots * kStageBytes;
static_assert(kBinOffRing % 128 == 0 && kBinSmem <= 232448, "binary layout fits one SM");

// Entry e = a + 16*b: the low nibble (codes 0..3) in a, the high one (codes
// 4..7) in b, sums A[a] + B[b]; thread q of a position writes b = q, q+4,
// q+8, q+12.
__device__ __forceinline__ void binary_rows(float* dst, const float (&xv)[8], int q) {
  float A[16], Bv[4];
#pragma unroll
  for (int a = 0; a < 16; ++a) {
    float v = (a & 1) ? xv[0] : -xv[0];
    v += (a & 2) ? xv[1] : -xv[1];
    v += (a & 4) ? xv[2] : -xv[2];
    v += (a & 8) ? xv[3] : -xv[3];
    A[a] = v;
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int bb = q + 4 * u;
    float v = (bb & 1) ? xv[4] : -xv[4];
    v += (bb & 2) ? xv[5] : -xv[5];
    v += (bb & 4) ? xv[6] : -xv[6];
    v += (bb & 8) ? xv[7] : -xv[7];
    Bv[u] = v;
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    float* rb = dst + 16 * 64 * (q + 4 * u);
#pragma unroll
    for (int a = 0; a < 16; ++a) rb[a * 64] = A[a] + Bv[u];
  }
}

__device__ __forceinline__ void build_tables_bin(const Params& p, uint8_t* smem, int s) {
  float* xs = reinterpret_cast<float*>(smem + kOffX);
  const int t = threadIdx.x;
  for (int i = t; i < kBinSliceCodes; i += kThreads) {
    const int kk = s * kBinSliceCodes + i;
    xs[i] = kk < p.k ? __half2float(p.x[kk]) : 0.f;
  }
  __syncthreads();
  const int pos = t & 127, q = t >> 7;
  const int pj = pos >> 5, pl = pos & 31;
  const int byte = 4 * pl + pj;
  float xv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) xv[i] = xs[8 * byte + i];
  binary_rows(reinterpret_cast<float*>(smem + kOffT + (pj >> 1) * kPairBytes + (pj & 1) * 128) + pl,
              xv, q);
}

__global__ void __launch_bounds__(kThreads, 1)
    gemv_bin_lut_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const int s = blockIdx.x % p.S, c = blockIdx.x / p.S;
  const int row0 = c * p.rc;
  const int rows = min(p.rc, p.n - row0);
  const int nst = (rows + kRows - 1) / kRows;
  const int mine = nst > warp ? (nst - warp + kWarps - 1) / kWarps : 0;  // stages warp, warp+16, ..
  const int sx = 8 * s;  // the slice's eight groups: one 16-byte scale piece per row
  const uint32_t ring = sbase + kBinOffRing + warp * kWarpSlots * kStageBytes;
  pdl_launch_dependents();

  // weights never depend on earlier work on the stream: with the prefetch
  // flag the first stages stream in while the previous kernel finishes
  const StageCopy cpy(p, row0, s, sx, lane);
  if (!p.prefetch) pdl_wait();
  for (int d = 0; d < kDepth; ++d) {
    if (d < mine) cpy.issue(ring + d * kStageBytes, warp + kWarps * d, lane);
    cp_commit();
  }

  // lane constants: table address of byte j as for ternary; the lane's 32
  // codes are one quarter of a group, so one scale per row and no hand-over
  const uint32_t tb0 = sbase + kOffT, tb1 = tb0 + kPairBytes;
  const uint32_t c0 = 4u * lane, c1 = 128u + 4u * lane;
  const uint32_t so = 2u * uint32_t(lane >> 2);

  pdl_wait();  // x, y and the workspace are used by earlier work on the stream
  build_tables_bin(p, smem, s);
  __syncthreads();

  float* part = p.ws + (size_t)(c * p.S + s) * p.rc;
  // One stage's rows: every shared-memory load of the 8 rows first, then the
  // arithmetic.
  struct Loads {
    float v0[kRows], v1[kRows], v2[kRows], v3[kRows], sc[kRows];
  };
  auto stage_loads = [&](uint32_t st, Loads& L) {
    uint32_t w[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) w[r] = lds_u32(st + r * kSliceBytes + 4 * lane);
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      L.v0[r] = lds_f32(tb0 + prmt(w[r], c0, 0x5504u));
      L.v1[r] = lds_f32(tb0 + prmt(w[r], c1, 0x5514u));
      L.v2[r] = lds_f32(tb1 + prmt(w[r], c0, 0x5524u));
      L.v3[r] = lds_f32(tb1 + prmt(w[r], c1, 0x5534u));
      L.sc[r] = lds_h2f(st + kStageW + r * kScaleRow + so);
    }
  };
  auto stage_values = [&](const Loads& L, float (&cr)[kRows]) {
#pragma unroll
    for (int r = 0; r < kRows; ++r) cr[r] = L.sc[r] * ((L.v0[r] + L.v1[r]) + (L.v2[r] + L.v3[r]));
  };
  // transposed butterfly over the 32 lanes (lanes 4R..4R+3 end with row R)
  // and the stage's 8 partial sums to the workspace
  const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4;
  auto reduce_store = [&](const float (&cr)[kRows], int stage) {
    float t4[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float keep = h16 ? cr[q + 4] : cr[q];
      const float send = h16 ? cr[q] : cr[q + 4];
      t4[q] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
    }
    float t2[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const float keep = h8 ? t4[q + 2] : t4[q];
      const float send = h8 ? t4[q] : t4[q + 2];
      t2[q] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 8);
    }
    float v = (h4 ? t2[1] : t2[0]) + __shfl_xor_sync(0xFFFFFFFFu, h4 ? t2[0] : t2[1], 4);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
    if ((lane & 3) == 0) part[stage * kRows + (lane >> 2)] = v;
  };
  // software pipeline: stage j's lookups, then stage j-1's butterfly, so the
  // butterfly's dependent shuffles overlap the next stage's loads
  float prev[kRows];
  for (int j = 0; j < mine; ++j) {
    const int jn = j + kDepth;
    if (jn < mine) cpy.issue(ring + (jn % kWarpSlots) * kStageBytes, warp + kWarps * jn, lane);
    cp_commit();
    cp_wait<kDepth>();  // this lane's copies of stage j have landed
    __syncwarp();       // and every other lane's
    Loads L;
    stage_loads(ring + (j % kWarpSlots) * kStageBytes + opaque_zero(), L);
    if (j > 0) reduce_store(prev, warp + kWarps * (j - 1));  // overlaps the loads
    float cur[kRows];
    stage_values(L, cur);
#pragma unroll
    for (int r = 0; r < kRows; ++r) prev[r] = cur[r];
    __syncwarp();  // the slot is refilled by the next iteration's copies
  }
  if (mine > 0) reduce_store(prev, warp + kWarps * (mine - 1));
  cp_wait<0>();
  __syncthreads();  // every partial of the CTA is written (program order)

  // arrivals: one counter per part of the chunk's rows. Release: the CTA's
  // partials before the arrival; acquire: the other CTAs' partials after it
  // (the barrier below extends both to the whole CTA).
  unsigned int* flags = reinterpret_cast<unsigned int*>(smem + kBinOffFlags);
  if (threadIdx.x < p.S) {
    unsigned int* ctr = p.cnt + c * p.S + threadIdx.x;
    unsigned int old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;"
                 : "=r"(old)
                 : "l"(ctr)
                 : "memory");
    const bool last = old == unsigned(p.S - 1);
    if (last) *ctr = 0u;  // every CTA of the chunk has arrived: re-arm for the next call
    flags[threadIdx.x] = last ? 1u : 0u;
  }
  __syncthreads();
  // the parts this CTA completed, all rows at once
  const float* base = p.ws + (size_t)c * p.S * p.rc;
  int nf = 0;
  for (int q = 0; q < p.S; ++q) nf += flags[q] ? 1 : 0;
  const int span = p.swiglu ? p.part_rows / 2 : p.part_rows;  // outputs per part
  const int total = nf * span;
  // two outputs per thread and pass, all their partials loaded at once (one
  // L2 round trip), each output's partials added in slice order
  for (int o0 = threadIdx.x; o0 < total; o0 += 2 * kThreads) {
    int rr[2], ff[2];
    bool ok[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int o = o0 + t * kThreads;
      ok[t] = false;
      rr[t] = ff[t] = 0;
      if (o < total) {
        int q = -1;
        for (int u = o / span; u >= 0; --u)  // the (o/span)-th completed part
          do ++q; while (!flags[q]);
        // row of the output (the gate row with swiglu: 8 gate rows, then the
        // 8 up rows of the same features, per 16-row block)
        ff[t] = q * span + (o - (o / span) * span);
        rr[t] = p.swiglu ? (ff[t] >> 3) * 16 + (ff[t] & 7) : ff[t];
        ok[t] = rr[t] < rows;
      }
    }
    float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};  // [output][gate or plain, up]
    for (int j0 = 0; j0 < p.S; j0 += 8) {
      float v[2][2][8];
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const bool in = ok[t] && j0 + u < p.S && (hh == 0 || p.swiglu);
            v[t][hh][u] = in ? __ldcg(base + (size_t)(j0 + u) * p.rc + rr[t] + 8 * hh) : 0.f;
          }
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int u = 0; u < 8; ++u) acc[t][hh] += v[t][hh][u];
    }
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if (!ok[t]) continue;
      if (p.swiglu) p.y[row0 / 2 + ff[t]] = __float2half_rn(silu(acc[t][0]) * acc[t][1]);
      else p.y[row0 + rr[t]] = __float2half_rn(acc[t][0]);
    }
  }
}

struct Shape {
  int S, C, rc, part_rows;
};

}  // namespace lut

// Rows per CTA below which the streaming kernel is faster: the tables and the
// cross-block sums cost ~3.5-4 us per launch (measured on B300, ternary:
// ~6.5 ns per row of 640 codes in the loop, 12.6 us for 976 rows against
// 13.9 us for the streaming kernel), so only products of about a thousand
// rows per block and slice gain. A binary row of a slice (1024 codes) costs
// less than half a ternary one, against a streaming binary kernel that is
// itself faster per code (measured: 9.0 against 8.75 us at 608 rows per
// block, N=17408 K=5120; the 64-layer binary decode gains 16% with gate/up
// and down on the tables).
constexpr int kLutMinRowsTer = 768;
constexpr int kLutMinRowsBin = 640;

static bool lut_shape(const bonsai_weights* w, lut::Shape& sh) {
  using namespace lut;
  const bool bin = w->format == BONSAI_FMT_BINARY;
  const int64_t k = w->k, n = w->n;
  if ((k / 128) % 8) return false;  // the scale rows' pitch must be 16-byte aligned
  const int sms = device_sm_count();
  if (device_max_smem_optin() < (bin ? kBinSmem : kSmem)) return false;
  const int64_t sc = bin ? kBinSliceCodes : kSliceCodes;
  const int64_t S = (k + sc - 1) / sc;
  if (S > sms || S > kMaxSlices) return false;
  int64_t C = sms / S;
  int64_t rc = ((n + C - 1) / C + 15) / 16 * 16;
  if (rc < (bin ? kLutMinRowsBin : kLutMinRowsTer)) return false;
  C = (n + rc - 1) / rc;
  if (C * S * rc > (int64_t(1) << 31)) return false;
  sh.S = (int)S;
  sh.C = (int)C;
  sh.rc = (int)rc;
  sh.part_rows = (int)(((rc + S - 1) / S + 15) / 16 * 16);
  return true;
}

static int64_t lut_ws_bytes(const lut::Shape& sh) {
  const int64_t parts = (int64_t)sh.C * sh.S * sh.rc * 4;
  return (parts + (int64_t)sh.C * sh.S * 4 + 255) / 256 * 256;
}

int64_t gemv_lut_workspace_bytes(const bonsai_weights* w) {
  lut::Shape sh;
  return lut_shape(w, sh) ? lut_ws_bytes(sh) : 0;
}

// UNSUPPORTED when the shape does not take the tables or the workspace is
// smaller than gemv_lut_workspace_bytes (nothing launched then).
bonsai_status gemv_lut_launch(const bonsai_weights* w, const uint16_t* x, uint16_t* y,
                              bool swiglu, void* ws, int64_t ws_bytes, cudaStream_t stream) {
  using namespace lut;
  Shape sh;
  if (!ws || !lut_shape(w, sh) || ws_bytes < lut_ws_bytes(sh)) return BONSAI_ERR_UNSUPPORTED;
  Params p{};
  p.packed = static_cast<const uint8_t*>(w->packed);
  p.scales = reinterpret_cast<const __half*>(w->scales);
  p.x = reinterpret_cast<const __half*>(x);
  p.y = reinterpret_cast<__half*>(y);
  p.ws = static_cast<float*>(ws);
  p.cnt = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(ws) +
                                          (int64_t)sh.C * sh.S * sh.rc * 4);
  p.row_bytes = w->row_bytes;
  p.n = (int)w->n;
  p.k = (int)w->k;
  p.G = (int)(w->k / 128);
  p.S = sh.S;
  p.C = sh.C;
  p.rc = sh.rc;
  p.part_rows = sh.part_rows;
  p.prefetch = (w->flags & BONSAI_WEIGHTS_PREFETCH) ? 1 : 0;
  p.swiglu = swiglu ? 1 : 0;
  const bool bin = w->format == BONSAI_FMT_BINARY;
  const void* fn = bin ? (const void*)gemv_bin_lut_kernel : (const void*)gemv_ter_lut_kernel;
  const int smem = bin ? kBinSmem : kSmem;
  if (ensure_dynamic_smem(fn, smem) != cudaSuccess) return BONSAI_ERR_CUDA;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(sh.C * sh.S);
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
