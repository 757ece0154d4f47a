/*
 * bonsai.h -- C ABI of libbonsai: matrix products of FP16 activations with
 * sub-bit weights (binary {-1,+1} or ternary {-1,0,+1}) that share one FP16
 * scale per group of 128 weights along K.
 *
 *   y[m][n] = sum_k x[m][k] * s[n][k/128] * w[n][k]              (FP32 accumulate)
 *
 * Sources (the "Bonsai" pages):
 *   - "1-bit diffusion ... WebGPU" (richmindsetzone), section "1-bit 嘅數學":
 *     each weight is binary and every group of weights shares one FP16 scale;
 *     1.125 effective bits per binary weight, about 1.71 for ternary
 *     {-1,0,+1}; a binary GEMM can be done with XOR + popcount.
 *   - "OpenBonsai" (ainewscove), section "工作原理": one FP16 group scale per
 *     128 weights, ternary codes {-1,0,+1}.
 *   - "三值权重压缩" (kongchang), section "三值权重到底做了什么" and its
 *     background paragraph: ternary multiplication reduces to addition and a
 *     sign flip.
 *   - "Bonsai 27B on phone" (xiaohu.ai), sections "第一の壁" and "速度は二層":
 *     token-by-token decode re-streams every weight per token and is bound by
 *     memory bandwidth at small batch.
 * The pages fix no byte layout; the layout below is this library's own and is
 * stated exactly so that any other implementation can produce it.
 *
 * ------------------------------------------------------------------------
 * Data layout (all matrices row-major, PyTorch Linear convention W[n][k]):
 *   x       FP16 bits, [m][k], row stride k elements.
 *   scales  FP16 bits, [n][k/128], row stride k/128 elements; scale of
 *           weight (n,k) is scales[n][k/128] (groups are contiguous runs of
 *           128 along K). Effective weight = scale * code (a product).
 *   y       FP16 bits, [m][n], row stride n elements; FP32 result rounded to
 *           nearest-even.
 *   BINARY  packed row n occupies row_bytes bytes at packed + n*row_bytes;
 *           bit i (LSB first) of little-endian 32-bit word j holds code
 *           k = 32*j + i; bit 1 means +1, bit 0 means -1. Bytes from k/8 to
 *           row_bytes are padding (pack writes 0).
 *   TERNARY byte b of row n holds the five codes k = 5b .. 5b+4 as the
 *           base-3 number  sum_{i<5} (code(5b+i) + 1) * 3^i  (least
 *           significant digit first, digit = code + 1 in {0,1,2}); codes past
 *           k are 0 (digit 1). Valid bytes are 0..242; all -1 -> 0, all 0 ->
 *           121, all +1 -> 242. Bytes from ceil(k/5) to row_bytes are padding
 *           holding 121 (five zero codes). A byte may hold codes of two
 *           adjacent 128-groups; the scale is applied per code.
 *
 * Size requirements checked on the host before any launch:
 *   k % 128 == 0, k > 0, n > 0, m > 0.
 *   BINARY : row_bytes >= k/8 and row_bytes % 16 == 0.
 *   TERNARY: row_bytes >= 64*ceil(ceil(k/5)/64) and row_bytes % 64 == 0.
 *   All device pointers 16-byte aligned.
 *
 * Conventions:
 *   - Every pointer passed to a compute call is a DEVICE pointer owned by the
 *     caller. The library allocates no device memory and keeps no pointer
 *     after the call returns. Its device state is one 32-bit status word per
 *     device, a file-scope __device__ variable, written by kernels that
 *     detect bad input codes or a bounded wait that ran out, plus the fixed
 *     scratch array of bonsai_gemv_splitk_static (declared below).
 *   - Calls enqueue work on `stream` and return without synchronising (the
 *     compute calls other than bonsai_gemv_splitk_static can be captured in
 *     a CUDA graph). A non-OK return means nothing was launched. Kernel-side
 *     problems are reported by bonsai_check_async.
 *   - Compute calls use programmatic dependent launch: a kernel may be
 *     scheduled while the previous kernel on the stream is still running,
 *     but it reads x (and writes y) only after that kernel has finished.
 *     It also waits before reading its weights, unless the weights carry
 *     BONSAI_WEIGHTS_PREFETCH: then it streams them at once, overlapping the
 *     previous kernel's tail (decode loops whose weights never change).
 *   - No C++ exceptions cross this interface.
 * ------------------------------------------------------------------------
 */
#ifndef BONSAI_H
#define BONSAI_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle; identical to cudaStream_t. NULL = legacy stream. */
typedef struct CUstream_st* bonsai_stream;

typedef enum {
  BONSAI_OK = 0,
  BONSAI_ERR_INVALID_ARG = 1,  /* null pointer, unknown enum, negative size   */
  BONSAI_ERR_SHAPE = 2,        /* k % 128 != 0, row_bytes too small, ...       */
  BONSAI_ERR_ALIGN = 3,        /* a pointer or row stride is not 16-B aligned  */
  BONSAI_ERR_FORMAT = 4,       /* wrong weight format for this call            */
  BONSAI_ERR_CUDA = 5,         /* a CUDA runtime call failed                   */
  BONSAI_ERR_UNSUPPORTED = 6,  /* valid request this build does not handle     */
  BONSAI_ERR_TIMEOUT = 7,      /* a bounded device-side wait ran out           */
  BONSAI_ERR_BAD_CODE = 8      /* pack saw a code outside the format's set     */
} bonsai_status;

enum { BONSAI_FMT_BINARY = 1, BONSAI_FMT_TERNARY = 2 };

/* bonsai_weights.flags bits. */
enum {
  /* The packed bytes and scales are not written by the kernel launched just
   * before this call on the same stream, so they may be read before that
   * kernel has finished. */
  BONSAI_WEIGHTS_PREFETCH = 1
};

/* A packed weight matrix W[n][k] with its FP16 group scales. */
typedef struct {
  int32_t format;          /* BONSAI_FMT_BINARY or BONSAI_FMT_TERNARY        */
  int64_t n;               /* output features (rows of W)                    */
  int64_t k;               /* input features, multiple of 128                */
  int64_t row_bytes;       /* bytes per packed row (see layout above)        */
  const void* packed;      /* device, n * row_bytes bytes                    */
  const uint16_t* scales;  /* device, FP16 bits [n][k/128]                   */
  int32_t flags;           /* BONSAI_WEIGHTS_* bits, 0 if none. Last, so a
                              caller that fills only the six fields above
                              (zero-initialised struct) gets flags = 0      */
} bonsai_weights;

/* Canonical packed row size: BINARY k/8; TERNARY 64*ceil(ceil(k/5)/64).
 * Returns -1 for an unknown format or k <= 0 or k % 128 != 0. Host only. */
int64_t bonsai_packed_row_bytes(int32_t format, int64_t k);

/* Pack int8 codes [rows][k] (row stride k) into the BINARY layout.
 * codes: device, values must be -1 or +1; out: device, rows*row_bytes bytes.
 * A code outside {-1,+1} sets BONSAI_ERR_BAD_CODE in the device status word
 * (the affected output word is unspecified); bonsai_check_async reports it.
 * Follows the binary-weight-with-group-scale format ("1-bit 嘅數學"). */
bonsai_status bonsai_pack_binary(const int8_t* codes, int64_t rows, int64_t k,
                                 void* out, int64_t row_bytes,
                                 bonsai_stream stream);

/* Pack int8 codes [rows][k] into the TERNARY layout (5 codes per byte,
 * base 3) including the 121-valued padding. Codes outside {-1,0,+1} set
 * BONSAI_ERR_BAD_CODE. Follows the ternary value set of the OpenBonsai page
 * ("工作原理") and "三值权重到底做了什么". */
bonsai_status bonsai_pack_ternary(const int8_t* codes, int64_t rows, int64_t k,
                                  void* out, int64_t row_bytes,
                                  bonsai_stream stream);

/* Batch-1 decode product y[n] = sum_k x[k] * s[n][k/128] * w[n][k].
 * w: binary or ternary weights; x: device FP16 [k]; y: device FP16 [n].
 * Packed bytes must be valid codes (ternary bytes <= 242, padding 121):
 * kernels do not re-check them. Decode is memory-bandwidth bound
 * ("第一の壁"): the kernel streams each packed byte once. Rows too long for
 * the decode kernel's on-chip activation table (beyond roughly 30K codes
 * ternary or 75K binary) run on the tensor-core kernel of bonsai_gemm. */
bonsai_status bonsai_gemv(const bonsai_weights* w, const uint16_t* x,
                          uint16_t* y, bonsai_stream stream);

/* bonsai_gemv with the activations and the result in host memory: enqueues
 * on `stream` the copy x_host -> x_dev (k FP16 values), the decode product
 * into y_dev, and the copy y_dev -> y_host (n FP16 values), then returns.
 * For a decode loop that samples on the host: one call per token, no other
 * API call in between. Synchronise the stream (or call bonsai_check_async)
 * before reading y_host. With page-locked, 16-byte aligned host buffers
 * (cudaHostAlloc / pinned tensors) no copy engine is used: a small kernel
 * reads x_host through its device mapping into x_dev, and the product
 * kernel writes y straight into y_host (y_dev is then left untouched).
 * Other host memory is copied with cudaMemcpyAsync (each copy then waits
 * for the host). x_dev, y_dev: device buffers of k and n FP16 values,
 * 16-byte aligned, owned by the caller (the library allocates nothing).
 * Errors as bonsai_gemv; BONSAI_ERR_CUDA if a copy cannot be enqueued. */
bonsai_status bonsai_gemv_host(const bonsai_weights* w, const uint16_t* x_host,
                               uint16_t* x_dev, uint16_t* y_dev, uint16_t* y_host,
                               bonsai_stream stream);

/* Workspace variants of bonsai_gemv and bonsai_gemv_host. For weights of a
 * shape that takes it (k/128 a multiple of 8, and enough rows to keep every
 * SM busy; bonsai_gemv_workspace_bytes says which), the product runs on a
 * kernel that needs no operand per code: a packed ternary byte holds five
 * codes (a binary byte eight), so x . w over them is one of 243 (256) sums
 * fixed by x alone ("multiplication degenerates to addition and sign flip",
 * 三值权重 page). K is split into slices of 640 (1024) codes across thread
 * blocks; each block tabulates the sums of its slice in FP32 and then
 * spends one table lookup and one add per packed byte. Its FP32 partial
 * sums per row go to the
 * workspace, and the block that completes a part of the rows adds them in
 * slice order and rounds once to FP16. Results of two calls with the same
 * inputs are bit-identical; they differ from bonsai_gemv's only by the
 * order of the FP32 additions (same error bound).
 *   workspace        device, 256-byte aligned, zero-filled before its first
 *                    use; a completed call leaves its arrival counters zero
 *                    again, so one workspace serves call after call. Calls
 *                    that may overlap on the GPU (other streams) need
 *                    separate workspaces; calls ordered on one stream may
 *                    share one. After BONSAI_ERR_TIMEOUT, zero it again.
 *   workspace_bytes  its size; below bonsai_gemv_workspace_bytes(w) (or
 *                    workspace NULL) the call runs bonsai_gemv's kernels.
 * Other arguments, errors and behaviour as bonsai_gemv / bonsai_gemv_host,
 * plus BONSAI_ERR_ALIGN for a workspace not 256-byte aligned.
 * bonsai_gemv_workspace_bytes returns 0 when the shape does not take the
 * table kernel (k/128 not a multiple of 8, too few rows per block) or w is
 * invalid. bonsai_gemm_workspace_bytes(w, 1) returns the same size, and
 * bonsai_gemm_ws / bonsai_gemm_swiglu_ws with m = 1 run the same kernel
 * (with swiglu, its final sums give silu(g) * u). */
int64_t bonsai_gemv_workspace_bytes(const bonsai_weights* w);
bonsai_status bonsai_gemv_ws(const bonsai_weights* w, const uint16_t* x, uint16_t* y,
                             void* workspace, int64_t workspace_bytes,
                             bonsai_stream stream);
bonsai_status bonsai_gemv_host_ws(const bonsai_weights* w, const uint16_t* x_host,
                                  uint16_t* x_dev, uint16_t* y_dev, uint16_t* y_host,
                                  void* workspace, int64_t workspace_bytes,
                                  bonsai_stream stream);

/* Decode product with K split across thread blocks, for matrices with few
 * rows (n <= 8192), computing the same y as bonsai_gemv (to the same error
 * bound, not bit-identically: the sums are ordered differently). The pages
 * have no counterpart of this call; it exists for callers that cannot
 * allocate device memory at call time -- a serving loop that must not stall
 * on cudaMalloc/cudaFree, which synchronise the device, or a process whose
 * device memory is budgeted up front -- yet need per-call scratch for the
 * split sums. The scratch is a fixed file-scope device array of 1 MiB of FP32
 * partial sums (at most 32 splits x 8192 rows) and 512 arrival counters;
 * nothing is allocated, ever.
 *   w, x, y: as bonsai_gemv (device pointers, 16-byte aligned).
 *   Returns BONSAI_ERR_UNSUPPORTED for n > 8192 (the scratch holds no more
 *   rows), with nothing launched; BONSAI_ERR_CUDA if the scratch address
 *   cannot be obtained.
 * The first call on a device looks up the scratch address
 * (cudaGetSymbolAddress) and enqueues a clear of the counters on `stream`.
 * Calls share the scratch: two calls that overlap in time
 * (different streams, or different host threads on one device) corrupt each
 * other's sums, so order them on one stream or synchronise between them.
 * Results of two ordered calls with the same inputs are bit-identical.
 * Unlike the other compute calls, this one uses neither programmatic
 * dependent launch nor BONSAI_WEIGHTS_PREFETCH: its kernel is an ordinary
 * launch that starts after the previous work on the stream has finished. */
bonsai_status bonsai_gemv_splitk_static(const bonsai_weights* w, const uint16_t* x,
                                        uint16_t* y, bonsai_stream stream);

/* ------------------------------------------------------------------------
 * Decode plans: the one-token products of a whole decoder token in ONE
 * persistent launch. Token-by-token decode re-streams every weight per token
 * and is bound by memory bandwidth ("第一の壁", "速度は二層"); a token of a
 * deep decoder is hundreds of small products, and as separate launches each
 * pays a launch, a grid-wide dependency wait and its table prologue. A plan
 * walks its products in order inside one kernel: the weights of the next
 * product stream while the current one finishes, and a product whose x is an
 * earlier product's y waits (on the device, bounded) until that product is
 * complete on every thread block.
 *
 * A step: the product y = x . (s (.) W)^T of `w` with one token, or with
 * swiglu = 1 the gated feed-forward input of bonsai_gemm_swiglu (w holds 2F
 * rows interleaved in 16-row blocks, y holds F values). `after` is the index
 * of an EARLIER step whose y this step reads as x (directly or through
 * memory written by it), or -1. Steps that reuse a buffer another step
 * reads must be ordered through `after` as well (a plan runs its products
 * concurrently where `after` allows).
 * This build: TERNARY weights, every step's x table must fit on chip
 * (K up to ~30K); w.flags is ignored (a plan always streams weights ahead:
 * they must not be written while the plan runs). x, y: device, 16-byte
 * aligned. */
typedef struct {
  bonsai_weights w;
  const uint16_t* x;   /* device FP16 [k]                      */
  uint16_t* y;         /* device FP16 [n], or [n/2] with swiglu */
  int32_t swiglu;      /* 0 or 1                               */
  int32_t after;       /* earlier step index, or -1            */
} bonsai_decode_step;

/* Bytes of device memory a plan of `count` steps needs (count >= 1), or -1. */
int64_t bonsai_decode_plan_bytes(int64_t count);

/* Checks the steps and writes the plan into `plan` (device memory owned by
 * the caller, 128-byte aligned, plan_bytes >= bonsai_decode_plan_bytes(count)):
 * per step the TMA descriptors of its weights and its parameters, and zeroed
 * completion counters. Enqueued on `stream` (the host copy is staged before
 * the call returns). Do not capture this call in a CUDA graph; capture
 * bonsai_decode_run. Errors: INVALID_ARG (null pointer, `after` not an
 * earlier step, count < 1 or > 4096), FORMAT (a binary step), SHAPE /
 * ALIGN as bonsai_gemv, UNSUPPORTED (a step's x table does not fit). */
bonsai_status bonsai_decode_plan_init(const bonsai_decode_step* steps, int64_t count,
                                      void* plan, int64_t plan_bytes, bonsai_stream stream);

/* Runs an initialised plan: one launch on `stream` computes every step's y.
 * `steps` and `count` must be those the plan was initialised with (the launch
 * geometry is recomputed from them; nothing else is read on the host). The
 * last thread block of the run resets the completion counters, so runs of
 * one plan may follow each other on a stream (or in a CUDA graph); two runs
 * of the same plan must not overlap. A dependency wait that runs out (2 s)
 * is reported as BONSAI_ERR_TIMEOUT by bonsai_check_async. */
bonsai_status bonsai_decode_run(const bonsai_decode_step* steps, int64_t count, void* plan,
                                bonsai_stream stream);

/* Self-test of the plan's dependency wait: one thread waits on a completion
 * counter that nothing increments, with a limit of limit_ns (1 us .. 100 ms,
 * else BONSAI_ERR_INVALID_ARG); the wait gives up and the next
 * bonsai_check_async reports BONSAI_ERR_TIMEOUT. No fault is involved. */
bonsai_status bonsai_selftest_plan_wait(uint64_t limit_ns, bonsai_stream stream);

/* Multi-token product Y[m][n] = sum_k X[m][k] * s[n][k/128] * w[n][k],
 * X FP16 [m][k], Y FP16 [m][n]. m <= 8 runs the streaming decode kernel with
 * m columns (speculative verification, prefill of a few tokens); larger m
 * runs the tensor-core GEMM that expands weight tiles to FP16 in on-chip
 * memory (prompt processing and diffusion-transformer image tokens). */
bonsai_status bonsai_gemm(const bonsai_weights* w, const uint16_t* x,
                          int64_t m, uint16_t* y, bonsai_stream stream);

/* Gated feed-forward input of a decode layer, gate and up projections in
 * one pass over one weight matrix, with the SwiGLU product applied before
 * the store:
 *   h[m][f] = silu(g) * u,  silu(g) = g / (1 + e^-g),
 *   g = x[m] . (s (.) W_gate[f]),  u = x[m] . (s (.) W_up[f]).
 * The pages (OpenBonsai page: Qwen3.5-9B) run Qwen-family models, whose
 * feed-forward block has this form; they do not write it out.
 *   w  BINARY or TERNARY weights with n = 2F rows, F a multiple of 8, stored
 *      interleaved in 16-row blocks: rows 16t..16t+7 are gate rows
 *      8t..8t+7 and rows 16t+8..16t+15 are up rows 8t..8t+7 (scales in the
 *      same row order). A tile of the product then holds both factors of
 *      its outputs, and g and u never leave the chip.
 *   x  device FP16 [m][k];  h: device FP16 [m][F] (the down projection's x).
 * g and u are FP32 sums (as in bonsai_gemm); silu and the product are FP32,
 * and h is rounded once to FP16. m <= 8 runs the streaming decode kernel,
 * larger m the tensor-core GEMM. Returns BONSAI_ERR_SHAPE if n % 16 != 0. */
bonsai_status bonsai_gemm_swiglu(const bonsai_weights* w, const uint16_t* x,
                                 int64_t m, uint16_t* h, bonsai_stream stream);

/* bonsai_gemm and bonsai_gemm_swiglu with a caller workspace for a
 * stream-K schedule. Products whose 128-feature x 256-token tiles fill the
 * SMs unevenly (prompt processing with N=5120: 80 tiles on 148 SMs) keep
 * their whole waves of tiles and cut the last wave's k-steps into equal
 * ranges, one per SM; a tile split over several SMs sums their FP32 partial
 * tiles (fixed order, the first range's own sums first, the rest in SM order)
 * before the one FP16 rounding, so results stay within the same 2e-3 norm
 * bound. The pages' prompt-processing workload is pp512 (Bonsai 27B on
 * phone page, "速度は二層"), whose N=5120 products are the uneven case.
 *   workspace        device memory, 256-byte aligned, zero-filled before its
 *                    first use; every call that completes leaves it zeroed
 *                    again (its counters), so it can be reused call after
 *                    call and inside CUDA graphs. Calls that may overlap on
 *                    the GPU need separate workspaces. After a call that
 *                    reported BONSAI_ERR_TIMEOUT, zero it again.
 *   workspace_bytes  its size; below bonsai_gemm_workspace_bytes(w, m) (or
 *                    workspace NULL) the call runs the plain schedule.
 * With m = 1 the workspace serves the one-token table kernel of
 * bonsai_gemv_ws instead (bonsai_gemm_workspace_bytes(w, 1) is its size).
 * Same results and errors as bonsai_gemm / bonsai_gemm_swiglu otherwise,
 * plus BONSAI_ERR_ALIGN for a workspace not 256-byte aligned. */
int64_t bonsai_gemm_workspace_bytes(const bonsai_weights* w, int64_t m);
bonsai_status bonsai_gemm_ws(const bonsai_weights* w, const uint16_t* x, int64_t m,
                             uint16_t* y, void* workspace, int64_t workspace_bytes,
                             bonsai_stream stream);
bonsai_status bonsai_gemm_swiglu_ws(const bonsai_weights* w, const uint16_t* x,
                                    int64_t m, uint16_t* h, void* workspace,
                                    int64_t workspace_bytes, bonsai_stream stream);

/* XNOR-popcount product of +-1 activations with +-1 weights ("1-bit 嘅數學":
 * binary GEMM via XOR + popcount). bonsai_xnor_gemm computes it on the
 * tensor cores: +-1 codes (and +-s, the scale times a code) are exact FP16
 * operands and every sum of up to 2^24 products of +-1 is exact in the FP32
 * accumulator, so D equals k - 2*popc(a XOR w) bit for bit; Y's FP32 sum
 * rounds once to FP16 after the a_scale product. bonsai_xnor_gemm_popc is
 * the literal XOR + popcount kernel (same arguments, same results).
 *   a_bits  device uint32 [m][k/32], same bit layout as BINARY weights
 *           (bit 1 = +1); row stride k/32 words.
 *   a_scale device FP16 [m], one scale per activation row.
 *   w       BINARY weights [n][k] with group scales.
 *   d_out   device int32 [m][n] or NULL: D = sum_k a*w = k - 2*popc(a XOR w),
 *           exact.
 *   y_out   device FP16 [m][n] or NULL:
 *           Y = a_scale[m] * sum_g s[n][g] * (128 - 2*popc over group g).
 * At least one of d_out / y_out must be non-NULL. */
bonsai_status bonsai_xnor_gemm(const uint32_t* a_bits, const uint16_t* a_scale,
                               int64_t m, const bonsai_weights* w,
                               int32_t* d_out, uint16_t* y_out,
                               bonsai_stream stream);
bonsai_status bonsai_xnor_gemm_popc(const uint32_t* a_bits, const uint16_t* a_scale,
                                    int64_t m, const bonsai_weights* w,
                                    int32_t* d_out, uint16_t* y_out,
                                    bonsai_stream stream);

/* Activation binarisation: the +-1 A operand of bonsai_xnor_gemm, made from
 * FP16 activation rows in one pass over x. The pages ("1-bit 嘅數學") use
 * XOR + popcount for +-1 operands but give no rule for the activation side;
 * this library's rule is
 *   code a[r][k] = +1 where x[r][k] >= 0 (+0 and -0 included; NaN gives -1),
 *   scale a_s[r] = (1/k) * sum_k |x[r][k]|,
 * the least-squares scale for those codes: it minimises
 * sum_k (x[r][k] - a_s * a[r][k])^2.
 *   x       device FP16 [m][k], row-major, 16-byte aligned.
 *   m       rows, >= 1.  k: multiple of 128.
 *   a_bits  device uint32 [m][k/32], written in the BINARY weight layout
 *           (bit (k%32) of word k/32, bit 1 = +1), 16-byte aligned.
 *   a_scale device FP16 [m] (round to nearest even of the FP32 mean of |x|;
 *           within 2^-11 + k*2^-24 of the exact mean, relative), 16-byte
 *           aligned.
 * Codes are exact (no arithmetic decides them). A row holding a NaN gets a
 * NaN scale; an infinite entry gives an infinite scale. */
bonsai_status bonsai_binarize_activations(const uint16_t* x, int64_t m, int64_t k,
                                          uint32_t* a_bits, uint16_t* a_scale,
                                          bonsai_stream stream);

/* Signed Hadamard rotation of activation rows, for weights that were
 * rotated offline (OpenBonsai page, "工作原理": a signed Hadamard rotation is
 * one of its compression steps; the pages give neither its size nor where
 * the activations are rotated). Block-diagonal along K with power-of-two
 * blocks, orthonormal:
 *   out[r][b0 + i] = block^(-1/2) * sum_{j<block} H[i][j] * s[b0+j] * x[r][b0+j],
 *   H[i][j] = (-1)^popcount(i & j)   (Sylvester's Hadamard matrix),
 * for b0 = 0, block, 2*block, ...
 *   x      device FP16 [m][k], 16-byte aligned.
 *   m      rows, >= 1.   k: multiple of 128 and of block.
 *   block  8, 16, ..., 1024 (else BONSAI_ERR_UNSUPPORTED).
 *   signs  device uint32 [k/32], bit (k%32) of word k/32 = 1 for s = +1,
 *          0 for s = -1 (the BINARY weight layout); NULL for all +1.
 *   out    device FP16 [m][k], 16-byte aligned; may equal x (in place) but
 *          must not otherwise overlap it (BONSAI_ERR_INVALID_ARG).
 * FP32 butterflies (log2(block) stages), one FP16 rounding of each output. */
bonsai_status bonsai_hadamard(const uint16_t* x, int64_t m, int64_t k, int32_t block,
                              const uint32_t* signs, uint16_t* out, bonsai_stream stream);

/* Self-test of the failure path: launches one thread that waits on a
 * barrier nothing completes, with the same bounded wait the product kernels
 * use on their barriers but a limit of `limit_ns` nanoseconds of wall-clock
 * time (1 us .. 100 ms, else BONSAI_ERR_INVALID_ARG). The wait gives up, the
 * kernel records BONSAI_ERR_TIMEOUT and returns; the next
 * bonsai_check_async on the stream reports it (and clears it), and the
 * device stays usable. No fault or trap is involved. */
bonsai_status bonsai_selftest_wait_timeout(uint64_t limit_ns, bonsai_stream stream);

/* Synchronises `stream`, then returns and clears the device status word of
 * the current device: BONSAI_OK, BONSAI_ERR_BAD_CODE or BONSAI_ERR_TIMEOUT.
 * Returns BONSAI_ERR_CUDA if the stream reported a CUDA error. */
bonsai_status bonsai_check_async(bonsai_stream stream);

/* Static, human-readable name of a status code. Never NULL. */
const char* bonsai_status_string(bonsai_status status);

#ifdef __cplusplus
}
#endif

#endif /* BONSAI_H */
