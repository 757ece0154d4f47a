// api.cu -- the C ABI of libbonsai (declared in include/bonsai.h): argument
// checks on the host, then one asynchronous launch on the caller's stream.
#include <mutex>

#include "common.cuh"

namespace bonsai {

// Launchers and status readers of the other translation units.
bonsai_status pack_binary_launch(const int8_t*, int64_t, int64_t, void*, int64_t, cudaStream_t);
bonsai_status pack_ternary_launch(const int8_t*, int64_t, int64_t, void*, int64_t, cudaStream_t);
bonsai_status gemv_launch(const bonsai_weights*, const uint16_t*, int64_t, uint16_t*, bool,
                          cudaStream_t);
bonsai_status splitk_launch(const bonsai_weights*, const uint16_t*, uint16_t*, cudaStream_t);
bonsai_status stage_x_launch(const uint16_t*, uint16_t*, int64_t, cudaStream_t);
bonsai_status gemm_launch(const bonsai_weights*, const uint16_t*, int64_t, uint16_t*, bool,
                          cudaStream_t, void* ws = nullptr, int64_t ws_bytes = 0);
int64_t gemm_workspace_bytes(const bonsai_weights*, int64_t);
int64_t gemv_lut_workspace_bytes(const bonsai_weights*);
bonsai_status gemv_lut_launch(const bonsai_weights*, const uint16_t*, uint16_t*, bool, void*,
                              int64_t, cudaStream_t);
bonsai_status xnor_launch(const uint32_t*, const uint16_t*, int64_t, const bonsai_weights*,
                          int32_t*, uint16_t*, cudaStream_t);
bonsai_status xnor_tc_launch(const uint32_t*, const uint16_t*, int64_t, const bonsai_weights*,
                             int32_t*, uint16_t*, cudaStream_t);
bonsai_status binarize_launch(const uint16_t*, int64_t, int64_t, uint32_t*, uint16_t*,
                              cudaStream_t);
bonsai_status hadamard_launch(const uint16_t*, int64_t, int64_t, int32_t, const uint32_t*,
                              uint16_t*, cudaStream_t);
bonsai_status selftest_wait_timeout_launch(uint64_t, cudaStream_t);
int64_t gemv_plan_bytes(int64_t);
bonsai_status gemv_plan_init(const bonsai_decode_step*, int64_t, void*, cudaStream_t);
bonsai_status gemv_plan_run(const bonsai_decode_step*, int64_t, void*, cudaStream_t);
bonsai_status plan_wait_selftest_launch(uint64_t, cudaStream_t);
unsigned int read_clear_status_selftest();
unsigned int read_clear_status_pack();
unsigned int read_clear_status_gemv();
unsigned int read_clear_status_gemm();
unsigned int read_clear_status_xnor();
unsigned int read_clear_status_xnor_tc();
unsigned int read_clear_status_lut();

namespace {
constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices];
int g_smem[kMaxDevices];
std::once_flag g_once[kMaxDevices];

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  return dev;
}

void query(int dev) {
  std::call_once(g_once[dev], [dev] {
    cudaDeviceGetAttribute(&g_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&g_smem[dev], cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  });
}
}  // namespace

int device_sm_count() {
  const int dev = current_device();
  query(dev);
  return g_sms[dev] > 0 ? g_sms[dev] : 1;
}

int device_max_smem_optin() {
  const int dev = current_device();
  query(dev);
  return g_smem[dev];
}

cudaError_t ensure_dynamic_smem(const void* kernel, int bytes) {
  struct Entry { const void* fn; int dev; int bytes; };
  static std::mutex mu;
  static Entry table[256];
  static int used = 0;
  const int dev = current_device();
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i) {
    if (table[i].fn == kernel && table[i].dev == dev) {
      if (table[i].bytes >= bytes) return cudaSuccess;
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      if (e == cudaSuccess) table[i].bytes = bytes;
      return e;
    }
  }
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && used < 256) table[used++] = Entry{kernel, dev, bytes};
  return e;
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType type, void* base, uint64_t dim0,
                          uint64_t dim1, uint64_t stride1_bytes, uint32_t box0, uint32_t box1,
                          CUtensorMapSwizzle swizzle) {
  static EncodeTiled fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<EncodeTiled>(f);
  }();
  if (!fn) return false;
  // A map depends only on these arguments, so the maps of recent calls are
  // kept (a decode loop encodes the same weights every token). A reused
  // address with the same shape gets the same, still correct, map.
  struct Key {
    CUtensorMapDataType type;
    void* base;
    uint64_t dim0, dim1, stride1;
    uint32_t box0, box1;
    CUtensorMapSwizzle swizzle;
    bool operator==(const Key& o) const {
      return type == o.type && base == o.base && dim0 == o.dim0 && dim1 == o.dim1 &&
             stride1 == o.stride1 && box0 == o.box0 && box1 == o.box1 && swizzle == o.swizzle;
    }
  };
  struct Entry { Key key; CUtensorMap map; bool used; };
  constexpr int kEntries = 64;
  static Entry cache[kEntries];
  static int next = 0;
  static std::mutex mu;
  const Key key{type, base, dim0, dim1, stride1_bytes, box0, box1, swizzle};
  {
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry& e : cache)
      if (e.used && e.key == key) {
        *map = e.map;
        return true;
      }
  }
  const cuuint64_t gdim[2] = {dim0, dim1};
  const cuuint64_t gstride[1] = {stride1_bytes};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  if (fn(map, type, 2, base, gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lock(mu);
  cache[next] = Entry{key, *map, true};
  next = (next + 1) % kEntries;
  return true;
}

}  // namespace bonsai

namespace {

using namespace bonsai;

constexpr int64_t kMaxK = 1 << 20;
constexpr int64_t kMaxN = 1 << 30;
constexpr int64_t kMaxM = 1 << 24;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bonsai_status check_workspace(const void* ws, int64_t ws_bytes) {
  if (ws_bytes < 0 || (ws_bytes > 0 && !ws)) return BONSAI_ERR_INVALID_ARG;
  if (ws && (reinterpret_cast<uintptr_t>(ws) & 255u)) return BONSAI_ERR_ALIGN;
  return BONSAI_OK;
}

bonsai_status check_row_bytes(int32_t format, int64_t k, int64_t row_bytes) {
  if (format == BONSAI_FMT_BINARY) {
    if (row_bytes < k / 8 || row_bytes % 16) return BONSAI_ERR_SHAPE;
  } else {
    if (row_bytes < bonsai_packed_row_bytes(BONSAI_FMT_TERNARY, k) || row_bytes % 64)
      return BONSAI_ERR_SHAPE;
  }
  return BONSAI_OK;
}

bonsai_status check_weights(const bonsai_weights* w) {
  if (!w || !w->packed || !w->scales) return BONSAI_ERR_INVALID_ARG;
  if (w->format != BONSAI_FMT_BINARY && w->format != BONSAI_FMT_TERNARY)
    return BONSAI_ERR_INVALID_ARG;
  if (w->flags & ~int32_t(BONSAI_WEIGHTS_PREFETCH)) return BONSAI_ERR_INVALID_ARG;
  if (w->n <= 0 || w->k <= 0 || w->row_bytes <= 0) return BONSAI_ERR_INVALID_ARG;
  if (w->k % 128) return BONSAI_ERR_SHAPE;
  if (w->k > kMaxK || w->n > kMaxN) return BONSAI_ERR_UNSUPPORTED;
  bonsai_status st = check_row_bytes(w->format, w->k, w->row_bytes);
  if (st != BONSAI_OK) return st;
  if (!aligned16(w->packed) || !aligned16(w->scales)) return BONSAI_ERR_ALIGN;
  return BONSAI_OK;
}

bonsai_status check_pack(const int8_t* codes, int64_t rows, int64_t k, void* out,
                         int64_t row_bytes, int32_t format) {
  if (!codes || !out) return BONSAI_ERR_INVALID_ARG;
  if (rows < 0 || k <= 0 || row_bytes <= 0) return BONSAI_ERR_INVALID_ARG;
  if (k % 128) return BONSAI_ERR_SHAPE;
  if (k > kMaxK || rows > kMaxN) return BONSAI_ERR_UNSUPPORTED;
  bonsai_status st = check_row_bytes(format, k, row_bytes);
  if (st != BONSAI_OK) return st;
  if (!aligned16(codes) || !aligned16(out)) return BONSAI_ERR_ALIGN;
  return BONSAI_OK;
}

}  // namespace

extern "C" {

int64_t bonsai_packed_row_bytes(int32_t format, int64_t k) {
  if (k <= 0 || k % 128) return -1;
  if (format == BONSAI_FMT_BINARY) return k / 8;
  if (format == BONSAI_FMT_TERNARY) {
    const int64_t data = (k + 4) / 5;
    return 64 * ((data + 63) / 64);
  }
  return -1;
}

bonsai_status bonsai_pack_binary(const int8_t* codes, int64_t rows, int64_t k, void* out,
                                 int64_t row_bytes, bonsai_stream stream) {
  bonsai_status st = check_pack(codes, rows, k, out, row_bytes, BONSAI_FMT_BINARY);
  if (st != BONSAI_OK) return st;
  return pack_binary_launch(codes, rows, k, out, row_bytes, stream);
}

bonsai_status bonsai_pack_ternary(const int8_t* codes, int64_t rows, int64_t k, void* out,
                                  int64_t row_bytes, bonsai_stream stream) {
  bonsai_status st = check_pack(codes, rows, k, out, row_bytes, BONSAI_FMT_TERNARY);
  if (st != BONSAI_OK) return st;
  return pack_ternary_launch(codes, rows, k, out, row_bytes, stream);
}

// One token on the device: the table kernel when a large enough workspace
// is given and the shape takes it, else the streaming decode kernel, else
// (very long rows: the decode kernel's per-CTA x table no longer fits in
// shared memory) the tensor-core kernel, which takes any K.
static bonsai_status gemv_any(const bonsai_weights* w, const uint16_t* x, uint16_t* y,
                              void* ws, int64_t ws_bytes, cudaStream_t stream) {
  bonsai_status st = gemv_lut_launch(w, x, y, false, ws, ws_bytes, stream);
  if (st != BONSAI_ERR_UNSUPPORTED) return st;
  st = gemv_launch(w, x, 1, y, false, stream);
  if (st == BONSAI_ERR_UNSUPPORTED) st = gemm_launch(w, x, 1, y, false, stream);
  return st;
}

static bonsai_status gemv_common(const bonsai_weights* w, const uint16_t* x, uint16_t* y,
                                 void* ws, int64_t ws_bytes, bonsai_stream stream) {
  bonsai_status st = check_weights(w);
  if (st != BONSAI_OK) return st;
  if (!x || !y) return BONSAI_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y)) return BONSAI_ERR_ALIGN;
  st = check_workspace(ws, ws_bytes);
  if (st != BONSAI_OK) return st;
  return gemv_any(w, x, y, ws, ws_bytes, stream);
}

bonsai_status bonsai_gemv(const bonsai_weights* w, const uint16_t* x, uint16_t* y,
                          bonsai_stream stream) {
  return gemv_common(w, x, y, nullptr, 0, stream);
}

int64_t bonsai_gemv_workspace_bytes(const bonsai_weights* w) {
  if (check_weights(w) != BONSAI_OK) return 0;
  return gemv_lut_workspace_bytes(w);
}

bonsai_status bonsai_gemv_ws(const bonsai_weights* w, const uint16_t* x, uint16_t* y,
                             void* workspace, int64_t workspace_bytes, bonsai_stream stream) {
  return gemv_common(w, x, y, workspace, workspace_bytes, stream);
}

static bonsai_status gemv_host_common(const bonsai_weights* w, const uint16_t* x_host,
                                      uint16_t* x_dev, uint16_t* y_dev, uint16_t* y_host,
                                      void* ws, int64_t ws_bytes, bonsai_stream stream) {
  bonsai_status st = check_weights(w);
  if (st != BONSAI_OK) return st;
  if (!x_host || !x_dev || !y_dev || !y_host) return BONSAI_ERR_INVALID_ARG;
  if (!aligned16(x_dev) || !aligned16(y_dev)) return BONSAI_ERR_ALIGN;
  st = check_workspace(ws, ws_bytes);
  if (st != BONSAI_OK) return st;
  // Page-locked host buffers are mapped into the device address space: the
  // activations are then read by a small kernel and the result is written by
  // the product kernel itself, so no copy-engine transfer (with its fixed
  // latency) sits between the launches. Other host memory goes through
  // cudaMemcpyAsync.
  auto mapped = [](const void* p) -> const void* {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
      cudaGetLastError();  // an unknown pointer is not an error here
      return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
  };
  const void* xm = aligned16(x_host) ? mapped(x_host) : nullptr;
  void* ym = aligned16(y_host) ? const_cast<void*>(mapped(y_host)) : nullptr;
  if (xm) {
    st = stage_x_launch(static_cast<const uint16_t*>(xm), x_dev, w->k, stream);
  } else {
    st = cudaMemcpyAsync(x_dev, x_host, (size_t)w->k * 2, cudaMemcpyHostToDevice, stream) ==
                 cudaSuccess ? BONSAI_OK : BONSAI_ERR_CUDA;
  }
  if (st != BONSAI_OK) return st;
  uint16_t* y_out = ym ? static_cast<uint16_t*>(ym) : y_dev;
  st = gemv_any(w, x_dev, y_out, ws, ws_bytes, stream);
  if (st != BONSAI_OK || ym) return st;
  if (cudaMemcpyAsync(y_host, y_dev, (size_t)w->n * 2, cudaMemcpyDeviceToHost, stream) !=
      cudaSuccess)
    return BONSAI_ERR_CUDA;
  return BONSAI_OK;
}

bonsai_status bonsai_gemv_host(const bonsai_weights* w, const uint16_t* x_host,
                               uint16_t* x_dev, uint16_t* y_dev, uint16_t* y_host,
                               bonsai_stream stream) {
  return gemv_host_common(w, x_host, x_dev, y_dev, y_host, nullptr, 0, stream);
}

bonsai_status bonsai_gemv_host_ws(const bonsai_weights* w, const uint16_t* x_host,
                                  uint16_t* x_dev, uint16_t* y_dev, uint16_t* y_host,
                                  void* workspace, int64_t workspace_bytes,
                                  bonsai_stream stream) {
  return gemv_host_common(w, x_host, x_dev, y_dev, y_host, workspace, workspace_bytes, stream);
}

bonsai_status bonsai_gemv_splitk_static(const bonsai_weights* w, const uint16_t* x, uint16_t* y,
                                        bonsai_stream stream) {
  bonsai_status st = check_weights(w);
  if (st != BONSAI_OK) return st;
  if (!x || !y) return BONSAI_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y)) return BONSAI_ERR_ALIGN;
  return splitk_launch(w, x, y, stream);
}

// bonsai_gemm / bonsai_gemm_swiglu, with or without a stream-K workspace
static bonsai_status gemm_common(const bonsai_weights* w, const uint16_t* x, int64_t m,
                                 uint16_t* y, bool swiglu, void* ws, int64_t ws_bytes,
                                 bonsai_stream stream) {
  bonsai_status st = check_weights(w);
  if (st != BONSAI_OK) return st;
  if (!x || !y || m <= 0) return BONSAI_ERR_INVALID_ARG;
  if (swiglu && w->n % 16) return BONSAI_ERR_SHAPE;
  if (m > kMaxM) return BONSAI_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(y)) return BONSAI_ERR_ALIGN;
  st = check_workspace(ws, ws_bytes);
  if (st != BONSAI_OK) return st;
  if (m == 1) {
    st = gemv_lut_launch(w, x, y, swiglu, ws, ws_bytes, stream);
    if (st != BONSAI_ERR_UNSUPPORTED) return st;
  }
  if (m <= 8) {
    st = gemv_launch(w, x, m, y, swiglu, stream);
    if (st != BONSAI_ERR_UNSUPPORTED) return st;
  }
  return gemm_launch(w, x, m, y, swiglu, stream, ws, ws_bytes);
}

bonsai_status bonsai_gemm(const bonsai_weights* w, const uint16_t* x, int64_t m, uint16_t* y,
                          bonsai_stream stream) {
  return gemm_common(w, x, m, y, false, nullptr, 0, stream);
}

bonsai_status bonsai_gemm_swiglu(const bonsai_weights* w, const uint16_t* x, int64_t m,
                                 uint16_t* h, bonsai_stream stream) {
  return gemm_common(w, x, m, h, true, nullptr, 0, stream);
}

int64_t bonsai_gemm_workspace_bytes(const bonsai_weights* w, int64_t m) {
  if (check_weights(w) != BONSAI_OK || m < 1 || m > kMaxM) return 0;
  if (m == 1) return gemv_lut_workspace_bytes(w);
  if (m <= 8) return 0;
  return gemm_workspace_bytes(w, m);
}

bonsai_status bonsai_gemm_ws(const bonsai_weights* w, const uint16_t* x, int64_t m, uint16_t* y,
                             void* workspace, int64_t workspace_bytes, bonsai_stream stream) {
  return gemm_common(w, x, m, y, false, workspace, workspace_bytes, stream);
}

bonsai_status bonsai_gemm_swiglu_ws(const bonsai_weights* w, const uint16_t* x, int64_t m,
                                    uint16_t* h, void* workspace, int64_t workspace_bytes,
                                    bonsai_stream stream) {
  return gemm_common(w, x, m, h, true, workspace, workspace_bytes, stream);
}

static bonsai_status check_xnor(const uint32_t* a_bits, const uint16_t* a_scale, int64_t m,
                                const bonsai_weights* w, int32_t* d_out, uint16_t* y_out) {
  bonsai_status st = check_weights(w);
  if (st != BONSAI_OK) return st;
  if (w->format != BONSAI_FMT_BINARY) return BONSAI_ERR_FORMAT;
  if (!a_bits || !a_scale || m <= 0 || (!d_out && !y_out)) return BONSAI_ERR_INVALID_ARG;
  if (m > kMaxM) return BONSAI_ERR_UNSUPPORTED;
  if (!aligned16(a_bits) || !aligned16(a_scale) || (d_out && !aligned16(d_out)) ||
      (y_out && !aligned16(y_out)))
    return BONSAI_ERR_ALIGN;
  return BONSAI_OK;
}

bonsai_status bonsai_xnor_gemm(const uint32_t* a_bits, const uint16_t* a_scale, int64_t m,
                               const bonsai_weights* w, int32_t* d_out, uint16_t* y_out,
                               bonsai_stream stream) {
  const bonsai_status st = check_xnor(a_bits, a_scale, m, w, d_out, y_out);
  if (st != BONSAI_OK) return st;
  return xnor_tc_launch(a_bits, a_scale, m, w, d_out, y_out, stream);
}

bonsai_status bonsai_xnor_gemm_popc(const uint32_t* a_bits, const uint16_t* a_scale, int64_t m,
                                    const bonsai_weights* w, int32_t* d_out, uint16_t* y_out,
                                    bonsai_stream stream) {
  const bonsai_status st = check_xnor(a_bits, a_scale, m, w, d_out, y_out);
  if (st != BONSAI_OK) return st;
  return xnor_launch(a_bits, a_scale, m, w, d_out, y_out, stream);
}

bonsai_status bonsai_binarize_activations(const uint16_t* x, int64_t m, int64_t k,
                                          uint32_t* a_bits, uint16_t* a_scale,
                                          bonsai_stream stream) {
  if (!x || !a_bits || !a_scale || m <= 0) return BONSAI_ERR_INVALID_ARG;
  if (k <= 0 || k % 128) return BONSAI_ERR_SHAPE;
  if (m > kMaxM || k > kMaxK) return BONSAI_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(a_bits) || !aligned16(a_scale)) return BONSAI_ERR_ALIGN;
  return binarize_launch(x, m, k, a_bits, a_scale, stream);
}

bonsai_status bonsai_hadamard(const uint16_t* x, int64_t m, int64_t k, int32_t block,
                              const uint32_t* signs, uint16_t* out, bonsai_stream stream) {
  if (!x || !out || m <= 0) return BONSAI_ERR_INVALID_ARG;
  if (block < 8 || block > 1024 || (block & (block - 1))) return BONSAI_ERR_UNSUPPORTED;
  if (k <= 0 || k % 128 || k % block) return BONSAI_ERR_SHAPE;
  if (m > kMaxM || k > kMaxK) return BONSAI_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(out) || (reinterpret_cast<uintptr_t>(signs) & 3u))
    return BONSAI_ERR_ALIGN;
  if (x != out) {  // distinct buffers must not overlap
    const uintptr_t a = reinterpret_cast<uintptr_t>(x), b = reinterpret_cast<uintptr_t>(out);
    const uintptr_t bytes = static_cast<uintptr_t>(m) * static_cast<uintptr_t>(k) * 2u;
    if (a < b + bytes && b < a + bytes) return BONSAI_ERR_INVALID_ARG;
  }
  return hadamard_launch(x, m, k, block, signs, out, stream);
}

// ---------------------------------------------------------------- plans
namespace {
constexpr int64_t kMaxPlanSteps = 4096;

bonsai_status check_plan_steps(const bonsai_decode_step* steps, int64_t count) {
  if (!steps || count < 1) return BONSAI_ERR_INVALID_ARG;
  if (count > kMaxPlanSteps) return BONSAI_ERR_INVALID_ARG;
  for (int64_t j = 0; j < count; ++j) {
    const bonsai_decode_step& st = steps[j];
    bonsai_status e = check_weights(&st.w);
    if (e != BONSAI_OK) return e;
    if (st.w.format != BONSAI_FMT_TERNARY) return BONSAI_ERR_FORMAT;
    if (!st.x || !st.y) return BONSAI_ERR_INVALID_ARG;
    if (st.swiglu != 0 && st.swiglu != 1) return BONSAI_ERR_INVALID_ARG;
    if (st.after < -1 || st.after >= j) return BONSAI_ERR_INVALID_ARG;
    if (st.swiglu && st.w.n % 16) return BONSAI_ERR_SHAPE;
    if (!aligned16(st.x) || !aligned16(st.y)) return BONSAI_ERR_ALIGN;
  }
  return BONSAI_OK;
}
}  // namespace

int64_t bonsai_decode_plan_bytes(int64_t count) {
  if (count < 1 || count > kMaxPlanSteps) return -1;
  return gemv_plan_bytes(count);
}

bonsai_status bonsai_decode_plan_init(const bonsai_decode_step* steps, int64_t count,
                                      void* plan, int64_t plan_bytes, bonsai_stream stream) {
  bonsai_status st = check_plan_steps(steps, count);
  if (st != BONSAI_OK) return st;
  if (!plan) return BONSAI_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(plan) % 128) return BONSAI_ERR_ALIGN;
  if (plan_bytes < gemv_plan_bytes(count)) return BONSAI_ERR_INVALID_ARG;
  return gemv_plan_init(steps, count, plan, stream);
}

bonsai_status bonsai_decode_run(const bonsai_decode_step* steps, int64_t count, void* plan,
                                bonsai_stream stream) {
  bonsai_status st = check_plan_steps(steps, count);
  if (st != BONSAI_OK) return st;
  if (!plan) return BONSAI_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(plan) % 128) return BONSAI_ERR_ALIGN;
  return gemv_plan_run(steps, count, plan, stream);
}

bonsai_status bonsai_selftest_plan_wait(uint64_t limit_ns, bonsai_stream stream) {
  if (limit_ns < 1000 || limit_ns > 100000000) return BONSAI_ERR_INVALID_ARG;
  return plan_wait_selftest_launch(limit_ns, stream);
}

bonsai_status bonsai_selftest_wait_timeout(uint64_t limit_ns, bonsai_stream stream) {
  if (limit_ns < 1000 || limit_ns > 100000000) return BONSAI_ERR_INVALID_ARG;
  return selftest_wait_timeout_launch(limit_ns, stream);
}

bonsai_status bonsai_check_async(bonsai_stream stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return BONSAI_ERR_CUDA;
  const unsigned int codes[7] = {read_clear_status_pack(),    read_clear_status_gemv(),
                                 read_clear_status_gemm(),    read_clear_status_xnor(),
                                 read_clear_status_xnor_tc(), read_clear_status_lut(),
                                 read_clear_status_selftest()};
  if (cudaGetLastError() != cudaSuccess) return BONSAI_ERR_CUDA;
  for (unsigned int c : codes)
    if (c != 0) return static_cast<bonsai_status>(c);
  return BONSAI_OK;
}

const char* bonsai_status_string(bonsai_status status) {
  switch (status) {
    case BONSAI_OK: return "BONSAI_OK";
    case BONSAI_ERR_INVALID_ARG: return "BONSAI_ERR_INVALID_ARG";
    case BONSAI_ERR_SHAPE: return "BONSAI_ERR_SHAPE";
    case BONSAI_ERR_ALIGN: return "BONSAI_ERR_ALIGN";
    case BONSAI_ERR_FORMAT: return "BONSAI_ERR_FORMAT";
    case BONSAI_ERR_CUDA: return "BONSAI_ERR_CUDA";
    case BONSAI_ERR_UNSUPPORTED: return "BONSAI_ERR_UNSUPPORTED";
    case BONSAI_ERR_TIMEOUT: return "BONSAI_ERR_TIMEOUT";
    case BONSAI_ERR_BAD_CODE: return "BONSAI_ERR_BAD_CODE";
  }
  return "BONSAI_ERR_UNKNOWN";
}

}  // extern "C"
