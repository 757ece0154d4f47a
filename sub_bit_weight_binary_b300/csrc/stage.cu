// stage.cu -- activations from page-locked host memory into a device buffer,
// for bonsai_gemv_host.
#include "common.cuh"

namespace bonsai {
namespace stage {

// Copy of the activations from page-locked host memory (read through its
// device mapping) into the device x buffer, for bonsai_gemv_host: one small
// grid instead of a copy-engine transfer, so the decode kernel that follows
// can start under programmatic dependent launch. Waits for earlier work on the
// stream first: the previous decode step may still read x_dev.
__global__ void __launch_bounds__(256) stage_x_kernel(const uint4* src, uint4* dst, int n16) {
  pdl_wait();
  pdl_launch_dependents();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += gridDim.x * blockDim.x)
    dst[i] = src[i];
}

}  // namespace stage

bonsai_status stage_x_launch(const uint16_t* src_mapped, uint16_t* dst, int64_t k,
                             cudaStream_t stream) {
  const int n16 = (int)(k / 8);  // k % 128 == 0
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)((n16 + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cuda_status(cudaLaunchKernelEx(&cfg, stage::stage_x_kernel,
                                        reinterpret_cast<const uint4*>(src_mapped),
                                        reinterpret_cast<uint4*>(dst), n16));
}

}  // namespace bonsai
