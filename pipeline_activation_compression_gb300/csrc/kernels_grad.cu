// kernels_grad.cu -- helpers of the projector gradient of the backward pass.
//
// Backward pass of MAPL §3.2 (the gradient of the boundary is routed through
// the same projector A): with X_res = X - E[tids] P, Z = X_res A and
// gZ = dL/dX_hat A, the Euclidean gradient that feeds SPEL is
//     dL/dA = X_res^T gZ + dL/dX_hat^T Z
//           = X^T gZ + dL/dX_hat^T Z - P^T (E[tids]^T gZ).
// The products are plain GEMMs (cuBLAS); this file gathers the anchor rows
// E[tids] into a dense N x r operand and widens P to fp32 for the last one.
#include "mapl_internal.h"

namespace mapl {

namespace {

// Eg[n] = E[tids[n]] (zero rows for ids outside [0, V)), 16 bytes per thread.
__global__ void k_gather_rows(const int32_t* __restrict__ tids, const uint4* __restrict__ E,
                              int N, int V, int row16, uint4* __restrict__ Eg) {
  const size_t x = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (x >= static_cast<size_t>(N) * row16) return;
  const int n = static_cast<int>(x / row16), c = static_cast<int>(x % row16);
  const int t = tids[n];
  Eg[x] = (t >= 0 && t < V) ? E[static_cast<size_t>(t) * row16 + c] : make_uint4(0u, 0u, 0u, 0u);
}

__global__ void k_widen(const __nv_bfloat16* __restrict__ a, size_t n, float* __restrict__ b) {
  const size_t x = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (x < n) b[x] = __bfloat162float(a[x]);
}

}  // namespace

cudaError_t launch_gather_rows(const int32_t* tids, const __nv_bfloat16* E, int N, int V, int r,
                               __nv_bfloat16* Eg, cudaStream_t s) {
  const int row16 = r / 8;   // r is a multiple of 64 on the tensor-core path
  const size_t total = static_cast<size_t>(N) * row16;
  k_gather_rows<<<static_cast<unsigned>((total + 255) / 256), 256, 0, s>>>(
      tids, reinterpret_cast<const uint4*>(E), N, V, row16, reinterpret_cast<uint4*>(Eg));
  return cudaGetLastError();
}

cudaError_t launch_widen(const __nv_bfloat16* a, size_t n, float* b, cudaStream_t s) {
  k_widen<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(a, n, b);
  return cudaGetLastError();
}

}  // namespace mapl
