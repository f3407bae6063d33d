// kernels_grad.cu -- helpers of the projector gradient of the backward pass.
//
// Backward pass of MAPL §3.2 (the gradient of the boundary is routed through
// the same projector A): with X_res = X - E[tids] P, Z = X_res A and
// gZ = dL/dX_hat A, the Euclidean gradient that feeds SPEL is
//     dL/dA = X_res^T gZ + dL/dX_hat^T Z
//           = X^T gZ + dL/dX_hat^T Z - P^T (E[tids]^T gZ).
// The products are plain GEMMs (cuBLAS); this file gathers the anchor rows
// E[tids] into a dense N x r operand and widens P to fp32 for the last one.
// It also lays out the first-boundary anchor table (Fig. 2: the first stage
// subtracts the original token embeddings): (E_emb A)[tids] as three bf16
// terms multiplied by -[I; I; I] in the compress kernel's anchor fold.
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

// First-boundary anchor table: row v of T = E_emb A (fp32, V x r) as three
// bf16 terms side by side, [hi | mid | lo] (V x 3r), the remainder of each
// term carried into the next.
__global__ void k_split3(const float* __restrict__ T, size_t V, int r, __nv_bfloat16* __restrict__ Tb) {
  const size_t x = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (x >= V * r) return;
  const size_t v = x / r;
  const int j = static_cast<int>(x % r);
  float rem = T[x];
  for (int s = 0; s < 3; ++s) {
    const __nv_bfloat16 b = __float2bfloat16_rn(rem);
    Tb[v * 3 * r + s * r + j] = b;
    rem -= __bfloat162float(b);
  }
}

// -[I; I; I]^T as the K-major B operand of the anchor fold (r x 3r):
// entry (j, k) is -1 where k mod r == j.
__global__ void k_neg_identity3(int r, __nv_bfloat16* __restrict__ M) {
  const int x = blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= 3 * r * r) return;
  const int j = x / (3 * r), k = x % (3 * r);
  M[x] = __float2bfloat16_rn(k % r == j ? -1.f : 0.f);
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

cudaError_t launch_split3(const float* T, size_t V, int r, __nv_bfloat16* Tb, cudaStream_t s) {
  const size_t n = V * static_cast<size_t>(r);
  k_split3<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(T, V, r, Tb);
  return cudaGetLastError();
}

cudaError_t launch_neg_identity3(int r, __nv_bfloat16* M, cudaStream_t s) {
  k_neg_identity3<<<(3 * r * r + 255) / 256, 256, 0, s>>>(r, M);
  return cudaGetLastError();
}

cudaError_t launch_widen(const __nv_bfloat16* a, size_t n, float* b, cudaStream_t s) {
  k_widen<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(a, n, b);
  return cudaGetLastError();
}

}  // namespace mapl
