// kernels_grad.cu -- operand layouts of the first-boundary anchor (Fig. 2:
// the first stage subtracts the original token embeddings): the table
// (E_emb A)[tids] as three bf16 terms, multiplied by -[I; I; I] in the
// compress kernel's anchor fold.
#include "mapl_internal.h"

namespace mapl {

namespace {

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

}  // namespace

cudaError_t launch_split3(const float* T, size_t V, int r, __nv_bfloat16* Tb, cudaStream_t s) {
  const size_t n = V * static_cast<size_t>(r);
  k_split3<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(T, V, r, Tb);
  return cudaGetLastError();
}

cudaError_t launch_neg_identity3(int r, __nv_bfloat16* M, cudaStream_t s) {
  k_neg_identity3<<<(3 * r * r + 255) / 256, 256, 0, s>>>(r, M);
  return cudaGetLastError();
}

}  // namespace mapl
