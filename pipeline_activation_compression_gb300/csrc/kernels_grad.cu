// kernels_grad.cu -- anchor term of the Euclidean gradient of the projector.
//
// Backward pass of MAPL §3.2 (the gradient of the boundary is routed through
// the same projector A): with X_res = X - E[tids] P, Z = X_res A and
// gZ = dL/dX_hat A, the Euclidean gradient that feeds SPEL is
//     dL/dA = X_res^T gZ + dL/dX_hat^T Z
//           = X^T gZ + dL/dX_hat^T Z - P^T (E[tids]^T gZ).
// The two dense products are plain GEMMs (cuBLAS, bf16 in, fp32 out); this
// file computes the anchor correction: S = E[tids]^T gZ (r x r, fp32) and
// dA -= P^T S.
#include "mapl_internal.h"

namespace mapl {

namespace {

constexpr int kOT = 128;     // S tile (kOT x kOT) per block
constexpr int kTokBatch = 16;

// S[i][j] += sum_n E[t_n][i] * gZ[n][j] over a chunk of tokens, one 128 x 128
// tile of S per block (blockIdx.y: tile), fp32 accumulation, atomics at the end.
__global__ void __launch_bounds__(256) k_anchor_outer(const int32_t* __restrict__ tids,
                                                      const __nv_bfloat16* __restrict__ E,
                                                      const __nv_bfloat16* __restrict__ gZ,
                                                      int N, int r, int V, int chunk,
                                                      float* __restrict__ S) {
  __shared__ float es[kTokBatch][kOT];
  __shared__ float gs[kTokBatch][kOT];
  const int ntj = (r + kOT - 1) / kOT;
  const int i0 = (blockIdx.y / ntj) * kOT, j0 = (blockIdx.y % ntj) * kOT;
  const int ti = threadIdx.x / 16, tj = threadIdx.x % 16;   // 8 x 8 sub-tile each
  float acc[8][8];
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) acc[a][b] = 0.f;
  const int n0 = blockIdx.x * chunk, n1 = min(N, n0 + chunk);
  for (int nb = n0; nb < n1; nb += kTokBatch) {
    __syncthreads();
    for (int x = threadIdx.x; x < kTokBatch * kOT; x += blockDim.x) {
      const int k = x / kOT, c = x % kOT, n = nb + k;
      float ev = 0.f, gv = 0.f;
      if (n < n1) {
        int t = tids[n];
        if (t >= 0 && t < V) {
          if (i0 + c < r) ev = __bfloat162float(E[static_cast<size_t>(t) * r + i0 + c]);
        }
        if (j0 + c < r) gv = __bfloat162float(gZ[static_cast<size_t>(n) * r + j0 + c]);
      }
      es[k][c] = ev;
      gs[k][c] = gv;
    }
    __syncthreads();
#pragma unroll 4
    for (int k = 0; k < kTokBatch; ++k) {
      float e8[8], g8[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) e8[a] = es[k][ti * 8 + a];
#pragma unroll
      for (int b = 0; b < 8; ++b) g8[b] = gs[k][tj * 8 + b];
#pragma unroll
      for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[a][b] = fmaf(e8[a], g8[b], acc[a][b]);
    }
  }
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int i = i0 + ti * 8 + a, j = j0 + tj * 8 + b;
      if (i < r && j < r) atomicAdd(S + static_cast<size_t>(i) * r + j, acc[a][b]);
    }
}

// dA[i][j] -= sum_k P[k][i] * S[k][j]   (P: r x d, dA: d x r, row-major)
__global__ void k_anchor_apply(const __nv_bfloat16* __restrict__ P, const float* __restrict__ S,
                               int d, int r, float* __restrict__ dA) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  const int i = blockIdx.y;
  if (j >= r || i >= d) return;
  float s = 0.f;
  for (int k = 0; k < r; ++k)
    s = fmaf(__bfloat162float(P[static_cast<size_t>(k) * d + i]), S[static_cast<size_t>(k) * r + j], s);
  dA[static_cast<size_t>(i) * r + j] -= s;
}

}  // namespace

cudaError_t launch_anchor_grad(const int32_t* tids, const __nv_bfloat16* E,
                               const __nv_bfloat16* gZ, const __nv_bfloat16* P, int N, int d,
                               int r, int V, int num_sms, float* S, float* dA, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(S, 0, static_cast<size_t>(r) * r * sizeof(float), s);
  if (e != cudaSuccess) return e;
  const int ntile = ((r + kOT - 1) / kOT) * ((r + kOT - 1) / kOT);
  int nblk = num_sms * 2 / ntile;
  if (nblk < 1) nblk = 1;
  int chunk = (N + nblk - 1) / nblk;
  chunk = (chunk + kTokBatch - 1) / kTokBatch * kTokBatch;
  nblk = (N + chunk - 1) / chunk;
  k_anchor_outer<<<dim3(nblk, ntile), 256, 0, s>>>(tids, E, gZ, N, r, V, chunk, S);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_anchor_apply<<<dim3((r + 127) / 128, d), 128, 0, s>>>(P, S, d, r, dA);
  return cudaGetLastError();
}

}  // namespace mapl
