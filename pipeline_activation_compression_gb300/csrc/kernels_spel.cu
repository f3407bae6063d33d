// kernels_spel.cu -- SPEL projector update (MAPL §3.3 eqs. (4)-(7)), fp32.
//
// For each of `batch` independent boundaries (A, G, m are d x r):
//   H   = sym(A^T G)                       r x r   (split-K over d, then sym)
//   m   = beta m + (1 - beta)(G - A H)     eq. (4) + (5), fused epilogue
//   Y   = m / (||m||_F + 1e-7)
//   repeat n_lmo:  S = Y^T Y; Q = aI + bS + cS^2; Y = Y Q      eq. (6)
//   Y   = A - lr Y
//   repeat n_retr: same polynomial step                         eq. (7)
//   A   = Y
// When d and r are multiples of 128, A^T G and the three products of each
// polynomial step run on the tensor cores in emulated fp32
// (kernels_spel_tc.cu); A H with its momentum epilogue, and every product of
// other shapes, run in the tiled fp32 CUDA-core kernel below (32 x 32 output
// tiles, sequential fp32 accumulation per output).  r x r reductions over d
// use a fixed split-K followed by an ordered sum, so results are run-to-run
// deterministic.
#include "mapl_internal.h"
#include "pdl.cuh"

namespace mapl {

namespace {

constexpr int BK = 16;

enum Epi { kStore = 0, kMomentum = 1, kPoly = 2, kRefresh = 3 };

struct EpiArgs {
  const float* G;     // kMomentum: gradient
  float* m;           // kMomentum: momentum (read-modify-write)
  const float* S;     // kPoly: S
  float beta, a, b, c;
  long sG, sm, sS;    // batch strides
  RefreshTable rt;    // kRefresh: bf16 plan operands written beside C
};

// C[z] = op(A) B for z = blockIdx.z / ksplit; with ksplit > 1 each split
// writes its partial product to C + split * M * N (per batch).  TM x TM
// output tile per block of 64 threads (an 8 x 8 thread grid), each thread a
// (TM/8) x (TM/8) micro-tile read from shared memory as float4s.  TM = 32
// keeps the GEMMs of SPEL (r x r outputs, d x r with K = r) in enough blocks
// to fill the GPU.  Requires lda, ldb, N multiples of 4 (d, r are) and, for
// the non-transposed A, a split start that is a multiple of 4 (ksplit 1).
template <bool TA, int EPI, int TM>
__global__ void __launch_bounds__(64)
    k_sgemm(const float* __restrict__ A, const float* __restrict__ B, float* __restrict__ C,
            int M, int N, int K, int lda, int ldb, long sA, long sB, long sC, int ksplit,
            EpiArgs e) {
  pdl_enter();
  constexpr int MT = TM / 8;          // outputs per thread per dimension
  constexpr int V4 = TM / 16;         // float4 loads per thread per operand tile
  constexpr int R4 = TM / 4;          // float4s in a TM-wide row
  __shared__ __align__(16) float As[2][BK][TM + 4];
  __shared__ __align__(16) float Bs[2][BK][TM + 4];
  const int z = blockIdx.z / ksplit, ks = blockIdx.z % ksplit;
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TM;
  const int kbeg = static_cast<int>(static_cast<long>(K) * ks / ksplit);
  const int kend = static_cast<int>(static_cast<long>(K) * (ks + 1) / ksplit);
  A += z * sA;
  B += z * sB;
  const int t = threadIdx.x;
  const int ty = t >> 3, tx = t & 7;
  float acc[MT][MT];
#pragma unroll
  for (int i = 0; i < MT; ++i)
#pragma unroll
    for (int j = 0; j < MT; ++j) acc[i][j] = 0.f;
  auto load4 = [](const float* src, int valid) {
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (valid >= 4) {
      x = *reinterpret_cast<const float4*>(src);
    } else {
      if (valid > 0) x.x = src[0];
      if (valid > 1) x.y = src[1];
      if (valid > 2) x.z = src[2];
    }
    return x;
  };
  // the next K-tile is fetched into registers while the current one is
  // multiplied out of the other shared-memory buffer
  float4 ra[V4], rb[V4];
  auto fetch = [&](int k0) {
#pragma unroll
    for (int v = 0; v < V4; ++v) {
      if (TA) {   // A is K x M (row-major, ld lda): rows k, m contiguous
        const int kk = t / R4 + (64 / R4) * v, mm = (t % R4) * 4;
        const int gk = k0 + kk, gm = m0 + mm;
        ra[v] = gk < kend ? load4(A + static_cast<long>(gk) * lda + gm, M - gm)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
      } else {    // A is M x K: rows m, k contiguous
        const int mm = t % TM, kk = 4 * (t / TM + (64 / TM) * v);
        const int gm = m0 + mm, gk = k0 + kk;
        ra[v] = gm < M ? load4(A + static_cast<long>(gm) * lda + gk, kend - gk)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      const int kk = t / R4 + (64 / R4) * v, nn = (t % R4) * 4;   // B is K x N
      const int gk = k0 + kk, gn = n0 + nn;
      rb[v] = gk < kend ? load4(B + static_cast<long>(gk) * ldb + gn, N - gn)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  auto stash = [&](int buf) {
#pragma unroll
    for (int v = 0; v < V4; ++v) {
      if (TA) {
        const int kk = t / R4 + (64 / R4) * v, mm = (t % R4) * 4;
        *reinterpret_cast<float4*>(&As[buf][kk][mm]) = ra[v];
      } else {
        const int mm = t % TM, kk = 4 * (t / TM + (64 / TM) * v);
        As[buf][kk][mm] = ra[v].x;
        As[buf][kk + 1][mm] = ra[v].y;
        As[buf][kk + 2][mm] = ra[v].z;
        As[buf][kk + 3][mm] = ra[v].w;
      }
      const int kk = t / R4 + (64 / R4) * v, nn = (t % R4) * 4;
      *reinterpret_cast<float4*>(&Bs[buf][kk][nn]) = rb[v];
    }
  };
  int buf = 0;
  if (kbeg < kend) {
    fetch(kbeg);
    stash(0);
  }
  __syncthreads();
  for (int k0 = kbeg; k0 < kend; k0 += BK) {
    const bool more = k0 + BK < kend;
    if (more) fetch(k0 + BK);
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float av[MT], bv[MT];
#pragma unroll
      for (int q = 0; q < MT / 4; ++q) {
        const float4 a4 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * MT + 4 * q]);
        const float4 b4 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * MT + 4 * q]);
        av[4 * q] = a4.x; av[4 * q + 1] = a4.y; av[4 * q + 2] = a4.z; av[4 * q + 3] = a4.w;
        bv[4 * q] = b4.x; bv[4 * q + 1] = b4.y; bv[4 * q + 2] = b4.z; bv[4 * q + 3] = b4.w;
      }
#pragma unroll
      for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int j = 0; j < MT; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    if (more) stash(buf ^ 1);
    __syncthreads();
    buf ^= 1;
  }
#pragma unroll
  for (int i = 0; i < MT; ++i) {
    const int gm = m0 + ty * MT + i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < MT; ++j) {
      const int gn = n0 + tx * MT + j;
      if (gn >= N) continue;
      const long o = static_cast<long>(gm) * N + gn;
      if (EPI == kStore) {
        C[z * sC + static_cast<long>(ks) * M * N + o] = acc[i][j];
      } else if (EPI == kRefresh) {
        // the new A (M = d rows, N = r columns) and, for a refreshed plan,
        // its bf16 rounding as A^T (r x d) and as columns [0, r) of [A | P^T]
        C[z * sC + o] = acc[i][j];
        if (z < e.rt.n && e.rt.At[z] != nullptr) {
          const __nv_bfloat16 v = __float2bfloat16_rn(acc[i][j]);
          e.rt.At[z][static_cast<long>(gn) * M + gm] = v;
          e.rt.Bcat[z][static_cast<long>(gm) * 2 * N + gn] = v;
        }
      } else if (EPI == kMomentum) {
        float* mp = e.m + z * e.sm + o;
        const float gR = e.G[z * e.sG + o] - acc[i][j];
        *mp = e.beta * (*mp) + (1.f - e.beta) * gR;
      } else {
        const float sv = e.S[z * e.sS + o];
        C[z * sC + o] = (gm == gn ? e.a : 0.f) + e.b * sv + e.c * acc[i][j];
      }
    }
  }
}

// Q = a I + b S + c (sum of `ksplit` partials of S^2, ordered)
__global__ void k_reduce_poly(const float* __restrict__ part, const float* __restrict__ S,
                              float* __restrict__ Q, int n, int ksplit, float a, float b,
                              float c, long sP, long sO) {
  pdl_enter();
  const int z = blockIdx.y;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n * n) return;
  const float* p = part + z * sP;
  float v = 0.f;
  for (int s = 0; s < ksplit; ++s) v += p[static_cast<long>(s) * n * n + idx];
  const int i = idx / n, j = idx % n;
  Q[z * sO + idx] = (i == j ? a : 0.f) + b * S[z * sO + idx] + c * v;
}

// out = sum of `ksplit` partials (ordered); optionally symmetrised.
__global__ void k_reduce(const float* __restrict__ part, float* __restrict__ out, int n,
                         int ksplit, int sym, long sP, long sO) {
  pdl_enter();
  const int z = blockIdx.y;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n * n) return;
  const float* p = part + z * sP;
  float v = 0.f;
  for (int s = 0; s < ksplit; ++s) v += p[static_cast<long>(s) * n * n + idx];
  if (sym) {
    const int i = idx / n, j = idx % n;
    float w = 0.f;
    for (int s = 0; s < ksplit; ++s) w += p[static_cast<long>(s) * n * n + j * n + i];
    v = 0.5f * (v + w);
  }
  out[z * sO + idx] = v;
}

// per-block partial sums of squares, then an ordered final sum
__global__ void k_sumsq_partial(const float* __restrict__ x, long n, float* part, long sX,
                                int nblk) {
  pdl_enter();
  __shared__ float red[256];
  const int z = blockIdx.y;
  const float* p = x + z * sX;
  float s = 0.f;
  for (long i = blockIdx.x * 256L + threadIdx.x; i < n; i += 256L * nblk) s = fmaf(p[i], p[i], s);
  red[threadIdx.x] = s;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) part[z * nblk + blockIdx.x] = red[0];
}

// m = beta m + (1 - beta)(G - AH) in place (AH = A H from the tensor-core
// product), with the per-block partial sums of squares of the new m in the
// same pass (same element order and block sums as k_sumsq_partial)
__global__ void k_momentum_sumsq(float* __restrict__ m, const float* __restrict__ G,
                                 const float* __restrict__ AH, float beta, long n,
                                 float* part, long sX, int nblk) {
  pdl_enter();
  __shared__ float red[256];
  const int z = blockIdx.y;
  float* mp = m + z * sX;
  const float* g = G + z * sX;
  const float* c = AH + z * sX;
  float s = 0.f;
  for (long i = blockIdx.x * 256L + threadIdx.x; i < n; i += 256L * nblk) {
    const float v = beta * mp[i] + (1.f - beta) * (g[i] - c[i]);
    mp[i] = v;
    s = fmaf(v, v, s);
  }
  red[threadIdx.x] = s;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) part[z * nblk + blockIdx.x] = red[0];
}

__global__ void k_sumsq_final(const float* part, int nblk, float* inv) {
  pdl_enter();
  const int z = blockIdx.x;
  if (threadIdx.x != 0) return;
  float s = 0.f;
  for (int i = 0; i < nblk; ++i) s += part[z * nblk + i];
  inv[z] = 1.f / (sqrtf(s) + 1e-7f);
}

// y = alpha_z * x (alpha from a per-batch array) or y = A - lr * x
__global__ void k_scale(const float* __restrict__ x, const float* __restrict__ inv, float* y,
                        long n, long sX) {
  pdl_enter();
  const int z = blockIdx.y;
  const float a = inv[z];
  for (long i = blockIdx.x * 256L + threadIdx.x; i < n; i += 256L * gridDim.x)
    y[z * sX + i] = a * x[z * sX + i];
}

__global__ void k_axpy(const float* __restrict__ A, const float* __restrict__ D, float lr,
                       float* y, long n, long sX) {
  pdl_enter();
  const int z = blockIdx.y;
  for (long i = blockIdx.x * 256L + threadIdx.x; i < n; i += 256L * gridDim.x)
    y[z * sX + i] = A[z * sX + i] - lr * D[z * sX + i];
}

constexpr int TM = 32;   // output tile of the SPEL GEMMs

inline dim3 gemm_grid(int M, int N, int zdim) {
  return dim3((N + TM - 1) / TM, (M + TM - 1) / TM, zdim);
}

// splits of the r-long sum in S^2 (bounded by the partial buffer's ks)
inline int choose_ksplit_r(int r, int ks) {
  int k = r / 64;
  if (k < 1) k = 1;
  return k < ks ? k : ks;
}

int choose_ksplit(int d) {
  int ks = d / 128;
  if (ks < 1) ks = 1;
  if (ks > 16) ks = 16;
  return ks;
}

struct Ws {
  float *Y0, *Y1, *S, *Q, *part, *nrm_part, *inv;
  long dr, rr;   // packed per-boundary strides of the d x r and r x r buffers
  int ks;
  bool tc;       // the products of the step fit the tensor-core kernel
};

constexpr int kNormBlocks = 64;

inline size_t al64(size_t x) { return (x + 63) & ~static_cast<size_t>(63); }

Ws carve(void* ws, int d, int r, int batch) {
  Ws w;
  w.dr = static_cast<long>(d) * r;
  w.rr = static_cast<long>(r) * r;
  w.ks = choose_ksplit(d);
  w.tc = gemm3_supported(r, r, d, w.ks) && gemm3_supported(r, r, r, choose_ksplit_r(r, w.ks)) &&
         gemm3_supported(d, r, r, 1);
  float* p = reinterpret_cast<float*>(ws);
  w.Y0 = p; p += al64(w.dr * batch);
  w.Y1 = p; p += al64(w.dr * batch);
  w.S = p; p += al64(w.rr * batch);
  w.Q = p; p += al64(w.rr * batch);
  w.part = p; p += al64(w.rr * w.ks * batch);
  w.nrm_part = p; p += al64(static_cast<size_t>(kNormBlocks) * batch);
  w.inv = p;
  return w;
}

// bf16 operands of the refreshed plans from an fp32 A (used when the step
// has no retraction product to carry them)
__global__ void k_refresh_AB(const float* __restrict__ A, int d, int r, long sA, RefreshTable rt) {
  pdl_enter();
  const int z = blockIdx.y;
  if (z >= rt.n || rt.At[z] == nullptr) return;
  for (long x = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x;
       x < static_cast<long>(d) * r; x += static_cast<long>(gridDim.x) * blockDim.x) {
    const int k = static_cast<int>(x / r), j = static_cast<int>(x % r);
    const __nv_bfloat16 v = __float2bfloat16_rn(A[z * sA + x]);
    rt.At[z][static_cast<long>(j) * d + k] = v;
    rt.Bcat[z][static_cast<long>(k) * 2 * r + j] = v;
  }
}

// Y_out = Y_in (a I + b S + c S^2), S = Y_in^T Y_in; with rt the final
// product also writes the refreshed plans' bf16 operands.  The three products
// run on the tensor cores (launch_gemm3) when the shapes allow it, else on the
// CUDA cores; the reductions and the polynomial are the same either way.
cudaError_t pe_step(const float* Yin, float* Yout, const float* co, const Ws& w, int d, int r,
                    int batch, cudaStream_t s, const RefreshTable* rt = nullptr) {
  EpiArgs none{};
  const int kr = choose_ksplit_r(r, w.ks);
  const bool tc = w.tc;
  cudaError_t e = cudaSuccess;
  if (tc) {   // S partials: (Y^T)(Y^T)^T, both operands Y read with rows contiguous
    e = launch_gemm3({Yin, r, w.dr, 1}, {Yin, r, w.dr, 1}, w.part, r, w.rr * w.ks, w.rr, r, r,
                     d, batch, w.ks, s);
    if (e != cudaSuccess) return e;
  } else {
    if ((e = launch_chained(k_sgemm<true, kStore, TM>, gemm_grid(r, r, batch * w.ks), dim3(64), 0,
        s, Yin, Yin, w.part, r, r, d, r, r, w.dr, w.dr, w.rr * w.ks, w.ks,
        none)) != cudaSuccess) return e;
  }
  if ((e = launch_chained(k_reduce, dim3((r * r + 255) / 256, batch), dim3(256), 0, s, w.part, w.S,
      r, w.ks, 0, w.rr * w.ks, w.rr)) != cudaSuccess) return e;
  // S^2 in split-K partials (a 4-aligned split of K = r for the plain A),
  // then Q = a I + b S + c S^2 in the ordered reduction
  if (tc) {
    e = launch_gemm3({w.S, r, w.rr, 0}, {w.S, r, w.rr, 1}, w.part, r, w.rr * w.ks, w.rr, r, r,
                     r, batch, kr, s);
    if (e != cudaSuccess) return e;
  } else {
    if ((e = launch_chained(k_sgemm<false, kStore, TM>, gemm_grid(r, r, batch * kr), dim3(64), 0,
        s, w.S, w.S, w.part, r, r, r, r, r, w.rr, w.rr, w.rr * w.ks, kr,
        none)) != cudaSuccess) return e;
  }
  if ((e = launch_chained(k_reduce_poly, dim3((r * r + 255) / 256, batch), dim3(256), 0, s, w.part,
      w.S, w.Q, r, kr, co[0], co[1], co[2], w.rr * w.ks, w.rr)) != cudaSuccess) return e;
  if (tc) {   // Y Q: Q read with rows contiguous (its transpose's rows)
    e = launch_gemm3({Yin, r, w.dr, 0}, {w.Q, r, w.rr, 1}, Yout, r, w.dr, 0, d, r, r, batch, 1,
                     s);
    if (e != cudaSuccess) return e;
    if (rt && (e = launch_chained(k_refresh_AB, dim3(256, batch), dim3(256), 0, s, Yout, d, r,
        w.dr, *rt)) != cudaSuccess) return e;
  } else if (rt) {
    EpiArgs re{};
    re.rt = *rt;
    if ((e = launch_chained(k_sgemm<false, kRefresh, TM>, gemm_grid(d, r, batch), dim3(64), 0, s,
        Yin, w.Q, Yout, d, r, r, r, r, w.dr, w.rr, w.dr, 1, re)) != cudaSuccess) return e;
  } else {
    if ((e = launch_chained(k_sgemm<false, kStore, TM>, gemm_grid(d, r, batch), dim3(64), 0, s,
        Yin, w.Q, Yout, d, r, r, r, r, w.dr, w.rr, w.dr, 1, none)) != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace

size_t spel_workspace_bytes(int64_t d, int64_t r, int32_t batch) {
  const size_t dr = static_cast<size_t>(d) * r, rr = static_cast<size_t>(r) * r;
  const int ks = choose_ksplit(static_cast<int>(d));
  const size_t floats = 2 * al64(dr * batch) + 2 * al64(rr * batch) + al64(rr * ks * batch) +
                        al64(static_cast<size_t>(kNormBlocks) * batch) + al64(batch);
  return floats * sizeof(float);
}

cudaError_t launch_spel(float* A, const float* G, float* m, int d, int r, int batch, float lr,
                        float beta, const float* coeffs, int n_lmo, int n_retr, void* ws,
                        cudaStream_t s, const RefreshTable* rt) {
  const Ws w = carve(ws, d, r, batch);
  EpiArgs none{};
  // H = sym(A^T G)
  cudaError_t e = cudaSuccess;
  if (w.tc) {
    e = launch_gemm3({A, r, w.dr, 1}, {G, r, w.dr, 1}, w.part, r, w.rr * w.ks, w.rr, r, r, d,
                     batch, w.ks, s);
    if (e != cudaSuccess) return e;
  } else {
    if ((e = launch_chained(k_sgemm<true, kStore, TM>, gemm_grid(r, r, batch * w.ks), dim3(64), 0,
        s, A, G, w.part, r, r, d, r, r, w.dr, w.dr, w.rr * w.ks, w.ks,
        none)) != cudaSuccess) return e;
  }
  if ((e = launch_chained(k_reduce, dim3((r * r + 255) / 256, batch), dim3(256), 0, s, w.part, w.S,
      r, w.ks, 1, w.rr * w.ks, w.rr)) != cudaSuccess) return e;
  // m = beta m + (1 - beta)(G - A H)
  EpiArgs mo{};
  mo.G = G;
  mo.m = m;
  mo.sG = w.dr;
  mo.sm = w.dr;
  mo.beta = beta;
  if (w.tc) {
    // A H on the tensor cores into the (still free) Y1 buffer, then the
    // momentum update fused with the first pass of ||m||_F
    e = launch_gemm3({A, r, w.dr, 0}, {w.S, r, w.rr, 1}, w.Y1, r, w.dr, 0, d, r, r, batch, 1, s);
    if (e != cudaSuccess) return e;
    if ((e = launch_chained(k_momentum_sumsq, dim3(kNormBlocks, batch), dim3(256), 0, s, m, G,
        w.Y1, beta, w.dr, w.nrm_part, w.dr, kNormBlocks)) != cudaSuccess) return e;
  } else {
    if ((e = launch_chained(k_sgemm<false, kMomentum, TM>, gemm_grid(d, r, batch), dim3(64), 0, s,
        A, w.S, nullptr, d, r, r, r, r, w.dr, w.rr, 0, 1, mo)) != cudaSuccess) return e;
    if ((e = launch_chained(k_sumsq_partial, dim3(kNormBlocks, batch), dim3(256), 0, s, m, w.dr,
        w.nrm_part, w.dr, kNormBlocks)) != cudaSuccess) return e;
  }
  // Y = m / (||m||_F + 1e-7)
  if ((e = launch_chained(k_sumsq_final, batch, dim3(32), 0, s, w.nrm_part, kNormBlocks,
      w.inv)) != cudaSuccess) return e;
  if ((e = launch_chained(k_scale, dim3(256, batch), dim3(256), 0, s, m, w.inv, w.Y0, w.dr,
      w.dr)) != cudaSuccess) return e;
  float* cur = w.Y0;
  float* nxt = w.Y1;
  for (int t = 0; t < n_lmo; ++t) {
    e = pe_step(cur, nxt, coeffs + 3 * t, w, d, r, batch, s);
    if (e != cudaSuccess) return e;
    float* tmp = cur; cur = nxt; nxt = tmp;
  }
  // retraction input A - lr D
  if ((e = launch_chained(k_axpy, dim3(256, batch), dim3(256), 0, s, A, cur, lr, nxt, w.dr,
      w.dr)) != cudaSuccess) return e;
  { float* tmp = cur; cur = nxt; nxt = tmp; }
  for (int t = 0; t < n_retr; ++t) {
    const bool last = t == n_retr - 1;
    float* out = last ? A : nxt;
    e = pe_step(cur, out, coeffs + 3 * (n_lmo + t), w, d, r, batch, s, last ? rt : nullptr);
    if (e != cudaSuccess) return e;
    float* tmp = cur; cur = out; nxt = tmp;
  }
  if (n_retr == 0) {
    if ((e = cudaMemcpyAsync(A, cur, sizeof(float) * w.dr * batch, cudaMemcpyDeviceToDevice,
                             s)) != cudaSuccess) return e;
    if (rt && (e = launch_chained(k_refresh_AB, dim3(256, batch), dim3(256), 0, s, A, d, r, w.dr,
        *rt)) != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace mapl

// ---------------------------------------------------------------------------
// Fixed-scratch variant of the SPEL step for callers that cannot allocate.
//
// The scratch lives in this file-scope device array, reserved on every GPU
// that loads the library for as long as the process runs.  Host code cannot
// hand the array's name to a kernel (in host code it is only a stand-in, not
// a device address); its device address is looked up with
// cudaGetSymbolAddress on every call, with the caller's device current.  No
// address is cached: after a device reset or a primary-context teardown the
// module is loaded again and a remembered address would point at freed
// memory.  The lookup itself is a table read once the module is loaded.
// ---------------------------------------------------------------------------
namespace mapl {

namespace {

__device__ __align__(256) unsigned char g_spel_scratch[kSpelStaticScratchBytes];

}  // namespace

cudaError_t spel_static_scratch(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_spel_scratch);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

}  // namespace mapl
