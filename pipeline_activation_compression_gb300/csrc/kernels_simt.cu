// kernels_simt.cu -- plan preparation kernels and the fp32 CUDA-core codec.
//
// Plan preparation (once per projector update, MAPL §3.3 "send the updated
// A_p ... after every optimizer step"):
//   M = P_send A (r x r) in compensated fp32 (exact products by fma split,
//   sums kept as unevaluated pairs, about 48 significant bits); for the bf16
//   tensor-core path -M is split into three bf16 terms hi + mid + lo (about
//   24 significant bits), stored transposed as K-major B operands; A^T and
//   [A | P_recv^T] are laid out as K-major B operands; codebook squared norms
//   and per-book maximum norm are computed.
//
// fp32 path (plan dtype MAPL_F32): one warp per token.
//   compress:   z = x A - E[t] M, then residual VQ with exact fp32 distances
//   decompress: x_hat = z_hat A^T + E'[t] P'
#include "mapl_internal.h"
#include "ptx.cuh"

namespace mapl {

namespace {

__device__ __forceinline__ double ld_f64(const void* p, size_t i, bool bf) {
  return bf ? static_cast<double>(__bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]))
            : static_cast<double>(reinterpret_cast<const float*>(p)[i]);
}

// ------------------------------------------------------------------ prep
__device__ __forceinline__ float ld_f32(const void* p, size_t i, bool bf) {
  return bf ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i])
            : reinterpret_cast<const float*>(p)[i];
}

__device__ __forceinline__ void two_sum_f(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

// fp32 plans: M[i][j] = sum_k P_send[i][k] A[k][j].  One block (8 warps) per row i and
// 32 columns (lane = column, reads of A coalesced, P broadcast); warp w sums
// k in its eighth of [0, d) with four independent compensated sums (k mod 4),
// each term an exact product split by fma; the pairs are combined in shared
// memory.
__device__ __forceinline__ void prep_M_block(const void* Ps, const void* A, int d, int r, bool bf,
                                             float* M32) {
  __shared__ float ph[8][32], pl[8][32];
  const int nj = (r + 31) / 32;
  const int i = blockIdx.x / nj, j = (blockIdx.x % nj) * 32 + (threadIdx.x & 31);
  const int w = threadIdx.x >> 5;
  const int kc = (d + 7) / 8, kb = w * kc, ke = min(d, kb + kc);
  float h[4] = {0.f, 0.f, 0.f, 0.f}, l[4] = {0.f, 0.f, 0.f, 0.f};
  // 32 k per pass: lane q fetches P[i][k0 + q] (coalesced, then broadcast by
  // shuffle) and every lane its 32 A values, all loads in flight together.
  // Terms past the end are 0 * 0, which leaves a compensated sum unchanged,
  // so chain k mod 4 sees the same terms in the same order as a plain loop.
  const int lane = threadIdx.x & 31;
  const bool jv = j < r;
  for (int k0 = kb; k0 < ke; k0 += 32) {
    const int kp = k0 + lane;
    const float pv = kp < ke ? ld_f32(Ps, static_cast<size_t>(i) * d + kp, bf) : 0.f;
    float av[32];
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      const int k = k0 + u;
      float b = 0.f;
      if (jv && k < ke) {
        b = ld_f32(A, static_cast<size_t>(k) * r + j, bf);
      }
      av[u] = b;
    }
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      const float a = __shfl_sync(0xffffffffu, pv, u);
      const float p = a * av[u], pe = fmaf(a, av[u], -p);
      float t, te;
      two_sum_f(h[u & 3], p, t, te);
      h[u & 3] = t;
      l[u & 3] += te + pe;
    }
  }
  float s01, e01, s23, e23, hi, e;
  two_sum_f(h[0], h[1], s01, e01);
  two_sum_f(h[2], h[3], s23, e23);
  two_sum_f(s01, s23, hi, e);
  ph[w][threadIdx.x & 31] = hi;
  pl[w][threadIdx.x & 31] = (l[0] + l[1]) + (l[2] + l[3]) + (e01 + e23) + e;
  __syncthreads();
  if (w != 0 || j >= r) return;
  const int c = threadIdx.x & 31;
  hi = ph[0][c];
  float lo = pl[0][c];
  for (int x = 1; x < 8; ++x) {
    float t, te;
    two_sum_f(hi, ph[x][c], t, te);
    hi = t;
    lo += pl[x][c] + te;
  }
  two_sum_f(hi, lo, hi, lo);
  M32[i * r + j] = hi + lo;
}

__global__ void __launch_bounds__(256) k_prep_M(const void* Ps, const void* A, int d, int r,
                                                bool bf, float* M32) {
  prep_M_block(Ps, A, d, r, bf, M32);
}

// -M^T as three bf16 terms (the K-major B operand of the anchor fold) from
// the fp32 M of a bf16 plan: term s holds the bf16 rounding of what the
// terms before it left; each remainder is exact in fp32.
__global__ void k_split_negMt(const float* __restrict__ M, int r, __nv_bfloat16* __restrict__ Mts) {
  const int x = blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= r * r) return;
  const int i = x / r, j = x % r;
  float v = -M[x];
  for (int t = 0; t < kNumSplit; ++t) {
    const __nv_bfloat16 b = __float2bfloat16_rn(v);
    Mts[(static_cast<size_t>(t) * r + j) * r + i] = b;
    v -= __bfloat162float(b);
  }
}

__global__ void k_prep_At(const __nv_bfloat16* A, int d, int r, __nv_bfloat16* At) {
  const size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
  if (idx >= static_cast<size_t>(d) * r) return;
  const int j = static_cast<int>(idx / d), i = static_cast<int>(idx % d);
  At[idx] = A[static_cast<size_t>(i) * r + j];
}

__global__ void k_prep_Bcat(const __nv_bfloat16* A, const __nv_bfloat16* Pr, int d, int r,
                            __nv_bfloat16* Bcat) {
  const size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
  const int w = 2 * r;
  if (idx >= static_cast<size_t>(d) * w) return;
  const int n = static_cast<int>(idx / w), k = static_cast<int>(idx % w);
  Bcat[idx] = k < r ? A[static_cast<size_t>(n) * r + k] : Pr[static_cast<size_t>(k - r) * d + n];
}

__global__ void k_copy_f32(const float* src, float* dst, size_t n) {
  const size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
  if (idx < n) dst[idx] = src[idx];
}

__global__ void k_prep_At32(const float* A, int d, int r, float* At) {
  const size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
  if (idx >= static_cast<size_t>(d) * r) return;
  const int j = static_cast<int>(idx / d), i = static_cast<int>(idx % d);
  At[idx] = A[static_cast<size_t>(i) * r + j];
}

// Norm row of a code for the distance MMA: h = cn / 2 (exact) as three bf16
// terms h_hi = bf16(h), h_mid = bf16(h - h_hi), h_lo = bf16(h - h_hi -
// h_mid) (each remainder is exact in fp32, and the three terms carry h's 24
// significant bits), then 13 zeros: 32 bytes, two 16-byte stores.
__device__ __forceinline__ void write_norm_row(float cn, __nv_bfloat16* row) {
  const float h = 0.5f * cn;
  const __nv_bfloat16 hi = __float2bfloat16_rn(h);
  const float r1 = h - __bfloat162float(hi);
  const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
  const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
  const uint32_t w0 = static_cast<uint32_t>(__bfloat16_as_ushort(hi)) |
                      (static_cast<uint32_t>(__bfloat16_as_ushort(mid)) << 16);
  const uint32_t w1 = static_cast<uint32_t>(__bfloat16_as_ushort(lo));
  uint4* d = reinterpret_cast<uint4*>(row);
  d[0] = make_uint4(w0, w1, 0u, 0u);
  d[1] = make_uint4(0u, 0u, 0u, 0u);
}

// ||c||^2 of bf16 values in fp32: every square is exact in fp32 (8-bit
// significands), the squares are added in index order with Knuth's two-sum
// and the rounding errors carried beside the sum, and the pair is rounded
// once at the end, so the result is the fp32 rounding of the exact value up
// to a relative 2^-40 or so.  The plan's preparation and the streaming
// update both use it, in the same order, so they give the same bits.
struct Norm2 {
  float s = 0.f, e = 0.f;
  __device__ __forceinline__ void add(float x) {
    const float p = x * x;
    const float t = s + p;
    const float bp = t - s;
    e += (s - (t - bp)) + (p - bp);
    s = t;
  }
  __device__ __forceinline__ void add8(const uint4& w) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(h[k]);
      add(f.x);
      add(f.y);
    }
  }
  __device__ __forceinline__ float value() const { return s + e; }
};

__global__ void k_prep_codes(const void* C, int nbooks, int K, int gd, bool bf,
                             __nv_bfloat16* Cb, __nv_bfloat16* Hs, float* C32, float* cnorm) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;   // code id over all books
  if (idx >= nbooks * K) return;
  if (bf) {
    const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(C) + static_cast<size_t>(idx) * gd;
    Norm2 n;
    for (int i = 0; i < gd; ++i) {
      n.add(__bfloat162float(src[i]));
      if (Cb) Cb[static_cast<size_t>(idx) * gd + i] = src[i];
    }
    cnorm[idx] = n.value();
    if (Hs) write_norm_row(n.value(), Hs + static_cast<size_t>(idx) * 16);
    return;
  }
  double s = 0.0;
  for (int i = 0; i < gd; ++i) {
    const double v = ld_f64(C, static_cast<size_t>(idx) * gd + i, false);
    s = fma(v, v, s);
    if (C32) C32[static_cast<size_t>(idx) * gd + i] = static_cast<float>(v);
  }
  cnorm[idx] = static_cast<float>(s);
}

// max_k ||c_k|| of each book, rounded up: one warp per book (the maximum of
// the fp32 norms is exact in any order; the correctly rounded fp32 square
// root, within half an ulp, times 1 + 2^-20 is above the exact root).
__device__ __forceinline__ float round_up_root(float m) { return sqrtf(m) * (1.f + 0x1p-20f); }

__device__ __forceinline__ void book_max_warp(const float* cnorm, int b, int K, int lane,
                                              float* cmax) {
  float m = 0.f;
#pragma unroll 8
  for (int k = lane; k < K; k += 32) m = fmaxf(m, __ldcg(cnorm + static_cast<size_t>(b) * K + k));
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) cmax[b] = round_up_root(m);
}

__global__ void k_prep_cmax(const float* cnorm, int nbooks, int K, float* cmax) {
  const int b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (b < nbooks) book_max_warp(cnorm, b, K, threadIdx.x & 31, cmax);
}

inline unsigned blocks_for(size_t n, int t) { return static_cast<unsigned>((n + t - 1) / t); }

// ------------------------------------------------------------ fp32 codec
constexpr int kWarpsPerBlock = 8;

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    k_compress_f32(const float* __restrict__ X, const int32_t* __restrict__ tids,
                   const float* __restrict__ A, const float* __restrict__ M,
                   const float* __restrict__ E, const float* __restrict__ C, void* out, int* err,
                   int N, int d, int r, int V, int G, int R, int K, int gd, int mode) {
  extern __shared__ float zs_all[];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * kWarpsPerBlock + w;
  if (n >= N) return;
  float* zs = zs_all + w * r;
  int t = tids[n];
  const bool bad = t < 0 || t >= V;
  if (bad && lane == 0) atomicOr(err, kErrBadToken);
  const float* x = X + static_cast<size_t>(n) * d;
  for (int j = lane; j < r; j += 32) {
    float acc = 0.f;
    for (int i = 0; i < d; ++i) acc = fmaf(x[i], A[static_cast<size_t>(i) * r + j], acc);
    if (!bad) {
      const float* e = E + static_cast<size_t>(t) * r;
      for (int k = 0; k < r; ++k) acc = fmaf(-e[k], M[static_cast<size_t>(k) * r + j], acc);
    }
    zs[j] = bad ? 0.f : acc;
  }
  __syncwarp();
  if (mode != kModeVQ) {
    float* o = reinterpret_cast<float*>(out) + static_cast<size_t>(n) * r;
    for (int j = lane; j < r; j += 32) o[j] = zs[j];
    return;
  }
  uint8_t* io = reinterpret_cast<uint8_t*>(out) + static_cast<size_t>(n) * R * G;
  for (int rho = 0; rho < R; ++rho) {
    for (int g = 0; g < G; ++g) {
      const float* book = C + static_cast<size_t>(rho * G + g) * K * gd;
      const float* u = zs + g * gd;
      float best = __int_as_float(0x7f800000);
      int bk = 0x7fffffff;
      for (int k = lane; k < K; k += 32) {
        float D = 0.f;
        for (int i = 0; i < gd; ++i) {
          const float df = u[i] - book[static_cast<size_t>(k) * gd + i];
          D = fmaf(df, df, D);
        }
        if (D < best) {
          best = D;
          bk = k;
        }
      }
      for (int off = 16; off > 0; off >>= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, best, off);
        const int ok = __shfl_xor_sync(0xffffffffu, bk, off);
        if (ob < best || (ob == best && ok < bk)) {
          best = ob;
          bk = ok;
        }
      }
      if (lane == 0) io[rho * G + g] = bad ? 0 : static_cast<uint8_t>(bk);
      __syncwarp();
      for (int i = lane; i < gd; i += 32) zs[g * gd + i] -= book[static_cast<size_t>(bk) * gd + i];
      __syncwarp();
    }
  }
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    k_decompress_f32(const void* in, const int32_t* __restrict__ tids,
                     const float* __restrict__ At, const float* __restrict__ Pr,
                     const float* __restrict__ E, const float* __restrict__ C, float* Xh,
                     int* err, int N, int d, int r, int V, int G, int R, int K, int gd, int vq) {
  extern __shared__ float zs_all[];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * kWarpsPerBlock + w;
  if (n >= N) return;
  float* zs = zs_all + w * r;
  const int t = tids[n];
  const bool bad = t < 0 || t >= V;
  if (bad && lane == 0) atomicOr(err, kErrBadToken);
  if (vq) {
    const uint8_t* ip = reinterpret_cast<const uint8_t*>(in) + static_cast<size_t>(n) * R * G;
    for (int j = lane; j < r; j += 32) {
      const int g = j / gd, i = j % gd;
      float acc = 0.f;
      for (int rho = 0; rho < R; ++rho) {
        int k = ip[rho * G + g];
        if (k >= K) {   // not a valid code: flag it, never read past the book
          atomicOr(err, kErrBadIndex);
          k = K - 1;
        }
        acc += C[(static_cast<size_t>(rho * G + g) * K + k) * gd + i];
      }
      zs[j] = acc;
    }
  } else {
    const float* z = reinterpret_cast<const float*>(in) + static_cast<size_t>(n) * r;
    for (int j = lane; j < r; j += 32) zs[j] = z[j];
  }
  __syncwarp();
  float* o = Xh + static_cast<size_t>(n) * d;
  for (int j = lane; j < d; j += 32) {
    float acc = 0.f;
    for (int k = 0; k < r; ++k) acc = fmaf(zs[k], At[static_cast<size_t>(k) * d + j], acc);
    if (!bad) {
      const float* e = E + static_cast<size_t>(t) * r;
      for (int k = 0; k < r; ++k) acc = fmaf(e[k], Pr[static_cast<size_t>(k) * d + j], acc);
    }
    o[j] = bad ? 0.f : acc;
  }
}

}  // namespace

cudaError_t launch_prep_bf16(const mapl_config& c, const void* A, const void* Ps, const void* Pr,
                             const void* C, PlanDevice& p, bool A_only, cudaStream_t s) {
  const int d = static_cast<int>(c.d), r = static_cast<int>(c.r);
  const int T = 256;
  k_prep_At<<<blocks_for(static_cast<size_t>(d) * r, T), T, 0, s>>>(
      reinterpret_cast<const __nv_bfloat16*>(A), d, r, p.At);
  k_prep_Bcat<<<blocks_for(static_cast<size_t>(d) * 2 * r, T), T, 0, s>>>(
      reinterpret_cast<const __nv_bfloat16*>(A), reinterpret_cast<const __nv_bfloat16*>(Pr), d, r,
      p.Bcat);
  if (!A_only && c.G > 0) {
    const int nb = c.R * c.G, gd = static_cast<int>(c.r / c.G);
    k_prep_codes<<<blocks_for(static_cast<size_t>(nb) * c.K, T), T, 0, s>>>(
        C, nb, c.K, gd, true, p.Cb, p.Hs, nullptr, p.cnorm);
    k_prep_cmax<<<blocks_for(static_cast<size_t>(nb) * 32, 256), 256, 0, s>>>(p.cnorm, nb, c.K, p.cmax);
  }
  return cudaGetLastError();
}

// A bf16 codebook set (R x G x K x gd) copied into plan storage with its
// squared norms and per-book maxima (the gradient codebooks of §3.5).
cudaError_t launch_prep_books_bf16(const mapl_config& c, const void* C, __nv_bfloat16* Cb,
                                   __nv_bfloat16* Hs, float* cnorm, float* cmax, cudaStream_t s) {
  const int nb = c.R * c.G, gd = static_cast<int>(c.r / c.G);
  k_prep_codes<<<blocks_for(static_cast<size_t>(nb) * c.K, 256), 256, 0, s>>>(
      C, nb, c.K, gd, true, Cb, Hs, nullptr, cnorm);
  k_prep_cmax<<<blocks_for(static_cast<size_t>(nb) * 32, 256), 256, 0, s>>>(cnorm, nb, c.K, cmax);
  return cudaGetLastError();
}

cudaError_t launch_split_negMt(const float* M, int r, __nv_bfloat16* Mts, cudaStream_t s) {
  k_split_negMt<<<(r * r + 255) / 256, 256, 0, s>>>(M, r, Mts);
  return cudaGetLastError();
}

// One updated code: its values are read first (16-byte loads for bf16 rows
// of 16 or 32 values, issued together with the id's load), then written to
// the plan's table with ||c||^2 (the preparation's Norm2 for bf16 rows, fp64
// for fp32 rows) and, for bf16 plans, the norm row of the distance MMA.
// A bf16 row of 16 or 32 values already in registers (w) written to code id;
// returns its ||c||^2, or -1 (error word set) for an id outside the table.
__device__ __forceinline__ float apply_code_bf16(int id, const uint4 (&w)[4], int gd, int ncode,
                                                 __nv_bfloat16* __restrict__ Cb,
                                                 __nv_bfloat16* __restrict__ Hs,
                                                 float* __restrict__ cnorm, int* err) {
  if (id < 0 || id >= ncode) {
    atomicOr(err, kErrBadIndex);
    return -1.f;
  }
  uint4* dst = reinterpret_cast<uint4*>(Cb) + static_cast<size_t>(id) * (gd / 8);
  Norm2 n;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    if (c < gd / 8) {
      dst[c] = w[c];
      n.add8(w[c]);
    }
  cnorm[id] = n.value();
  if (Hs) write_norm_row(n.value(), Hs + static_cast<size_t>(id) * 16);
  return n.value();
}

__device__ __forceinline__ void load_code_bf16(const void* codes, int i, int gd, uint4 (&w)[4]) {
  const uint4* src = reinterpret_cast<const uint4*>(codes) + static_cast<size_t>(i) * (gd / 8);
#pragma unroll
  for (int c = 0; c < 4; ++c) w[c] = c < gd / 8 ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
}

__device__ __forceinline__ float update_one_code(int id, int i, const void* __restrict__ codes,
                                                int gd, int ncode, bool bf,
                                                __nv_bfloat16* __restrict__ Cb,
                                                __nv_bfloat16* __restrict__ Hs,
                                                float* __restrict__ C32, float* __restrict__ cnorm,
                                                int* err) {
  if (bf && (gd == 16 || gd == 32)) {
    uint4 w[4];
    load_code_bf16(codes, i, gd, w);
    return apply_code_bf16(id, w, gd, ncode, Cb, Hs, cnorm, err);
  }
  if (id < 0 || id >= ncode) {
    atomicOr(err, kErrBadIndex);
    return -1.f;
  }
  if (bf) {
    Norm2 n;
    for (int j = 0; j < gd; ++j) {
      const __nv_bfloat16 v =
          reinterpret_cast<const __nv_bfloat16*>(codes)[static_cast<size_t>(i) * gd + j];
      Cb[static_cast<size_t>(id) * gd + j] = v;
      n.add(__bfloat162float(v));
    }
    cnorm[id] = n.value();
    if (Hs) write_norm_row(n.value(), Hs + static_cast<size_t>(id) * 16);
    return n.value();
  }
  double s = 0.0;
  for (int j = 0; j < gd; ++j) {
    const float v = reinterpret_cast<const float*>(codes)[static_cast<size_t>(i) * gd + j];
    C32[static_cast<size_t>(id) * gd + j] = v;
    s = fma(static_cast<double>(v), static_cast<double>(v), s);
  }
  cnorm[id] = static_cast<float>(s);
  return static_cast<float>(s);
}

// Streaming codebook update (§3.5, App. F): code ids[i] (flat over R x G x
// K) takes the values codes[i] (gd entries, plan dtype); its squared norm is
// recomputed.  One thread per updated code; ids outside the table set the
// error word and are skipped.  Then every book's max ||c|| is recomputed,
// one warp per book, in the same launch:
//  * one block (at most kUpdThreads codes, a table whose norms fit in
//    shared memory): the block reads the table's old norms into shared
//    memory while the new codes load, overwrites the updated entries and
//    takes the maxima there, so the update costs one round trip to memory;
//  * else the last block to finish (a counter in the plan, left at zero)
//    reads the norms back from memory.
constexpr int kUpdThreads = 512;
constexpr int kUpdSmemCodes = 12288;   // 48 KB of norms

__global__ void __launch_bounds__(kUpdThreads) k_update_codes_block(
    const int32_t* ids, int count, const void* codes, int gd, int ncode, bool bf,
    __nv_bfloat16* Cb, __nv_bfloat16* Hs, float* C32, float* cnorm, int* err, int nbooks, int K,
    float* cmax) {
  extern __shared__ float nrm[];
  const int i = threadIdx.x;
  const bool fast = bf && (gd == 16 || gd == 32);
  // the id, the new values and the table's old norms, all loads in flight
  // together
  const int id = i < count ? __ldg(ids + i) : -1;
  uint4 w[4];
  if (fast && i < count) load_code_bf16(codes, i, gd, w);
  for (int k0 = 0; k0 < ncode; k0 += 8 * kUpdThreads) {
    float t[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int k = k0 + u * kUpdThreads + i;
      t[u] = k < ncode ? __ldcg(cnorm + k) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int k = k0 + u * kUpdThreads + i;
      if (k < ncode) nrm[k] = t[u];
    }
  }
  __syncthreads();
  if (i < count) {
    const float v = fast ? apply_code_bf16(id, w, gd, ncode, Cb, Hs, cnorm, err)
                         : update_one_code(id, i, codes, gd, ncode, bf, Cb, Hs, C32, cnorm, err);
    if (v >= 0.f) nrm[id] = v;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  for (int b = threadIdx.x >> 5; b < nbooks; b += blockDim.x >> 5) {
    float m = 0.f;
    for (int k = lane; k < K; k += 32) m = fmaxf(m, nrm[b * K + k]);
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) cmax[b] = round_up_root(m);
  }
}

__global__ void __launch_bounds__(kUpdThreads) k_update_codes(const int32_t* ids, int count,
                                                              const void* codes, int gd, int ncode,
                                                              bool bf, __nv_bfloat16* Cb,
                                                              __nv_bfloat16* Hs, float* C32,
                                                              float* cnorm, int* err, int nbooks,
                                                              int K, float* cmax,
                                                              unsigned int* ctr) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < count) update_one_code(__ldg(ids + i), i, codes, gd, ncode, bf, Cb, Hs, C32, cnorm, err);
  __shared__ bool last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(ctr, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int b = threadIdx.x >> 5; b < nbooks; b += blockDim.x >> 5)
    book_max_warp(cnorm, b, K, threadIdx.x & 31, cmax);
  if (threadIdx.x == 0) *ctr = 0u;
}


// Self-test of the bounded wait every kernel uses: one warp waits on an
// mbarrier that nothing arrives on, through the same mbar_wait, and reports
// the give-up exactly as a codec kernel would (the error word's timeout bit).
// Nothing is in flight while it waits, so giving up leaves nothing behind.
__global__ void k_wait_selftest(uint64_t budget_ns, int* err, unsigned long long* waited) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const uint64_t t0 = global_ns();
  const bool ok = mbar_wait(smem_u32(&bar), 0, &abort_flag, budget_ns);
  const uint64_t t1 = global_ns();
  if (threadIdx.x == 0) {
    if (!ok) atomicOr(err, kErrTimeout);
    *waited = t1 - t0;
  }
}

cudaError_t launch_wait_selftest(uint64_t budget_ns, int* err, unsigned long long* waited,
                                 cudaStream_t s) {
  k_wait_selftest<<<1, 32, 0, s>>>(budget_ns, err, waited);
  return cudaGetLastError();
}

cudaError_t launch_update_codes(const mapl_config& c, const int32_t* ids, int count,
                                const void* codes, PlanDevice& p, cudaStream_t s) {
  const int nb = c.R * c.G, gd = static_cast<int>(c.r / c.G), ncode = nb * c.K;
  const bool bf = c.dtype == MAPL_BF16;
  if (count <= kUpdThreads && ncode <= kUpdSmemCodes) {
    k_update_codes_block<<<1, kUpdThreads, static_cast<size_t>(ncode) * sizeof(float), s>>>(
        ids, count, codes, gd, ncode, bf, p.Cb, p.Hs, p.C32, p.cnorm, p.err, nb, c.K, p.cmax);
    return cudaGetLastError();
  }
  k_update_codes<<<blocks_for(static_cast<size_t>(count), kUpdThreads), kUpdThreads, 0, s>>>(
      ids, count, codes, gd, ncode, bf, p.Cb, p.Hs, p.C32, p.cnorm, p.err, nb, c.K, p.cmax,
      p.upd_ctr);
  return cudaGetLastError();
}

cudaError_t launch_prep_f32(const mapl_config& c, const void* A, const void* Ps, const void* Pr,
                            const void* C, PlanDevice& p, bool A_only, cudaStream_t s) {
  const int d = static_cast<int>(c.d), r = static_cast<int>(c.r);
  const int T = 256;
  const size_t dr = static_cast<size_t>(d) * r;
  k_copy_f32<<<blocks_for(dr, T), T, 0, s>>>(reinterpret_cast<const float*>(A), p.A32, dr);
  k_prep_At32<<<blocks_for(dr, T), T, 0, s>>>(reinterpret_cast<const float*>(A), d, r, p.At32);
  k_prep_M<<<r * ((r + 31) / 32), 256, 0, s>>>(Ps, A, d, r, false, p.M32);
  (void)Pr;   // the plan's P_recv copy is used in place (p.Pr32)
  if (!A_only) {
    if (c.G > 0) {
      const int nb = c.R * c.G, gd = static_cast<int>(c.r / c.G);
      k_prep_codes<<<blocks_for(static_cast<size_t>(nb) * c.K, T), T, 0, s>>>(
          C, nb, c.K, gd, false, nullptr, nullptr, p.C32, p.cnorm);
      k_prep_cmax<<<blocks_for(static_cast<size_t>(nb) * 32, 256), 256, 0, s>>>(p.cnorm, nb, c.K, p.cmax);
    }
  }
  return cudaGetLastError();
}

cudaError_t launch_compress_f32(const mapl_config& c, const PlanDevice& p, const float* X,
                                const int32_t* tids, int64_t N, const float* E, void* out,
                                int mode, cudaStream_t s) {
  const int r = static_cast<int>(c.r);
  const int gd = c.G ? r / c.G : 0;
  const unsigned grid = static_cast<unsigned>((N + kWarpsPerBlock - 1) / kWarpsPerBlock);
  const size_t smem = static_cast<size_t>(kWarpsPerBlock) * r * sizeof(float);
  k_compress_f32<<<grid, kWarpsPerBlock * 32, smem, s>>>(
      X, tids, p.A32, p.M32, E, p.C32, out, p.err, static_cast<int>(N), static_cast<int>(c.d), r,
      static_cast<int>(c.V), c.G, c.R, c.K, gd, mode);
  return cudaGetLastError();
}

cudaError_t launch_decompress_f32(const mapl_config& c, const PlanDevice& p, const void* in,
                                  const int32_t* tids, int64_t N, const float* E, float* Xh,
                                  cudaStream_t s) {
  const int r = static_cast<int>(c.r);
  const int gd = c.G ? r / c.G : 0;
  const unsigned grid = static_cast<unsigned>((N + kWarpsPerBlock - 1) / kWarpsPerBlock);
  const size_t smem = static_cast<size_t>(kWarpsPerBlock) * r * sizeof(float);
  k_decompress_f32<<<grid, kWarpsPerBlock * 32, smem, s>>>(
      in, tids, p.At32, p.Pr32, E, p.C32, Xh, p.err, static_cast<int>(N), static_cast<int>(c.d),
      r, static_cast<int>(c.V), c.G, c.R, c.K, gd, c.G > 0 ? 1 : 0);
  return cudaGetLastError();
}

// Write-rate probe: zeros over [dst, dst + 16 n16) with nothing read.
// Modes 0/1: 16-byte stores from a grid-stride loop, four stores in flight
// per thread (1: the streaming, evict-first hint).  Mode 2: bulk
// asynchronous copies of a zeroed 32 KB shared-memory buffer, one CTA per
// SM over a contiguous range, the copy path of the TMA store drain.
namespace {

template <bool kStream>
__global__ void __launch_bounds__(512) k_store_probe(uint4* __restrict__ dst, size_t n16) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (; i + 3 * stride < n16; i += 4 * stride) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (kStream) __stcs(dst + i + k * stride, z);
      else dst[i + k * stride] = z;
    }
  }
  for (; i < n16; i += stride) {
    if (kStream) __stcs(dst + i, z);
    else dst[i] = z;
  }
}

constexpr uint32_t kBulkBytes = 32768;

__global__ void __launch_bounds__(128) k_store_probe_bulk(uint8_t* __restrict__ dst, size_t n16) {
  __shared__ __align__(128) uint4 buf[kBulkBytes / 16];
  for (int i = threadIdx.x; i < static_cast<int>(kBulkBytes / 16); i += blockDim.x)
    buf[i] = make_uint4(0u, 0u, 0u, 0u);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  if (threadIdx.x != 0) return;
  const size_t b0 = n16 * blockIdx.x / gridDim.x * 16, b1 = n16 * (blockIdx.x + 1) / gridDim.x * 16;
  const uint32_t src = static_cast<uint32_t>(__cvta_generic_to_shared(buf));
  for (size_t o = b0; o < b1; o += kBulkBytes) {
    const uint32_t n = b1 - o < kBulkBytes ? static_cast<uint32_t>(b1 - o) : kBulkBytes;
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst + o),
                 "r"(src), "r"(n)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group.read 8;" ::: "memory");
  }
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

}  // namespace

cudaError_t launch_store_probe(void* dst, size_t bytes, int mode, int num_sms, cudaStream_t s) {
  const size_t n16 = bytes / 16;
  if (mode == 2) {
    k_store_probe_bulk<<<num_sms, 128, 0, s>>>(static_cast<uint8_t*>(dst), n16);
  } else if (mode == 1) {
    k_store_probe<true><<<4 * num_sms, 512, 0, s>>>(static_cast<uint4*>(dst), n16);
  } else {
    k_store_probe<false><<<4 * num_sms, 512, 0, s>>>(static_cast<uint4*>(dst), n16);
  }
  return cudaGetLastError();
}

}  // namespace mapl
