// kernels_spel_tc.cu -- fp32 matrix products of the SPEL step on the
// tcgen05 tensor cores.
//
// The SPEL step (MAPL §3.3 eqs. (4)-(7)) is fp32 arithmetic.  Each fp32
// operand element x is written to shared memory as three bf16 terms
//   hi = bf16(x),  mid = bf16(x - hi),  lo = bf16(x - hi - mid)
// (each remainder is exact in fp32, so hi + mid + lo carries x to about 2^-24),
// and the product is accumulated in fp32 in TMEM from the six term products
// whose magnitude is at least ~2^-16 of the leading one:
//   hi.hi + hi.mid + mid.hi + hi.lo + lo.hi + mid.mid.
// The three dropped products (mid.lo, lo.mid, lo.lo) are below 2^-24 of the
// leading term, the size of fp32 rounding itself.
//
// One CTA computes a 128 x 128 (or 128 x 64) tile of C[z] = opA[z] (M x K) * opB[z]^T
// (opB: N x K) over a K range (split-K writes partial tiles).  Sixteen warps
// load and split the fp32 operand tiles (64 K-columns per step) into two
// shared-memory buffers while thread 0 issues the MMAs of the other buffer;
// the warps then read the accumulator (TMEM lane = row) and store C.
// An operand is read either with K contiguous (element (row, k) at
// p[row * ld + k]) or with rows contiguous (element (row, k) at
// p[k * ld + row], i.e. the transpose of a row-major matrix).
#include "mapl_internal.h"
#include "ptx.cuh"
#include "pdl.cuh"

namespace mapl {

namespace {

constexpr int kGThreads = 512;
constexpr uint32_t kGTile = 128u * 128u;          // one bf16 term: 128 rows x 64 (128 B)
constexpr uint32_t kGBuf = 6u * kGTile;           // A hi/mid/lo + B hi/mid/lo
constexpr uint32_t kGSmem = 2u * kGBuf + 1024u;   // two buffers + alignment

struct GemmOp {
  const float* p;
  long ld;           // leading dimension of the stored matrix
  long sz;           // batch stride
  int rows_contig;   // 1: element (row, k) at p[k * ld + row]
};

// bf16 pair (a in the low half) -> its two fp32 values (exact)
__device__ __forceinline__ float lo_f(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float hi_f(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ uint32_t cvt_pair(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Three-term split of the pair (a, b): h + m + l carries each value, every
// remainder exact in fp32.  Each output packs a in its low 16 bits.
__device__ __forceinline__ void split_pair(float a, float b, uint32_t& h, uint32_t& m,
                                           uint32_t& l) {
  h = cvt_pair(a, b);
  const float ra = a - lo_f(h), rb = b - hi_f(h);
  m = cvt_pair(ra, rb);
  l = cvt_pair(ra - lo_f(m), rb - hi_f(m));
}

__device__ __forceinline__ void st_shared_v2(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void st_shared_f4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from shared to global memory, completion tracked by the bulk group.
__device__ __forceinline__ void bulk_store(float* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(src), "r"(bytes)
               : "memory");
}

constexpr uint32_t kGRowPitch = 528;   // staged C row: 512 bytes + 16 (spreads banks)

__device__ __forceinline__ float sel4(const float4& v, int j) {
  return j == 0 ? v.x : (j == 1 ? v.y : (j == 2 ? v.z : v.w));
}

// Global -> registers: rows [r0, r0 + ROWS) x K-columns [k0, k0 + 64) of an
// operand (ROWS = 128 or 64), ROWS / 32 float4 per thread (512 threads).
//  K contiguous: float4 i of thread t holds row (t >> 4) + 32 i, columns
//    4 (t & 15) .. + 3 (a half-warp reads one 256-byte row).
//  rows contiguous, ROWS = 128: float4 2 i + e holds K-column 2 kp + e + 32 i,
//    rows 4 rq .. + 3, rq = (lane & 7) | ((warp & 3) << 3),
//    kp = (lane >> 3) | ((warp >> 2) << 2) (a warp reads four 128-byte row
//    segments per load); ROWS = 64: float4 e holds K-column 2 kp + e,
//    rq = (lane & 7) | ((warp & 1) << 3), kp = (lane >> 3) | ((warp >> 1) << 2).
template <int ROWS>
__device__ __forceinline__ void fetch_tile(const GemmOp& op, const float* base, int r0, int k0,
                                           int tid, float4 (&v)[ROWS / 32]) {
  if (!op.rows_contig) {
    const float* p = base + static_cast<long>(r0 + (tid >> 4)) * op.ld + k0 + 4 * (tid & 15);
#pragma unroll
    for (int i = 0; i < ROWS / 32; ++i)
      v[i] = *reinterpret_cast<const float4*>(p + 32L * i * op.ld);
  } else {
    const int lane = tid & 31, warp = tid >> 5;
    const int rq = ROWS == 128 ? ((lane & 7) | ((warp & 3) << 3))
                               : ((lane & 7) | ((warp & 1) << 3));
    const int kp = ROWS == 128 ? ((lane >> 3) | ((warp >> 2) << 2))
                               : ((lane >> 3) | ((warp >> 1) << 2));
    const float* p = base + static_cast<long>(k0 + 2 * kp) * op.ld + r0 + 4 * rq;
#pragma unroll
    for (int i = 0; i < ROWS / 64; ++i) {
      v[2 * i] = *reinterpret_cast<const float4*>(p + 32L * i * op.ld);
      v[2 * i + 1] = *reinterpret_cast<const float4*>(p + (32L * i + 1) * op.ld);
    }
  }
}

// Registers -> shared memory: the three bf16 terms of the values fetch_tile
// read, at tiles t0, t0 + kGTile, t0 + 2 kGTile (K-major, 128-byte swizzle,
// row r at r * 128 bytes).  Both layouts store without bank conflicts: in the
// rows-contiguous one, the eight lanes that share a K pair write their four
// rows in a rotated order so that they hit eight different 16-byte chunks.
template <int ROWS>
__device__ __forceinline__ void stash_tile(const GemmOp& op, const float4 (&v)[ROWS / 32],
                                           uint32_t t0, int tid) {
  if (!op.rows_contig) {
    const int q = tid & 15;
#pragma unroll
    for (int i = 0; i < ROWS / 32; ++i) {
      const int row = (tid >> 4) + 32 * i;
      uint32_t h01, m01, l01, h23, m23, l23;
      split_pair(v[i].x, v[i].y, h01, m01, l01);
      split_pair(v[i].z, v[i].w, h23, m23, l23);
      const uint32_t off = sw128_off(static_cast<uint32_t>(row), static_cast<uint32_t>(q >> 1)) +
                           static_cast<uint32_t>(q & 1) * 8u;
      st_shared_v2(t0 + off, h01, h23);
      st_shared_v2(t0 + kGTile + off, m01, m23);
      st_shared_v2(t0 + 2u * kGTile + off, l01, l23);
    }
  } else {
    const int lane = tid & 31, warp = tid >> 5;
    const int rq = ROWS == 128 ? ((lane & 7) | ((warp & 3) << 3))
                               : ((lane & 7) | ((warp & 1) << 3));
    const int rot = (lane & 7) >> 1;
    const uint32_t kbyte = static_cast<uint32_t>(lane >> 3) * 4u;   // (2 kp mod 8) * 2 bytes
#pragma unroll
    for (int i = 0; i < ROWS / 64; ++i) {
      // k >> 3 of K-column 2 kp + e (+ 32 i)
      const uint32_t chunk = ROWS == 128 ? static_cast<uint32_t>((warp >> 2) | (i << 2))
                                         : static_cast<uint32_t>(warp >> 1);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int jj = (j + rot) & 3;
        uint32_t h, m, l;
        split_pair(sel4(v[2 * i], jj), sel4(v[2 * i + 1], jj), h, m, l);
        const uint32_t off = sw128_off(static_cast<uint32_t>(4 * rq + jj), chunk) + kbyte;
        st_shared_u32(t0 + off, h);
        st_shared_u32(t0 + kGTile + off, m);
        st_shared_u32(t0 + 2u * kGTile + off, l);
      }
    }
  }
}

// C[z] (+ ks * sS) = opA[z] * opB[z]^T over split ks of K, fp32, in
// 128 x TN output tiles (TN = 128, or 64 to give a small product twice the
// CTAs).  grid: (N / TN, M / 128, batch * ksplit); C row-major with leading
// dimension ldc and batch stride sC.  Every wait is bounded; a CTA that gives
// up writes NaN over its tile, so the failure reaches the caller's result.
template <int TN>
__global__ void __launch_bounds__(kGThreads, 1)
    k_gemm3(GemmOp A, GemmOp B, float* __restrict__ C, long ldc, long sC, long sS, int K,
            int ksplit, uint64_t budget_ns) {
  pdl_allow_next();
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t mma_done[2];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int z = blockIdx.z / ksplit, ks = blockIdx.z % ksplit;
  const int m0 = blockIdx.y * 128, n0 = blockIdx.x * TN;
  const int kbeg = static_cast<int>(static_cast<long>(K) * ks / ksplit);
  const int kend = static_cast<int>(static_cast<long>(K) * (ks + 1) / ksplit);
  const int nkb = (kend - kbeg) / 64;
  const float* pa = A.p + z * A.sz;
  const float* pb = B.p + z * B.sz;

  if (tid == 0) {
    mbar_init(smem_u32(&mma_done[0]), 1);
    mbar_init(smem_u32(&mma_done[1]), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(&tmem_base), TN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tacc = tmem_base;
  // the setup above overlapped the kernels before this one; the operands
  // they wrote are read only from here on
  pdl_wait_prior();
  constexpr uint32_t idesc = idesc_bf16(128, TN);
  bool ok = true;
  int issued = 0;
  float4 va[4], vb[TN / 32];   // this K block
  float4 na[4], nb[TN / 32];   // the next one, in flight while this one is split
  if (nkb > 0) {
    fetch_tile<128>(A, pa, m0, kbeg, tid, va);
    fetch_tile<TN>(B, pb, n0, kbeg, tid, vb);
  }

  for (int kb = 0; kb < nkb; ++kb) {
    const int b = kb & 1;
    const uint32_t buf = sbase + static_cast<uint32_t>(b) * kGBuf;
    // the loads do not touch shared memory: the next block's start before
    // this block waits for its buffer and is split into it
    if (kb + 1 < nkb) {
      fetch_tile<128>(A, pa, m0, kbeg + (kb + 1) * 64, tid, na);
      fetch_tile<TN>(B, pb, n0, kbeg + (kb + 1) * 64, tid, nb);
    }
    // the MMAs that read this buffer two steps ago have completed (one
    // thread waits; the barrier releases the rest)
    if (kb >= 2 && tid == 0)
      ok = mbar_wait(smem_u32(&mma_done[b]), ((kb >> 1) - 1) & 1, &abort_flag, budget_ns);
    ok = __syncthreads_and(ok) != 0;
    if (!ok) break;
    stash_tile<128>(A, va, buf, tid);
    stash_tile<TN>(B, vb, buf + 3u * kGTile, tid);
    fence_async_shared();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      // term pairs (A term, B term): hi.hi, hi.mid, mid.hi, hi.lo, lo.hi, mid.mid
#pragma unroll
      for (int pidx = 0; pidx < 6; ++pidx) {
        const uint32_t ta = pidx == 2 ? 1u : (pidx == 4 ? 2u : (pidx == 5 ? 1u : 0u));
        const uint32_t tb = pidx == 1 ? 1u : (pidx == 3 ? 2u : (pidx == 5 ? 1u : 0u));
        const uint64_t ad = sw128_desc(buf + ta * kGTile);
        const uint64_t bd = sw128_desc(buf + (3u + tb) * kGTile);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(tacc, ad + 2 * k, bd + 2 * k, idesc, (kb | pidx | k) != 0 ? 1u : 0u);
      }
      mma_commit(smem_u32(&mma_done[b]));
    }
    ++issued;
#pragma unroll
    for (int i = 0; i < 4; ++i) va[i] = na[i];
#pragma unroll
    for (int i = 0; i < TN / 32; ++i) vb[i] = nb[i];
  }
  // the last commit arrives once every MMA issued before it has completed
  if (issued > 0) {
    const int last = issued - 1;
    bool fin = true;
    if (tid == 0)
      fin = mbar_wait(smem_u32(&mma_done[last & 1]), (last >> 1) & 1, &abort_flag, budget_ns);
    ok = __syncthreads_and(ok && fin) != 0;
  }
  tc_fence_after();
  if (nkb > 0 && 32 * (warp >> 2) < TN) {
    // warp w reads TMEM lanes 32 (w & 3) .. + 31 (its lane quarter) and
    // accumulator columns 32 (w >> 2) .. + 31, and stages them row-major in
    // the (now idle) first operand buffer; rows then leave by bulk copies.
    const int row = 32 * (warp & 3) + lane, c0 = 32 * (warp >> 2);
    float v[32];
    if (ok) {
      tmem_ld32(tacc + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + static_cast<uint32_t>(c0),
                v);
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __int_as_float(0x7fc00000);
    }
    const uint32_t srow = sbase + static_cast<uint32_t>(row) * kGRowPitch + 4u * c0;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      st_shared_f4(srow + 16u * j, v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    fence_async_shared();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tacc, TN);
  if (nkb > 0 && tid < 128) {
    bulk_store(C + z * sC + ks * sS + static_cast<long>(m0 + tid) * ldc + n0,
               sbase + static_cast<uint32_t>(tid) * kGRowPitch, 4u * TN);
    bulk_commit();
    bulk_wait<0>();
  }
}

}  // namespace

bool gemm3_supported(int M, int N, int K, int ksplit) {
  return M > 0 && N > 0 && M % 128 == 0 && N % 128 == 0 && ksplit >= 1 && K > 0 &&
         K % (64 * ksplit) == 0;
}

cudaError_t launch_gemm3(const Gemm3Operand& a, const Gemm3Operand& b, float* C, long ldc,
                         long sC, long sS, int M, int N, int K, int batch, int ksplit,
                         cudaStream_t s) {
  if (!gemm3_supported(M, N, K, ksplit) || batch < 1 || batch * ksplit > 65535)
    return cudaErrorInvalidValue;
  // float4 loads and 16-byte bulk stores: 16-byte aligned rows and batches
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!al16(a.p) || !al16(b.p) || !al16(C) || ((a.ld | a.batch_stride | b.ld | b.batch_stride |
                                                 ldc | sC | sS) & 3) != 0)
    return cudaErrorInvalidValue;
  // 128 x 64 tiles when 128 x 128 tiles would leave more than half of the
  // SMs idle (the chain inside one CTA, not the tensor pipe, sets the time)
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long ctas128 = static_cast<long>(N / 128) * (M / 128) * batch * ksplit;
  const bool narrow = 2 * ctas128 <= sms;
  auto kern = narrow ? k_gemm3<64> : k_gemm3<128>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kGSmem));
  if (e != cudaSuccess) return e;
  const GemmOp ga{a.p, a.ld, a.batch_stride, a.rows_contig};
  const GemmOp gb{b.p, b.ld, b.batch_stride, b.rows_contig};
  const dim3 grid(static_cast<unsigned>(N / (narrow ? 64 : 128)), static_cast<unsigned>(M / 128),
                  static_cast<unsigned>(batch * ksplit));
  return launch_chained(kern, grid, dim3(kGThreads), kGSmem, s, ga, gb, C, ldc, sC, sS, K,
                        ksplit, kDefaultTimeoutNs);
}

}  // namespace mapl
