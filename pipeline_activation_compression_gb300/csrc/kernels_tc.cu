// kernels_tc.cu -- tcgen05 / TMA decompress kernel of the MAPL codec (bf16).
//
// decompress (eq. (2)):
//   X_hat = [Z_hat | E'[tids]] [A^T ; P']   one contraction with K = 2r
//
// One CTA owns a tile of 128 tokens (the MMA M).  Warp roles (192 threads):
//   warp 0 lane 0 : TMA producer of a ring of shared-memory stages
//   warp 1        : TMEM allocation; lane 0 issues every tcgen05.mma
//   warps 2..5    : gather of anchor rows, VQ / epilogue (TMEM lane = row)
// Every wait is bounded (mbar_wait); on give-up the CTA sets the device error
// word, writes nothing more and unwinds through the common exit.
#include "mapl_internal.h"
#include "pdl.cuh"
#include "ptx.cuh"

namespace mapl {

namespace {

constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr int kMaxStages = 8;
constexpr uint32_t kBlockBytes = kTile * 128;   // 128 rows x 64 bf16, swizzled
constexpr int kEpiBar = 1;                      // named barrier of the epilogue warps

struct Ctl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t zfull;     // compress: Z accumulator complete
  uint64_t uready;    // compress: VQ residual operand written
  uint64_t dready;    // compress: VQ distances in TMEM
  uint64_t aready;    // decompress: resident A operand built / loaded
  uint64_t tfull[2];  // decompress: accumulator ready
  uint64_t tempty[2]; // decompress: accumulator drained
  uint32_t tmem_base;
  int abort;
  int gate;           // anchor-gather items whose stage the producer has freed
  int32_t tids[kTile];
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

template <typename C>
__device__ __forceinline__ void give_up(C* ctl, int* err) {
  ctl->abort = 1;
  atomicOr(err, kErrTimeout);
}

// 8 consecutive threads copy one row's 64-element K-block of an anchor
// table into a swizzled 128-row tile.  Rows with a negative id get zeros.
__device__ __forceinline__ void gather_block(const __nv_bfloat16* __restrict__ E, int r,
                                             const int32_t* tids_s, int kb, uint32_t dst,
                                             int tid) {
#pragma unroll 4
  for (int q = tid; q < kTile * 8; q += kEpiThreads) {
    const int row = q >> 3, c = q & 7;
    const int t = tids_s[row];
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (t >= 0)
      v = __ldg(reinterpret_cast<const uint4*>(E + static_cast<size_t>(t) * r + kb * 64 + c * 8));
    st_shared_v4(dst + sw128_off(row, c), v);
  }
}

// Load the tile's token ids; out-of-range ids are recorded (-1) and flagged,
// rows past N get -2.  Both produce zero anchor rows.
__device__ __forceinline__ void load_tids(const int32_t* __restrict__ tids, int N, int V, int tile,
                                          int tid, int32_t* tids_s, int* err) {
  for (int q = tid; q < kTile; q += kEpiThreads) {
    const int n = tile * kTile + q;
    int t = -2;
    if (n < N) {
      t = tids[n];
      if (t < 0 || t >= V) {
        t = -1;
        atomicOr(err, kErrBadToken);
      }
    }
    tids_s[q] = t;
  }
}

// ======================================================================
// decompress
// ======================================================================
template <int GD>
__device__ __forceinline__ void decode_rows(const DecompressArgs& a, const int32_t* tids_s,
                                            uint32_t aop, int row, int n) {
  // Z_hat[n, g-block] = sum_rho C[rho][g][idx[n][rho][g]]  (fp32, then bf16)
  const int G = a.G, R = a.R, K = a.K;
  const bool live = n < a.N && tids_s[row] != -1;
  const uint8_t* ip = a.idx + static_cast<size_t>(n) * R * G;
  for (int g = 0; g < G; ++g) {
    float acc[GD];
#pragma unroll
    for (int i = 0; i < GD; ++i) acc[i] = 0.f;
    if (live) {
      for (int rho = 0; rho < R; ++rho) {
        int k = ip[rho * G + g];
        if (k >= K) {   // not a valid code: flag it, never read past the book
          atomicOr(a.err, kErrBadIndex);
          k = K - 1;
        }
        const uint4* cr = reinterpret_cast<const uint4*>(
            a.Cb + (static_cast<size_t>(rho * G + g) * K + k) * GD);
#pragma unroll
        for (int c = 0; c < GD / 8; ++c) {
          const uint4 w = __ldg(cr + c);
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h[e]);
            acc[c * 8 + 2 * e] += f.x;
            acc[c * 8 + 2 * e + 1] += f.y;
          }
        }
      }
    }
#pragma unroll
    for (int c = 0; c < GD / 8; ++c) {
      const int col = g * GD + c * 8;
      uint4 v;
      v.x = pack_bf16x2(acc[c * 8 + 0], acc[c * 8 + 1]);
      v.y = pack_bf16x2(acc[c * 8 + 2], acc[c * 8 + 3]);
      v.z = pack_bf16x2(acc[c * 8 + 4], acc[c * 8 + 5]);
      v.w = pack_bf16x2(acc[c * 8 + 6], acc[c * 8 + 7]);
      st_shared_v4(aop + (col >> 6) * kBlockBytes + sw128_off(row, (col & 63) >> 3), v);
    }
  }
}

template <int GD>
__global__ void __launch_bounds__(kThreads, 2)
    k_decompress_tc(const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmZ, const DecompressArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  const int nst = a.nstage;
  const uint32_t sb = a.stage_bytes;
  const uint32_t aop = smem_u32(base);               // resident A operand
  const uint32_t ring = aop + a.a_bytes;
  Ctl* ctl = reinterpret_cast<Ctl*>(base + a.a_bytes + nst * sb);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x;
  const int r = a.r, d = a.d;
  const int NC = a.nc;                            // output chunk
  const int nchunk = d / NC;
  const int nzb = r / 64;                          // K-blocks holding Z_hat
  const int nka = a.anchor ? 2 * nzb : nzb;        // K-blocks of [Z_hat | E'] (or Z_hat)
  const int nitems = nchunk * nka;
  const bool stream = a.a_stream != 0;
  const uint32_t a_slot = stream ? kBlockBytes : 0u;   // A block at stage start
  const uint32_t tmem_cols = 2u * NC < 32u ? 32u : 2u * NC;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 2);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    mbar_init(smem_u32(&ctl->aready), 2);
    ctl->gate = 0;
    for (int q = 0; q < 2; ++q) {
      mbar_init(smem_u32(&ctl->tfull[q]), 1);
      mbar_init(smem_u32(&ctl->tempty[q]), 1);
    }
    ctl->abort = 0;
    fence_mbar_init();
    fence_async_shared();
  }
  if (warp == 1) tmem_alloc(smem_u32(&ctl->tmem_base), tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmB);
      if (!a.vq) prefetch_tmap(&tmZ);
      if (!stream) {
        const uint32_t ab = smem_u32(&ctl->aready);
        if (!a.vq) {
          mbar_arrive_expect_tx(ab, nzb * kBlockBytes);
          for (int kb = 0; kb < nzb; ++kb)
            tma_load_2d(aop + kb * kBlockBytes, &tmZ, kb * 64, tile * kTile, ab);
        } else {
          mbar_arrive(ab);
        }
      }
      for (int i = 0; i < nitems; ++i) {
        const int s = i % nst, use = i / nst;
        const int c = i / nka, kb = i % nka;
        if (!mbar_wait(smem_u32(&ctl->empty[s]), (use & 1) ^ 1, &ctl->abort, a.timeout_ns)) {
          give_up(ctl, a.err);
          break;
        }
        const uint32_t st = ring + s * sb;
        const uint32_t fb = smem_u32(&ctl->full[s]);
        if (stream && kb < nzb) {
          mbar_arrive_expect_tx(fb, kBlockBytes + NC * 128u);
          tma_load_2d(st, &tmZ, kb * 64, tile * kTile, fb);
          tma_load_2d(st + a_slot, &tmB, kb * 64, c * NC, fb);
          mbar_arrive(fb);
        } else {
          mbar_arrive_expect_tx(fb, NC * 128u);
          tma_load_2d(st + a_slot, &tmB, kb * 64, c * NC, fb);
          if (!stream) {
            mbar_arrive(fb);
          } else {
            // streamed E' block: the stage is free for the builders, who
            // give the second arrival; gate counts such items in order
            gate_publish(smem_u32(&ctl->gate), c * nzb + (kb - nzb) + 1);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idc = idesc_bf16(kTile, NC);
      bool ok = true;
      if (!stream) ok = mbar_wait(smem_u32(&ctl->aready), 0, &ctl->abort, a.timeout_ns);
      if (!ok) give_up(ctl, a.err);
      for (int c = 0; c < nchunk && ok; ++c) {
        const int acc = c & 1;
        if (!mbar_wait(smem_u32(&ctl->tempty[acc]), ((c >> 1) & 1) ^ 1, &ctl->abort,
                       a.timeout_ns)) {
          give_up(ctl, a.err);
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < nka; ++kb) {
          const int i = c * nka + kb, s = i % nst, use = i / nst;
          if (!mbar_wait(smem_u32(&ctl->full[s]), use & 1, &ctl->abort, a.timeout_ns)) {
            give_up(ctl, a.err);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = ring + s * sb;
          const uint32_t aa = stream ? st : aop + kb * kBlockBytes;
          const uint32_t bb = st + a_slot;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16(tbase + acc * NC, sw128_desc(aa + k * 32), sw128_desc(bb + k * 32), idc,
                     (kb | k) != 0 ? 1u : 0u);
          mma_commit(smem_u32(&ctl->empty[s]));
        }
        if (ok) mma_commit(smem_u32(&ctl->tfull[acc]));
      }
    }
  } else {
    const int tid = threadIdx.x - 64;
    const int row = (warp & 3) * 32 + lane;
    const int n = tile * kTile + row;
    if (a.anchor) {
      load_tids(a.tids, a.N, a.V, tile, tid, ctl->tids, a.err);
    } else {
      for (int q = tid; q < kTile; q += kEpiThreads) ctl->tids[q] = tile * kTile + q < a.N ? 0 : -2;
    }
    named_bar_sync(kEpiBar, kEpiThreads);
    bool alive = true;
    if (!stream) {
      if (a.vq) {
        if constexpr (GD > 0) decode_rows<GD>(a, ctl->tids, aop, row, n);
      }
      if (a.anchor)
        for (int kb = 0; kb < nzb; ++kb)
          gather_block(a.E, r, ctl->tids, kb, aop + (nzb + kb) * kBlockBytes, tid);
      fence_async_shared();
      named_bar_sync(kEpiBar, kEpiThreads);
      if (tid == 0) mbar_arrive(smem_u32(&ctl->aready));
    }
    const uint32_t trow = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const bool store = n < a.N;
    const bool bad = ctl->tids[row] == -1;
    // streamed mode gathers the E' blocks of chunk c before draining chunk c-1
    for (int c = 0; c <= nchunk && alive; ++c) {
      if (stream && c < nchunk) {
        for (int kb = nzb; kb < nka; ++kb) {
          const int i = c * nka + kb, s = i % nst;
          bool ok = gate_wait(smem_u32(&ctl->gate), c * nzb + (kb - nzb), &ctl->abort,
                              a.timeout_ns);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) {
            give_up(ctl, a.err);
            alive = false;
            break;
          }
          gather_block(a.E, r, ctl->tids, kb - nzb, ring + s * sb, tid);
          fence_async_shared();
          named_bar_sync(kEpiBar, kEpiThreads);
          if (tid == 0) mbar_arrive(smem_u32(&ctl->full[s]));
        }
        if (!alive) break;
      }
      const int cd = stream ? c - 1 : c;       // chunk to drain now
      if (cd < 0 || cd >= nchunk) continue;
      const int acc = cd & 1;
      bool ok = mbar_wait(smem_u32(&ctl->tfull[acc]), (cd >> 1) & 1, &ctl->abort, a.timeout_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        give_up(ctl, a.err);
        alive = false;
        break;
      }
      tc_fence_after();
      for (int c0 = 0; c0 < NC; c0 += 32) {
        float v[32];
        __syncwarp();
        tmem_ld32(trow + acc * NC + c0, v);
        tmem_wait_ld();
        if (!store) continue;   // no collective operation follows in this iteration
        uint4* dst = reinterpret_cast<uint4*>(a.Xh + static_cast<size_t>(n) * d + cd * NC + c0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 w = make_uint4(0u, 0u, 0u, 0u);
          if (!bad)
            w = make_uint4(pack_bf16x2(v[8 * q + 0], v[8 * q + 1]),
                           pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                           pack_bf16x2(v[8 * q + 4], v[8 * q + 5]),
                           pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
          dst[q] = w;
        }
      }
      tc_fence_before();
      named_bar_sync(kEpiBar, kEpiThreads);
      if (tid == 0) mbar_arrive(smem_u32(&ctl->tempty[acc]));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tbase, tmem_cols);
  }
}

// ======================================================================
// decompress, persistent form (A operand in TMEM, r <= 256)
// ======================================================================
// One CTA per SM walks its own contiguous range of rows in tiles of up to
// 128 rows.  A tile's A operand [Z_hat | E'[tids]] (128 rows, K = 2r; K = r
// without the anchor term) lives in TMEM, two bf16 per 32-bit column (the
// lower K index in the low half), where the builder warps write it, and the
// tensor cores read it from there ([a-tmem] form).  Shared memory then holds
// only the [A^T | P'^T] ring, as deep as it fits (the ring is L2-latency
// bound), and the drain's staging.  TMEM columns: [acc 0 | acc 1 | A 0 |
// A 1] = NC, NC, K/2, K/2 (one A buffer when two do not fit).
// Warp roles (320 threads):
//   warp 0 lane 0 : TMA producer of the [A^T | P'^T] ring (NC x 64 blocks)
//   warp 1        : TMEM allocation; lane 0 issues every tcgen05.mma
//   warps 2..5    : builders: warp w writes TMEM lanes 32 (w % 4).. (its
//                   rows) of the next tile's A: the VQ decode (or the Z_hat
//                   payload row) and the E' row of the token's id
//   warps 6..9    : drain of the two TMEM accumulators (TMEM lane = row)
constexpr int kPtThreads = 320;
constexpr int kPtDrain0 = 6;      // first drain warp
constexpr int kPtMaxStages = 12;
constexpr uint32_t kPtStagingBytes = 4 * 4096;   // per drain warp: 32 rows x 128 B

struct CtlPt {
  uint64_t full[kPtMaxStages];
  uint64_t empty[kPtMaxStages];
  uint64_t afull[2];      // A operand written (one arrival per builder warp)
  uint64_t aempty[2];     // MMAs of the tile that used the buffer are complete
  uint64_t tfull[2];      // accumulator holds a finished chunk
  uint64_t tempty[2];     // accumulator drained (one arrival per drain warp)
  uint64_t done;          // every MMA of the CTA has completed
  uint64_t efull;         // first tile: E' rows written by the drain warps
  uint32_t tmem_base;
  int abort;
};

// Code index of (round rho, group g) in a VQ payload row; an index >= K is
// flagged and replaced by K - 1 (never read past the book).
__device__ __forceinline__ int code_index(const DecompressArgs& a, const uint8_t* ip, int rho,
                                          int g) {
  int k = ip[rho * a.G + g];
  if (k >= a.K) {
    atomicOr(a.err, kErrBadIndex);
    k = a.K - 1;
  }
  return k;
}

template <int GD>
__device__ __forceinline__ void load_code(const DecompressArgs& a, int rho, int g, int k,
                                          uint4 (&w)[GD / 8]) {
  const uint4* cr =
      reinterpret_cast<const uint4*>(a.Cb + (static_cast<size_t>(rho * a.G + g) * a.K + k) * GD);
#pragma unroll
  for (int c = 0; c < GD / 8; ++c) w[c] = __ldg(cr + c);
}

template <int GD>
__device__ __forceinline__ void add_code(const uint4 (&w)[GD / 8], float* acc) {
#pragma unroll
  for (int c = 0; c < GD / 8; ++c) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w[c]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      acc[c * 8 + 2 * e] += f.x;
      acc[c * 8 + 2 * e + 1] += f.y;
    }
  }
}

// Z_hat row n of the VQ payload into this thread's TMEM lane, columns
// [ta, ta + r / 2): per 64 elements (64 / GD groups), the code indices of
// every round first, then the codes of two rounds at a time in flight, each
// group summed over the rounds in order in fp32, then rounded to bf16.
template <int GD>
__device__ __forceinline__ void decode_row_tm(const DecompressArgs& a, uint32_t ta, int n,
                                              bool live) {
  constexpr int GP = 64 / GD;   // groups per 64 elements
  const int R = a.R;
  const uint8_t* ip = a.idx + static_cast<size_t>(n) * R * a.G;
  for (int g0 = 0; g0 < a.G; g0 += GP) {
    float v[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = 0.f;
    if (live) {
      for (int r0 = 0; r0 < R; r0 += 2) {
        int k[2][GP];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int x = 0; x < GP; ++x) k[j][x] = r0 + j < R ? code_index(a, ip, r0 + j, g0 + x) : 0;
        uint4 w[2][GP][GD / 8];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int x = 0; x < GP; ++x)
            if (r0 + j < R) load_code<GD>(a, r0 + j, g0 + x, k[j][x], w[j][x]);
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int x = 0; x < GP; ++x)
            if (r0 + j < R) add_code<GD>(w[j][x], v + x * GD);
      }
    }
    uint32_t u[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) u[c] = pack_bf16x2(v[2 * c], v[2 * c + 1]);
    tmem_st32u(ta + static_cast<uint32_t>(g0 * GD / 2), u);
  }
}

// A bf16 row (ncol 32-bit columns, a multiple of 32) into this thread's
// TMEM lane from `src` (16-byte aligned), or zeros when !live.
__device__ __forceinline__ void copy_row_tm(const __nv_bfloat16* src, int ncol, uint32_t ta,
                                            bool live) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  for (int c0 = 0; c0 < ncol; c0 += 32) {
    uint4 w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = live ? __ldg(s4 + c0 / 4 + j) : make_uint4(0u, 0u, 0u, 0u);
    uint32_t u[32];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      u[4 * j] = w[j].x;
      u[4 * j + 1] = w[j].y;
      u[4 * j + 2] = w[j].z;
      u[4 * j + 3] = w[j].w;
    }
    tmem_st32u(ta + static_cast<uint32_t>(c0), u);
  }
}

template <int GD>
__global__ void __launch_bounds__(kPtThreads, 1)
    k_decompress_pt(const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmXh, const DecompressArgs a) {
  // dependent launch: the setup below overlaps the kernel before this one;
  // nothing in memory is touched before pdl_wait_prior
  pdl_allow_next();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  const int nst = a.nstage, nab = a.nab;
  const uint32_t sb = a.stage_bytes;
  const uint32_t ring = smem_u32(base);
  const uint32_t stage0 = ring + nst * sb;                   // drain staging
  CtlPt* ctl = reinterpret_cast<CtlPt*>(base + nst * sb + kPtStagingBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NC = a.nc;
  const int nchunk = a.d / NC;
  const int nzb = a.r / 64;          // K-blocks of Z_hat (and of E')
  const int nka = a.anchor ? 2 * nzb : nzb;   // K-blocks of [Z_hat | E'] (or Z_hat alone)
  const uint32_t acol0 = 2u * static_cast<uint32_t>(NC);     // TMEM column of A buffer 0
  const uint32_t acols = static_cast<uint32_t>(nka) * 32u;   // TMEM columns of one A buffer
  // this CTA's rows: a contiguous run of 32-row blocks, [rbeg, rend), walked
  // in tiles of up to 128 rows, so every SM writes about the same number of
  // rows; tile edges fall on 32-row boxes, so no TMA store crosses into the
  // next CTA's rows
  const int nb32 = (a.N + 31) / 32;
  const int blk0 = static_cast<int>(static_cast<long long>(nb32) * blockIdx.x / gridDim.x);
  const int blk1 = static_cast<int>(static_cast<long long>(nb32) * (blockIdx.x + 1) / gridDim.x);
  const int rbeg = 32 * blk0, rend = 32 * blk1 < a.N ? 32 * blk1 : a.N;
  const int L = (blk1 - blk0 + 3) / 4;
  constexpr uint32_t tmem_cols = 512;
  const uint64_t bud = a.timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctl->afull[b]), 4);
      mbar_init(smem_u32(&ctl->aempty[b]), 1);
      mbar_init(smem_u32(&ctl->tfull[b]), 1);
      mbar_init(smem_u32(&ctl->tempty[b]), 4);
    }
    mbar_init(smem_u32(&ctl->done), 1);
    mbar_init(smem_u32(&ctl->efull), 4);
    ctl->abort = 0;
    fence_mbar_init();
    fence_async_shared();
  }
  if (warp == 1) tmem_alloc(smem_u32(&ctl->tmem_base), tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = ctl->tmem_base;
  // the payload (and the plan's tables) may come from the kernel before
  pdl_wait_prior();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------- B operand producer
      prefetch_tmap(&tmB);
      int s = 0, issued = 0;
      uint32_t ph = 0;
      bool ok = true;
      // a stage holds two 64-element K-blocks of NC rows: one 3-D box
      for (int it = 0; it < L && ok; ++it)
        for (int c = 0; c < nchunk && ok; ++c)
          for (int kb = 0; kb < nka; kb += 2) {
            if (!(ok = mbar_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, &ctl->abort, bud))) break;
            const uint32_t fb = smem_u32(&ctl->full[s]);
            mbar_arrive_expect_tx(fb, 2u * static_cast<uint32_t>(NC) * 128u);
            tma_load_3d(ring + s * sb, &tmB, 0, c * NC, kb, fb);
            ++issued;
            if (++s == nst) {
              s = 0;
              ph ^= 1u;
            }
          }
      if (!ok) {
        give_up(ctl, a.err);
        // let the copies in flight land before the CTA's memory goes away
        for (int x = 0; x < nst && x < issued; ++x) {
          const int i = issued - 1 - x, ss = i % nst;
          mbar_wait(smem_u32(&ctl->full[ss]), static_cast<uint32_t>(i / nst) & 1u, &ctl->abort,
                    bud / 16);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t idc = idesc_bf16(kTile, NC);
      const uint64_t r_d = sw128_desc(ring);
      int s = 0, cc = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int it = 0; it < L && ok; ++it) {
        const int ab = nab == 2 ? (it & 1) : 0;
        const int ause = nab == 2 ? (it >> 1) : it;
        if (!(ok = mbar_wait(smem_u32(&ctl->afull[ab]), ause & 1, &ctl->abort, bud))) break;
        if (it == 0 && a.anchor && !(ok = mbar_wait(smem_u32(&ctl->efull), 0, &ctl->abort, bud)))
          break;
        tc_fence_after();
        const uint32_t at = tbase + acol0 + static_cast<uint32_t>(ab) * acols;
        for (int c = 0; c < nchunk && ok; ++c, ++cc) {
          const int acc = cc & 1;
          if (!(ok = mbar_wait(smem_u32(&ctl->tempty[acc]), ((cc >> 1) & 1) ^ 1, &ctl->abort,
                               bud)))
            break;
          tc_fence_after();
          for (int kb = 0; kb < nka; kb += 2) {
            if (!(ok = mbar_wait(smem_u32(&ctl->full[s]), ph, &ctl->abort, bud))) break;
            tc_fence_after();
            for (int j = 0; j < 2 && kb + j < nka; ++j) {
              const uint64_t bd =
                  r_d + ((static_cast<uint32_t>(s) * sb + static_cast<uint32_t>(j * NC) * 128u) >> 4);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_bf16_ta(tbase + acc * NC, at + static_cast<uint32_t>((kb + j) * 32 + k * 8),
                            bd + 2 * k, idc, (kb + j + k) != 0 ? 1u : 0u);
            }
            mma_commit(smem_u32(&ctl->empty[s]));
            if (++s == nst) {
              s = 0;
              ph ^= 1u;
            }
          }
          if (ok) mma_commit(smem_u32(&ctl->tfull[acc]));
        }
        if (ok) mma_commit(smem_u32(&ctl->aempty[ab]));
      }
      if (!ok) give_up(ctl, a.err);
      // every MMA issued above has completed once `done` flips
      mma_commit(smem_u32(&ctl->done));
      mbar_wait(smem_u32(&ctl->done), 0, &ctl->abort, bud);
    }
  } else if (warp < kPtDrain0) {
    // ------------------------------------------------------------- builders
    const int row = (warp & 3) * 32 + lane;   // this thread's TMEM lane and tile row
    const uint32_t tq = static_cast<uint32_t>((warp & 3) * 32) << 16;
    for (int it = 0; it < L; ++it) {
      const int t0 = rbeg + it * kTile;
      const int cnt = rend - t0 < kTile ? rend - t0 : kTile;   // rows of this tile
      const int ab = nab == 2 ? (it & 1) : 0;
      const int ause = nab == 2 ? (it >> 1) : it;
      bool ok = mbar_wait(smem_u32(&ctl->aempty[ab]), (ause & 1) ^ 1, &ctl->abort, bud);
      ok = __all_sync(0xffffffffu, ok) && !ctl->abort;
      if (!ok) {
        if (lane == 0) give_up(ctl, a.err);
        break;
      }
      tc_fence_after();   // the MMAs that read this buffer have completed
      const int n = t0 + row;
      const uint32_t ta = tbase + tq + acol0 + static_cast<uint32_t>(ab) * acols;
      int t = 0;
      bool live = row < cnt;
      if (live && a.anchor) {
        t = __ldg(a.tids + n);
        if (t < 0 || t >= a.V) {
          atomicOr(a.err, kErrBadToken);
          live = false;
        }
      }
      if (a.vq) {
        if constexpr (GD > 0) decode_row_tm<GD>(a, ta, n, live);
      } else {
        copy_row_tm(a.Zp + static_cast<size_t>(live ? n : 0) * a.r, a.r / 2, ta, live);
      }
      if (a.anchor && it > 0)   // the first tile's E' rows come from the drain warps
        copy_row_tm(a.E + static_cast<size_t>(t) * a.r, a.r / 2, ta + static_cast<uint32_t>(a.r / 2),
                    live);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->afull[ab]));
    }
  } else {
    // ---------------------------------------------------------------- drain
    // TMEM -> bf16 -> a swizzled 32-row x 64-column staging tile -> TMA
    // store.  The tile is reused once the previous store has read it.
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t trow = tbase + (static_cast<uint32_t>(q * 32) << 16);
    if (a.anchor && L > 0) {
      // the first tile's anchor rows E'[tids], written beside the builders'
      // Z_hat so that the two chains of dependent loads run side by side
      const int cnt0 = rend - rbeg < kTile ? rend - rbeg : kTile;
      int t = 0;
      bool live = row < cnt0;
      if (live) {
        t = __ldg(a.tids + rbeg + row);
        live = t >= 0 && t < a.V;   // the builder flags a bad id
      }
      copy_row_tm(a.E + static_cast<size_t>(live ? t : 0) * a.r, a.r / 2,
                  trow + acol0 + static_cast<uint32_t>(a.r / 2), live);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->efull));
    }
    const uint32_t stg = stage0 + (warp - kPtDrain0) * 4096u;
    if (lane == 0) prefetch_tmap(&tmXh);
    int cc = 0;
    bool alive = true;
    for (int it = 0; it < L && alive; ++it) {
      const int t0 = rbeg + it * kTile;
      const int cnt = rend - t0 < kTile ? rend - t0 : kTile;   // rows of this tile
      const int n = t0 + row;
      const int row0 = t0 + q * 32;               // first row of this warp's box
      const bool any = q * 32 < cnt;
      bool bad = false;
      int t = 0;
      if (row < cnt && (a.anchor || a.Eadd)) {
        t = __ldg(a.tids + n);
        bad = t < 0 || t >= a.V;
        if (bad && !a.anchor) atomicOr(a.err, kErrBadToken);   // no builder saw this id
      }
      // first-boundary anchor: the full embedding row is added in fp32
      const __nv_bfloat16* erow =
          (a.Eadd && row < cnt && !bad) ? a.Eadd + static_cast<size_t>(t) * a.d : nullptr;
      for (int c = 0; c < nchunk; ++c, ++cc) {
        const int acc = cc & 1;
        bool ok = mbar_wait(smem_u32(&ctl->tfull[acc]), (cc >> 1) & 1, &ctl->abort, bud);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          give_up(ctl, a.err);
          alive = false;
          break;
        }
        tc_fence_after();
        for (int c0 = 0; c0 < NC; c0 += 64) {
          float v0[32], v1[32];
          uint4 ev[8];
          if (erow) {
            const uint4* src = reinterpret_cast<const uint4*>(erow + c * NC + c0);
#pragma unroll
            for (int j = 0; j < 8; ++j) ev[j] = __ldg(src + j);
          }
          __syncwarp();
          tmem_ld32(trow + acc * NC + c0, v0);
          tmem_ld32(trow + acc * NC + c0 + 32, v1);
          tmem_wait_ld();
          if (erow) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              float* vv = j < 4 ? v0 + 8 * j : v1 + 8 * (j - 4);
              const uint32_t w4[4] = {ev[j].x, ev[j].y, ev[j].z, ev[j].w};
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                vv[2 * h] += __uint_as_float(w4[h] << 16);
                vv[2 * h + 1] += __uint_as_float(w4[h] & 0xffff0000u);
              }
            }
          }
          if (!any) continue;   // no collective operation follows in this iteration
          if (lane == 0) bulk_wait_read<0>();   // the previous store has read the tile
          __syncwarp();
          const uint32_t buf = stg;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float* vv = j < 4 ? v0 + 8 * j : v1 + 8 * (j - 4);
            uint4 w = make_uint4(0u, 0u, 0u, 0u);
            if (!bad)
              w = make_uint4(pack_bf16x2(vv[0], vv[1]), pack_bf16x2(vv[2], vv[3]),
                             pack_bf16x2(vv[4], vv[5]), pack_bf16x2(vv[6], vv[7]));
            st_shared_v4(buf + sw128_off(lane, j), w);
          }
          fence_async_shared();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmXh, buf, c * NC + c0, row0);
            bulk_commit();
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[acc]));
      }
    }
    if (lane == 0) bulk_wait<0>();   // stores complete before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tbase, tmem_cols);
  }
}

template <typename KernelT>
cudaError_t set_smem(KernelT k, uint32_t bytes) {
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bytes));
}

}  // namespace

uint32_t decompress_ctl_bytes() { return static_cast<uint32_t>(sizeof(Ctl)); }
uint32_t decompress_pt_ctl_bytes() { return static_cast<uint32_t>(sizeof(CtlPt)) + kPtStagingBytes; }

cudaError_t launch_decompress_tc(const CUtensorMap& tmB, const CUtensorMap& tmZ,
                                 const DecompressArgs& a, uint32_t smem_bytes, int grid,
                                 cudaStream_t s) {
  cudaError_t e;
  switch (a.vq ? a.gd : 0) {
    case 0:
      e = set_smem(k_decompress_tc<0>, smem_bytes);
      if (e != cudaSuccess) return e;
      k_decompress_tc<0><<<grid, kThreads, smem_bytes, s>>>(tmB, tmZ, a);
      break;
    case 16:
      e = set_smem(k_decompress_tc<16>, smem_bytes);
      if (e != cudaSuccess) return e;
      k_decompress_tc<16><<<grid, kThreads, smem_bytes, s>>>(tmB, tmZ, a);
      break;
    case 32:
      e = set_smem(k_decompress_tc<32>, smem_bytes);
      if (e != cudaSuccess) return e;
      k_decompress_tc<32><<<grid, kThreads, smem_bytes, s>>>(tmB, tmZ, a);
      break;
    case 64:
      e = set_smem(k_decompress_tc<64>, smem_bytes);
      if (e != cudaSuccess) return e;
      k_decompress_tc<64><<<grid, kThreads, smem_bytes, s>>>(tmB, tmZ, a);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace mapl

namespace mapl {

cudaError_t launch_decompress_pt(const CUtensorMap& tmB, const CUtensorMap& tmXh,
                                 const DecompressArgs& a, uint32_t smem_bytes, int grid,
                                 cudaStream_t s) {
  cudaError_t e;
  switch (a.vq ? a.gd : 0) {
    case 0:
      e = set_smem(k_decompress_pt<0>, smem_bytes);
      if (e != cudaSuccess) return e;
      e = launch_chained(k_decompress_pt<0>, dim3(grid), dim3(kPtThreads), smem_bytes, s, tmB, tmXh,
                         a);
      if (e != cudaSuccess) return e;
      break;
    case 16:
      e = set_smem(k_decompress_pt<16>, smem_bytes);
      if (e != cudaSuccess) return e;
      e = launch_chained(k_decompress_pt<16>, dim3(grid), dim3(kPtThreads), smem_bytes, s, tmB, tmXh,
                         a);
      if (e != cudaSuccess) return e;
      break;
    case 32:
      e = set_smem(k_decompress_pt<32>, smem_bytes);
      if (e != cudaSuccess) return e;
      e = launch_chained(k_decompress_pt<32>, dim3(grid), dim3(kPtThreads), smem_bytes, s, tmB, tmXh,
                         a);
      if (e != cudaSuccess) return e;
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace mapl
